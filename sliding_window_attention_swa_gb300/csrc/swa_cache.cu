// swa_cache.cu -- the ring-buffer KV cache: appending tokens, and gathering a
// chunk's window history in position order for chunked prefill.
//
// Slot rule (lizeman.github.io llm-arch-kb, KV cache paragraph, after Mistral 7B
// section 2: token p goes to slot p mod W and overwrites what was there), with
// n_sink pinned sink slots in front: slot(p) = p for p < n_sink, else
// n_sink + (p - n_sink) mod (n_slots - n_sink).
//
// Both kernels are pure copies, bound by HBM, moving 16-byte pieces.
#include <atomic>
#include <climits>

#include "ptx.cuh"
#include "swa_internal.h"

namespace swa {
namespace {

__device__ unsigned int g_cache_err = 0;
constexpr unsigned int kErrBadPosition = 1u;    // a negative (or overflowing) position
constexpr unsigned int kErrCacheMismatch = 2u;  // a slot not holding the position needed
static_assert(kErrBadPosition == SWA_DEVERR_BAD_POSITION && kErrCacheMismatch == SWA_DEVERR_CACHE_MISMATCH,
              "device error bits");

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // independent 16-byte loads in flight per thread

// Division of 31-bit values by a divisor fixed for the launch, by a multiply-high and a
// shift (Granlund and Montgomery, "Division by invariant integers using multiplication",
// 1994): with s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1,
// x / d = (umulhi(x, m) + x) >> s for 0 <= x < 2^31.  The kernels' index arithmetic
// would otherwise spend more time in 64-bit division than in moving the data.
struct FastDiv {
    uint32_t d, m, s;
};
FastDiv fast_div(uint32_t d) {
    uint32_t s = 0;
    while ((uint64_t{1} << s) < d) ++s;
    const uint64_t m = ((uint64_t{1} << 32) * ((uint64_t{1} << s) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), s};
}
__device__ __forceinline__ uint32_t fdiv(uint32_t x, const FastDiv &f) { return (__umulhi(x, f.m) + x) >> f.s; }

// Divisors of the two kernels' flat indices.
struct CopyPlan {
    FastDiv hkv;   // H_kv
    FastDiv n;     // tokens per sequence (append: n; gather: W - 1 + C)
    FastDiv ring;  // ring slots n_slots - n_sink
    FastDiv sink;  // n_sink (gather)
};

// Both kernels walk a flat list of 16-byte pieces: piece c of (sequence, token, kv
// head) x is the c-th of the 2*D/8 pieces of its key row then its value row, so a
// warp's lanes cover consecutive pieces of the same rows (coalesced).  Each thread
// issues kUnroll loads before its stores.

template <int D>
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendArgs a, const CopyPlan pl) {
    constexpr int P = 2 * D / 8;
    const int64_t total = static_cast<int64_t>(a.B) * a.n * a.H_kv * P;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t R = a.n_slots - a.n_sink;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < total;
         base += kUnroll * stride) {
        uint4 val[kUnroll];
        uint4 *dst[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            dst[u] = nullptr;
            const int64_t f = base + u * stride;
            if (f >= total) continue;
            const int c = static_cast<int>(f % P);
            const uint32_t x = static_cast<uint32_t>(f / P);  // < 2^31 rows (checked at launch)
            const uint32_t bi = fdiv(x, pl.hkv);
            const int kvh = static_cast<int>(x - bi * pl.hkv.d);
            const uint32_t bq = fdiv(bi, pl.n);
            const int i = static_cast<int>(bi - bq * pl.n.d);
            const int b = static_cast<int>(bq);
            const int64_t p0 = __ldg(a.p0 + b);
            const int64_t p = p0 + i, last = p0 + a.n - 1;
            if (p0 < 0 || last > INT_MAX) {
                if (c == 0 && i == 0 && kvh == 0) atomicOr(&g_cache_err, kErrBadPosition);
                continue;
            }
            int64_t slot;
            if (p < a.n_sink) {
                slot = p;
            } else {
                if (last - p >= R) continue;  // a later token of this call takes the same ring slot
                const uint32_t pr = static_cast<uint32_t>(p - a.n_sink);
                slot = a.n_sink + (pr - fdiv(pr, pl.ring) * pl.ring.d);
            }
            const bool is_v = c >= P / 2;
            const int pc = is_v ? c - P / 2 : c;
            // debug build: the new row and its slot exist
            if (!SWA_IN_BOUNDS(b < a.B && i < a.n && kvh < a.H_kv && slot >= 0 && slot < a.n_slots, &g_cache_err))
                continue;
            const int64_t src = ((static_cast<int64_t>(b) * a.n + i) * a.H_kv + kvh) * D;
            const int64_t dsto = ((static_cast<int64_t>(b) * a.H_kv + kvh) * a.n_slots + slot) * D;
            val[u] = __ldg(reinterpret_cast<const uint4 *>((is_v ? a.vn : a.kn) + src) + pc);
            dst[u] = reinterpret_cast<uint4 *>((is_v ? a.vc : a.kc) + dsto) + pc;
            if (c == 0 && kvh == 0) a.slot_pos[static_cast<int64_t>(b) * a.n_slots + slot] = static_cast<int32_t>(p);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (dst[u]) *dst[u] = val[u];
    }
}

// Key index x of sequence b (0 <= x < Tk = W-1+C): x < W-1 is history position
// p0 - (W-1) + x, read from its slot (slot rule with n_sink sinks) when the cache holds
// it; x >= W-1 is chunk token x - (W-1).  Absent history rows are written as zeros and
// lie below kmin[b].  After the B*Tk*H_kv rows come the B*n_sink*H_kv sink rows: sink
// position s from its cache slot when s < p0, from the chunk when it lies in the
// chunk, else zeros (no query of this chunk reaches it).
template <int D>
__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherArgs a, const CopyPlan pl) {
    constexpr int P = 2 * D / 8;
    const int Tk = a.W - 1 + a.C;
    const int64_t rows_hist = static_cast<int64_t>(a.B) * Tk * a.H_kv;
    const int64_t total = (rows_hist + static_cast<int64_t>(a.B) * a.n_sink * a.H_kv) * P;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < a.n_sink; i += blockDim.x) a.sink_idx[i] = i;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < total;
         base += kUnroll * stride) {
        uint4 val[kUnroll];
        uint4 *dst[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            dst[u] = nullptr;
            const int64_t f = base + u * stride;
            if (f >= total) continue;
            const int c = static_cast<int>(f % P);
            const int64_t x = f / P;
            const bool is_v = c >= P / 2;
            const int pc = is_v ? c - P / 2 : c;
            val[u] = make_uint4(0, 0, 0, 0);
            if (x < rows_hist) {
                const uint32_t x32 = static_cast<uint32_t>(x);  // < 2^31 rows (checked at launch)
                const uint32_t bx = fdiv(x32, pl.hkv);
                const int kvh = static_cast<int>(x32 - bx * pl.hkv.d);
                const uint32_t bq = fdiv(bx, pl.n);
                const int xx = static_cast<int>(bx - bq * pl.n.d);
                const int b = static_cast<int>(bq);
                // debug build: the gathered row (b, key index, kv head) exists
                if (!SWA_IN_BOUNDS(b < a.B && xx < Tk && kvh < a.H_kv, &g_cache_err)) continue;
                const int64_t p0 = __ldg(a.p0 + b);
                // history positions present right before p0 (a sink cache's ring covers the window)
                const int64_t ring = a.n_sink == 0 ? a.n_slots : a.W - 1;
                const int64_t have = p0 < 0 ? 0 : min(min(p0, ring), static_cast<int64_t>(a.W - 1));
                if (xx == 0 && kvh == 0 && c == 0) {
                    a.kmin[b] = static_cast<int32_t>(a.W - 1 - have);
                    if (p0 < 0) atomicOr(&g_cache_err, kErrBadPosition);
                }
                if (xx >= a.W - 1) {
                    const int64_t src = ((static_cast<int64_t>(b) * a.C + (xx - (a.W - 1))) * a.H_kv + kvh) * D;
                    val[u] = __ldg(reinterpret_cast<const uint4 *>((is_v ? a.vn : a.kn) + src) + pc);
                } else if (xx >= a.W - 1 - have) {
                    const int64_t p = p0 - (a.W - 1) + xx;
                    const uint32_t pr = static_cast<uint32_t>(p - a.n_sink);
                    const int64_t slot = p < a.n_sink ? p : a.n_sink + (pr - fdiv(pr, pl.ring) * pl.ring.d);
                    if (!SWA_IN_BOUNDS(slot >= 0 && slot < a.n_slots, &g_cache_err)) continue;
                    if (__ldg(a.slot_pos + static_cast<int64_t>(b) * a.n_slots + slot) == p) {
                        const int64_t src = ((static_cast<int64_t>(b) * a.H_kv + kvh) * a.n_slots + slot) * D;
                        val[u] = __ldg(reinterpret_cast<const uint4 *>((is_v ? a.vc : a.kc) + src) + pc);
                    } else if (kvh == 0 && c == 0) {
                        atomicOr(&g_cache_err, kErrCacheMismatch);
                    }
                }
                const int64_t dsto = ((static_cast<int64_t>(b) * Tk + xx) * a.H_kv + kvh) * D;
                dst[u] = reinterpret_cast<uint4 *>((is_v ? a.vl : a.kl) + dsto) + pc;
            } else {
                const uint32_t y = static_cast<uint32_t>(x - rows_hist);  // (b, s, kvh)
                const uint32_t bs = fdiv(y, pl.hkv);
                const int kvh = static_cast<int>(y - bs * pl.hkv.d);
                const uint32_t bq = fdiv(bs, pl.sink);
                const int sidx = static_cast<int>(bs - bq * pl.sink.d);
                const int b = static_cast<int>(bq);
                // debug build: the sink row (b, sink, kv head) exists
                if (!SWA_IN_BOUNDS(b < a.B && sidx < a.n_sink && sidx < a.n_slots && kvh < a.H_kv, &g_cache_err))
                    continue;
                const int64_t p0 = __ldg(a.p0 + b);
                if (sidx < p0) {
                    if (__ldg(a.slot_pos + static_cast<int64_t>(b) * a.n_slots + sidx) == sidx) {
                        const int64_t src = ((static_cast<int64_t>(b) * a.H_kv + kvh) * a.n_slots + sidx) * D;
                        val[u] = __ldg(reinterpret_cast<const uint4 *>((is_v ? a.vc : a.kc) + src) + pc);
                    } else if (kvh == 0 && c == 0) {
                        atomicOr(&g_cache_err, kErrCacheMismatch);
                    }
                } else if (sidx < p0 + a.C) {
                    const int64_t src = ((static_cast<int64_t>(b) * a.C + (sidx - p0)) * a.H_kv + kvh) * D;
                    val[u] = __ldg(reinterpret_cast<const uint4 *>((is_v ? a.vn : a.kn) + src) + pc);
                }
                const int64_t dsto = ((static_cast<int64_t>(b) * a.n_sink + sidx) * a.H_kv + kvh) * D;
                dst[u] = reinterpret_cast<uint4 *>((is_v ? a.vs : a.ks) + dsto) + pc;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (dst[u]) *dst[u] = val[u];
    }
}

int sm_count() {
    static std::atomic<int> n[64];  // per device; 0 = not looked up yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int v = n[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        n[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

int copy_grid(int64_t pieces) {
    const int64_t blocks = (pieces + kThreads * kUnroll - 1) / (kThreads * kUnroll);
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;  // 8 blocks of 256 threads per SM
    return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_append(const AppendArgs &a, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(a.B) * a.n * a.H_kv;
    const int64_t pieces = rows * (2 * a.D / 8);
    if (pieces == 0) return cudaSuccess;
    if (rows >= (int64_t{1} << 31) || a.n_slots - a.n_sink < 1) return cudaErrorInvalidValue;
    CopyPlan pl{};
    pl.hkv = fast_div(static_cast<uint32_t>(a.H_kv));
    pl.n = fast_div(static_cast<uint32_t>(a.n));
    pl.ring = fast_div(static_cast<uint32_t>(a.n_slots - a.n_sink));
    pl.sink = fast_div(1);
    switch (a.D) {
        case 64: append_kernel<64><<<copy_grid(pieces), kThreads, 0, s>>>(a, pl); break;
        case 128: append_kernel<128><<<copy_grid(pieces), kThreads, 0, s>>>(a, pl); break;
        case 256: append_kernel<256><<<copy_grid(pieces), kThreads, 0, s>>>(a, pl); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_gather(const GatherArgs &a, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(a.B) * (a.W - 1 + a.C + a.n_sink) * a.H_kv;
    const int64_t pieces = rows * (2 * a.D / 8);
    if (rows >= (int64_t{1} << 31) || a.n_slots - a.n_sink < 1) return cudaErrorInvalidValue;
    CopyPlan pl{};
    pl.hkv = fast_div(static_cast<uint32_t>(a.H_kv));
    pl.n = fast_div(static_cast<uint32_t>(a.W - 1 + a.C));
    pl.ring = fast_div(static_cast<uint32_t>(a.n_slots - a.n_sink));
    pl.sink = fast_div(static_cast<uint32_t>(a.n_sink > 0 ? a.n_sink : 1));
    switch (a.D) {
        case 64: gather_kernel<64><<<copy_grid(pieces), kThreads, 0, s>>>(a, pl); break;
        case 128: gather_kernel<128><<<copy_grid(pieces), kThreads, 0, s>>>(a, pl); break;
        case 256: gather_kernel<256><<<copy_grid(pieces), kThreads, 0, s>>>(a, pl); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

unsigned int cache_read_clear_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_cache_err, sizeof v) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_cache_err, &z, sizeof z);
    return v;
}

}  // namespace swa
