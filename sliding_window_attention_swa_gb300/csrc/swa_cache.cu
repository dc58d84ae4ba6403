// swa_cache.cu -- the ring-buffer KV cache: appending tokens, and gathering a
// chunk's window history in position order for chunked prefill.
//
// Slot rule (lizeman.github.io llm-arch-kb, KV cache paragraph, after Mistral 7B
// section 2: token p goes to slot p mod W and overwrites what was there), with
// n_sink pinned sink slots in front: slot(p) = p for p < n_sink, else
// n_sink + (p - n_sink) mod (n_slots - n_sink).
//
// Both kernels are pure copies, bound by HBM: one warp moves one (sequence, token,
// kv head) pair of key and value rows in 16-byte pieces, grid-striding over pairs.
#include <climits>

#include "swa_internal.h"

namespace swa {
namespace {

__device__ unsigned int g_cache_err = 0;
constexpr unsigned int kErrBadPosition = 1u;    // a negative (or overflowing) position
constexpr unsigned int kErrCacheMismatch = 2u;  // a slot not holding the position needed

constexpr int kThreads = 256;

__device__ __forceinline__ void copy_rows(uint4 *kd, uint4 *vd, const uint4 *ks, const uint4 *vs, int pieces,
                                          int lane) {
    for (int c = lane; c < 2 * pieces; c += 32) {
        if (c < pieces) kd[c] = ks ? __ldg(ks + c) : make_uint4(0, 0, 0, 0);
        else vd[c - pieces] = vs ? __ldg(vs + c - pieces) : make_uint4(0, 0, 0, 0);
    }
}

__global__ void __launch_bounds__(kThreads) append_kernel(const AppendArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t total = static_cast<int64_t>(a.B) * a.n * a.H_kv;
    const int pieces = a.D / 8;
    const int64_t R = a.n_slots - a.n_sink;
    for (int64_t x = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; x < total; x += nw) {
        const int kvh = static_cast<int>(x % a.H_kv);
        const int64_t bi = x / a.H_kv;
        const int i = static_cast<int>(bi % a.n);
        const int b = static_cast<int>(bi / a.n);
        const int64_t p0 = __ldg(a.p0 + b);
        const int64_t p = p0 + i, last = p0 + a.n - 1;
        if (p0 < 0 || last > INT_MAX) {
            if (lane == 0 && i == 0 && kvh == 0) atomicOr(&g_cache_err, kErrBadPosition);
            continue;
        }
        int64_t slot;
        if (p < a.n_sink) {
            slot = p;
        } else {
            if (last - p >= R) continue;  // a later token of this call takes the same ring slot
            slot = a.n_sink + (p - a.n_sink) % R;
        }
        const int64_t src = ((static_cast<int64_t>(b) * a.n + i) * a.H_kv + kvh) * a.D;
        const int64_t dst = ((static_cast<int64_t>(b) * a.H_kv + kvh) * a.n_slots + slot) * a.D;
        copy_rows(reinterpret_cast<uint4 *>(a.kc + dst), reinterpret_cast<uint4 *>(a.vc + dst),
                  reinterpret_cast<const uint4 *>(a.kn + src), reinterpret_cast<const uint4 *>(a.vn + src), pieces,
                  lane);
        if (kvh == 0 && lane == 0) a.slot_pos[static_cast<int64_t>(b) * a.n_slots + slot] = static_cast<int32_t>(p);
    }
}

// Key index x of sequence b (0 <= x < Tk = W-1+C): x < W-1 is history position
// p0 - (W-1) + x, read from its ring slot when the cache holds it; x >= W-1 is chunk
// token x - (W-1).  Absent history rows are written as zeros and lie below kmin[b].
__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int Tk = a.W - 1 + a.C;
    const int64_t total = static_cast<int64_t>(a.B) * Tk * a.H_kv;
    const int pieces = a.D / 8;
    for (int64_t x = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; x < total; x += nw) {
        const int kvh = static_cast<int>(x % a.H_kv);
        const int64_t bx = x / a.H_kv;
        const int xx = static_cast<int>(bx % Tk);
        const int b = static_cast<int>(bx / Tk);
        const int64_t p0 = __ldg(a.p0 + b);
        const int64_t have = p0 < 0 ? 0 : min(min(p0, static_cast<int64_t>(a.n_slots)), static_cast<int64_t>(a.W - 1));
        if (xx == 0 && kvh == 0 && lane == 0) {
            a.kmin[b] = static_cast<int32_t>(a.W - 1 - have);
            if (p0 < 0) atomicOr(&g_cache_err, kErrBadPosition);
        }
        const uint16_t *ks = nullptr, *vs = nullptr;
        if (xx >= a.W - 1) {
            const int64_t src = ((static_cast<int64_t>(b) * a.C + (xx - (a.W - 1))) * a.H_kv + kvh) * a.D;
            ks = a.kn + src;
            vs = a.vn + src;
        } else if (xx >= a.W - 1 - have) {
            const int64_t p = p0 - (a.W - 1) + xx;
            const int64_t slot = p % a.n_slots;
            if (__ldg(a.slot_pos + static_cast<int64_t>(b) * a.n_slots + slot) == p) {
                const int64_t src = ((static_cast<int64_t>(b) * a.H_kv + kvh) * a.n_slots + slot) * a.D;
                ks = a.kc + src;
                vs = a.vc + src;
            } else if (kvh == 0 && lane == 0) {
                atomicOr(&g_cache_err, kErrCacheMismatch);
            }
        }
        const int64_t dst = ((static_cast<int64_t>(b) * Tk + xx) * a.H_kv + kvh) * a.D;
        copy_rows(reinterpret_cast<uint4 *>(a.kl + dst), reinterpret_cast<uint4 *>(a.vl + dst),
                  reinterpret_cast<const uint4 *>(ks), reinterpret_cast<const uint4 *>(vs), pieces, lane);
    }
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                      cudaSuccess)
            n = 148;
    }
    return n;
}

int copy_grid(int64_t warps) {
    const int64_t blocks = (warps + kThreads / 32 - 1) / (kThreads / 32);
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;  // 8 blocks of 8 warps per SM
    return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_append(const AppendArgs &a, cudaStream_t s) {
    const int64_t warps = static_cast<int64_t>(a.B) * a.n * a.H_kv;
    if (warps == 0) return cudaSuccess;
    append_kernel<<<copy_grid(warps), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gather(const GatherArgs &a, cudaStream_t s) {
    const int64_t warps = static_cast<int64_t>(a.B) * (a.W - 1 + a.C) * a.H_kv;
    gather_kernel<<<copy_grid(warps), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

unsigned int cache_read_clear_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_cache_err, sizeof v) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_cache_err, &z, sizeof z);
    return v;
}

}  // namespace swa
