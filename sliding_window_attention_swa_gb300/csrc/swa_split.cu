// swa_split.cu -- split-K attention of a few query rows against many key/value
// slots, and the log-sum-exp merge of the splits.
//
// Used for ring-buffer decode (one query token per sequence against its W cache
// slots, validity from the stored slot positions) and for the global rows of the
// prefill path (each global position attends to all T keys).  Work is
// HBM-bound: every valid key/value byte is read once.  A CTA owns 512 slots of
// one (batch, kv head, query block); 4 warps share a cp.async pipeline of
// 64-slot chunks (K and V, XOR-swizzled rows) and each warp scores 16 slots of
// every chunk with mma.sync (the query block's <= 16 rows -- a GQA group of
// heads -- are the M dimension).  Chunks without a valid slot are never loaded;
// invalid slots inside a loaded chunk are zero-filled, so uninitialised cache
// memory cannot leak into the result.  Each split writes (max, sum, weighted
// values); the merge kernel combines them (FlashAttention-style rescaling).
#include <cfloat>
#include <cmath>

#include "ptx.cuh"
#include "swa_internal.h"

namespace swa {
namespace {

template <int D>
struct SplitCfg {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kPieces = D / 8;  // 16-byte pieces per row
    static constexpr int kTileBytes = kSplitChunk * kRowBytes;
    static constexpr int kStages = D == 64 ? 4 : (D == 128 ? 3 : 2);
    static constexpr int kSmem = kStages * 2 * kTileBytes;
    static_assert(kSmem >= 4 * kSplitRows * D * 4, "combine buffer must fit in the stage memory");
};

__device__ __forceinline__ uint32_t swz(int row, int piece, int row_bytes) {
    return static_cast<uint32_t>(row * row_bytes + ((piece ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(128) split_attn_kernel(const SplitArgs a) {
    using C = SplitCfg<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint8_t valid[kSlotsPerSplit];
    __shared__ int chunk_list[kSlotsPerSplit / kSplitChunk];
    __shared__ int n_chunks_valid;
    __shared__ int cnt_total;
    __shared__ float red_m[4][kSplitRows];
    __shared__ float red_l[4][kSplitRows];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x;
    const int nqb = (a.NQ + a.q_per_cta - 1) / a.q_per_cta;
    const int kvh = blockIdx.y / nqb, qb = blockIdx.y % nqb;
    const int b = blockIdx.z;
    const int group = a.H_q / a.H_kv;
    const int slot0 = split * a.slots_per_split;
    const int nslots = min(a.n_slots, slot0 + a.slots_per_split) - slot0;

    // ---- 1. slot validity, valid count, and the list of chunks worth loading
    if (tid == 0) {
        cnt_total = 0;
        n_chunks_valid = 0;
    }
    __syncthreads();
    {
        const int64_t t = a.q_pos ? static_cast<int64_t>(a.q_pos[b]) : 0;
        int mine = 0;
        for (int i = tid; i < a.slots_per_split; i += 128) {
            bool ok = false;
            if (i < nslots) {
                if (a.slot_pos) {
                    const int64_t p = a.slot_pos[static_cast<int64_t>(b) * a.W + slot0 + i];
                    ok = p >= 0 && p > t - a.W && p <= t;
                } else {
                    ok = true;
                }
            }
            valid[i] = ok ? 1 : 0;
            mine += ok ? 1 : 0;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
        if (lane == 0) atomicAdd(&cnt_total, mine);
    }
    __syncthreads();
    if (warp == 0) {
        const int nch = (nslots + kSplitChunk - 1) / kSplitChunk;
        for (int c0 = 0; c0 < nch; c0 += 32) {
            const int c = c0 + lane;
            bool any = false;
            if (c < nch)
                for (int i = 0; i < kSplitChunk; ++i) any |= valid[c * kSplitChunk + i] != 0;
            const unsigned m = __ballot_sync(0xffffffffu, any);
            if (any) chunk_list[n_chunks_valid + __popc(m & ((1u << lane) - 1u))] = c;
            __syncwarp();
            if (lane == 0) n_chunks_valid += __popc(m);
            __syncwarp();
        }
    }
    __syncthreads();
    const int nvc = n_chunks_valid;

    // ---- 2. query fragments (rows r0 = lane/4, r1 = r0 + 8 of the 16-row M tile)
    const int rows = a.q_per_cta * group;
    uint32_t qa[D / 16][4];
    {
        const int rr[2] = {lane >> 2, (lane >> 2) + 8};
        const __nv_bfloat16 *qp[2];
        bool rv[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = rr[i];
            const int qs = qb * a.q_per_cta + r / group;
            rv[i] = r < rows && qs < a.NQ;
            const int h = kvh * group + r % group;
            int64_t tok = (rv[i] && a.q_tok) ? a.q_tok[qs] : 0;
            if (tok < 0 || tok >= a.tok_limit) {
                rv[i] = false;
                tok = 0;
            }
            qp[i] = static_cast<const __nv_bfloat16 *>(a.q) + static_cast<int64_t>(b) * a.q_sb + tok * a.q_st +
                    static_cast<int64_t>(h) * a.q_sh;
        }
        const int c = 2 * (lane & 3);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qa[kk][0] = rv[0] ? *reinterpret_cast<const uint32_t *>(qp[0] + kk * 16 + c) : 0u;
            qa[kk][1] = rv[1] ? *reinterpret_cast<const uint32_t *>(qp[1] + kk * 16 + c) : 0u;
            qa[kk][2] = rv[0] ? *reinterpret_cast<const uint32_t *>(qp[0] + kk * 16 + 8 + c) : 0u;
            qa[kk][3] = rv[1] ? *reinterpret_cast<const uint32_t *>(qp[1] + kk * 16 + 8 + c) : 0u;
        }
    }

    // ---- 3. pipelined loop over the valid chunks
    const uint32_t sbase = smem_u32(smem);
    const __nv_bfloat16 *kb = static_cast<const __nv_bfloat16 *>(a.k) + static_cast<int64_t>(b) * a.k_sb +
                              static_cast<int64_t>(kvh) * a.k_sh;
    const __nv_bfloat16 *vb = static_cast<const __nv_bfloat16 *>(a.v) + static_cast<int64_t>(b) * a.v_sb +
                              static_cast<int64_t>(kvh) * a.v_sh;

    auto issue = [&](int stage, int chunk) {
        const uint32_t kdst = sbase + stage * 2 * C::kTileBytes;
        const uint32_t vdst = kdst + C::kTileBytes;
        constexpr int kPer = kSplitChunk * C::kPieces;  // pieces per tile
#pragma unroll 4
        for (int idx = tid; idx < kPer; idx += 128) {
            const int r = idx / C::kPieces, pc = idx % C::kPieces;
            const int si = chunk * kSplitChunk + r;  // slot index within the split
            const bool ok = si < nslots && valid[si];
            const int64_t slot = ok ? slot0 + si : slot0;
            const uint32_t o = swz(r, pc, C::kRowBytes);
            cp_async16(kdst + o, kb + slot * a.k_ss + pc * 8, ok);
            cp_async16(vdst + o, vb + slot * a.v_ss + pc * 8, ok);
        }
    };

#pragma unroll
    for (int s = 0; s < C::kStages - 1; ++s) {
        if (s < nvc) issue(s, chunk_list[s]);
        cp_async_commit();
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

#pragma unroll 1
    for (int i = 0; i < nvc; ++i) {
        cp_async_wait<C::kStages - 2>();
        __syncthreads();
        {
            const int nx = i + C::kStages - 1;
            if (nx < nvc) issue(nx % C::kStages, chunk_list[nx]);
            cp_async_commit();
        }
        const int stage = i % C::kStages;
        const int chunk = chunk_list[i];
        const uint32_t ks = sbase + stage * 2 * C::kTileBytes;
        const uint32_t vs = ks + C::kTileBytes;

        // S = Q K^T for this warp's 16 slots (two n-tiles of 8)
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
            const int row = 16 * warp + 8 * nt + (lane & 7);
#pragma unroll
            for (int k2 = 0; k2 < D / 32; ++k2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(ks + swz(row, k2 * 4 + (lane >> 3), C::kRowBytes), b0, b1, b2, b3);
                mma_bf16_16816(sc[nt], qa[2 * k2], b0, b1);
                mma_bf16_16816(sc[nt], qa[2 * k2 + 1], b2, b3);
            }
        }
        // mask + scale (log2 domain)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int si = chunk * kSplitChunk + 16 * warp + 8 * nt + 2 * (lane & 3) + (e & 1);
                const bool ok = si < nslots && valid[si];
                sc[nt][e] = ok ? sc[nt][e] * a.scale_log2 : -INFINITY;
            }
            mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = mn0 == -INFINITY ? 1.f : ex2(m0 - mn0);
        const float al1 = mn1 == -INFINITY ? 1.f : ex2(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        float p[2][4];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            p[nt][0] = mn0 == -INFINITY ? 0.f : ex2(sc[nt][0] - mn0);
            p[nt][1] = mn0 == -INFINITY ? 0.f : ex2(sc[nt][1] - mn0);
            p[nt][2] = mn1 == -INFINITY ? 0.f : ex2(sc[nt][2] - mn1);
            p[nt][3] = mn1 == -INFINITY ? 0.f : ex2(sc[nt][3] - mn1);
            s0 += p[nt][0] + p[nt][1];
            s1 += p[nt][2] + p[nt][3];
        }
        l0 = l0 * al0 + s0;
        l1 = l1 * al1 + s1;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            acc[n][0] *= al0;
            acc[n][1] *= al0;
            acc[n][2] *= al1;
            acc[n][3] *= al1;
        }
        uint32_t pa[4];
        pa[0] = pack_bf16x2(p[0][0], p[0][1]);
        pa[1] = pack_bf16x2(p[0][2], p[0][3]);
        pa[2] = pack_bf16x2(p[1][0], p[1][1]);
        pa[3] = pack_bf16x2(p[1][2], p[1][3]);
        // O += P V (V^T fragments via transposing ldmatrix)
        const int vrow = 16 * warp + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
        for (int d2 = 0; d2 < D / 16; ++d2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vs + swz(vrow, 2 * d2 + (lane >> 4), C::kRowBytes), b0, b1, b2, b3);
            mma_bf16_16816(acc[2 * d2], pa, b0, b1);
            mma_bf16_16816(acc[2 * d2 + 1], pa, b2, b3);
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- 4. combine the 4 warps, write this split's partial result
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const int r0 = lane >> 2, r1 = r0 + 8;
    if ((lane & 3) == 0) {
        red_m[warp][r0] = m0;
        red_m[warp][r1] = m1;
        red_l[warp][r0] = l0;
        red_l[warp][r1] = l1;
    }
    __syncthreads();
    float *cbuf = reinterpret_cast<float *>(smem);  // [4][16][D]
    {
        float mw0 = -INFINITY, mw1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            mw0 = fmaxf(mw0, red_m[w][r0]);
            mw1 = fmaxf(mw1, red_m[w][r1]);
        }
        const float f0 = mw0 == -INFINITY ? 0.f : ex2(m0 - mw0);
        const float f1 = mw1 == -INFINITY ? 0.f : ex2(m1 - mw1);
        float *c0 = cbuf + (warp * kSplitRows + r0) * D;
        float *c1 = cbuf + (warp * kSplitRows + r1) * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            const int d = 8 * n + 2 * (lane & 3);
            *reinterpret_cast<float2 *>(c0 + d) = make_float2(acc[n][0] * f0, acc[n][1] * f0);
            *reinterpret_cast<float2 *>(c1 + d) = make_float2(acc[n][2] * f1, acc[n][3] * f1);
        }
    }
    __syncthreads();
    for (int idx = tid; idx < rows * D; idx += 128) {
        const int r = idx / D, d = idx % D;
        const int qs = qb * a.q_per_cta + r / group;
        if (qs >= a.NQ) continue;
        if (a.q_tok && (a.q_tok[qs] < 0 || a.q_tok[qs] >= a.tok_limit)) continue;
        const int h = kvh * group + r % group;
        float mw = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) mw = fmaxf(mw, red_m[w][r]);
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) s += cbuf[(w * kSplitRows + r) * D + d];
        const int64_t row = ((static_cast<int64_t>(b) * a.NQ + qs) * a.H_q + h) * a.n_splits + split;
        a.ws_acc[row * D + d] = s;
        if (d == 0) {
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                L += mw == -INFINITY ? 0.f : red_l[w][r] * ex2(red_m[w][r] - mw);
            a.ws_ml[row * 2 + 0] = mw;
            a.ws_ml[row * 2 + 1] = L;
        }
    }
    if (qb == 0 && tid == 0) a.ws_cnt[(static_cast<int64_t>(b) * a.H_kv + kvh) * a.n_splits + split] = cnt_total;
}

__global__ void __launch_bounds__(128) merge_kernel(const MergeArgs a) {
    const int qs = blockIdx.x / a.H_q, h = blockIdx.x % a.H_q, b = blockIdx.y;
    const int group = a.H_q / a.H_kv, kvh = h / group;
    const int64_t base = ((static_cast<int64_t>(b) * a.NQ + qs) * a.H_q + h) * a.n_splits;
    float M = -INFINITY;
    for (int s = 0; s < a.n_splits; ++s) M = fmaxf(M, a.ws_ml[(base + s) * 2]);
    float L = 0.f;
    if (M != -INFINITY)
        for (int s = 0; s < a.n_splits; ++s) L += a.ws_ml[(base + s) * 2 + 1] * exp2f(a.ws_ml[(base + s) * 2] - M);
    const int64_t tok = a.q_tok ? a.q_tok[qs] : 0;
    if (tok < 0 || tok >= a.tok_limit) return;
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o) + static_cast<int64_t>(b) * a.o_sb + tok * a.o_st +
                       static_cast<int64_t>(h) * a.o_sh;
    for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
        float acc = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < a.n_splits; ++s)
                acc += a.ws_acc[(base + s) * a.D + d] * exp2f(a.ws_ml[(base + s) * 2] - M);
            acc /= L;
        }
        o[d] = __float2bfloat16_rn(acc);
    }
    if (threadIdx.x == 0) {
        const float lse = M == -INFINITY ? -INFINITY : (M + log2f(L)) * 0.6931471805599453f;
        a.lse[static_cast<int64_t>(b) * a.lse_sb + static_cast<int64_t>(h) * a.lse_sh + tok * a.lse_st] = lse;
        if (a.counts) {
            int c = 0;
            for (int s = 0; s < a.n_splits; ++s) c += a.ws_cnt[(static_cast<int64_t>(b) * a.H_kv + kvh) * a.n_splits + s];
            a.counts[static_cast<int64_t>(b) * a.cnt_sb + static_cast<int64_t>(h) * a.cnt_sh + tok * a.cnt_st] = c;
        }
    }
}

template <int D>
cudaError_t launch_split_d(const SplitArgs &a, cudaStream_t s) {
    using C = SplitCfg<D>;
    static bool configured = false;  // idempotent attribute set; benign if raced
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(split_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int nqb = (a.NQ + a.q_per_cta - 1) / a.q_per_cta;
    dim3 grid(a.n_splits, a.H_kv * nqb, a.B);
    split_attn_kernel<D><<<grid, 128, C::kSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_split(const SplitArgs &a, cudaStream_t s) {
    switch (a.D) {
        case 64: return launch_split_d<64>(a, s);
        case 128: return launch_split_d<128>(a, s);
        case 256: return launch_split_d<256>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s) {
    dim3 grid(a.NQ * a.H_q, a.B);
    merge_kernel<<<grid, 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace swa
