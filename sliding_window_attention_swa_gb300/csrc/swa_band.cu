// swa_band.cu -- banded (sliding-window) attention prefill on 5th-generation
// tensor cores (sm_103a).
//
// Work unit: one (batch b, key/value head kvh, query tile).  A query tile is 128
// rows = TQ consecutive tokens x the G = H_q/H_kv query heads of the group
// (row = token_local * G + head_local), so every key/value tile is loaded once
// for the whole group.  The unit iterates only over the key tiles that intersect
// the union of its rows' bands
//     [max(0, t_first - wl), min(T-1, t_last + wr)]
// (keys outside the window are never loaded or scored; the production
// kernels described in "Sliding Window Attention", lizeman.github.io
// llm-arch-kb section 3, and in the superteams.ai glossary, iterate over the
// band only), followed by ceil(n_global / BN) "global column" tiles that hold the
// key/value rows of the global positions (prathamp.com "Sliding Window
// Attention: From Local Windows to Global Context", section 4.3).
//
// Roles (192 threads):
//   warp 0      TMA producer: Q once; K and V tiles into a STAGES-deep ring;
//               global-column tiles are gathered with plain loads into the same
//               swizzled layout.
//   warp 1      TMEM owner and MMA issuer (one thread):
//                 S[j&1] = Q K_j^T          (tcgen05.mma, M=128, N=BN, K=D)
//                 O     += P_{j-1} V_{j-1}  (tcgen05.mma, M=128, N=D, K=BN)
//               S is double-buffered in TMEM so S_{j+1} runs while the softmax
//               works on S_j.
//   warps 2..5  softmax (one TMEM lane = one row per thread): mask (edge tiles
//               and global tiles only), running max in the log2 domain, P =
//               2^(x - m) written as bf16 to shared memory (K-major, 128B
//               swizzle) for the PV MMA, running sum l.  The O accumulator in
//               TMEM is rescaled only when a row's max grows by more than 2^8
//               (the result is exact either way: numerator and denominator share
//               the stale max).  Epilogue: O / l -> bf16 -> TMA store; lse and
//               attended-key counts per row.
// Every wait is bounded; on expiry the CTA records an error word, drains its
// copies and MMAs, frees TMEM and returns.
#include <cfloat>
#include <cmath>

#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "swa_internal.h"

namespace swa {
namespace {

__device__ unsigned int g_band_err = 0;

constexpr int BM = 128;          // query rows per unit (TMEM lanes)
constexpr int kThreads = 192;    // 6 warps
constexpr float kRescaleTau = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

template <int D>
struct BandCfg {
    static constexpr int BN = D == 256 ? 64 : 128;          // keys per tile
    static constexpr int STAGES = D == 64 ? 4 : 2;           // K/V ring depth
    static constexpr int QBYTES = BM * D * 2;
    static constexpr int KVBYTES = BN * D * 2;               // one K (or V) tile
    static constexpr int PBYTES = BM * BN * 2;               // one P buffer
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + QBYTES;
    static constexpr int OFF_V = OFF_K + STAGES * KVBYTES;
    static constexpr int OFF_P = OFF_V + STAGES * KVBYTES;
    static constexpr int OFF_BAR = OFF_P + 2 * PBYTES;
    // barriers: q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], s_empty[2], p_full[2],
    // pv_done[2], drain
    static constexpr int NBAR = 1 + 3 * STAGES + 8 + 1;
    static constexpr int OFF_TMEMPTR = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_TMEMPTR + 16 + 1024;      // + slack for 1024-B alignment
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_O = 0;                       // O accumulator columns [0, D)
    static constexpr uint32_t TM_S = 256;                     // S buffers at 256 and 256 + BN
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(D <= 256 && TM_S + 2 * BN <= TMEM_COLS, "tensor memory budget");
};

struct BandKernelArgs {
    int B, T, H_q, H_kv, G, TQ, n_qtiles;
    int wl, wr;
    float scale_log2;
    const int32_t *global_idx;
    int n_global;
    const __nv_bfloat16 *k, *v;     // for the global-column gather
    int64_t k_st[3], v_st[3];
    float *lse;
    int32_t *counts;
};

// Every lane waits (each acquires the barrier); the warp proceeds only if all did,
// so the .sync.aligned tcgen05 instructions that follow stay convergent.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, abort, &g_band_err);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool in_band(int t, int s, int wl, int wr) {
    return (wl < 0 || s >= t - wl) && (wr < 0 || s <= t + wr);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    band_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const BandKernelArgs a) {
    using C = BandCfg<D>;
    constexpr int BN = C::BN, STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t *sgen = smem_raw + (sbase - sraw);

    const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sP = sbase + C::OFF_P;
    const uint32_t bars = sbase + C::OFF_BAR;
    auto bar_q = [&]() { return bars; };
    auto bar_kf = [&](int s) { return bars + 8u * (1 + s); };
    auto bar_vf = [&](int s) { return bars + 8u * (1 + STAGES + s); };
    auto bar_ke = [&](int s) { return bars + 8u * (1 + 2 * STAGES + s); };
    auto bar_sf = [&](int b) { return bars + 8u * (1 + 3 * STAGES + b); };
    auto bar_se = [&](int b) { return bars + 8u * (3 + 3 * STAGES + b); };
    auto bar_pf = [&](int b) { return bars + 8u * (5 + 3 * STAGES + b); };
    auto bar_pv = [&](int b) { return bars + 8u * (7 + 3 * STAGES + b); };
    const uint32_t bar_drain = bars + 8u * (9 + 3 * STAGES);
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(sgen + C::OFF_TMEMPTR);

    // ---- unit decode (longest units first: query tiles in decreasing order)
    const int bh = blockIdx.x % (a.B * a.H_kv);
    const int qt = a.n_qtiles - 1 - blockIdx.x / (a.B * a.H_kv);
    const int b = bh / a.H_kv, kvh = bh % a.H_kv;
    const int t0 = qt * a.TQ;
    const int t1 = min(a.T - 1, t0 + a.TQ - 1);
    const int kv_lo = a.wl < 0 ? 0 : max(0, t0 - a.wl);
    const int kv_hi = a.wr < 0 ? a.T - 1 : min(a.T - 1, t1 + a.wr);
    const int n_band = (kv_hi - kv_lo + BN) / BN;
    const int n_gt = (a.n_global + BN - 1) / BN;
    const int n_tiles = n_band + n_gt;

    // ---- setup: barriers, TMEM
    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar_q(), 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_kf(s), 1);
            mbar_init(bar_vf(s), 1);
            mbar_init(bar_ke(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_sf(i), 1);
            mbar_init(bar_se(i), 4);
            mbar_init(bar_pf(i), 4);
            mbar_init(bar_pv(i), 1);
        }
        mbar_init(bar_drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_holder)), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    volatile int *abort = &abort_flag;

    if (warp == 0) {
        // ============================ producer ============================
        int last_tile[STAGES];
#pragma unroll
        for (int s = 0; s < STAGES; ++s) last_tile[s] = -1;
        bool ok = true;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_q(), static_cast<uint32_t>(a.G * a.TQ * D * 2));
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(sQ + c * (BM * 128), &tm_q, bar_q(), c * 64, kvh * a.G, t0, b);
        }
#pragma unroll 1
        for (int j = 0; j < n_tiles && ok; ++j) {
            const int s = j % STAGES;
            if (j >= STAGES) ok = warp_wait(bar_ke(s), ((j / STAGES) - 1) & 1, abort);
            if (!ok) break;
            const uint32_t kd = sK + s * C::KVBYTES, vd = sV + s * C::KVBYTES;
            if (j < n_band) {
                if (lane == 0) {
                    const int k0 = kv_lo + j * BN;
                    mbar_arrive_expect_tx(bar_kf(s), C::KVBYTES);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) tma_load_4d(kd + c * (BN * 128), &tm_k, bar_kf(s), c * 64, kvh, k0, b);
                    mbar_arrive_expect_tx(bar_vf(s), C::KVBYTES);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) tma_load_4d(vd + c * (BN * 128), &tm_v, bar_vf(s), c * 64, kvh, k0, b);
                }
            } else {
                // global-column tile: gather rows global_idx[jg*BN + r] (zero rows past the list)
                const int g0 = (j - n_band) * BN;
                constexpr int kPieces = D / 8;
                for (int idx = lane; idx < BN * kPieces; idx += 32) {
                    const int r = idx / kPieces, pc = idx % kPieces;
                    const int gi = g0 + r;
                    int srow = -1;
                    if (gi < a.n_global) {
                        const int gs = a.global_idx[gi];
                        if (gs >= 0 && gs < a.T) srow = gs;
                    }
                    uint4 kx = make_uint4(0, 0, 0, 0), vx = make_uint4(0, 0, 0, 0);
                    if (srow >= 0) {
                        const int64_t eb = static_cast<int64_t>(b);
                        kx = *reinterpret_cast<const uint4 *>(a.k + eb * a.k_st[0] + static_cast<int64_t>(srow) * a.k_st[1] +
                                                              static_cast<int64_t>(kvh) * a.k_st[2] + pc * 8);
                        vx = *reinterpret_cast<const uint4 *>(a.v + eb * a.v_st[0] + static_cast<int64_t>(srow) * a.v_st[1] +
                                                              static_cast<int64_t>(kvh) * a.v_st[2] + pc * 8);
                    }
                    const uint32_t off = (pc >> 3) * (BN * 128) + r * 128 + (((pc & 7) ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(sgen + C::OFF_K + s * C::KVBYTES + off) = kx;
                    *reinterpret_cast<uint4 *>(sgen + C::OFF_V + s * C::KVBYTES + off) = vx;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_kf(s));
                    mbar_arrive(bar_vf(s));
                }
            }
            last_tile[s] = j;
        }
        if (!ok && lane == 0) {
            // drain the copies still in flight before the CTA exits
            mbar_drain(bar_q(), 0, &g_band_err);
#pragma unroll
            for (int s = 0; s < STAGES; ++s)
                if (last_tile[s] >= 0 && last_tile[s] < n_band) {
                    mbar_drain(bar_kf(s), (last_tile[s] / STAGES) & 1, &g_band_err);
                    mbar_drain(bar_vf(s), (last_tile[s] / STAGES) & 1, &g_band_err);
                }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(BM, D, false, true);
            bool ok = mbar_wait(bar_q(), 0, abort, &g_band_err);
            auto issue_pv = [&](int i) -> bool {
                const int s = i % STAGES, pb = i & 1;
                if (!mbar_wait(bar_pf(pb), (i >> 1) & 1, abort, &g_band_err)) return false;
                if (!mbar_wait(bar_vf(s), (i / STAGES) & 1, abort, &g_band_err)) return false;
                tc_fence_after();
                const uint32_t pbase = sP + pb * C::PBYTES, vbase = sV + s * C::KVBYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t ad = smem_desc(pbase + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024, kSwizzle128B);
                    const uint64_t bd = smem_desc(vbase + kk * 2048, BN * 128, 1024, kSwizzle128B);
                    tc_mma_ss(tmem + C::TM_O, ad, bd, idPV, (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar_pv(pb));
                tc_commit(bar_ke(s));
                return true;
            };
#pragma unroll 1
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j % STAGES, sb = j & 1;
                ok = mbar_wait(bar_kf(s), (j / STAGES) & 1, abort, &g_band_err);
                if (ok && j >= 2) ok = mbar_wait(bar_se(sb), ((j >> 1) - 1) & 1, abort, &g_band_err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kbase = sK + s * C::KVBYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ad = smem_desc(sQ + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024, kSwizzle128B);
                    const uint64_t bd = smem_desc(kbase + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024, kSwizzle128B);
                    tc_mma_ss(tmem + C::TM_S + sb * BN, ad, bd, idS, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar_sf(sb));
                if (j >= 1) ok = issue_pv(j - 1);
            }
            if (ok && n_tiles > 0) ok = issue_pv(n_tiles - 1);
            if (!ok) {
                tc_commit(bar_drain);
                mbar_drain(bar_drain, 0, &g_band_err);
            }
        }
        __syncwarp();
    } else {
        // ============================ softmax / epilogue ============================
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;             // row == TMEM lane
        const int tq = r / a.G, hj = r % a.G;
        const int t = t0 + tq;
        const bool row_ok = tq < a.TQ && t < a.T;
        const int h = kvh * a.G + hj;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        float m = -INFINITY, l = 0.f;
        int count = 0;
        bool ok = true;
#pragma unroll 1
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j & 1;
            if (!warp_wait(bar_sf(sb), (j >> 1) & 1, abort)) { ok = false; break; }
            tc_fence_after();
            float x[BN];
            {
                uint32_t raw[32];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    tmem_ld32(tmem + lane_addr + C::TM_S + sb * BN + c * 32, raw);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(raw[e]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_se(sb));

            // mask
            if (j < n_band) {
                const int k0 = kv_lo + j * BN;
                const bool interior = (a.wl < 0 || k0 >= t1 - a.wl) && (a.wr < 0 || k0 + BN - 1 <= t0 + a.wr) &&
                                      (k0 + BN - 1 <= a.T - 1);
                if (interior) {
                    count += BN;
                } else {
#pragma unroll
                    for (int c = 0; c < BN; ++c) {
                        const int sk = k0 + c;
                        const bool al = sk <= a.T - 1 && in_band(t, sk, a.wl, a.wr);
                        count += al ? 1 : 0;
                        x[c] = al ? x[c] : -INFINITY;
                    }
                }
            } else {
                const int g0 = (j - n_band) * BN;
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    const int gi = g0 + c;
                    bool al = false;
                    if (gi < a.n_global) {
                        const int gs = __ldg(a.global_idx + gi);
                        al = gs >= 0 && gs < a.T && !in_band(t, gs, a.wl, a.wr);
                    }
                    count += al ? 1 : 0;
                    x[c] = al ? x[c] : -INFINITY;
                }
            }
            // running max (log2 domain) with lazy rescale
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; ++c) mx = fmaxf(mx, x[c]);
            const float mt = mx * a.scale_log2;
            const bool need = mt > m + kRescaleTau;
            const float mu = need ? mt : m;
            const float alpha = need ? ex2(m - mu) : 1.f;  // m = -inf gives 0
            if (__any_sync(0xffffffffu, need) && j > 0) {
                // O holds PV_0 .. PV_{j-1}; wait for the last one, then rescale this warp's rows.
                if (!warp_wait(bar_pv((j - 1) & 1), ((j - 1) >> 1) & 1, abort)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tmem + lane_addr + C::TM_O + c * 32, ov);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    tmem_st32(tmem + lane_addr + C::TM_O + c * 32, ov);
                }
                tc_wait_st();
            }
            m = mu;
            const float msub = mu == -INFINITY ? 0.f : mu;
            float rs = 0.f;
            // P buffer sb was last read by PV_{j-2}
            if (j >= 2) {
                if (!warp_wait(bar_pv(sb), ((j - 2) >> 1) & 1, abort)) { ok = false; break; }
            }
            uint8_t *pdst = sgen + C::OFF_P + sb * C::PBYTES;
#pragma unroll
            for (int c8 = 0; c8 < BN / 8; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = ex2(fmaf(x[c8 * 8 + 2 * e], a.scale_log2, -msub));
                    const float p1 = ex2(fmaf(x[c8 * 8 + 2 * e + 1], a.scale_log2, -msub));
                    rs += p0 + p1;
                    w[e] = pack_bf16x2(p0, p1);
                }
                const uint32_t off = (c8 >> 3) * (BM * 128) + r * 128 + (((c8 & 7) ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(pdst + off) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            l = l * alpha + rs;
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pf(sb));
        }

        // ---- epilogue
        if (ok && n_tiles > 0) {
            ok = warp_wait(bar_pv((n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1, abort);
        }
        // all four softmax warps agree before touching the Q region (reused as O staging)
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const bool all_ok = *abort == 0 && ok;
        if (all_ok) {
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(tmem + lane_addr + C::TM_O + c * 32, ov);
                tc_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 2 * e]) * inv_l,
                                           __uint_as_float(ov[q4 * 8 + 2 * e + 1]) * inv_l);
                    const int pc = c * 4 + q4;  // 16-byte piece index along d
                    const uint32_t off = (pc >> 3) * (BM * 128) + r * 128 + (((pc & 7) ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(sgen + C::OFF_Q + off) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            if (row_ok) {
                const int64_t li = (static_cast<int64_t>(b) * a.H_q + h) * a.T + t;
                a.lse[li] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
                if (a.counts) a.counts[li] = count;
            }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (all_ok && warp == 2 && lane == 0) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_store_4d(&tm_o, sQ + c * (BM * 128), c * 64, kvh * a.G, t0, b);
            tma_store_commit();
            tma_store_wait_all();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 4-D bf16 map over (d, head, token, batch) with a (64, box_h, box_t, 1) box, 128-B swizzle.
bool make_map(CUtensorMap *m, const void *base, int D, int H, int T, int B, const int64_t st[3], int box_h,
              int box_t) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2, static_cast<cuuint64_t>(st[1]) * 2,
                             static_cast<cuuint64_t>(st[0]) * 2};
    cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(box_h), static_cast<cuuint32_t>(box_t), 1u};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_band_d(const BandArgs &x, cudaStream_t s) {
    using C = BandCfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(band_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int G = x.H_q / x.H_kv;
    const int TQ = BM / G;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, x.q, D, x.H_q, x.T, x.B, x.q_st, G, TQ) ||
        !make_map(&mk, x.k, D, x.H_kv, x.T, x.B, x.k_st, 1, C::BN) ||
        !make_map(&mv, x.v, D, x.H_kv, x.T, x.B, x.v_st, 1, C::BN) ||
        !make_map(&mo, x.o, D, x.H_q, x.T, x.B, x.o_st, G, TQ))
        return cudaErrorInvalidValue;
    BandKernelArgs a{};
    a.B = x.B;
    a.T = x.T;
    a.H_q = x.H_q;
    a.H_kv = x.H_kv;
    a.G = G;
    a.TQ = TQ;
    a.n_qtiles = (x.T + TQ - 1) / TQ;
    a.wl = x.wl;
    a.wr = x.wr;
    a.scale_log2 = x.scale_log2;
    a.global_idx = x.global_idx;
    a.n_global = x.n_global;
    a.k = static_cast<const __nv_bfloat16 *>(x.k);
    a.v = static_cast<const __nv_bfloat16 *>(x.v);
    for (int i = 0; i < 3; ++i) {
        a.k_st[i] = x.k_st[i];
        a.v_st[i] = x.v_st[i];
    }
    a.lse = x.lse;
    a.counts = x.counts;
    const long long units = static_cast<long long>(x.B) * x.H_kv * a.n_qtiles;
    if (units <= 0 || units > 0x7fffffffLL) return cudaErrorInvalidValue;
    band_fwd_kernel<D><<<static_cast<unsigned>(units), kThreads, C::SMEM, s>>>(mq, mk, mv, mo, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_band(const BandArgs &x, cudaStream_t s) {
    switch (x.D) {
        case 64: return launch_band_d<64>(x, s);
        case 128: return launch_band_d<128>(x, s);
        case 256: return launch_band_d<256>(x, s);
        default: return cudaErrorInvalidValue;
    }
}

unsigned int band_read_clear_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_band_err, sizeof v) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_band_err, &z, sizeof z);
    return v;
}

}  // namespace swa
