// swa_band.cu -- banded (sliding-window) attention prefill on 5th-generation
// tensor cores (sm_103a).
//
// Work unit: one (batch b, key/value head kvh, group of NQT query tiles).  A query
// tile is 128 rows = TQ consecutive tokens x the G = H_q/H_kv query heads of the
// group (row = token_local * G + head_local), so every key/value tile is loaded
// once for the whole group.  The unit iterates only over the key tiles that
// intersect the union of its rows' bands
//     [max(0, t_first - wl), min(T-1, t_last + wr)]
// -- keys outside the window are never loaded or scored, as in the production
// kernels described by "Sliding Window Attention" (lizeman.github.io llm-arch-kb,
// section 3) and the superteams.ai glossary -- followed by ceil(n_global / BN)
// "global column" tiles holding the key/value rows of the global positions
// (prathamp.com "Sliding Window Attention: From Local Windows to Global Context",
// section 4.3).
//
// Persistent: one CTA per SM walks the units (longest first, dealt in rounds of the grid
// size in alternating directions); TMEM and the mbarriers are set up once and every
// barrier phase runs on across units.
// Roles:
//   warp 0        K/V producer: K_0, V_0, K_1, V_1, ... of every unit into a ring of
//                 NSLOT shared-memory slots (TMA for band tiles, plain gathers into
//                 the same 128B-swizzled layout for global tiles).  V_j and K_{j+1} are
//                 copied together and signal one barrier (that of K_{j+1}'s slot): with
//                 two query tiles the MMA warp then waits once per key tile, before
//                 P_A V_j, and S_A(j+1) needs no wait of its own; with one query tile the
//                 wait before S(j+1) covers V_j's P V.  With two query tiles, ring slots
//                 are released by key fills (a value fill's last reader precedes the next
//                 key fill's); without global positions that release is an arrive by
//                 softmax warpgroup B once it sees S_B(j) done.
//   warp 1        TMEM owner and MMA issuer (warp-uniform loop, one elected lane issues):
//                   S_X   = Q_X K_j^T   (tcgen05.mma, A/B from shared memory; at head dim
//                                        256 A = Q from tensor memory)
//                   O_X  += P_X V_j     (tcgen05.mma, A = P from tensor memory)
//   warp 2        Q loader: a unit's query tiles once the previous unit's last S MMA
//                 from that tile has completed (its only readers; with global positions,
//                 once the previous unit's epilogue has seen all its MMAs complete).
//   softmax WGs   NQT warpgroups; one row per thread (TMEM lane).  Scores are masked
//                 only on band-edge and global tiles; the running max is kept in the
//                 log2 domain; P = 2^(x - m) is written back as bf16 over the S
//                 columns it came from; O is rescaled in TMEM only when a row's max
//                 grows by more than 2^8 (numerator and denominator share the stale
//                 max, so the result is exact either way).  Epilogue: O / l -> bf16
//                 stored straight from registers; lse and attended-key counts.
// NQT = 2 (head dim <= 128): two query tiles ping-pong -- while one warpgroup turns
// S_A into P_A the tensor cores run S_B and P_B V -- with TMEM S_A | S_B | O_A | O_B.
// NQT = 1 (head dim 256): one query tile, S double-buffered, TMEM S0 | S1 | Q | O.
// Builds per head dim: with and without global-position code (kGlob), and for long and
// short bands (kShort: at most kShortTiles key tiles per unit, where most tiles are band
// edges or lie beyond one query tile's band).  At most kNarrow global positions take one
// kNarrow-key global-column tile (S with N = kNarrow, P V with K = kNarrow).
// Every wait is bounded; on expiry the CTA records an error word, drains its
// copies and MMAs, frees TMEM and returns.
#include <atomic>
#include <cfloat>
#include <climits>
#include <cmath>

#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "swa_internal.h"

namespace swa {
namespace {

__device__ unsigned int g_band_err = 0;
static_assert(kErrWaitTimeout == SWA_DEVERR_WAIT_TIMEOUT && kErrDrainTimeout == SWA_DEVERR_DRAIN_TIMEOUT &&
                  kErrBadGlobalList == SWA_DEVERR_GLOBAL_LIST,
              "device error bits");

constexpr int BM = 128;              // query rows per tile (TMEM lanes)
constexpr int kNarrow = 32;          // width of a narrow global-column tile
constexpr int kShortTiles = 8;       // key tiles per unit at most for the short-band kernel
constexpr float kRescaleTau = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

template <int D>
struct BandCfg {
    static constexpr int NQT = D <= 128 ? 2 : 1;     // query tiles per unit
    static constexpr int BN = D == 256 ? 64 : 128;  // keys per K/V tile
    // NQT = 2: warpgroup 0 = K/V producer warp, MMA warp, Q loader warp, one idle
    // warp; warpgroups 1, 2 = softmax.  Twelve warps put three on each SM
    // sub-partition, whose 16K-register file caps the launch at 168 registers a
    // thread; setmaxnreg then moves registers from warpgroup 0 (104) to the softmax
    // warpgroups (200):  128 * 104 + 256 * 200 = 64512 = 384 * 168.  (Neither side
    // spills; control warps below 104 spill in the producer's gather.)
    // NQT = 1: the same warpgroup 0, then one softmax warpgroup (256 threads).
    static constexpr int THREADS = NQT == 2 ? 384 : 256;
    static constexpr int SOFTMAX_WARP0 = 4;
    static constexpr int REG_CTRL = 104, REG_SOFTMAX = 200;
    static_assert(NQT == 1 || 128 * REG_CTRL + 256 * REG_SOFTMAX <= THREADS * 168, "register split");
    static constexpr int QBYTES = BM * D * 2;  // one query tile
    static constexpr int TBYTES = BN * D * 2;  // one K or V tile
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = NQT * QBYTES;
    // K/V ring: as deep as shared memory allows, except at head dim 64, where six 16 KB slots
    // (three tiles in flight) measured best (Longformer shape, with and without global
    // positions: +2.1% / +1.6% over twelve; 4, 5, 7 slots slower, 8-10 as six with globals)
    static constexpr int NSLOT = D == 64 ? 6 : (232448 - 2048 - OFF_RING) / TBYTES;
    static constexpr int OFF_BAR = OFF_RING + NSLOT * TBYTES;
    // q_full[2], q_empty[2], kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2],
    // o_done[2], o_free[2], two unused words, drain
    static constexpr int NBAR = 2 * NSLOT + 15;
    static constexpr int OFF_TMEMPTR = OFF_BAR + NBAR * 8;
    // global positions of a list of at most BN entries, staged once per CTA
    static constexpr int OFF_GPOS = (OFF_TMEMPTR + 16 + 15) & ~15;
    static constexpr int SMEM = OFF_GPOS + BN * 4 + 1024;  // + slack for 1024-B alignment
    static_assert(OFF_GPOS + BN * 4 - OFF_BAR <= 2048, "barriers and staged positions exceed the reserve");
    static constexpr uint32_t TMEM_COLS = 512;
    __host__ __device__ static constexpr uint32_t tm_s(int slot) { return static_cast<uint32_t>(slot * BN); }
    __host__ __device__ static constexpr uint32_t tm_o(int tile) { return 256u + static_cast<uint32_t>(tile * 128); }
    // One query tile (head dim 256): the tile is copied into tensor memory once per unit
    // (sixteen tcgen05.cp of 128 rows x 256 bits, issued in order by the MMA warp, which then
    // releases the tile's shared memory with one commit) into the 128 columns between
    // S0 | S1 and O, and every S MMA takes its A operand from there, reading only its K slice
    // from shared memory (2 KB instead of 6 KB per 128x64x16 MMA): Gemma-local 1138 -> 1198
    // TFLOP/s in an A/B.
    static constexpr bool QTM = NQT == 1;
    static constexpr uint32_t TM_Q = 128;
    static_assert(NSLOT >= 3, "K/V ring too shallow");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(!QTM || (tm_s(1) + BN <= TM_Q && TM_Q + D / 2 <= tm_o(0)), "query tile in tensor memory");
    static_assert(tm_o(NQT - 1) + D <= TMEM_COLS && tm_s(1) + BN <= 256, "tensor memory budget");
};

struct BandKernelArgs {
    int B, T, H_q, H_kv, G, TQ, n_units_t, n_units;
    // Keys live in their own index space of Tk positions: query row t sits at key
    // index t + q_off, and keys below kmin[b] (when kmin is set) do not exist.
    int Tk, q_off;
    const int32_t *kmin;
    // key index q_off of sequence b is position p0[b] (nullptr: 0); global positions are
    // positions, and with gcol_list_rows their K/V rows are the k/v rows in list order
    const int32_t *p0;
    int gcol_list_rows;
    int gcol_hi;  // global positions at or above gcol_hi are not keys (Tk; no bound with a row list)
    int wl, wr;
    float scale_log2;
    const int32_t *global_idx;
    int n_global;
    int sink;  // global columns are attention sinks: kept only left of a row's band
    int sep;   // separate global projections: band tiles drop global columns, the
               // global-column tiles keep all of them
    const __nv_bfloat16 *k, *v;  // for the global-column gather (k_g, v_g when sep)
    int64_t k_st[3], v_st[3], o_st[3];
    __nv_bfloat16 *o;
    int o_align32;  // o and its strides are 32-byte aligned: rows stored 32 bytes at a time
    float *lse;
    int32_t *counts;
    int64_t lse_st[3];
    // at most kNarrow global positions: their one column tile is kNarrow keys wide (S with
    // N = kNarrow, P V with K = kNarrow, a kNarrow-column softmax) instead of BN
    int gcol_narrow;
    // planted fault of the failure-detection tests: the K/V producer of every CTA issues
    // no ring fill numbered at or past this (INT_MAX: off), so the other roles' waits run out
    int fault_stop_fill;
};

// Index of the first entry >= k0 of the sorted list g[0..n) (n if none).
__device__ __forceinline__ int first_at_least(const int32_t *g, int n, int k0) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(g + mid) < k0) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Geometry of work unit u (units are numbered longest first).
struct Unit {
    int b, kvh, t0, kv_lo, n_band, n_tiles, kmin;
    int pos_off;  // position of key index x is x + pos_off
};

template <int NQT, int BN>
__device__ __forceinline__ Unit unit_of(int u, const BandKernelArgs &a) {
    Unit w;
    const int bh = u % (a.B * a.H_kv);
    const int ut = a.n_units_t - 1 - u / (a.B * a.H_kv);
    w.b = bh / a.H_kv;
    w.kvh = bh % a.H_kv;
    w.t0 = ut * NQT * a.TQ;
    const int t1 = min(a.T - 1, w.t0 + NQT * a.TQ - 1);
    w.kmin = a.kmin ? __ldg(a.kmin + w.b) : 0;
    w.pos_off = a.p0 ? __ldg(a.p0 + w.b) - a.q_off : 0;
    w.kv_lo = a.wl < 0 ? w.kmin : max(w.kmin, w.t0 + a.q_off - a.wl);
    const int kv_hi = a.wr < 0 ? a.Tk - 1 : min(a.Tk - 1, t1 + a.q_off + a.wr);
    w.n_band = (kv_hi - w.kv_lo + BN) / BN;
    w.n_tiles = w.n_band + (a.n_global + BN - 1) / BN;
    return w;
}

// Every lane waits (each acquires the barrier); the warp proceeds only if all did,
// so the .sync.aligned tcgen05 instructions that follow stay convergent.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, abort, &g_band_err);
    return __all_sync(0xffffffffu, ok);
}

// kGlob: the launch has global positions (global-column tiles).  kShort: the band spans at
// most kShortTiles key tiles per unit, so most tiles are band edges (or, with two query
// tiles, beyond one tile's band): their masks take the cheaper forms below.
template <int D, bool kGlob, bool kShort>
__global__ void __launch_bounds__(BandCfg<D>::THREADS, 1)
    band_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const BandKernelArgs a) {
    using C = BandCfg<D>;
    constexpr int BN = C::BN, NSLOT = C::NSLOT, NQT = C::NQT;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t *sgen = smem_raw + (sbase - sraw);

    const uint32_t sQ = sbase + C::OFF_Q, sRing = sbase + C::OFF_RING;
    const uint32_t bars = sbase + C::OFF_BAR;
    auto bar_qf = [&](int x) { return bars + 8u * x; };
    auto bar_qe = [&](int x) { return bars + 8u * (2 + x); };
    auto bar_full = [&](int s) { return bars + 8u * (4 + s); };
    auto bar_empty = [&](int s) { return bars + 8u * (4 + NSLOT + s); };
    auto bar_sf = [&](int i) { return bars + 8u * (4 + 2 * NSLOT + i); };
    auto bar_pf = [&](int i) { return bars + 8u * (6 + 2 * NSLOT + i); };
    auto bar_od = [&](int i) { return bars + 8u * (8 + 2 * NSLOT + i); };
    auto bar_of = [&](int i) { return bars + 8u * (10 + 2 * NSLOT + i); };
    const uint32_t bar_drain = bars + 8u * (14 + 2 * NSLOT);
    // NQT = 1: only value fills release their slot (a tile's S MMAs precede its P V, so the
    // release of V_j also frees K_j's slot).  With an odd ring, a slot alternates key and
    // value fills, so its barrier counts value fills only: the phase of value fill p.
    static_assert(NQT == 2 || NSLOT % 2 == 1, "value-only slot releases need an odd ring");
    auto vpar = [&](int p) -> uint32_t {
        const int sl = p % NSLOT, i = p / NSLOT;
        return static_cast<uint32_t>(((i - ((1 + sl) & 1)) / 2) & 1);
    };
    // NQT = 2: only key fills release their slot (V_j's last reader, P V_B(j), is issued
    // before K_{j+1}'s, S_B(j+1)), so a value fill's slot is free once the next key fill's
    // is.  The phase of key fill p on its slot's barrier: an odd ring alternates key and
    // value fills per slot, an even one keeps them in slots of their own.
    // (Not in the long-band build with global positions, where a unit's last value slot,
    // held across the boundary until the next unit's first key is released, cost 1.8%.)
    constexpr bool kKeyRel = NQT == 2 && !(kGlob && !kShort);
    // Paired fills: V_j and K_{j+1} are copied together on K_{j+1}'s slot barrier, so one
    // wait covers both: before P V_A(j) with two query tiles (S_A(j+1) follows), before
    // S(j+1) with one (P V(j) follows).  A slot barrier then completes only for key fills
    // (and for the CTA's last value fill, which has no key fill after it): fpar(q) is the
    // parity of owner fill q's completion.  A global-column tile is gathered by the
    // producer warp: its part of a pair is counted by one plain arrival once its stores are
    // visible to the async proxy, the TMA part by expected bytes.
    // kSoftRel (no global positions, two query tiles): softmax warpgroup B, which waits for
    // S_B(j) anyway, releases K_j's slot instead of a commit by the MMA warp
    constexpr bool kSoftRel = !kGlob && NQT == 2;
    auto fpar = [&](int q) -> uint32_t {
        const int sl = q % NSLOT, i = q / NSLOT;
        const int n = NSLOT % 2 == 1 ? (i - (sl & 1) + 1) / 2 : (sl % 2 == 0 ? i : 0);
        return static_cast<uint32_t>(n & 1);
    };
    // This CTA's i-th unit.  Units are numbered longest first and dealt in rounds of
    // gridDim.x, in alternating directions (a CTA that takes a round's longest unit takes
    // the next round's shortest), so the per-CTA totals of the shorter units at the end
    // even out.
    auto unit_at = [&](int i) -> int {
        const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
        return i * G + ((i & 1) ? G - 1 - c : c);
    };
    // key tiles of this CTA over all its units: ring fills 0 .. 2 * count - 1
    auto count_cta_tiles = [&]() -> int {
        int c = 0;
        for (int i = 0; unit_at(i) < a.n_units; ++i) c += unit_of<NQT, BN>(unit_at(i), a).n_tiles;
        return c;
    };
    auto kpar = [&](int p) -> uint32_t {
        const int sl = p % NSLOT, i = p / NSLOT;
        return static_cast<uint32_t>((NSLOT % 2 == 1 ? (i - (sl & 1)) / 2 : i) & 1);
    };
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(sgen + C::OFF_TMEMPTR);
    int *gpos = reinterpret_cast<int *>(sgen + C::OFF_GPOS);
    // A list of at most BN positions is staged in shared memory for the global-column mask.
    const bool gpos_staged = kGlob && a.n_global > 0 && a.n_global <= BN;
    if (gpos_staged)
        for (int i = tid; i < a.n_global; i += C::THREADS) gpos[i] = a.global_idx[i];
    if constexpr (kGlob) {
        // The list's contract (strictly increasing, within [0, Tk)), checked across the
        // grid and reported on the host as an invalid argument.  Every read below stays in
        // bounds whatever the list holds (gathers and searches are clamped), but a list
        // that breaks the contract gives undefined outputs.  A sink list built by the
        // library (row-list mode) holds positions, not key indices, and is not checked.
        if (!a.gcol_list_rows)
            for (int i = blockIdx.x * C::THREADS + tid; i < a.n_global; i += gridDim.x * C::THREADS) {
                const int gi = __ldg(a.global_idx + i);
                if (gi < 0 || gi >= a.Tk || (i + 1 < a.n_global && __ldg(a.global_idx + i + 1) <= gi))
                    atomicOr(&g_band_err, kErrBadGlobalList);
            }
    }

    // ---- setup: barriers, TMEM (once per CTA)
    if (tid == 0) {
        abort_flag = 0;
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar_qf(x), 1);
            // the four warps of the tile's softmax warpgroup; with the tile in tensor memory,
            // the MMA warp's one commit after the copy
            mbar_init(bar_qe(x), C::QTM ? 1 : 4);
            mbar_init(bar_sf(x), 1);
            mbar_init(bar_pf(x), 4);
            mbar_init(bar_od(x), 1);
            mbar_init(bar_of(x), 4);
        }
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
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
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    volatile int *abort = &abort_flag;
    // a dependent grid launched behind this one (the global-row pass, only with global
    // positions) reads none of its outputs: it may take SMs as soon as this grid's CTAs
    // leave them
    if constexpr (kGlob) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ============================ K/V producer ============================
        if constexpr (NQT == 2) regs_dec<C::REG_CTRL>();
        int g = 0;  // ring fills issued so far (all units)
        bool ok = true;
        // a fill's slot is free once its last occupant (a key fill), or the key fill after
        // its last occupant (a value fill), has been released
        auto slot_free = [&](int p) -> bool {
            if (p < NSLOT) return true;
            const int prev = p - NSLOT;
            if constexpr (NQT == 1) {
                const int vp = (prev & 1) ? prev : prev + 1;  // value fills release
                return warp_wait(bar_empty(vp % NSLOT), vpar(vp), abort);
            } else if constexpr (kKeyRel) {
                const int kp = (prev & 1) ? prev + 1 : prev;  // key fills release
                return warp_wait(bar_empty(kp % NSLOT), kpar(kp), abort);
            } else {
                return warp_wait(bar_empty(p % NSLOT), ((p / NSLOT) - 1) & 1, abort);  // every fill
            }
        };
        auto tma_tile = [&](const Unit &w, int j, bool is_v, int slot, uint32_t bar) {
            const int k0 = w.kv_lo + j * BN;
            // debug build: the tile starts inside the key rows of an existing (b, kv head)
            (void)SWA_IN_BOUNDS(k0 >= 0 && k0 < a.Tk && w.b >= 0 && w.b < a.B && w.kvh >= 0 && w.kvh < a.H_kv,
                                &g_band_err);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(sRing + slot * C::TBYTES + c * (BN * 128), is_v ? &tm_v : &tm_k, bar, c * 64, w.kvh,
                            k0, w.b);
        };
        // global-column tile: rows global_idx[g0 + r] (zero rows past the list), gathered by
        // the warp into the 128B-swizzled layout a TMA copy would have written
        auto gather_tile = [&](const Unit &w, int j, bool is_v, int slot) {
            if constexpr (kGlob) {
                const int g0 = (j - w.n_band) * BN;
                const __nv_bfloat16 *src = is_v ? a.v : a.k;
                const int64_t *st = is_v ? a.v_st : a.k_st;
                constexpr int kPieces = D / 8;
                const int rows = a.gcol_narrow ? kNarrow : BN;  // rows the MMAs read
                for (int idx = lane; idx < rows * kPieces; idx += 32) {
                    const int r = idx / kPieces, pc = idx % kPieces;
                    const int gi = g0 + r;
                    int srow = -1;
                    if (gi < a.n_global) {
                        if (a.gcol_list_rows) {
                            srow = gi;
                        } else {
                            const int gs = a.global_idx[gi];
                            if (gs >= 0 && gs < a.Tk) srow = gs;
                        }
                    }
                    uint4 val = make_uint4(0, 0, 0, 0);
                    if (srow >= 0 && SWA_IN_BOUNDS(srow < (a.gcol_list_rows ? a.n_global : a.Tk) && w.b < a.B &&
                                                       w.kvh < a.H_kv && pc * 8 < D,
                                                   &g_band_err))
                        val = *reinterpret_cast<const uint4 *>(src + static_cast<int64_t>(w.b) * st[0] +
                                                               static_cast<int64_t>(srow) * st[1] +
                                                               static_cast<int64_t>(w.kvh) * st[2] + pc * 8);
                    const uint32_t off = (pc >> 3) * (BN * 128) + r * 128 + (((pc & 7) ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(sgen + C::OFF_RING + slot * C::TBYTES + off) = val;
                }
            }
        };
        // one barrier phase for tile (wa, ja) and, if `two`, key tile (wb, jb): band tiles by
        // TMA (their bytes expected on the barrier), global tiles gathered by the warp, whose
        // one arrival comes only after its stores are visible to the tensor cores
        auto fill = [&](const Unit &wa, int ja, bool va, int sa, bool two, const Unit &wb, int jb, int sb,
                        uint32_t bar) {
            const bool ta = !kGlob || ja < wa.n_band, tb = two && (!kGlob || jb < wb.n_band);
            const bool gath = !ta || (two && !tb);
            const uint32_t tx = (ta ? 1u : 0u) + (tb ? 1u : 0u);
            if (lane == 0) {
                if (!gath)
                    mbar_arrive_expect_tx(bar, tx * C::TBYTES);
                else if (tx > 0)
                    mbar_expect_tx(bar, tx * C::TBYTES);
                if (ta) tma_tile(wa, ja, va, sa, bar);
                if (tb) tma_tile(wb, jb, false, sb, bar);
            }
            if (gath) {
                if (!ta) gather_tile(wa, ja, va, sa);
                if (two && !tb) gather_tile(wb, jb, false, sb);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar);
            }
            __syncwarp();
        };
        const int cta_tiles = count_cta_tiles(), nfill = 2 * cta_tiles;
        int ui = 0, u = unit_at(0), j = 0;  // unit ordinal, unit, tile within it
        Unit w{};
        if (u < a.n_units) w = unit_of<NQT, BN>(u, a);
        // planted fault: only the steps whose fills all lie below a.fault_stop_fill run
        // (step t issues fills up to 2t + 2; the last step, fill nfill - 1 alone)
        const int n_steps = a.fault_stop_fill >= nfill ? cta_tiles : max(0, (a.fault_stop_fill - 1) / 2);
        const bool k0 = nfill > 0 && a.fault_stop_fill > 0;
        if (k0) fill(w, 0, false, 0, false, w, 0, 0, bar_full(0));  // K_0 alone
        g = k0 ? 1 : 0;
        ok = n_steps == cta_tiles;
#pragma unroll 1
        for (int t = 0; t < n_steps; ++t) {
            // the tile after (u, j), possibly the next unit's first
            int u2 = u, j2 = j + 1, ui2 = ui;
            if (j2 >= w.n_tiles) {
                ui2 = ui + 1;
                u2 = unit_at(ui2);
                j2 = 0;
            }
            const bool has_next = t + 1 < cta_tiles;
            const Unit w2 = has_next && u2 != u ? unit_of<NQT, BN>(u2, a) : w;
            const int pv = 2 * t + 1, own = has_next ? pv + 1 : pv;
            if (!(slot_free(pv) && (!has_next || slot_free(own)))) {
                ok = false;
                break;
            }
            fill(w, j, true, pv % NSLOT, has_next, w2, j2, own % NSLOT, bar_full(own % NSLOT));
            g = own + 1;
            u = u2;
            ui = ui2;
            j = j2;
            w = w2;
        }
        if (!ok && lane == 0) {
            // drain the owner barriers of the copies that may still be in flight.  Fills
            // below g - NSLOT have landed: fill q + NSLOT was issued only once the key
            // (NQT = 2) or value (NQT = 1) fill that releases q's slot was released, and
            // its readers waited for the owner barrier of q.  So only fills g - NSLOT ..
            // g - 1 -- one per slot -- can be in flight; their owners are the key fills
            // among them, and the CTA's last fill, which owns its own barrier.
            for (int q = max(0, g - NSLOT); q < g; ++q)
                if ((q & 1) == 0 || q + 1 == nfill) mbar_drain(bar_full(q % NSLOT), fpar(q), &g_band_err);
        }
    } else if (warp == 2) {
        // ============================ Q loader ============================
        if constexpr (NQT == 2) regs_dec<C::REG_CTRL>();
        int k = 0;
        int issued[2] = {0, 0};  // query loads issued per tile
        bool ok = true;
#pragma unroll 1
        for (int u = unit_at(0); u < a.n_units && ok; ++k, u = unit_at(k)) {
            const Unit w = unit_of<NQT, BN>(u, a);
#pragma unroll 1
            for (int x = 0; x < NQT && ok; ++x) {
                // the previous unit's S MMAs are done with this tile's shared memory
                if (k >= 1) ok = warp_wait(bar_qe(x), (k - 1) & 1, abort);
                if (!ok) break;
                if (lane == 0) {
                    const int tx = w.t0 + x * a.TQ;
                    if (tx < a.T) {
                        // debug build: the tile's tokens and its group's heads exist
                        (void)SWA_IN_BOUNDS(tx >= 0 && (w.kvh + 1) * a.G <= a.H_q && w.b < a.B, &g_band_err);
                        mbar_arrive_expect_tx(bar_qf(x), static_cast<uint32_t>(a.G * a.TQ * D * 2));
#pragma unroll
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_4d(sQ + x * C::QBYTES + c * (BM * 128), &tm_q, bar_qf(x), c * 64, w.kvh * a.G,
                                        tx, w.b);
                    } else {
                        mbar_arrive(bar_qf(x));  // tile past the sequence end: nothing to load
                    }
                }
                __syncwarp();
                ++issued[x];
            }
        }
        if (!ok && lane == 0) {
            // drain the last query copy of each tile before exit
            for (int x = 0; x < NQT; ++x)
                if (issued[x] > 0) mbar_drain(bar_qf(x), (issued[x] - 1) & 1, &g_band_err);
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if constexpr (NQT == 2) regs_dec<C::REG_CTRL>();
        // Every lane of the warp runs the MMA issuer's loop, so its control flow and the
        // descriptor and index arithmetic stay warp-uniform; inside each tcgen05 instruction's
        // asm, elect.sync picks the one lane that issues it (always the same lane, so each
        // commit tracks all MMAs before it).  The same loop run by lane 0 alone, in a
        // divergent branch, measured 7.7% slower on the Mistral shape, 6.8% on Gemma-local
        // and 10% on the Longformer shape.
        {
            constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idS_narrow = idesc_bf16_f32(BM, kNarrow, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(BM, D, false, true);
            bool ok = true;
            int J = 0;  // key tiles of this CTA's previous units
            int k = 0;  // units of this CTA so far
            int cta_tiles = 0;
            cta_tiles = count_cta_tiles();
            // S into TMEM slot `slot` from query tile `qt` and the K tile of global tile index jg.
            // The query tiles never move: the A descriptor of every K slice of each is built once
            // here, a constant of the CTA, since the MMA warp's instruction count per tile is
            // part of the tile period (Mistral +1.3%, Longformer +1.7% in A/B runs).  With the
            // query tile in tensor memory (one query tile) the S MMAs take no A descriptor.
            constexpr bool kQDesc = !C::QTM;
            uint64_t qdesc[NQT][D / 16];
#pragma unroll
            for (int qt = 0; qt < NQT; ++qt)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    qdesc[qt][kk] = kQDesc ? smem_desc(sQ + qt * C::QBYTES + (kk >> 2) * (BM * 128) + (kk & 3) * 32,
                                                       16, 1024, kSwizzle128B)
                                           : 0ull;
            // The V slice descriptors of value tile jg: with two query tiles both P V of a tile
            // step read one V tile, so the set is built once per tile step (Mistral +2.7%,
            // Mistral with sinks +1.3%, the Longformer shape without globals +1.2% in an A/B).
            // Sharing the K slice descriptors of the two S MMAs as well made the head-dim-128
            // MMA warp spill and ran slower.
            constexpr bool kShareV = NQT == 2;
            uint64_t vd[BN / 16];
            auto v_descs = [&](int jg) {
                const uint64_t v0 = smem_desc(sRing + ((2 * jg + 1) % NSLOT) * C::TBYTES, BN * 128, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) vd[kk] = desc_offset(v0, kk * 2048);
            };
            auto mma_s = [&](int slot, int qt, int jg, bool wait_k, bool narrow = false) -> bool {
                const int fi = 2 * jg, s = fi % NSLOT;
                // paired fills: a key fill owns its barrier (with V_{jg-1} on it); with two
                // query tiles only the CTA's first key tile is waited for here (phase 0)
                const uint32_t kpty = NQT == 1 ? fpar(fi) : static_cast<uint32_t>((fi / NSLOT) & 1);
                if (wait_k && !warp_wait(bar_full(s), kpty, abort)) return false;
                tc_fence_after();
                const uint32_t qb = sQ + qt * C::QBYTES, kb = sRing + s * C::TBYTES;
                // one descriptor per operand tile; a K slice is a constant byte offset from it
                const uint64_t a0 = smem_desc(qb, 16, 1024, kSwizzle128B), b0 = smem_desc(kb, 16, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ad =
                        kQDesc ? qdesc[qt][kk] : desc_offset(a0, (kk >> 2) * (BM * 128) + (kk & 3) * 32);
                    const uint64_t bd = desc_offset(b0, (kk >> 2) * (BN * 128) + (kk & 3) * 32);
                    uint32_t id = idS;
                    if constexpr (kGlob) id = narrow ? idS_narrow : idS;
                    if constexpr (C::QTM) tc_mma_ts_e(tmem + C::tm_s(slot), tmem + C::TM_Q + kk * 8, bd, id, kk > 0 ? 1u : 0u);
                    else tc_mma_ss_e(tmem + C::tm_s(slot), ad, bd, id, kk > 0 ? 1u : 0u);
                }
                return true;
            };
            // O_tile (+)= P(slot) V of global tile index jg; `first` starts a fresh O.
            auto mma_pv = [&](int slot, int otile, int jg, uint32_t p_parity, bool wait_v, bool first,
                              bool narrow = false, bool have_vd = false) -> bool {
                const int fi = 2 * jg + 1, s = fi % NSLOT;
                if (!warp_wait(bar_pf(slot), p_parity, abort)) return false;
                // V_jg arrives on the barrier of the key fill after it (K_{jg+1}), if any
                const int own = jg + 1 < cta_tiles ? fi + 1 : fi;
                if (wait_v && !warp_wait(bar_full(own % NSLOT), fpar(own), abort)) return false;
                // the previous unit's epilogue has read this O accumulator out
                if (first && k >= 1 && !warp_wait(bar_of(otile), (k - 1) & 1, abort)) return false;
                tc_fence_after();
                const uint32_t vb = sRing + s * C::TBYTES;
                const uint64_t v0 = smem_desc(vb, BN * 128, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    if constexpr (kGlob) {
                        if (narrow && kk >= kNarrow / 16) break;
                    }
                    const uint64_t bd = have_vd ? vd[kk] : desc_offset(v0, kk * 2048);
                    tc_mma_ts_e(tmem + C::tm_o(otile), tmem + C::tm_s(slot) + kk * 8, bd, idPV,
                              (!first || kk > 0) ? 1u : 0u);
                }
                return true;
            };
            auto kslot = [&](int jg) { return (2 * jg) % NSLOT; };
            auto vslot = [&](int jg) { return (2 * jg + 1) % NSLOT; };
#pragma unroll 1
            for (int u = unit_at(0); u < a.n_units && ok; ++k, u = unit_at(k)) {
                const int n = unit_of<NQT, BN>(u, a).n_tiles;
                // tile jj of the unit is the narrow global-column tile
                const int nb = kGlob ? unit_of<NQT, BN>(u, a).n_band : n;
                auto narrow = [&](int jj) { return kGlob && a.gcol_narrow && jj >= nb; };
                // each query tile is waited for just before its first S MMA
                ok = warp_wait(bar_qf(0), k & 1, abort);
                if (!ok) break;
                if constexpr (NQT == 2) {
                    // paired fills: K_J came with V_{J-1}, waited for before that tile's P V
                    ok = mma_s(0, 0, J, J == 0, narrow(0));
                    if (ok) {
                        tc_commit_e(bar_sf(0));
                        ok = warp_wait(bar_qf(1), k & 1, abort);
                    }
                    if (ok) ok = mma_s(1, 1, J, false, narrow(0));
                    if (ok) {
                        tc_commit_e(bar_sf(1));
                        if constexpr (!kSoftRel) tc_commit_e(bar_empty(kslot(J)));
                    }
#pragma unroll 1
                    for (int j = 0; j < n && ok; ++j) {
                        const int jg = J + j;
                        if constexpr (kShareV) v_descs(jg);
                        ok = mma_pv(0, 0, jg, jg & 1, true, j == 0, narrow(j), kShareV);
                        if (!ok) break;
                        if (j + 1 < n) {
                            ok = mma_s(0, 0, jg + 1, false, narrow(j + 1));
                            if (!ok) break;
                            tc_commit_e(bar_sf(0));
                        } else {
                            tc_commit_e(bar_od(0));
                        }
                        ok = mma_pv(1, 1, jg, jg & 1, false, j == 0, narrow(j), kShareV);
                        if (!ok) break;
                        if constexpr (!kKeyRel) tc_commit_e(bar_empty(vslot(jg)));
                        if (j + 1 < n) {
                            ok = mma_s(1, 1, jg + 1, false, narrow(j + 1));
                            if (!ok) break;
                            tc_commit_e(bar_sf(1));
                            if constexpr (!kSoftRel) tc_commit_e(bar_empty(kslot(jg + 1)));
                        } else {
                            tc_commit_e(bar_od(1));
                        }
                    }
                } else {
                    if constexpr (C::QTM) {
                        // the unit's query tile into tensor memory, 16 columns per copy (the
                        // previous unit's last S MMA precedes the copies in the tensor pipe);
                        // its shared memory is free for the next unit once they complete
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            tc_cp_128x256b_e(tmem + C::TM_Q + kk * 8,
                                             smem_desc(sQ + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024, kSwizzle128B));
                        tc_commit_e(bar_qe(0));
                    }
                    ok = mma_s(J & 1, 0, J, true, narrow(0));
                    if (ok) {
                        tc_commit_e(bar_sf(J & 1));
                    }
#pragma unroll 1
                    for (int j = 0; j < n && ok; ++j) {
                        const int jg = J + j;
                        if (j + 1 < n) {
                            // slot (jg+1)&1 last held P of tile jg-1, consumed by its P V issued earlier
                            ok = mma_s((jg + 1) & 1, 0, jg + 1, true, narrow(j + 1));
                            if (!ok) break;
                            tc_commit_e(bar_sf((jg + 1) & 1));
                        }
                        // paired fills: V_jg came with K_{jg+1}, waited for by S(jg+1) just above
                        ok = mma_pv(jg & 1, 0, jg, (jg >> 1) & 1, j + 1 == n, j == 0, narrow(j));
                        if (!ok) break;
                        tc_commit_e(bar_empty(vslot(jg)));
                        if (j + 1 == n) tc_commit_e(bar_od(0));
                    }
                }
                J += n;
            }
            if (!ok) {
                tc_commit_e(bar_drain);
                mbar_drain(bar_drain, 0, &g_band_err);
            }
        }
        __syncwarp();
    } else if (warp >= C::SOFTMAX_WARP0) {
        // ============================ softmax / epilogue ============================
        if constexpr (NQT == 2) regs_inc<C::REG_SOFTMAX>();
        const int wg = (warp - C::SOFTMAX_WARP0) >> 2;  // query tile of this warpgroup
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // row == TMEM lane
        const int tq = r / a.G, hj = r % a.G;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t o_addr = tmem + lane_addr + C::tm_o(wg);
        bool ok = true;
        int J = 0, k = 0;
#pragma unroll 1
        for (int u = unit_at(0); u < a.n_units && ok; ++k, u = unit_at(k)) {
            const Unit w = unit_of<NQT, BN>(u, a);
            const int tx = w.t0 + wg * a.TQ;  // first token of this warpgroup's query tile
            const int t = tx + tq;
            const int h = w.kvh * a.G + hj;
            // (debug build: a real row's O, lse and count addresses lie inside their tensors)
            const bool row_ok =
                tq < a.TQ && t < a.T && SWA_IN_BOUNDS(t >= 0 && h < a.H_q && w.b < a.B, &g_band_err);
            // key-index positions of this tile's first and last rows and of this row
            const int tlo = tx + a.q_off, thi = min(a.T - 1, tx + a.TQ - 1) + a.q_off;
            const int tk = t + a.q_off;
            // this row's band, clipped to [kmin, Tk)
            const int lo_abs = a.wl < 0 ? w.kmin : max(w.kmin, tk - a.wl);
            const int hi_abs = a.wr < 0 ? a.Tk - 1 : min(a.Tk - 1, tk + a.wr);
            float m = -INFINITY, l = 0.f;
            int count = 0;
#pragma unroll 1
            for (int j = 0; j < w.n_tiles; ++j) {
                const int jg = J + j;
                const int slot = NQT == 2 ? wg : (jg & 1);
                const uint32_t parity = NQT == 2 ? (jg & 1) : ((jg >> 1) & 1);
                if (!warp_wait(bar_sf(slot), parity, abort)) {
                    ok = false;
                    break;
                }
                // Without global positions the query tile is released here, at the unit's
                // last S MMA from it (its only readers), so the next unit's rows load while
                // this tile's last softmax, P V and epilogue run: Mistral +0.9% in an A/B.
                // The builds with global positions release it after the epilogue: there the
                // early release measured 4-7% slower (Longformer, Mistral with sinks).
                if (!kGlob && !C::QTM && j + 1 == w.n_tiles && lane == 0) mbar_arrive(bar_qe(wg));
                if constexpr (kSoftRel) {
                    // S_B(jg) was the last MMA issued before this commit: every reader of
                    // K_jg (and of V_{jg-1}) is done, so the key fill's slot is released here
                    // rather than by another commit of the MMA warp
                    if (wg == 1 && quarter == 0 && lane == 0) mbar_arrive(bar_empty((2 * jg) % NSLOT));
                }
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_addr + C::tm_s(slot);
                if constexpr (kGlob) {
                    if (a.gcol_narrow && j >= w.n_band) {
                        // the unit's one global-column tile, at most kNarrow keys wide: the
                        // staged positions left of the row's band are a prefix [0, nl) of the
                        // sorted list and those right of it a suffix [nr, n); sinks keep only
                        // the prefix, separate projections keep every column
                        float xn[kNarrow];
                        {
                            uint32_t raw[32];
                            tmem_ld32(s_addr, raw);
                            tc_wait_ld();
#pragma unroll
                            for (int e = 0; e < kNarrow; ++e) xn[e] = __uint_as_float(raw[e]);
                        }
                        const int n = a.n_global;
                        const int lo_pos = lo_abs + w.pos_off, hi_pos = hi_abs + w.pos_off;
                        int nl = 0, nr = 0;
#pragma unroll
                        for (int step = kNarrow; step >= 1; step >>= 1) {
                            if (nl + step <= n && gpos[nl + step - 1] < lo_pos) nl += step;
                            if (nr + step <= n && gpos[nr + step - 1] <= hi_pos) nr += step;
                        }
                        if (a.sink) nr = n;
                        if (a.sep) nl = nr = n;
                        count += nl + (n - nr);
#pragma unroll
                        for (int c = 0; c < kNarrow; ++c)
                            xn[c] = (c < nl) | ((c >= nr) & (c < n)) ? xn[c] : -INFINITY;
                        float mx8[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            mx8[i] = fmaxf(fmax3(xn[i], xn[8 + i], xn[16 + i]), xn[24 + i]);
                        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                               fmaxf(mx8[6], mx8[7]));
                        const float mt = mx * a.scale_log2;
                        const bool need = mt > m + kRescaleTau;
                        const float mu = need ? mt : m;
                        const float alpha = need ? ex2(m - mu) : 1.f;  // m = -inf gives 0
                        if (__any_sync(0xffffffffu, need) && j > 0) {
                            // O holds P V of tiles 0 .. j-1 of this unit and must be complete:
                            // the release of tile j-1's V slot (fill 2(j-1)+1) is committed
                            // right after that P V
                            if constexpr (NQT == 1) {
                                if (!warp_wait(bar_empty((2 * (jg - 1) + 1) % NSLOT), vpar(2 * (jg - 1) + 1),
                                               abort)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                            }
#pragma unroll 1
                            for (int c = 0; c < D / 32; ++c) {
                                uint32_t ov[32];
                                tmem_ld32(o_addr + c * 32, ov);
                                tc_wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                                tmem_st32(o_addr + c * 32, ov);
                            }
                        }
                        m = mu;
                        const float msub = mu == -INFINITY ? 0.f : mu;
                        const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2), nm2 = f2_pack(-msub, -msub);
                        uint64_t rs2[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) rs2[i] = f2_pack(0.f, 0.f);
                        uint32_t pk[kNarrow / 2];
#pragma unroll
                        for (int e = 0; e < kNarrow / 2; ++e) {
                            float t0, t1;
                            f2_unpack(f2_fma(f2_pack(xn[2 * e], xn[2 * e + 1]), sc2, nm2), t0, t1);
                            const float p0 = ex2(t0), p1 = ex2(t1);
                            rs2[e & 3] = f2_add(rs2[e & 3], f2_pack(p0, p1));
                            pk[e] = pack_bf16x2(p0, p1);
                        }
                        tmem_st16(s_addr, pk);
                        tc_wait_st();
                        float rsum;
                        {
                            const uint64_t r01 = f2_add(rs2[0], rs2[1]), r23 = f2_add(rs2[2], rs2[3]);
                            float lo, hi;
                            f2_unpack(f2_add(r01, r23), lo, hi);
                            rsum = lo + hi;
                        }
                        l = l * alpha + rsum;
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_pf(slot));
                        continue;
                    }
                }
                if (kGlob && kShort && j < w.n_band) {
                    // a band tile that none of this warp's rows reaches (the other query tile's
                    // part of the unit's key range): P = 0 for these rows, nothing else changes
                    const int k0 = w.kv_lo + j * BN;
                    if (__all_sync(0xffffffffu, hi_abs < k0 || lo_abs > k0 + BN - 1 || hi_abs < lo_abs)) {
#pragma unroll
                        for (int hlf = 0; hlf < BN / 64; ++hlf) tmem_fill32(s_addr + hlf * 32, 0u);
                        tc_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_pf(slot));
                        continue;
                    }
                }
                float x[BN];
                {
                    uint32_t raw[BN / 32][32];
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_addr + c * 32, raw[c]);
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(raw[c][e]);
                }
                // ---- mask (branch-free; only band-edge and global tiles)
                if (!kGlob || j < w.n_band) {
                    const int k0 = w.kv_lo + j * BN;
                    const bool interior = (a.wl < 0 || k0 >= thi - a.wl) && (a.wr < 0 || k0 + BN - 1 <= tlo + a.wr) &&
                                          (k0 + BN - 1 <= a.Tk - 1);
                    if (interior) {
                        count += BN;
                    } else {
                        // allowed columns of this row form one run [lo, lo + len)
                        const int lo = min(max(lo_abs - k0, 0), BN);
                        const int hi = min(max(hi_abs - k0 + 1, 0), BN);
                        const int len = max(hi - lo, 0);
                        count += len;
                        // short bands: one compare per column where the warp's rows are cut on
                        // one side only
                        if (kShort && __all_sync(0xffffffffu, hi == BN)) {
#pragma unroll
                            for (int c = 0; c < BN; ++c) x[c] = c >= lo ? x[c] : -INFINITY;
                        } else if (kShort && __all_sync(0xffffffffu, lo == 0)) {
#pragma unroll
                            for (int c = 0; c < BN; ++c) x[c] = c < hi ? x[c] : -INFINITY;
                        } else {
#pragma unroll
                            for (int c = 0; c < BN; ++c)
                                x[c] = static_cast<unsigned>(c - lo) < static_cast<unsigned>(len) ? x[c] : -INFINITY;
                        }
                    }
                    if (kGlob && a.sep) {
                        // with separate global projections a global key is scored (with
                        // k_g) in the global-column tiles only: drop it here, 32 columns at
                        // a time (the sorted list is scanned once from its first entry >= k0)
                        int gi = first_at_least(a.global_idx, a.n_global, k0);
#pragma unroll
                        for (int wd = 0; wd < BN / 32; ++wd) {
                            uint32_t bits = 0u;
                            while (gi < a.n_global) {
                                const int c = __ldg(a.global_idx + gi) - k0 - 32 * wd;
                                if (c >= 32) break;
                                bits |= 1u << c;
                                ++gi;
                            }
                            if (bits) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) {
                                    const bool g = (bits >> e) & 1u;
                                    count -= (g && x[32 * wd + e] != -INFINITY) ? 1 : 0;
                                    x[32 * wd + e] = g ? -INFINITY : x[32 * wd + e];
                                }
                            }
                        }
                    }
                } else if (gpos_staged) {
                    // global columns, one tile of n <= BN sorted positions: those left of the
                    // row's band form a prefix [0, nl) and those right of it a suffix [nr, n)
                    // (two branch-free binary searches over the staged list); sinks keep only
                    // the prefix, separate projections keep every column
                    const int n = a.n_global;
                    // (positions: the band's key indices shifted by the sequence's offset)
                    const int lo_pos = lo_abs + w.pos_off, hi_pos = hi_abs + w.pos_off;
                    int nl = 0, nr = 0;
#pragma unroll
                    for (int step = BN; step >= 1; step >>= 1) {
                        if (nl + step <= n && gpos[nl + step - 1] < lo_pos) nl += step;
                        if (nr + step <= n && gpos[nr + step - 1] <= hi_pos) nr += step;
                    }
                    if (a.sink) nr = n;
                    if (a.sep) nl = nr = n;
                    count += nl + (n - nr);
                    if (n <= 32) {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            x[c] = (c < nl) | ((c >= nr) & (c < n)) ? x[c] : -INFINITY;
#pragma unroll
                        for (int c = 32; c < BN; ++c) x[c] = -INFINITY;
                    } else {
#pragma unroll
                        for (int c = 0; c < BN; ++c)
                            x[c] = (c < nl) | ((c >= nr) & (c < n)) ? x[c] : -INFINITY;
                    }
                } else {
                    // global columns of a longer list: each lane loads BN/32 of this tile's
                    // positions, shuffles broadcast them; keep the ones outside the row's band
                    const int g0 = (j - w.n_band) * BN;
                    int gv[BN / 32];
#pragma unroll
                    for (int i = 0; i < BN / 32; ++i) {
                        const int gi = g0 + i * 32 + lane;
                        gv[i] = gi < a.n_global ? __ldg(a.global_idx + gi) : -1;
                    }
                    int cnt4[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int c = 0; c < BN; ++c) {
                        const int gs = __shfl_sync(0xffffffffu, gv[c >> 5], c & 31);
                        // kept: outside the row's band (sinks: left of it); with separate
                        // projections every global key is scored here
                        const bool outside =
                            (gs < lo_abs + w.pos_off) | ((gs > hi_abs + w.pos_off) & !a.sink);
                        const bool valid = (gs >= 0) & (gs < a.gcol_hi);
                        const bool al = valid & (outside | (a.sep != 0));
                        cnt4[c & 3] += al ? 1 : 0;
                        x[c] = al ? x[c] : -INFINITY;
                    }
                    count += (cnt4[0] + cnt4[1]) + (cnt4[2] + cnt4[3]);
                }
                // ---- running max (log2 domain): eight chains of three-input maxima
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = x[i];
#pragma unroll
                for (int c = 8; c + 8 < BN; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], x[c + i], x[c + 8 + i]);
                if constexpr ((BN / 8) % 2 == 0) {  // one column block of 8 left over
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], x[BN - 8 + i]);
                }
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]));
                const float mt = mx * a.scale_log2;
                const bool need = mt > m + kRescaleTau;
                const float mu = need ? mt : m;
                const float alpha = need ? ex2(m - mu) : 1.f;  // m = -inf gives 0
                if (__any_sync(0xffffffffu, need) && j > 0) {
                    // O holds P V of tiles 0 .. j-1 of this unit and must be complete: the
                    // release of tile j-1's V slot (fill 2(j-1)+1) is committed right after
                    // that P V (no commit of its own by the MMA warp)
                    if constexpr (NQT == 1) {
                        if (!warp_wait(bar_empty((2 * (jg - 1) + 1) % NSLOT), vpar(2 * (jg - 1) + 1),
                                       abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(o_addr + c * 32, ov);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(o_addr + c * 32, ov);
                    }
                }
                m = mu;
                const float msub = mu == -INFINITY ? 0.f : mu;
                // ---- P = 2^(x*scale_log2 - m) as bf16 pairs over the first BN/2 S columns;
                // the scale-and-shift and the row sum run on column pairs (fp32x2)
                const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2), nm2 = f2_pack(-msub, -msub);
                uint64_t rs2[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) rs2[i] = f2_pack(0.f, 0.f);
#pragma unroll
                for (int hlf = 0; hlf < BN / 64; ++hlf) {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float t0, t1;
                        f2_unpack(f2_fma(f2_pack(x[hlf * 64 + 2 * e], x[hlf * 64 + 2 * e + 1]), sc2, nm2), t0, t1);
                        const float p0 = ex2(t0), p1 = ex2(t1);
                        rs2[e & 3] = f2_add(rs2[e & 3], f2_pack(p0, p1));
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(s_addr + hlf * 32, pk);
                }
                tc_wait_st();
                float rsum;
                {
                    const uint64_t r01 = f2_add(rs2[0], rs2[1]), r23 = f2_add(rs2[2], rs2[3]);
                    float lo, hi;
                    f2_unpack(f2_add(r01, r23), lo, hi);
                    rsum = lo + hi;
                }
                l = l * alpha + rsum;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_pf(slot));
            }
            if (!ok) break;

            // ---- epilogue: O is final once this tile's last P V completes
            if (!warp_wait(bar_od(wg), k & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // every MMA of this unit has completed: the Q loader may refill this tile
            if (kGlob && !C::QTM && lane == 0) mbar_arrive(bar_qe(wg));
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *orow = a.o + static_cast<int64_t>(w.b) * a.o_st[0] + static_cast<int64_t>(t) * a.o_st[1] +
                                  static_cast<int64_t>(h) * a.o_st[2];
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(o_addr + c * 32, ov);
                tc_wait_ld();
                if (row_ok && a.o_align32) {
                    // 32-byte stores: each lane of a store writes one whole sector of its row
#pragma unroll
                    for (int q8 = 0; q8 < 2; ++q8) {
                        uint32_t wv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            wv[e] = pack_bf16x2(__uint_as_float(ov[q8 * 16 + 2 * e]) * inv_l,
                                                __uint_as_float(ov[q8 * 16 + 2 * e + 1]) * inv_l);
                        st_global_v8(orow + c * 32 + q8 * 16, wv);
                    }
                } else if (row_ok) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t wv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            wv[e] = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 2 * e]) * inv_l,
                                                __uint_as_float(ov[q4 * 8 + 2 * e + 1]) * inv_l);
                        *reinterpret_cast<uint4 *>(orow + c * 32 + q4 * 8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                }
            }
            // O has been read out: the next unit's first P V may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_of(wg));
            if (row_ok) {
                const int64_t li = static_cast<int64_t>(w.b) * a.lse_st[0] + static_cast<int64_t>(h) * a.lse_st[1] +
                                   static_cast<int64_t>(t) * a.lse_st[2];
                a.lse[li] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
                if (a.counts) a.counts[li] = count;
            }
            J += w.n_tiles;
        }
    } else {
        // idle warp of warpgroup 0 gives its registers to the softmax warpgroups
        if constexpr (NQT == 2) regs_dec<C::REG_CTRL>();
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

int band_sm_count() {
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

template <int D>
cudaError_t launch_band_d(const BandArgs &x, cudaStream_t s) {
    using C = BandCfg<D>;
    // launches without global positions take the kernel built without their code paths;
    // bands of at most kShortTiles key tiles per unit the one built for short bands
    const bool glob = x.n_global > 0;
    const int G = x.H_q / x.H_kv;
    const int TQ = BM / G;
    const bool shrt = x.wl >= 0 && x.wr >= 0 &&
                      (static_cast<long long>(C::NQT) * TQ - 1 + x.wl + x.wr) / C::BN + 2 <= kShortTiles;
    auto kernel = glob ? (shrt ? band_fwd_kernel<D, true, true> : band_fwd_kernel<D, true, false>)
                       : (shrt ? band_fwd_kernel<D, false, true> : band_fwd_kernel<D, false, false>);
    // the dynamic shared-memory limit is a per-device function attribute: set once per device
    static std::atomic<bool> configured[64][2][2];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) dev = -1;
    if (dev < 0 || !configured[dev][glob][shrt].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0) configured[dev][glob][shrt].store(true, std::memory_order_release);
    }
    CUtensorMap mq, mk, mv;
    const int Tk = x.Tk > 0 ? x.Tk : x.T;
    if (!make_map(&mq, x.q, D, x.H_q, x.T, x.B, x.q_st, G, TQ) ||
        !make_map(&mk, x.k, D, x.H_kv, Tk, x.B, x.k_st, 1, C::BN) ||
        !make_map(&mv, x.v, D, x.H_kv, Tk, x.B, x.v_st, 1, C::BN))
        return cudaErrorInvalidValue;
    BandKernelArgs a{};
    a.B = x.B;
    a.T = x.T;
    a.Tk = Tk;
    a.q_off = x.q_off;
    a.kmin = x.kmin;
    a.p0 = x.p0;
    a.gcol_list_rows = x.gcol_list_rows ? 1 : 0;
    a.gcol_hi = x.gcol_list_rows ? INT_MAX : Tk;
    a.H_q = x.H_q;
    a.H_kv = x.H_kv;
    a.G = G;
    a.TQ = TQ;
    const int n_qtiles = (x.T + TQ - 1) / TQ;
    a.n_units_t = (n_qtiles + C::NQT - 1) / C::NQT;
    a.wl = x.wl;
    a.wr = x.wr;
    a.scale_log2 = x.scale_log2;
    a.global_idx = x.global_idx;
    a.n_global = x.n_global;
    a.sink = x.gmode == SWA_GLOBAL_SINK ? 1 : 0;
    a.sep = x.sep ? 1 : 0;
    a.gcol_narrow = glob && x.n_global <= kNarrow ? 1 : 0;
    const FaultPlan fp = fault_plan();
    a.fault_stop_fill = fp.band_stop_fill;
    // global-column rows come from kg / vg with separate projections or a row list
    const bool gsrc = x.sep || x.gcol_list_rows;
    a.k = static_cast<const __nv_bfloat16 *>(gsrc ? x.kg : x.k);
    a.v = static_cast<const __nv_bfloat16 *>(gsrc ? x.vg : x.v);
    for (int i = 0; i < 3; ++i) {
        a.k_st[i] = gsrc ? x.kg_st[i] : x.k_st[i];
        a.v_st[i] = gsrc ? x.vg_st[i] : x.v_st[i];
        a.o_st[i] = x.o_st[i];
        a.lse_st[i] = x.lse_st[i];
    }
    a.o = static_cast<__nv_bfloat16 *>(x.o);
    a.o_align32 = (reinterpret_cast<uintptr_t>(x.o) % 32 == 0) && (x.o_st[0] % 16 == 0) && (x.o_st[1] % 16 == 0) &&
                  (x.o_st[2] % 16 == 0);
    a.lse = x.lse;
    a.counts = x.counts;
    const long long units = static_cast<long long>(x.B) * x.H_kv * a.n_units_t;
    if (units <= 0 || units > 0x7fffffffLL) return cudaErrorInvalidValue;
    a.n_units = static_cast<int>(units);
    const int grid = static_cast<int>(units < band_sm_count() ? units : band_sm_count());
    kernel<<<grid, C::THREADS, C::SMEM, s>>>(mq, mk, mv, a);
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
