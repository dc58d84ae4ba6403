// swa_split.cu -- split-K attention of a few query rows against many key/value
// slots, and the log-sum-exp merge of the splits.
//
// Used for ring-buffer decode (one query token per sequence against its W cache
// slots; a slot is valid when its stored position lies in the query's window,
// Gemma 3 note, ai-engineer-exhaustive.pages.dev "How it works") and for the
// global rows of the prefill path (each global position attends to all T keys,
// prathamp.com "Sliding Window Attention: From Local Windows to Global Context",
// section 4.3).  The work is HBM-bound: every valid key/value byte is read once.
//
// Persistent kernel, two CTAs per SM for head dim <= 128 (one for 256), five warps:
//   warp 0     producer.  Walks this CTA's work items (batch, kv head, query block,
//              split of at most 1024 slots) in a static round-robin order.  For each item it
//              reads the slot positions, builds one 64-bit validity mask per
//              64-slot chunk, writes the split's valid count, and streams the K and
//              V of every chunk that has a valid slot into a ring of NST stages
//              with TMA (128B swizzle); chunks without a valid slot are never read.
//   warps 1-4  consumers.  Each scores 16 slots of every chunk with mma.sync (the
//              query block's <= 16 rows -- a GQA group of heads -- are the M
//              dimension), keeps a running (max, sum, weighted values) per row, and
//              at the end of an item the four warps combine through shared memory
//              and write the split's partial.  Value rows of invalid slots are
//              zeroed before P V, so whatever an unwritten slot holds (even NaN)
//              never reaches the result.
// The merge kernel combines the splits of a row (log-sum-exp rescaling).  It is launched
// as a programmatic dependent of the split pass, and the global-row split pass as one
// of the band kernel before it (it reads only q/k/v); griddepcontrol.wait orders each
// consumer after the grid whose results it reads.
// Every wait is bounded; on expiry the CTA records an error word, drains its
// copies and returns.
#include <atomic>
#include <cfloat>
#include <climits>
#include <cmath>

#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "swa_internal.h"

namespace swa {
namespace {

__device__ unsigned int g_split_err = 0;

constexpr int CH = kSplitChunk;                 // slots per chunk (64)
constexpr int MAX_CHUNKS = kSlotsPerSplit / CH;  // chunks per split (16)
constexpr int kThreads = 160;

struct StageHdr {
    int item, chunk, last, pad;
    unsigned long long mask;  // bit i: slot chunk*64 + i of the split is valid
    unsigned long long pad2;
};

// Several CTAs share an SM where shared memory and registers allow -- three at head dim
// 64 (three 16 KB stages each), two at 128 -- so one CTA's end-of-item combine and its
// consumers' latency-bound chains overlap the others' streaming.  (Three at d = 64 took the
// Longformer global rows' pass, two query rows per head, from 46.6% of the DRAM peak; at
// d = 128 a third CTA would leave one stage each.)
template <int D>
struct StreamCfg {
    static constexpr int STAGE = 2 * CH * D * 2;        // K + V of one chunk
    static constexpr int CROW = D + 8;  // padded row: float2 stores of 4 rows per half-warp hit distinct banks
    static constexpr int CBUF = 4 * kSplitRows * CROW * 4;  // combine buffer [4 warps][16 rows][CROW] fp32
    static constexpr int CTAS_PER_SM = D <= 64 ? 3 : D <= 128 ? 2 : 1;
    static constexpr int NST_RAW = (232448 / CTAS_PER_SM - 2048 - CBUF) / STAGE;
    static constexpr int NST = NST_RAW > 8 ? 8 : NST_RAW;
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_CBUF = NST * STAGE;
    static constexpr int OFF_HDR = OFF_CBUF + CBUF;
    static constexpr int OFF_RED = OFF_HDR + NST * static_cast<int>(sizeof(StageHdr));  // red_m, red_l [4][16]
    static constexpr int OFF_BAR = OFF_RED + 2 * 4 * kSplitRows * 4;
    // full[NST], empty[NST], cmb_full, cmb_done
    static constexpr int NBAR = 2 * NST + 2;
    static constexpr int SMEM = OFF_BAR + NBAR * 8 + 1024;
    static_assert(NST >= 2, "ring too shallow");
    static_assert(SMEM * CTAS_PER_SM <= 232448, "shared memory budget");
};

// Offset of 16-byte piece `pc` of row `row` in a 128B-swizzled tile of `rows` rows
// written by TMA boxes of 64 elements (one 128-byte row per box row).
__device__ __forceinline__ uint32_t sw128(int rows, int row, int pc) {
    return static_cast<uint32_t>((pc >> 3) * (rows * 128) + row * 128 + (((pc & 7) ^ (row & 7)) << 4));
}

struct StreamKernelArgs {
    SplitArgs s;
    int n_items;
    int nqb;
    // planted fault of the failure-detection tests: the producer of every CTA emits no
    // stage numbered at or past this (INT_MAX: off), so the consumers' waits run out
    int fault_stop_stage;
};

// Registers: two 5-warp CTAs put three warps on two of the SM's sub-partitions,
// whose 16K-register files then allow at most 168 registers a thread; three CTAs put
// four warps on three of them (at most 128).
template <int D>
__global__ void __maxnreg__(StreamCfg<D>::CTAS_PER_SM == 3 ? 128 : StreamCfg<D>::CTAS_PER_SM == 2 ? 168 : 255)
    stream_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const StreamKernelArgs ka) {
    using C = StreamCfg<D>;
    constexpr int NST = C::NST;
    const SplitArgs &a = ka.s;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t *sgen = smem_raw + (sbase - sraw);
    StageHdr *hdr = reinterpret_cast<StageHdr *>(sgen + C::OFF_HDR);
    float *cbuf = reinterpret_cast<float *>(sgen + C::OFF_CBUF);
    float *red_m = reinterpret_cast<float *>(sgen + C::OFF_RED);
    float *red_l = red_m + 4 * kSplitRows;
    const uint32_t bars = sbase + C::OFF_BAR;
    auto bar_full = [&](int s) { return bars + 8u * s; };
    auto bar_empty = [&](int s) { return bars + 8u * (NST + s); };
    const uint32_t bar_cf = bars + 8u * (2 * NST), bar_cd = bars + 8u * (2 * NST + 1);
    const int group = a.H_q / a.H_kv;
    const int Y = a.H_kv * ka.nqb;

    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 4);
        }
        mbar_init(bar_cf, 4);
        mbar_init(bar_cd, 4);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    __syncthreads();
    volatile int *abort = &abort_flag;
    // the merge grid may be scheduled from here on: its blocks wait (griddepcontrol.wait)
    // for this grid to complete before they read the partials
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ============================ producer ============================
        int seq = 0;          // stages emitted so far
        bool ok = true;
        // Slot positions of an item, 16 per lane (slot i*32 + lane of the split); the
        // loads for item i + grid are issued before item i's chunks are streamed.
        auto load_pos = [&](int item, int (&pv)[2 * MAX_CHUNKS]) {
            if (item >= ka.n_items) return;
            const int split = item % a.n_splits;
            const int b = item / (a.n_splits * Y);
            const int slot0 = split * a.slots_per_split;
            const int nslots = min(a.n_slots, slot0 + a.slots_per_split) - slot0;
            const int32_t *row = a.slot_pos ? a.slot_pos + static_cast<int64_t>(b) * a.n_slots + slot0 : nullptr;
#pragma unroll
            for (int i = 0; i < 2 * MAX_CHUNKS; ++i) {
                const int si = i * 32 + lane;
                pv[i] = si >= nslots ? INT_MIN : (row ? __ldg(row + si) : 0);
            }
        };
        int pos_cur[2 * MAX_CHUNKS], pos_next[2 * MAX_CHUNKS];
        load_pos(blockIdx.x, pos_cur);
        for (int item = blockIdx.x; item < ka.n_items && ok; item += gridDim.x) {
            const int split = item % a.n_splits;
            const int y = (item / a.n_splits) % Y;
            const int b = item / (a.n_splits * Y);
            const int kvh = y / ka.nqb, qb = y % ka.nqb;
            const int slot0 = split * a.slots_per_split;
            // debug build: the item is a (sequence, kv head, query block, split) that exists
            (void)SWA_IN_BOUNDS(b < a.B && kvh < a.H_kv && qb < ka.nqb && slot0 < a.n_slots, &g_split_err);
            const int64_t t = a.q_pos ? static_cast<int64_t>(a.q_pos[b]) : 0;
            // decode with append: the current token goes to slot(t) before it is read;
            // si_new is that slot's index in this split (-1: not in this split)
            int si_new = -1, s_new = 0;
            if (a.k_new && t >= 0) {
                s_new = t < a.n_sink ? static_cast<int>(t)
                                     : a.n_sink + static_cast<int>((t - a.n_sink) % (a.n_slots - a.n_sink));
                const int rel = s_new - slot0;
                if (rel >= 0 && rel < a.slots_per_split && s_new < a.n_slots) si_new = rel;
            }
            load_pos(item + gridDim.x, pos_next);
            // validity of the item's slots, 64 per chunk (two ballots)
            bool v[2 * MAX_CHUNKS];
#pragma unroll
            for (int i = 0; i < 2 * MAX_CHUNKS; ++i) {
                const int64_t p = pos_cur[i];
                v[i] = pos_cur[i] != INT_MIN &&
                       (!a.slot_pos || (p >= 0 && p <= t && (p > t - a.W || p < a.n_sink)));
                v[i] = v[i] || (i * 32 + lane == si_new);  // the appended token, position t
            }
            unsigned long long mask[MAX_CHUNKS];
            int count = 0;
#pragma unroll
            for (int c = 0; c < MAX_CHUNKS; ++c) {
                const unsigned lo = __ballot_sync(0xffffffffu, v[2 * c]);
                const unsigned hi = __ballot_sync(0xffffffffu, v[2 * c + 1]);
                mask[c] = static_cast<unsigned long long>(lo) | (static_cast<unsigned long long>(hi) << 32);
                count += __popcll(mask[c]);
            }
#pragma unroll
            for (int i = 0; i < 2 * MAX_CHUNKS; ++i) pos_cur[i] = pos_next[i];
            if (qb == 0 && lane == 0 &&
                SWA_IN_BOUNDS(b < a.B && kvh < a.H_kv && split < a.n_splits, &g_split_err))
                a.ws_cnt[(static_cast<int64_t>(b) * a.H_kv + kvh) * a.n_splits + split] = count;
            if (si_new >= 0 && kvh == 0 && qb == 0 && lane == 0 &&
                SWA_IN_BOUNDS(s_new >= 0 && s_new < a.n_slots && b < a.B, &g_split_err))
                a.slot_pos_w[static_cast<int64_t>(b) * a.n_slots + s_new] = static_cast<int32_t>(t);
            int last_c = -1;
#pragma unroll
            for (int c = 0; c < MAX_CHUNKS; ++c)
                if (mask[c]) last_c = c;
            // emit the chunks with a valid slot (one empty stage if there is none)
#pragma unroll 1
            for (int c = 0; c < MAX_CHUNKS && ok; ++c) {
                const bool emit = mask[c] != 0 || (last_c < 0 && c == 0);
                if (!emit) continue;
                if (seq >= ka.fault_stop_stage) {  // planted fault: this stage is never emitted
                    ok = false;
                    break;
                }
                const int st = seq % NST;
                if (seq >= NST) {
                    ok = __all_sync(0xffffffffu, mbar_wait<true>(bar_empty(st), ((seq / NST) - 1) & 1, abort, &g_split_err));
                    if (!ok) break;
                }
                if (si_new >= 0 && c == si_new / CH) {
                    // write the current token's key and value rows into its slot, then make
                    // those generic-proxy stores visible to the TMA load of this chunk
                    const uint4 *ks = reinterpret_cast<const uint4 *>(a.k_new + (static_cast<int64_t>(b) * a.H_kv + kvh) * D);
                    const uint4 *vs = reinterpret_cast<const uint4 *>(a.v_new + (static_cast<int64_t>(b) * a.H_kv + kvh) * D);
                    uint4 *kd = reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(a.k)) +
                                                          b * a.k_sb + static_cast<int64_t>(s_new) * a.k_ss + kvh * a.k_sh);
                    uint4 *vd = reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(a.v)) +
                                                          b * a.v_sb + static_cast<int64_t>(s_new) * a.v_ss + kvh * a.v_sh);
                    if (SWA_IN_BOUNDS(s_new >= 0 && s_new < a.n_slots && b < a.B && kvh < a.H_kv, &g_split_err))
                        for (int pc = lane; pc < 2 * (D / 8); pc += 32) {
                            if (pc < D / 8) kd[pc] = __ldg(ks + pc);
                            else vd[pc - D / 8] = __ldg(vs + pc - D / 8);
                        }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __syncwarp();
                }
                if (lane == 0) {
                    StageHdr &h = hdr[st];
                    h.item = item;
                    h.chunk = c;
                    h.last = (c == last_c || last_c < 0) ? 1 : 0;
                    h.mask = mask[c];
                    if (mask[c]) {
                        const uint32_t kd = sbase + C::OFF_RING + st * C::STAGE;
                        const uint32_t vd = kd + C::STAGE / 2;
                        mbar_arrive_expect_tx(bar_full(st), C::STAGE);
                        const int srow = slot0 + c * CH;
                        (void)SWA_IN_BOUNDS(srow < a.n_slots, &g_split_err);  // debug build: chunk inside the slots
#pragma unroll
                        for (int pc = 0; pc < D / 64; ++pc) {
                            tma_load_4d(kd + pc * (CH * 128), &tm_k, bar_full(st), pc * 64, srow, kvh, b);
                            tma_load_4d(vd + pc * (CH * 128), &tm_v, bar_full(st), pc * 64, srow, kvh, b);
                        }
                    } else {
                        mbar_arrive(bar_full(st));
                    }
                }
                __syncwarp();
                ++seq;
            }
        }
        if (!ok && lane == 0) {
            // drain the copies still in flight (at most the last NST stages)
            for (int s = max(0, seq - NST); s < seq; ++s) mbar_drain(bar_full(s % NST), (s / NST) & 1, &g_split_err);
        }
    } else {
        // ============================ consumers ============================
        const int w = warp - 1;  // slots [16w, 16w + 16) of every chunk
        const int rows = a.q_per_cta * group;
        const int r0 = lane >> 2, r1 = r0 + 8;
        const int kq = 2 * (lane & 3);
        uint32_t qa[D / 16][4];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        float acc[D / 8][4];
        int cur = -1, n_done = 0;
        bool ok = true;
#pragma unroll 1
        for (int seq = 0; ok; ++seq) {
            const int st = seq % NST;
            if (!__all_sync(0xffffffffu, mbar_wait<true>(bar_full(st), (seq / NST) & 1, abort, &g_split_err))) {
                ok = false;
                break;
            }
            const int item = hdr[st].item, chunk = hdr[st].chunk, last = hdr[st].last;
            const unsigned long long mask = hdr[st].mask;
            const int split = item % a.n_splits;
            const int y = (item / a.n_splits) % Y;
            const int b = item / (a.n_splits * Y);
            const int kvh = y / ka.nqb, qb = y % ka.nqb;
            if (item != cur) {
                // new item: query fragments of its rows (r0, r1 of the 16-row M tile), fresh state
                cur = item;
                const int rr[2] = {r0, r1};
                const __nv_bfloat16 *qp[2];
                bool rv[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = rr[i];
                    const int qs = qb * a.q_per_cta + r / group;
                    rv[i] = r < rows && qs < a.NQ;
                    int64_t tok = (rv[i] && a.q_tok) ? a.q_tok[qs] : 0;
                    if (tok < 0 || tok >= a.tok_limit) {
                        rv[i] = false;
                        tok = 0;
                    }
                    const int h = kvh * group + r % group;
                    if (rv[i] && !SWA_IN_BOUNDS(h < a.H_q && b < a.B, &g_split_err)) rv[i] = false;
                    qp[i] = static_cast<const __nv_bfloat16 *>(a.q) + static_cast<int64_t>(b) * a.q_sb + tok * a.q_st +
                            static_cast<int64_t>(h) * a.q_sh;
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    qa[kk][0] = rv[0] ? __ldg(reinterpret_cast<const unsigned *>(qp[0] + kk * 16 + kq)) : 0u;
                    qa[kk][1] = rv[1] ? __ldg(reinterpret_cast<const unsigned *>(qp[1] + kk * 16 + kq)) : 0u;
                    qa[kk][2] = rv[0] ? __ldg(reinterpret_cast<const unsigned *>(qp[0] + kk * 16 + 8 + kq)) : 0u;
                    qa[kk][3] = rv[1] ? __ldg(reinterpret_cast<const unsigned *>(qp[1] + kk * 16 + 8 + kq)) : 0u;
                }
                m0 = m1 = -INFINITY;
                l0 = l1 = 0.f;
#pragma unroll
                for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
            }
            const unsigned wmask = static_cast<unsigned>(mask >> (16 * w)) & 0xffffu;  // this warp's 16 slots
            if (wmask) {
                const uint32_t ks = sbase + C::OFF_RING + st * C::STAGE;
                const uint32_t vs = ks + C::STAGE / 2;
                if (wmask != 0xffffu) {
                    // zero the value rows of this warp's invalid slots
                    uint8_t *vg = sgen + C::OFF_RING + st * C::STAGE + C::STAGE / 2;
                    for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
                        const int rr = idx / (D / 8), pc = idx % (D / 8);
                        if (!((wmask >> rr) & 1u))
                            *reinterpret_cast<uint4 *>(vg + sw128(CH, 16 * w + rr, pc)) = make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }
                // S = Q K^T over this warp's 16 slots (two n-tiles of 8)
                float sc[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                    const int row = 16 * w + 8 * nt + (lane & 7);
#pragma unroll
                    for (int k2 = 0; k2 < D / 32; ++k2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(ks + sw128(CH, row, k2 * 4 + (lane >> 3)), b0, b1, b2, b3);
                        mma_bf16_16816(sc[nt], qa[2 * k2], b0, b1);
                        mma_bf16_16816(sc[nt], qa[2 * k2 + 1], b2, b3);
                    }
                }
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int bit = 8 * nt + kq + (e & 1);
                        sc[nt][e] = ((wmask >> bit) & 1u) ? sc[nt][e] * a.scale_log2 : -INFINITY;
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
                const int vrow = 16 * w + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
                for (int d2 = 0; d2 < D / 16; ++d2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vs + sw128(CH, vrow, 2 * d2 + (lane >> 4)), b0, b1, b2, b3);
                    mma_bf16_16816(acc[2 * d2], pa, b0, b1);
                    mma_bf16_16816(acc[2 * d2 + 1], pa, b2, b3);
                }
                // order this warp's generic writes (zeroed rows) before the next TMA into the stage
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty(st));
            (void)chunk;

            if (last) {
                // ---- combine the four warps and write this split's partial
                float ls0 = l0, ls1 = l1;
#pragma unroll
                for (int o = 1; o <= 2; o <<= 1) {
                    ls0 += __shfl_xor_sync(0xffffffffu, ls0, o);
                    ls1 += __shfl_xor_sync(0xffffffffu, ls1, o);
                }
                if (n_done > 0 && !__all_sync(0xffffffffu, mbar_wait<true>(bar_cd, (n_done - 1) & 1, abort, &g_split_err))) {
                    ok = false;
                    break;
                }
                if ((lane & 3) == 0) {
                    red_m[w * kSplitRows + r0] = m0;
                    red_m[w * kSplitRows + r1] = m1;
                    red_l[w * kSplitRows + r0] = ls0;
                    red_l[w * kSplitRows + r1] = ls1;
                }
                if (r0 < rows) {
#pragma unroll
                    for (int n = 0; n < D / 8; ++n)
                        *reinterpret_cast<float2 *>(cbuf + (w * kSplitRows + r0) * C::CROW + 8 * n + kq) =
                            make_float2(acc[n][0], acc[n][1]);
                }
                if (r1 < rows) {
#pragma unroll
                    for (int n = 0; n < D / 8; ++n)
                        *reinterpret_cast<float2 *>(cbuf + (w * kSplitRows + r1) * C::CROW + 8 * n + kq) =
                            make_float2(acc[n][2], acc[n][3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_cf);
                if (!__all_sync(0xffffffffu, mbar_wait<true>(bar_cf, n_done & 1, abort, &g_split_err))) {
                    ok = false;
                    break;
                }
                // eight threads per row: the row's split weights once, then float4 columns
                // interleaved so each 8-thread phase reads 128 contiguous bytes
                {
                    const int t = w * 32 + lane;
                    const int r = t >> 3, part = t & 7;
                    const int qs = qb * a.q_per_cta + r / group;
                    bool live = r < rows && qs < a.NQ;
                    if (live && a.q_tok && (a.q_tok[qs] < 0 || a.q_tok[qs] >= a.tok_limit)) live = false;
                    // debug build: the partial's row (b, query, head, split) exists
                    if (live && !SWA_IN_BOUNDS(b < a.B && kvh * group + r % group < a.H_q && split < a.n_splits,
                                               &g_split_err))
                        live = false;
                    if (live) {
                        const int h = kvh * group + r % group;
                        float mw = -INFINITY;
#pragma unroll
                        for (int ww = 0; ww < 4; ++ww) mw = fmaxf(mw, red_m[ww * kSplitRows + r]);
                        float f[4], L = 0.f;
#pragma unroll
                        for (int ww = 0; ww < 4; ++ww) {
                            f[ww] = mw == -INFINITY ? 0.f : ex2(red_m[ww * kSplitRows + r] - mw);
                            L += red_l[ww * kSplitRows + r] * f[ww];
                        }
                        const int64_t row = ((static_cast<int64_t>(b) * a.NQ + qs) * a.H_q + h) * a.n_splits + split;
#pragma unroll
                        for (int k4 = 0; k4 < D / 32; ++k4) {
                            const int col = k4 * 32 + part * 4;
                            float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                            for (int ww = 0; ww < 4; ++ww) {
                                const float4 c4 =
                                    *reinterpret_cast<const float4 *>(cbuf + (ww * kSplitRows + r) * C::CROW + col);
                                acc4.x += c4.x * f[ww];
                                acc4.y += c4.y * f[ww];
                                acc4.z += c4.z * f[ww];
                                acc4.w += c4.w * f[ww];
                            }
                            *reinterpret_cast<float4 *>(a.ws_acc + row * D + col) = acc4;
                        }
                        if (part == 0) {
                            a.ws_ml[row * 2 + 0] = mw;
                            a.ws_ml[row * 2 + 1] = L;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_cd);
                ++n_done;
                cur = -1;
                if (item + static_cast<int>(gridDim.x) >= ka.n_items) break;  // this CTA's last item
            }
        }
    }
    // After the band kernel of the same call (global rows): complete only once that grid has,
    // so the merge, which waits for this grid, overwrites the band kernel's rows after it.
    // (Without a programmatic launch this returns at once.)
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Sum (kMax: max) of v over the block's 128 threads; every thread gets the result.
template <bool kMax>
__device__ __forceinline__ float block_reduce128(float v, float *red) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = kMax ? fmaxf(v, w) : v + w;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    v = kMax ? fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])) : (red[0] + red[1]) + (red[2] + red[3]);
    __syncthreads();  // red is reused by the next reduction
    return v;
}

// Integer sum over the block's 128 threads (exact), every thread gets it.
__device__ __forceinline__ int block_sum128_int(int v, int *red) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    v = (red[0] + red[1]) + (red[2] + red[3]);
    __syncthreads();
    return v;
}

// One block per output row (b, query, head): the log-sum-exp merge of the row's splits,
// so that the row's work is a few dependent load latencies, not one per split.
//   At most kMergeFewSplits splits (decode): every thread loads all the (max, sum) pairs at
//   once and derives the weights 2^(m_s - M) itself, then loads its columns' partials of
//   all splits at once -- no block-wide reduction.
//   More splits (the global rows of long sequences): the block's threads read the pairs in
//   parallel and reduce them across the block; the weights go to shared memory and each
//   thread combines its columns over the splits four loads at a time.
constexpr int kMergeFewSplits = 8;
constexpr int kMergeCachedSplits = 512;  // split weights kept in shared memory (more: recomputed)

__global__ void __launch_bounds__(128) merge_kernel(const MergeArgs a) {
    // launched as a programmatic dependent of the pass that wrote the partials: wait for
    // that grid's completion (and its writes) before reading them
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float red[4];
    __shared__ int ired[4];
    __shared__ float wsplit[kMergeCachedSplits];
    const int qs = blockIdx.x / a.H_q, h = blockIdx.x % a.H_q, b = blockIdx.y;
    const int group = a.H_q / a.H_kv, kvh = h / group;
    const int tid = threadIdx.x, ns = a.n_splits;
    // debug build: the block's row (b, query, head) exists (the grid is NQ * H_q x B)
    if (!SWA_IN_BOUNDS(qs < a.NQ && h < a.H_q && b < a.B, &g_split_err)) return;
    const int64_t base = ((static_cast<int64_t>(b) * a.NQ + qs) * a.H_q + h) * ns;
    const float2 *ml = reinterpret_cast<const float2 *>(a.ws_ml) + base;  // (max in log2 units, sum)
    if (ns <= kMergeFewSplits) {
        float2 v[kMergeFewSplits];
#pragma unroll
        for (int i = 0; i < kMergeFewSplits; ++i) v[i] = i < ns ? ml[i] : make_float2(-INFINITY, 0.f);
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < kMergeFewSplits; ++i) M = fmaxf(M, v[i].x);
        float wgt[kMergeFewSplits], L = 0.f;
#pragma unroll
        for (int i = 0; i < kMergeFewSplits; ++i) {
            wgt[i] = M == -INFINITY || i >= ns ? 0.f : exp2f(v[i].x - M);
            L += v[i].y * wgt[i];
        }
        const int64_t tok = a.q_tok ? a.q_tok[qs] : 0;
        if (tok < 0 || tok >= a.tok_limit) return;
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o) + static_cast<int64_t>(b) * a.o_sb + tok * a.o_st +
                           static_cast<int64_t>(h) * a.o_sh;
        const float inv_l = L > 0.f ? 1.f / L : 0.f;
        for (int d = tid; d < a.D; d += blockDim.x) {
            const float *col = a.ws_acc + base * a.D + d;
            float x[kMergeFewSplits];
#pragma unroll
            for (int i = 0; i < kMergeFewSplits; ++i) x[i] = i < ns ? col[static_cast<int64_t>(i) * a.D] : 0.f;
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kMergeFewSplits; ++i) acc += x[i] * wgt[i];
            o[d] = __float2bfloat16_rn(acc * inv_l);
        }
        if (tid == 0) {
            const float lse = M == -INFINITY ? -INFINITY : (M + log2f(L)) * 0.6931471805599453f;
            a.lse[static_cast<int64_t>(b) * a.lse_sb + static_cast<int64_t>(h) * a.lse_sh + tok * a.lse_st] = lse;
            if (a.counts) {
                const int32_t *cn = a.ws_cnt + (static_cast<int64_t>(b) * a.H_kv + kvh) * ns;
                int c = 0;
#pragma unroll
                for (int i = 0; i < kMergeFewSplits; ++i) c += i < ns ? cn[i] : 0;
                a.counts[static_cast<int64_t>(b) * a.cnt_sb + static_cast<int64_t>(h) * a.cnt_sh + tok * a.cnt_st] =
                    c;
            }
        }
        return;
    }
    float M = -INFINITY;
    for (int s = tid; s < ns; s += blockDim.x) M = fmaxf(M, ml[s].x);
    M = block_reduce128<true>(M, red);
    float L = 0.f;
    int c = 0;
    for (int s = tid; s < ns; s += blockDim.x) {
        const float2 v = ml[s];
        const float wgt = M == -INFINITY ? 0.f : exp2f(v.x - M);
        if (s < kMergeCachedSplits) wsplit[s] = wgt;
        L += v.y * wgt;
        if (a.counts) c += a.ws_cnt[(static_cast<int64_t>(b) * a.H_kv + kvh) * ns + s];
    }
    L = block_reduce128<false>(L, red);  // (its barriers also publish wsplit)
    if (a.counts) c = block_sum128_int(c, ired);
    const int64_t tok = a.q_tok ? a.q_tok[qs] : 0;
    if (tok < 0 || tok >= a.tok_limit) return;
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o) + static_cast<int64_t>(b) * a.o_sb + tok * a.o_st +
                       static_cast<int64_t>(h) * a.o_sh;
    const float inv_l = L > 0.f ? 1.f / L : 0.f;
    auto weight = [&](int s) { return s < kMergeCachedSplits ? wsplit[s] : exp2f(ml[s].x - M); };
    for (int d = tid; d < a.D; d += blockDim.x) {
        const float *col = a.ws_acc + base * a.D + d;
        float acc = 0.f;
        if (M != -INFINITY) {
            int s = 0;
            for (; s + 4 <= ns; s += 4) {
                float v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = col[static_cast<int64_t>(s + i) * a.D];
#pragma unroll
                for (int i = 0; i < 4; ++i) acc += v[i] * weight(s + i);
            }
            for (; s < ns; ++s) acc += col[static_cast<int64_t>(s) * a.D] * weight(s);
        }
        o[d] = __float2bfloat16_rn(acc * inv_l);
    }
    if (tid == 0) {
        const float lse = M == -INFINITY ? -INFINITY : (M + log2f(L)) * 0.6931471805599453f;
        a.lse[static_cast<int64_t>(b) * a.lse_sb + static_cast<int64_t>(h) * a.lse_sh + tok * a.lse_st] = lse;
        if (a.counts) a.counts[static_cast<int64_t>(b) * a.cnt_sb + static_cast<int64_t>(h) * a.cnt_sh + tok * a.cnt_st] = c;
    }
}

// ---------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 4-D bf16 map over (d, slot, kv head, batch) -- any element strides -- with a
// (64, 64, 1, 1) box and 128-B swizzle.
bool slot_map(CUtensorMap *m, const void *base, int D, int n_slots, int H, int B, int64_t s_slot, int64_t s_head,
              int64_t s_batch) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(n_slots), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(s_slot) * 2, static_cast<cuuint64_t>(s_head) * 2,
                             static_cast<cuuint64_t>(s_batch) * 2};
    cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(CH), 1u, 1u};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

template <int D>
cudaError_t launch_stream_d(const SplitArgs &a, cudaStream_t s) {
    using C = StreamCfg<D>;
    // the dynamic shared-memory limit is a per-device function attribute: set once per device
    static std::atomic<bool> configured[64];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) dev = -1;
    if (dev < 0 || !configured[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(stream_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0) configured[dev].store(true, std::memory_order_release);
    }
    if (a.slots_per_split <= 0 || a.slots_per_split > kSlotsPerSplit || a.slots_per_split % CH != 0 ||
        static_cast<int64_t>(a.slots_per_split) * a.n_splits < a.n_slots)
        return cudaErrorInvalidValue;
    CUtensorMap mk, mv;
    if (!slot_map(&mk, a.k, D, a.n_slots, a.H_kv, a.B, a.k_ss, a.k_sh, a.k_sb) ||
        !slot_map(&mv, a.v, D, a.n_slots, a.H_kv, a.B, a.v_ss, a.v_sh, a.v_sb))
        return cudaErrorInvalidValue;
    StreamKernelArgs ka{};
    ka.s = a;
    ka.nqb = (a.NQ + a.q_per_cta - 1) / a.q_per_cta;
    const FaultPlan fp = fault_plan();
    ka.fault_stop_stage = fp.split_stop_stage;
    const long long items = static_cast<long long>(a.B) * a.H_kv * ka.nqb * a.n_splits;
    if (items <= 0 || items > 0x7fffffffLL) return cudaErrorInvalidValue;
    ka.n_items = static_cast<int>(items);
    const int slots = sm_count() * C::CTAS_PER_SM;
    const int grid = static_cast<int>(items < slots ? items : slots);
    if (!a.after_band) {
        stream_attn_kernel<D><<<grid, kThreads, C::SMEM, s>>>(mk, mv, ka);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_attn_kernel<D>, mk, mv, ka);
}

}  // namespace

int split_grid(int D) {
    return sm_count() * (D <= 64    ? StreamCfg<64>::CTAS_PER_SM
                         : D <= 128 ? StreamCfg<128>::CTAS_PER_SM
                                    : StreamCfg<256>::CTAS_PER_SM);
}

cudaError_t launch_split(const SplitArgs &a, cudaStream_t s) {
    switch (a.D) {
        case 64: return launch_stream_d<64>(a, s);
        case 128: return launch_stream_d<128>(a, s);
        case 256: return launch_stream_d<256>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s) {
    // programmatic dependent launch: the merge grid is launched while the split pass
    // before it on the stream drains, instead of after it
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.NQ * a.H_q, a.B);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel, a);
}

unsigned int split_read_clear_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_split_err, sizeof v) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_split_err, &z, sizeof z);
    return v;
}

}  // namespace swa
