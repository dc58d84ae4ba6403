// swa_internal.h -- host-side interface between the C ABI (swa_abi.cu) and the
// kernel translation units.  Not installed; the public surface is include/swa.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "swa.h"

namespace swa {

// One query row set attended against a list of key/value "slots".
//   decode:      slots are the cache slots, a slot is valid iff its stored position p
//                satisfies 0 <= p <= t and (t - W < p or p < n_sink) (t = q_pos[b]);
//   global rows: slots are the T key positions, all valid; the queries are the
//                rows of the global positions (q_tok[qs]).
// Rows packed into one CTA: q_per_cta query tokens x the H_q/H_kv heads of a group.
struct SplitArgs {
    const void *q;
    int64_t q_sb, q_st, q_sh;  // query element address: b*q_sb + tok*q_st + h*q_sh
    const void *k;
    const void *v;
    int64_t k_sb, k_ss, k_sh;     // key element address: b*k_sb + slot*k_ss + kvh*k_sh
    int64_t v_sb, v_ss, v_sh;     // value element address, likewise
    const int32_t *slot_pos;      // [B, n_slots] (decode) or nullptr (every slot < n_slots valid)
    const int32_t *q_pos;         // [B] (decode) or nullptr
    const int32_t *q_tok;         // [NQ] token of each query (global rows) or nullptr (token 0)
    int tok_limit;                // q_tok entries outside [0, tok_limit) are skipped
    int B, NQ, H_q, H_kv, D;
    int n_slots;  // cache slots (decode) or T (global rows)
    int W;        // window for the position test (decode)
    int n_sink;   // positions below n_sink pass the position test whatever the window
    float scale_log2;
    int slots_per_split, n_splits, q_per_cta;
    float *ws_ml;     // [B, NQ, H_q, n_splits, 2]   (max in log2 units, sum)
    float *ws_acc;    // [B, NQ, H_q, n_splits, D]   unnormalised weighted values
    int32_t *ws_cnt;  // [B, H_kv, n_splits]         valid slots per split
    // Decode only: the current token's key/value rows [B, H_kv, D] to write into slot
    // slot(q_pos[b]) before it is read (nullptr: none), and slot_pos to update there.
    const uint16_t *k_new, *v_new;
    int32_t *slot_pos_w;
    // Global rows: launched as a programmatic dependent of the band kernel before it on
    // the stream (it reads only q/k/v, so it may start on SMs the band kernel has left);
    // the grid then waits for that kernel before completing.
    int after_band;
};

struct MergeArgs {
    const float *ws_ml;
    const float *ws_acc;
    const int32_t *ws_cnt;
    int B, NQ, H_q, H_kv, D, n_splits;
    const int32_t *q_tok;  // as in SplitArgs
    int tok_limit;
    void *o;
    int64_t o_sb, o_st, o_sh;
    float *lse;
    int64_t lse_sb, lse_sh, lse_st;
    int32_t *counts;  // may be nullptr
    int64_t cnt_sb, cnt_sh, cnt_st;
};

// Split geometry shared by the workspace-size query and the launch.
constexpr int kSplitChunk = 64;         // slots per pipeline stage
constexpr int kSlotsPerSplit = 1024;    // slots per work item (larger items amortise the per-item combine)
constexpr int kSplitRows = 16;          // mma.sync M: query rows per CTA

inline int split_q_per_cta(int group) { return group >= kSplitRows ? 1 : kSplitRows / group; }
inline int split_count(int n_slots) { return (n_slots + kSlotsPerSplit - 1) / kSlotsPerSplit; }
// Slots per split: the fewest whole chunks that still cover n_slots with split_count
// splits, so the last split is not left nearly empty (4100 slots: 5 x 832, not 4 x 1024 + 4).
inline int split_size(int n_slots) {
    const int ns = split_count(n_slots);
    const int per = (n_slots + ns - 1) / ns;
    return (per + kSplitChunk - 1) / kSplitChunk * kSplitChunk;
}
// Slots per split for a pass whose items are `pairs` (batch, kv head, query block)
// groups times the splits of n_slots, dealt round-robin to `grid` persistent CTAs.
// Among whole-chunk splits from 256 slots up to kSlotsPerSplit (each balanced like
// split_size), take the one that finishes in the fewest slot-times, counting about
// 96 slots of fixed cost per item (its end-of-item combine).  A pass of few groups
// (the global rows of a short sequence) gets smaller splits so the last wave of items
// is not left half empty.
inline int split_size_for_grid(int n_slots, long long pairs, int grid) {
    const int ns_min = split_count(n_slots);
    const int ns_max = ns_min > (n_slots + 255) / 256 ? ns_min : (n_slots + 255) / 256;
    int best = split_size(n_slots);
    long long best_t = -1;
    for (int ns = ns_min; ns <= ns_max; ++ns) {
        const int per = (n_slots + ns - 1) / ns;
        const int sz = (per + kSplitChunk - 1) / kSplitChunk * kSplitChunk;
        if (sz > kSlotsPerSplit) continue;
        const long long items = pairs * ((n_slots + sz - 1) / sz);
        const long long t = (items + grid - 1) / grid * (sz + 96);
        if (best_t < 0 || t < best_t) {
            best_t = t;
            best = sz;
        }
    }
    return best;
}
// Workspace of a split pass with ns splits: ml, acc and cnt, each 256-byte aligned.
inline size_t split_workspace_bytes(int B, int NQ, int H_q, int H_kv, int D, int ns) {
    const size_t rows = static_cast<size_t>(B) * NQ * H_q * ns;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    return up(rows * 2 * sizeof(float)) + up(rows * D * sizeof(float)) +
           up(static_cast<size_t>(B) * H_kv * ns * sizeof(int32_t));
}
inline void split_carve(void *ws, int B, int NQ, int H_q, int D, int ns, float **ml, float **acc, int32_t **cnt) {
    const size_t rows = static_cast<size_t>(B) * NQ * H_q * ns;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    char *p = static_cast<char *>(ws);
    *ml = reinterpret_cast<float *>(p);
    p += up(rows * 2 * sizeof(float));
    *acc = reinterpret_cast<float *>(p);
    p += up(rows * D * sizeof(float));
    *cnt = reinterpret_cast<int32_t *>(p);
}

// Persistent CTAs of the split pass at head dim D on the current device.
int split_grid(int D);
cudaError_t launch_split(const SplitArgs &a, cudaStream_t s);
cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s);
unsigned int split_read_clear_error();

// Banded prefill (tcgen05 path).
struct BandArgs {
    const void *q, *k, *v;
    int64_t q_st[3], k_st[3], v_st[3], o_st[3];  // element strides (b, t, h)
    int B, T, H_q, H_kv, D;
    int wl, wr;  // < 0: unbounded
    float scale_log2;
    const int32_t *global_idx;
    int n_global;
    int gmode;           // SWA_GLOBAL_FULL / SWA_GLOBAL_SINK
    bool sep;            // separate global projections: global keys come from kg, vg only
    const void *kg, *vg; // key/value rows of the global-column tiles (k, v unless sep)
    int64_t kg_st[3], vg_st[3];
    void *o;
    float *lse;
    int32_t *counts;
    int64_t lse_st[3];  // element strides (b, h, t) of lse and counts
    // Keys in their own index space (chunked prefill): Tk key rows (0: T), query row t
    // at key index t + q_off, keys below kmin[b] absent (kmin: device [B] or nullptr).
    int Tk, q_off;
    const int32_t *kmin;
    // Chunked prefill with sinks: key index q_off of sequence b is position p0[b] (global
    // positions are then true positions); global-column rows are kg/vg rows in list order.
    const int32_t *p0;
    bool gcol_list_rows;
};
cudaError_t launch_band(const BandArgs &a, cudaStream_t s);

// Ring-buffer cache (swa_cache.cu).  Slot rule: p < n_sink -> p, else
// n_sink + (p - n_sink) mod (n_slots - n_sink).
struct AppendArgs {
    uint16_t *kc, *vc;     // [B, H_kv, n_slots, D] bf16 bits
    int32_t *slot_pos;     // [B, n_slots]
    int B, H_kv, D, n_slots, n_sink;
    const uint16_t *kn, *vn;  // [B, n, H_kv, D]
    int n;
    const int32_t *p0;     // [B] position of token 0
};
cudaError_t launch_append(const AppendArgs &a, cudaStream_t s);

// Window history of a chunk in position order, then the chunk: kl/vl [B, W-1+C, H_kv, D]
// and kmin[b], the first key index present.  With n_sink pinned sinks also their rows,
// ks/vs [B, n_sink, H_kv, D] (from the cache, or from the chunk for sinks inside it).
struct GatherArgs {
    const uint16_t *kc, *vc;
    const int32_t *slot_pos;
    int B, H_kv, D, n_slots, n_sink;
    const uint16_t *kn, *vn;  // [B, C, H_kv, D]
    int C, W;
    const int32_t *p0;
    uint16_t *kl, *vl;
    int32_t *kmin;
    uint16_t *ks, *vs;
    int32_t *sink_idx;  // [n_sink] positions 0 .. n_sink-1 (the band kernel's column list)
};
cudaError_t launch_gather(const GatherArgs &a, cudaStream_t s);
unsigned int cache_read_clear_error();  // bit 0: bad position, bit 1: cache mismatch

// Host-side helpers of the C ABI shared with the allocation-free decode entry point.
swa_status validate_decode(const swa_decode_params *p);  // the checks swa_decode applies
// Bytes of split partials a decode of `p` needs, and the split + merge launches of a
// validated decode into workspace `ws` (at least that many bytes, 256-byte aligned).
size_t decode_workspace_bytes(const swa_decode_params *p);
// k_new / v_new (bf16 [B, H_kv, d_h]) non-null: the current token is appended first.
cudaError_t run_decode(const swa_decode_params *p, void *ws, cudaStream_t s, const void *k_new = nullptr,
                       const void *v_new = nullptr);
bool record_cuda_failure(cudaError_t e);                  // true (and recorded) if e failed
unsigned int band_read_clear_error();

// Planted faults of the failure-detection tests (swa_debug_set_faults), read by every
// band and split launch: a producer that stops issuing copies (INT_MAX: off).
struct FaultPlan {
    int band_stop_fill;
    int split_stop_stage;
};
FaultPlan fault_plan();

}  // namespace swa
