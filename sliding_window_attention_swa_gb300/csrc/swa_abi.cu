// swa_abi.cu -- the extern "C" entry points of libswa.so: argument validation on
// the host, workspace sizing, and the kernel launches on the caller's stream.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>

#include "swa_internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }
bool strides_ok(const int64_t st[3]) {
    for (int i = 0; i < 3; ++i)
        if (st[i] <= 0 || (st[i] % 8) != 0) return false;
    return true;
}
bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }
constexpr float kLog2e = 1.4426950408889634f;

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

// Planted faults (swa_debug_set_faults); INT_MAX / 0 = off.
std::atomic<int> g_band_stop{INT_MAX};
std::atomic<int> g_split_stop{INT_MAX};

// Records a failed CUDA call for swa_last_error_string(); true if `e` is a failure.
bool failed(cudaError_t e) {
    if (e == cudaSuccess) return false;
    t_last_cuda_error = e;
    return true;
}

// Separate global projections given (all three) or not (none); a partial set is invalid.
bool has_sep(const swa_fwd_params *p) { return p->q_g || p->k_g || p->v_g; }

swa_status fwd_check(const swa_fwd_params *p) {
    if (!p || !p->q || !p->k || !p->v || !p->o || !p->lse) return SWA_ERR_INVALID_ARG;
    if (p->B < 1 || p->T < 1 || p->H_q < 1 || p->H_kv < 1 || p->d_h < 1) return SWA_ERR_INVALID_ARG;
    if (p->H_q % p->H_kv != 0) return SWA_ERR_INVALID_ARG;
    if (p->n_global < 0 || p->n_global > p->T) return SWA_ERR_INVALID_ARG;
    if (p->n_global > 0 && !p->global_idx) return SWA_ERR_INVALID_ARG;
    if (!std::isfinite(p->scale)) return SWA_ERR_INVALID_ARG;
    if (p->global_mode != SWA_GLOBAL_FULL && p->global_mode != SWA_GLOBAL_SINK) return SWA_ERR_INVALID_ARG;
    if (has_sep(p)) {
        if (!p->q_g || !p->k_g || !p->v_g || p->global_mode != SWA_GLOBAL_FULL) return SWA_ERR_INVALID_ARG;
        if (!strides_ok(p->qg_strides) || !strides_ok(p->kg_strides) || !strides_ok(p->vg_strides) ||
            !aligned16(p->q_g) || !aligned16(p->k_g) || !aligned16(p->v_g))
            return SWA_ERR_UNSUPPORTED;
    }
    if (p->dilation) {
        bool dilated = false;
        for (int h = 0; h < p->H_q; ++h) {
            if (p->dilation[h] < 1) return SWA_ERR_INVALID_ARG;
            dilated |= p->dilation[h] > 1;
        }
        if (dilated && p->n_global > 0) return SWA_ERR_UNSUPPORTED;
    }
    if (!head_dim_ok(p->d_h)) return SWA_ERR_UNSUPPORTED;
    if (p->H_q / p->H_kv > swa::kSplitRows) return SWA_ERR_UNSUPPORTED;
    if (!scale_ok(p->scale)) return SWA_ERR_UNSUPPORTED;
    if (!strides_ok(p->q_strides) || !strides_ok(p->k_strides) || !strides_ok(p->v_strides) ||
        !strides_ok(p->o_strides))
        return SWA_ERR_UNSUPPORTED;
    if (!aligned16(p->q) || !aligned16(p->k) || !aligned16(p->v) || !aligned16(p->o) ||
        (p->global_idx && (reinterpret_cast<uintptr_t>(p->global_idx) & 3u)) ||
        (reinterpret_cast<uintptr_t>(p->lse) & 3u) || (reinterpret_cast<uintptr_t>(p->row_counts) & 3u))
        return SWA_ERR_UNSUPPORTED;
    return SWA_OK;
}

swa_status decode_check(const swa_decode_params *p) {
    if (!p || !p->q || !p->k_cache || !p->v_cache || !p->slot_pos || !p->q_pos || !p->o || !p->lse)
        return SWA_ERR_INVALID_ARG;
    if (p->B < 1 || p->H_q < 1 || p->H_kv < 1 || p->d_h < 1 || p->W < 1) return SWA_ERR_INVALID_ARG;
    if (p->H_q % p->H_kv != 0) return SWA_ERR_INVALID_ARG;
    if (!std::isfinite(p->scale)) return SWA_ERR_INVALID_ARG;
    if (p->window < 0 || p->n_sink < 0) return SWA_ERR_INVALID_ARG;
    if (!head_dim_ok(p->d_h)) return SWA_ERR_UNSUPPORTED;
    if (p->H_q / p->H_kv > swa::kSplitRows) return SWA_ERR_UNSUPPORTED;
    if (!scale_ok(p->scale)) return SWA_ERR_UNSUPPORTED;
    if (!aligned16(p->q) || !aligned16(p->k_cache) || !aligned16(p->v_cache) || !aligned16(p->o) ||
        (reinterpret_cast<uintptr_t>(p->slot_pos) & 3u) || (reinterpret_cast<uintptr_t>(p->q_pos) & 3u) ||
        (reinterpret_cast<uintptr_t>(p->lse) & 3u) || (reinterpret_cast<uintptr_t>(p->row_counts) & 3u))
        return SWA_ERR_UNSUPPORTED;
    return SWA_OK;
}

swa_status cache_check(const swa_cache_params *c) {
    if (!c || !c->k_cache || !c->v_cache || !c->slot_pos) return SWA_ERR_INVALID_ARG;
    if (c->B < 1 || c->H_kv < 1 || c->d_h < 1 || c->n_slots < 1) return SWA_ERR_INVALID_ARG;
    if (c->n_sink < 0 || c->n_sink >= c->n_slots) return SWA_ERR_INVALID_ARG;
    if (!head_dim_ok(c->d_h)) return SWA_ERR_UNSUPPORTED;
    if (!aligned16(c->k_cache) || !aligned16(c->v_cache) || (reinterpret_cast<uintptr_t>(c->slot_pos) & 3u))
        return SWA_ERR_UNSUPPORTED;
    return SWA_OK;
}

swa_status chunk_check(const swa_chunk_params *p, const swa_cache_params *c) {
    swa_status st = cache_check(c);
    if (st != SWA_OK) return st;
    if (!p || !p->q || !p->k_new || !p->v_new || !p->p0 || !p->o || !p->lse) return SWA_ERR_INVALID_ARG;
    if (p->B < 1 || p->C < 1 || p->H_q < 1 || p->H_kv < 1 || p->d_h < 1 || p->window < 1) return SWA_ERR_INVALID_ARG;
    if (p->H_q % p->H_kv != 0 || p->B != c->B || p->H_kv != c->H_kv || p->d_h != c->d_h) return SWA_ERR_INVALID_ARG;
    if (!std::isfinite(p->scale)) return SWA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(p->window) - 1 + p->C > (1 << 30)) return SWA_ERR_INVALID_ARG;
    // a sink cache's ring must cover the window (its history is then contiguous)
    if (c->n_sink > 0 && c->n_slots - c->n_sink < p->window - 1) return SWA_ERR_UNSUPPORTED;
    if (c->n_sink > 128) return SWA_ERR_UNSUPPORTED;
    // the gather's index arithmetic is 32-bit
    if (static_cast<int64_t>(p->B) * (static_cast<int64_t>(p->window) - 1 + p->C + c->n_sink) * p->H_kv >=
        (int64_t{1} << 31))
        return SWA_ERR_UNSUPPORTED;
    if (!head_dim_ok(p->d_h)) return SWA_ERR_UNSUPPORTED;
    if (p->H_q / p->H_kv > swa::kSplitRows) return SWA_ERR_UNSUPPORTED;
    if (!scale_ok(p->scale)) return SWA_ERR_UNSUPPORTED;
    if (!aligned16(p->q) || !aligned16(p->k_new) || !aligned16(p->v_new) || !aligned16(p->o) ||
        (reinterpret_cast<uintptr_t>(p->p0) & 3u) || (reinterpret_cast<uintptr_t>(p->lse) & 3u) ||
        (reinterpret_cast<uintptr_t>(p->row_counts) & 3u))
        return SWA_ERR_UNSUPPORTED;
    return SWA_OK;
}

// Workspace of a chunked prefill: gathered keys and values, kmin, sink rows, sink list.
struct ChunkWs {
    size_t kv_bytes, kmin_bytes, sink_bytes, total;
};
ChunkWs chunk_ws(const swa_chunk_params *p, const swa_cache_params *c) {
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t rows = static_cast<size_t>(p->B) * (static_cast<size_t>(p->window) - 1 + p->C) * p->H_kv;
    const size_t kv = up(rows * p->d_h * 2);
    const size_t km = up(static_cast<size_t>(p->B) * 4);
    const size_t sk = up(static_cast<size_t>(p->B) * c->n_sink * p->H_kv * p->d_h * 2);
    return {kv, km, sk, 2 * kv + km + 2 * sk + up(static_cast<size_t>(c->n_sink) * 4)};
}

swa::AppendArgs append_args(const swa_cache_params *c, const void *k_new, const void *v_new, int n,
                            const int32_t *p0) {
    swa::AppendArgs a{};
    a.kc = static_cast<uint16_t *>(c->k_cache);
    a.vc = static_cast<uint16_t *>(c->v_cache);
    a.slot_pos = c->slot_pos;
    a.B = c->B;
    a.H_kv = c->H_kv;
    a.D = c->d_h;
    a.n_slots = c->n_slots;
    a.n_sink = c->n_sink;
    a.kn = static_cast<const uint16_t *>(k_new);
    a.vn = static_cast<const uint16_t *>(v_new);
    a.n = n;
    a.p0 = p0;
    return a;
}

swa_status workspace_ok(void *ws, size_t have, size_t need) {
    if (need == 0) return SWA_OK;
    if (!ws || have < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return SWA_ERR_WORKSPACE;
    return SWA_OK;
}

// Global rows (attending to every key) exist only for SWA_GLOBAL_FULL.
bool has_global_rows(const swa_fwd_params *p) { return p->n_global > 0 && p->global_mode == SWA_GLOBAL_FULL; }

// Split size and count of the global-row pass: its items are (batch, kv head, query
// block) groups times the splits of T, sized to the persistent grid.
int global_row_split_size(const swa_fwd_params *p) {
    const int qpc = swa::split_q_per_cta(p->H_q / p->H_kv);
    const long long pairs = static_cast<long long>(p->B) * p->H_kv * ((p->n_global + qpc - 1) / qpc);
    return swa::split_size_for_grid(p->T, pairs, swa::split_grid(p->d_h));
}
int global_row_splits(const swa_fwd_params *p) {
    const int sz = global_row_split_size(p);
    return (p->T + sz - 1) / sz;
}

// Band launches of swa_fwd.  A dilated head attends, within each residue class
// t = r (mod d), to the ordinary band of that subsequence (keys t + k*d), so every
// (dilation, residue) pair is one launch over strided views of q, k, v, o, lse and
// counts: token stride d * stride, T' = ceil((T - r) / d), window sides unchanged.
// Heads sharing a dilation are taken in runs of whole GQA groups; a head whose
// group mixes dilations is launched alone (one query head over its kv head).
cudaError_t launch_band_views(const swa_fwd_params *p, const swa::BandArgs &base, cudaStream_t s) {
    auto dil = [&](int h) { return p->dilation ? p->dilation[h] : 1; };
    const int G = p->H_q / p->H_kv;
    bool uniform = true;
    for (int h = 1; h < p->H_q; ++h) uniform &= dil(h) == dil(0);
    if (uniform && dil(0) == 1) return swa::launch_band(base, s);
    auto launch = [&](int h0, int nh, int kvh0, int nkv, int d) -> cudaError_t {
        for (int r = 0; r < d && r < p->T; ++r) {
            swa::BandArgs v = base;
            const auto *q = static_cast<const uint16_t *>(p->q);
            const auto *k = static_cast<const uint16_t *>(p->k);
            const auto *vv = static_cast<const uint16_t *>(p->v);
            auto *o = static_cast<uint16_t *>(p->o);
            v.q = q + r * p->q_strides[1] + static_cast<int64_t>(h0) * p->q_strides[2];
            v.k = k + r * p->k_strides[1] + static_cast<int64_t>(kvh0) * p->k_strides[2];
            v.v = vv + r * p->v_strides[1] + static_cast<int64_t>(kvh0) * p->v_strides[2];
            v.o = o + r * p->o_strides[1] + static_cast<int64_t>(h0) * p->o_strides[2];
            v.q_st[1] = d * p->q_strides[1];
            v.k_st[1] = d * p->k_strides[1];
            v.v_st[1] = d * p->v_strides[1];
            v.o_st[1] = d * p->o_strides[1];
            v.T = (p->T - r + d - 1) / d;
            v.H_q = nh;
            v.H_kv = nkv;
            const int64_t off = static_cast<int64_t>(h0) * base.lse_st[1] + r * base.lse_st[2];
            v.lse = p->lse + off;
            v.counts = p->row_counts ? p->row_counts + off : nullptr;
            v.lse_st[2] = d * base.lse_st[2];
            const cudaError_t e = swa::launch_band(v, s);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    };
    int g = 0;
    while (g < p->H_kv) {
        bool whole = true;
        for (int h = g * G + 1; h < (g + 1) * G; ++h) whole &= dil(h) == dil(g * G);
        if (!whole) {
            for (int h = g * G; h < (g + 1) * G; ++h) {
                const cudaError_t e = launch(h, 1, g, 1, dil(h));
                if (e != cudaSuccess) return e;
            }
            ++g;
            continue;
        }
        int g1 = g + 1;  // extend the run over following whole groups of the same dilation
        while (g1 < p->H_kv) {
            bool same = true;
            for (int h = g1 * G; h < (g1 + 1) * G; ++h) same &= dil(h) == dil(g * G);
            if (!same) break;
            ++g1;
        }
        const cudaError_t e = launch(g * G, (g1 - g) * G, g, g1 - g, dil(g * G));
        if (e != cudaSuccess) return e;
        g = g1;
    }
    return cudaSuccess;
}

}  // namespace

swa::FaultPlan swa::fault_plan() {
    FaultPlan f;
    f.band_stop_fill = g_band_stop.load(std::memory_order_relaxed);
    f.split_stop_stage = g_split_stop.load(std::memory_order_relaxed);
    return f;
}

swa_status swa::validate_decode(const swa_decode_params *p) { return decode_check(p); }
bool swa::record_cuda_failure(cudaError_t e) { return failed(e); }

size_t swa::decode_workspace_bytes(const swa_decode_params *p) {
    return split_workspace_bytes(p->B, 1, p->H_q, p->H_kv, p->d_h, split_count(p->W));
}

cudaError_t swa::run_decode(const swa_decode_params *p, void *ws, cudaStream_t s, const void *k_new,
                            const void *v_new) {
    const int64_t D = p->d_h, W = p->W;
    SplitArgs sa{};
    sa.q = p->q;
    sa.q_sb = static_cast<int64_t>(p->H_q) * D;
    sa.q_st = 0;
    sa.q_sh = D;
    sa.k = p->k_cache;
    sa.v = p->v_cache;
    sa.k_sb = sa.v_sb = static_cast<int64_t>(p->H_kv) * W * D;
    sa.k_ss = sa.v_ss = D;
    sa.k_sh = sa.v_sh = W * D;
    sa.slot_pos = p->slot_pos;
    sa.q_pos = p->q_pos;
    sa.q_tok = nullptr;
    sa.tok_limit = 1;
    sa.B = p->B;
    sa.NQ = 1;
    sa.H_q = p->H_q;
    sa.H_kv = p->H_kv;
    sa.D = p->d_h;
    sa.n_slots = p->W;
    sa.W = p->window > 0 ? p->window : p->W;
    sa.n_sink = p->n_sink;
    sa.scale_log2 = p->scale * kLog2e;
    sa.slots_per_split = split_size(p->W);
    sa.n_splits = split_count(p->W);
    sa.q_per_cta = split_q_per_cta(p->H_q / p->H_kv);
    split_carve(ws, p->B, 1, p->H_q, p->d_h, sa.n_splits, &sa.ws_ml, &sa.ws_acc, &sa.ws_cnt);
    sa.k_new = static_cast<const uint16_t *>(k_new);
    sa.v_new = static_cast<const uint16_t *>(v_new);
    sa.slot_pos_w = const_cast<int32_t *>(p->slot_pos);
    cudaError_t e = launch_split(sa, s);
    if (e != cudaSuccess) return e;

    MergeArgs ma{};
    ma.ws_ml = sa.ws_ml;
    ma.ws_acc = sa.ws_acc;
    ma.ws_cnt = sa.ws_cnt;
    ma.B = p->B;
    ma.NQ = 1;
    ma.H_q = p->H_q;
    ma.H_kv = p->H_kv;
    ma.D = p->d_h;
    ma.n_splits = sa.n_splits;
    ma.q_tok = nullptr;
    ma.tok_limit = 1;
    ma.o = p->o;
    ma.o_sb = static_cast<int64_t>(p->H_q) * D;
    ma.o_st = 0;
    ma.o_sh = D;
    ma.lse = p->lse;
    ma.lse_sb = p->H_q;
    ma.lse_sh = 1;
    ma.lse_st = 0;
    ma.counts = p->row_counts;
    ma.cnt_sb = p->H_q;
    ma.cnt_sh = 1;
    ma.cnt_st = 0;
    return launch_merge(ma, s);
}

extern "C" {

int32_t swa_abi_version(void) { return SWA_ABI_VERSION; }

const char *swa_last_error_string(void) { return cudaGetErrorString(t_last_cuda_error); }

const char *swa_status_string(swa_status s) {
    switch (s) {
        case SWA_OK: return "ok";
        case SWA_ERR_INVALID_ARG: return "invalid argument";
        case SWA_ERR_UNSUPPORTED: return "unsupported configuration (head dim, group size, scale or alignment)";
        case SWA_ERR_CUDA: return "CUDA launch or runtime error";
        case SWA_ERR_TIMEOUT: return "a kernel's bounded wait expired";
        case SWA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    }
    return "unknown status";
}

size_t swa_fwd_workspace_size(const swa_fwd_params *p) {
    if (fwd_check(p) != SWA_OK || !has_global_rows(p)) return 0;
    return swa::split_workspace_bytes(p->B, p->n_global, p->H_q, p->H_kv, p->d_h, global_row_splits(p));
}

swa_status swa_fwd(const swa_fwd_params *p, void *workspace, size_t workspace_bytes, swa_stream_t stream) {
    swa_status st = fwd_check(p);
    if (st != SWA_OK) return st;
    st = workspace_ok(workspace, workspace_bytes, swa_fwd_workspace_size(p));
    if (st != SWA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float scale_log2 = p->scale * kLog2e;
    const bool sep = has_sep(p);

    swa::BandArgs ba{};
    ba.q = p->q;
    ba.k = p->k;
    ba.v = p->v;
    ba.o = p->o;
    for (int i = 0; i < 3; ++i) {
        ba.q_st[i] = p->q_strides[i];
        ba.k_st[i] = p->k_strides[i];
        ba.v_st[i] = p->v_strides[i];
        ba.o_st[i] = p->o_strides[i];
        ba.kg_st[i] = sep ? p->kg_strides[i] : p->k_strides[i];
        ba.vg_st[i] = sep ? p->vg_strides[i] : p->v_strides[i];
    }
    ba.B = p->B;
    ba.T = p->T;
    ba.H_q = p->H_q;
    ba.H_kv = p->H_kv;
    ba.D = p->d_h;
    ba.wl = p->window_left < 0 ? -1 : p->window_left;
    ba.wr = p->window_right < 0 ? -1 : p->window_right;
    ba.scale_log2 = scale_log2;
    ba.global_idx = p->n_global > 0 ? p->global_idx : nullptr;
    ba.n_global = p->n_global;
    ba.gmode = p->global_mode;
    ba.sep = sep && p->n_global > 0;
    ba.kg = sep ? p->k_g : p->k;
    ba.vg = sep ? p->v_g : p->v;
    ba.lse = p->lse;
    ba.counts = p->row_counts;
    ba.lse_st[0] = static_cast<int64_t>(p->H_q) * p->T;
    ba.lse_st[1] = p->T;
    ba.lse_st[2] = 1;
    if (failed(launch_band_views(p, ba, s))) return SWA_ERR_CUDA;

    if (has_global_rows(p)) {
        // Global rows attend to all T keys: split-K over T, merged by log-sum-exp,
        // overwriting the rows the band kernel wrote for those positions.  With
        // separate projections they read q_g, k_g and v_g only.
        const void *gq = sep ? p->q_g : p->q, *gk = sep ? p->k_g : p->k, *gv = sep ? p->v_g : p->v;
        const int64_t *qs = sep ? p->qg_strides : p->q_strides;
        const int64_t *ks = sep ? p->kg_strides : p->k_strides;
        const int64_t *vs = sep ? p->vg_strides : p->v_strides;
        swa::SplitArgs sa{};
        sa.q = gq;
        sa.q_sb = qs[0];
        sa.q_st = qs[1];
        sa.q_sh = qs[2];
        sa.k = gk;
        sa.v = gv;
        sa.k_sb = ks[0];
        sa.k_ss = ks[1];
        sa.k_sh = ks[2];
        sa.v_sb = vs[0];
        sa.v_ss = vs[1];
        sa.v_sh = vs[2];
        sa.slot_pos = nullptr;
        sa.q_pos = nullptr;
        sa.q_tok = p->global_idx;
        sa.tok_limit = p->T;
        sa.B = p->B;
        sa.NQ = p->n_global;
        sa.H_q = p->H_q;
        sa.H_kv = p->H_kv;
        sa.D = p->d_h;
        sa.n_slots = p->T;
        sa.W = p->T;
        sa.n_sink = 0;
        sa.scale_log2 = scale_log2;
        sa.slots_per_split = global_row_split_size(p);
        sa.n_splits = (p->T + sa.slots_per_split - 1) / sa.slots_per_split;
        sa.q_per_cta = swa::split_q_per_cta(p->H_q / p->H_kv);
        swa::split_carve(workspace, p->B, p->n_global, p->H_q, p->d_h, sa.n_splits, &sa.ws_ml, &sa.ws_acc,
                         &sa.ws_cnt);
        sa.after_band = 1;
        if (failed(swa::launch_split(sa, s))) return SWA_ERR_CUDA;
        swa::MergeArgs ma{};
        ma.ws_ml = sa.ws_ml;
        ma.ws_acc = sa.ws_acc;
        ma.ws_cnt = sa.ws_cnt;
        ma.B = p->B;
        ma.NQ = p->n_global;
        ma.H_q = p->H_q;
        ma.H_kv = p->H_kv;
        ma.D = p->d_h;
        ma.n_splits = sa.n_splits;
        ma.q_tok = p->global_idx;
        ma.tok_limit = p->T;
        ma.o = p->o;
        ma.o_sb = p->o_strides[0];
        ma.o_st = p->o_strides[1];
        ma.o_sh = p->o_strides[2];
        ma.lse = p->lse;
        ma.lse_sb = static_cast<int64_t>(p->H_q) * p->T;
        ma.lse_sh = p->T;
        ma.lse_st = 1;
        ma.counts = p->row_counts;
        ma.cnt_sb = ma.lse_sb;
        ma.cnt_sh = ma.lse_sh;
        ma.cnt_st = 1;
        if (failed(swa::launch_merge(ma, s))) return SWA_ERR_CUDA;
    }
    return SWA_OK;
}

size_t swa_decode_workspace_size(const swa_decode_params *p) {
    if (decode_check(p) != SWA_OK) return 0;
    return swa::decode_workspace_bytes(p);
}

swa_status swa_decode(const swa_decode_params *p, void *workspace, size_t workspace_bytes, swa_stream_t stream) {
    swa_status st = decode_check(p);
    if (st != SWA_OK) return st;
    st = workspace_ok(workspace, workspace_bytes, swa_decode_workspace_size(p));
    if (st != SWA_OK) return st;
    if (failed(swa::run_decode(p, workspace, reinterpret_cast<cudaStream_t>(stream)))) return SWA_ERR_CUDA;
    return SWA_OK;
}

swa_status swa_cache_append(const swa_cache_params *c, const void *k_new, const void *v_new, int32_t n_new,
                            const int32_t *p0, swa_stream_t stream) {
    swa_status st = cache_check(c);
    if (st != SWA_OK) return st;
    if (n_new < 0 || (n_new > 0 && (!k_new || !v_new || !p0))) return SWA_ERR_INVALID_ARG;
    if (n_new == 0) return SWA_OK;
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(p0) & 3u)) return SWA_ERR_UNSUPPORTED;
    // the append kernel's index arithmetic is 32-bit
    if (static_cast<int64_t>(c->B) * n_new * c->H_kv >= (int64_t{1} << 31)) return SWA_ERR_UNSUPPORTED;
    if (failed(swa::launch_append(append_args(c, k_new, v_new, n_new, p0), reinterpret_cast<cudaStream_t>(stream))))
        return SWA_ERR_CUDA;
    return SWA_OK;
}

swa_status swa_decode_append(const swa_decode_params *p, const void *k_new, const void *v_new, void *workspace,
                             size_t workspace_bytes, swa_stream_t stream) {
    swa_status st = decode_check(p);
    if (st != SWA_OK) return st;
    if (!k_new || !v_new || p->n_sink >= p->W) return SWA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return SWA_ERR_UNSUPPORTED;
    st = workspace_ok(workspace, workspace_bytes, swa_decode_workspace_size(p));
    if (st != SWA_OK) return st;
    if (failed(swa::run_decode(p, workspace, reinterpret_cast<cudaStream_t>(stream), k_new, v_new)))
        return SWA_ERR_CUDA;
    return SWA_OK;
}

size_t swa_prefill_chunk_workspace_size(const swa_chunk_params *p, const swa_cache_params *c) {
    if (chunk_check(p, c) != SWA_OK) return 0;
    return chunk_ws(p, c).total;
}

swa_status swa_prefill_chunk(const swa_chunk_params *p, const swa_cache_params *c, void *workspace,
                             size_t workspace_bytes, swa_stream_t stream) {
    swa_status st = chunk_check(p, c);
    if (st != SWA_OK) return st;
    const ChunkWs ws = chunk_ws(p, c);
    st = workspace_ok(workspace, workspace_bytes, ws.total);
    if (st != SWA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int W = p->window, C = p->C, Tk = W - 1 + C;
    char *w = static_cast<char *>(workspace);
    uint16_t *kl = reinterpret_cast<uint16_t *>(w);
    uint16_t *vl = reinterpret_cast<uint16_t *>(w + ws.kv_bytes);
    int32_t *kmin = reinterpret_cast<int32_t *>(w + 2 * ws.kv_bytes);
    uint16_t *ksink = reinterpret_cast<uint16_t *>(w + 2 * ws.kv_bytes + ws.kmin_bytes);
    uint16_t *vsink = reinterpret_cast<uint16_t *>(w + 2 * ws.kv_bytes + ws.kmin_bytes + ws.sink_bytes);
    int32_t *sink_idx = reinterpret_cast<int32_t *>(w + 2 * ws.kv_bytes + ws.kmin_bytes + 2 * ws.sink_bytes);
    const int ns = c->n_sink;

    // 1. the window history (positions p0-W+1 .. p0-1) in position order, then the chunk
    swa::GatherArgs ga{};
    ga.kc = static_cast<const uint16_t *>(c->k_cache);
    ga.vc = static_cast<const uint16_t *>(c->v_cache);
    ga.slot_pos = c->slot_pos;
    ga.B = p->B;
    ga.H_kv = p->H_kv;
    ga.D = p->d_h;
    ga.n_slots = c->n_slots;
    ga.n_sink = ns;
    ga.ks = ksink;
    ga.vs = vsink;
    ga.sink_idx = sink_idx;
    ga.kn = static_cast<const uint16_t *>(p->k_new);
    ga.vn = static_cast<const uint16_t *>(p->v_new);
    ga.C = C;
    ga.W = W;
    ga.p0 = p->p0;
    ga.kl = kl;
    ga.vl = vl;
    ga.kmin = kmin;
    if (failed(swa::launch_gather(ga, s))) return SWA_ERR_CUDA;

    // 2. the causal window over that key sequence: query i sits at key index W-1+i
    const int64_t D = p->d_h;
    swa::BandArgs ba{};
    ba.q = p->q;
    ba.k = kl;
    ba.v = vl;
    ba.o = p->o;
    const int64_t qs[3] = {static_cast<int64_t>(C) * p->H_q * D, p->H_q * D, D};
    const int64_t ks[3] = {static_cast<int64_t>(Tk) * p->H_kv * D, p->H_kv * D, D};
    for (int i = 0; i < 3; ++i) {
        ba.q_st[i] = ba.o_st[i] = qs[i];
        ba.k_st[i] = ba.v_st[i] = ba.kg_st[i] = ba.vg_st[i] = ks[i];
    }
    ba.B = p->B;
    ba.T = C;
    ba.Tk = Tk;
    ba.q_off = W - 1;
    ba.kmin = kmin;
    ba.H_q = p->H_q;
    ba.H_kv = p->H_kv;
    ba.D = p->d_h;
    ba.wl = W - 1;
    ba.wr = 0;
    ba.scale_log2 = p->scale * kLog2e;
    ba.kg = kl;
    ba.vg = vl;
    if (ns > 0) {
        // the sinks as pinned key columns: true positions 0 .. ns-1 against each row's band
        // (key index W-1 is position p0[b]); their rows are the gathered sink rows
        ba.global_idx = sink_idx;
        ba.n_global = ns;
        ba.gmode = SWA_GLOBAL_SINK;
        ba.p0 = p->p0;
        ba.gcol_list_rows = true;
        ba.kg = ksink;
        ba.vg = vsink;
        const int64_t ss[3] = {static_cast<int64_t>(ns) * p->H_kv * D, p->H_kv * D, D};
        for (int i = 0; i < 3; ++i) ba.kg_st[i] = ba.vg_st[i] = ss[i];
    }
    ba.lse = p->lse;
    ba.counts = p->row_counts;
    ba.lse_st[0] = static_cast<int64_t>(p->H_q) * C;
    ba.lse_st[1] = C;
    ba.lse_st[2] = 1;
    if (failed(swa::launch_band(ba, s))) return SWA_ERR_CUDA;

    // 3. the chunk joins the cache
    if (p->append &&
        failed(swa::launch_append(append_args(c, p->k_new, p->v_new, C, p->p0), s)))
        return SWA_ERR_CUDA;
    return SWA_OK;
}

swa_status swa_read_device_errors(swa_stream_t stream, swa_device_errors *out) {
    if (out) *out = swa_device_errors{};
    if (failed(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)))) return SWA_ERR_CUDA;
    swa_device_errors e;
    e.prefill = swa::band_read_clear_error();
    e.split = swa::split_read_clear_error();
    e.cache = swa::cache_read_clear_error();
    if (out) *out = e;
    constexpr uint32_t kTimeout = SWA_DEVERR_WAIT_TIMEOUT | SWA_DEVERR_DRAIN_TIMEOUT;
    if ((e.prefill | e.split) & kTimeout) return SWA_ERR_TIMEOUT;
    if ((e.prefill & SWA_DEVERR_GLOBAL_LIST) || ((e.prefill | e.split) & SWA_DEVERR_BOUNDS) || e.cache)
        return SWA_ERR_INVALID_ARG;
    return SWA_OK;
}

swa_status swa_check_device_error(swa_stream_t stream) { return swa_read_device_errors(stream, nullptr); }

swa_status swa_debug_set_faults(const swa_debug_faults *f) {
    if (f && (f->band_stop_fill < -1 || f->split_stop_stage < -1)) return SWA_ERR_INVALID_ARG;
    g_band_stop.store(f && f->band_stop_fill >= 0 ? f->band_stop_fill : INT_MAX, std::memory_order_relaxed);
    g_split_stop.store(f && f->split_stop_stage >= 0 ? f->split_stop_stage : INT_MAX, std::memory_order_relaxed);
    return SWA_OK;
}

}  // extern "C"
