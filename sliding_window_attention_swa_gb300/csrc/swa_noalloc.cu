// swa_noalloc.cu -- ring-buffer decode for callers that cannot allocate device
// memory at the call site.
//
// swa_decode needs a workspace for its split partials, which the caller normally
// allocates.  Some callers can't: a serving loop that must not allocate once it is
// running (cudaMalloc may synchronise the device and can fail under memory
// pressure), or a plugin interface that hands the kernel only its inputs and
// outputs.  swa_decode_noalloc runs the same two kernels (split-K scoring, then the
// log-sum-exp merge) with the partials in a fixed scratch array compiled into the
// library, so it allocates nothing.
#include <mutex>

#include "swa_internal.h"

namespace {

// The scratch array: SWA_DECODE_NOALLOC_SCRATCH_BYTES of device memory on every GPU
// that loads the library, held until the process exits.  In host code its name is
// only a host-side stand-in; kernels get the device address from scratch_address().
static __device__ __align__(256) unsigned char g_decode_scratch[SWA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};  // device address of g_decode_scratch, per device

// Device address of the scratch array on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" swa_status swa_decode_noalloc(const swa_decode_params *p, swa_stream_t stream) {
    const swa_status st = swa::validate_decode(p);
    if (st != SWA_OK) return st;
    const size_t need = swa::split_workspace_bytes(p->B, 1, p->H_q, p->H_kv, p->d_h, p->W);
    if (need > SWA_DECODE_NOALLOC_SCRATCH_BYTES) return SWA_ERR_WORKSPACE;
    void *ws = nullptr;
    if (swa::record_cuda_failure(scratch_address(&ws))) return SWA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t D = p->d_h, W = p->W;

    // Every partial the merge reads is written by the split kernel of the same call,
    // so the scratch needs no clearing between calls.
    swa::SplitArgs sa{};
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
    sa.W = p->W;
    sa.scale_log2 = p->scale * 1.4426950408889634f;
    sa.slots_per_split = swa::kSlotsPerSplit;
    sa.n_splits = swa::split_count(p->W);
    sa.q_per_cta = swa::split_q_per_cta(p->H_q / p->H_kv);
    swa::split_carve(ws, p->B, 1, p->H_q, p->H_kv, p->d_h, p->W, &sa.ws_ml, &sa.ws_acc, &sa.ws_cnt);
    if (swa::record_cuda_failure(swa::launch_split(sa, s))) return SWA_ERR_CUDA;

    swa::MergeArgs ma{};
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
    if (swa::record_cuda_failure(swa::launch_merge(ma, s))) return SWA_ERR_CUDA;
    return SWA_OK;
}
