/*
 * swa.h -- C ABI of the sliding-window attention library (libswa.so, sm_103a).
 *
 * Operations
 * ----------
 * swa_fwd     Prefill / encoder attention over a band:
 *               o_t = sum over allowed s of softmax_s(scale * q_t . k_s) v_s
 *             Allowed keys of query t: window_left / window_right bound the band
 *             t - window_left <= s <= t + window_right (a negative value leaves that
 *             side unbounded), clipped to [0, T).  The causal window of W keys,
 *             N_t = [max(0, t-W+1), t] (Sliding Window Attention,
 *             lizeman.github.io llm-arch-kb, section 2 "Derivation"), is
 *             window_left = W-1, window_right = 0.  The bidirectional window
 *             |t - s| <= r (prathamp.com "Sliding Window Attention: From Local
 *             Windows to Global Context", section 1.1) is window_left =
 *             window_right = r.  Global positions (same page, section 4.3) attend
 *             to every key and are attended by every query; a global key already
 *             inside a query's band is counted once.  Variants:
 *               - global_mode SWA_GLOBAL_SINK: the listed positions are attention
 *                 sinks (lizeman page, "Failure mode 1", after StreamingLLM): key
 *                 columns that every query sees unless they lie right of its band
 *                 (for a causal window: in its future); their rows are ordinary.
 *               - separate global projections q_g, k_g, v_g (prathamp.com page,
 *                 section 5.2): a global row scores q_g[t] against k_g of every key
 *                 and averages v_g; a local row scores q[t] against k_g, v_g at the
 *                 global positions and against k, v elsewhere.
 *               - dilation d per query head (same page, section 3.1; lizeman page,
 *                 "Dilation"): the band becomes {t + k*d : -window_left <= k <=
 *                 window_right}, clipped to [0, T); the window sides count steps
 *                 of d.
 * swa_decode  One query token per sequence against a ring-buffer KV cache of W
 *             slots.  Token p is stored in slot p mod W (lizeman page, KV cache
 *             paragraph) and every slot carries its true token position; the
 *             window is evaluated on positions, not slot offsets (Gemma 3 note,
 *             ai-engineer-exhaustive.pages.dev, "How it works"): slot j is attended
 *             by the query at position t iff 0 <= pos_j <= t and either
 *             t - window < pos_j or pos_j < n_sink (the first n_sink positions
 *             pinned as attention sinks; window defaults to W).
 *
 * Conventions
 * -----------
 * - Element types: q, k, v, o are bf16; lse is fp32 (natural log of the softmax
 *   normaliser of the scaled scores, i.e. lse_t = log sum_s exp(scale q_t . k_s));
 *   row_counts are int32 numbers of attended keys.
 * - Grouped-query attention: H_q must be a multiple of H_kv; query head h reads
 *   key/value head h / (H_q / H_kv).
 * - Ownership: every pointer is device memory owned by the caller (unless stated
 *   otherwise); the library allocates nothing and keeps no pointer after return.
 * - Asynchrony: work is enqueued on `stream` and the call returns without
 *   synchronising.  Argument errors are detected on the host and returned before
 *   anything is launched.  SWA_ERR_CUDA reports a failed launch.
 * - Bounded waits: every wait inside a kernel has a time limit; on expiry the
 *   kernel records an error word in device memory, drains its own copies and
 *   tensor-core work, frees its tensor memory and returns, so the CUDA context stays
 *   usable.  The words are read (and cleared) by swa_check_device_error() or
 *   swa_read_device_errors().  They are per device, shared by every stream and
 *   every call on it.
 * - Thread safety: calls may be made from several host threads on different
 *   streams; workspaces must not be shared between calls that overlap in time.
 *   One-time per-device setup (kernel attributes, SM counts) is cached in atomics,
 *   so one process may also drive several devices (the current device is used).
 */
#ifndef SWA_H
#define SWA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SWA_API __attribute__((visibility("default")))
#else
#define SWA_API
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st *swa_stream_t;

/* Modes of swa_fwd's global position list. */
#define SWA_GLOBAL_FULL 0 /* global tokens: their rows see every key, every row sees them */
#define SWA_GLOBAL_SINK 1 /* attention sinks: key columns only, never right of a row's band */

typedef enum swa_status {
    SWA_OK = 0,
    SWA_ERR_INVALID_ARG = 1, /* a null pointer, a bad size, stride or window */
    SWA_ERR_UNSUPPORTED = 2, /* valid but not built: head dim, group size, alignment */
    SWA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    SWA_ERR_TIMEOUT = 4,     /* a kernel's bounded wait expired (see swa_check_device_error) */
    SWA_ERR_WORKSPACE = 5    /* workspace null or smaller than the *_workspace_size answer */
} swa_status;

/*
 * swa_fwd parameters.
 *   q           bf16 [B, T, H_q, d_h]; q_strides = element strides of (b, t, h); d_h contiguous.
 *   k, v        bf16 [B, T, H_kv, d_h]; k_strides / v_strides likewise.
 *   o           bf16 [B, T, H_q, d_h]; o_strides likewise.
 *   lse         fp32 [B, H_q, T], contiguous.
 *   row_counts  optional int32 [B, H_q, T], contiguous (NULL: not written).
 *   global_idx  optional int32 [n_global] device array of global positions, strictly
 *               increasing, each in [0, T) (NULL with n_global = 0: none).  The prefill
 *               kernel checks this on the device: a list that breaks it is reported by
 *               swa_check_device_error as SWA_ERR_INVALID_ARG (bit
 *               SWA_DEVERR_GLOBAL_LIST); that call's outputs are then undefined, but
 *               no memory outside its own buffers is read or written.
 *   global_mode SWA_GLOBAL_FULL (0) or SWA_GLOBAL_SINK (1): how global_idx is used.
 *   q_g, k_g, v_g  optional separate global projections, laid out like q, k, v with
 *               their own strides (all three or none; SWA_GLOBAL_FULL only).
 *   dilation    optional HOST int32 [H_q]: band dilation of each query head, >= 1
 *               (NULL: 1 for every head).  A dilation above 1 requires n_global = 0.
 * Requirements: d_h in {64, 128, 256}; H_q % H_kv == 0 and H_q / H_kv <= 16;
 * every base pointer 16-byte aligned; strides multiples of 8 elements; T >= 1.
 * Fields after row_counts were added in ABI version 2; zero them for the version 1
 * behaviour.
 */
typedef struct swa_fwd_params {
    const void *q;
    const void *k;
    const void *v;
    int64_t q_strides[3];
    int64_t k_strides[3];
    int64_t v_strides[3];
    int32_t B, T, H_q, H_kv, d_h;
    int32_t window_left;
    int32_t window_right;
    float scale;
    const int32_t *global_idx;
    int32_t n_global;
    void *o;
    int64_t o_strides[3];
    float *lse;
    int32_t *row_counts;
    int32_t global_mode;
    const void *q_g;
    const void *k_g;
    const void *v_g;
    int64_t qg_strides[3];
    int64_t kg_strides[3];
    int64_t vg_strides[3];
    const int32_t *dilation;
} swa_fwd_params;

/* Bytes of device workspace swa_fwd needs (0 without global rows); 0 for invalid params. */
SWA_API size_t swa_fwd_workspace_size(const swa_fwd_params *p);

/*
 * Banded attention (plus global rows and columns).  workspace: device memory of at
 * least swa_fwd_workspace_size(p) bytes, 256-byte aligned (may be NULL when that is 0).
 * Errors: SWA_ERR_INVALID_ARG / SWA_ERR_UNSUPPORTED / SWA_ERR_WORKSPACE before any
 * launch; SWA_ERR_CUDA if a launch fails.
 */
SWA_API swa_status swa_fwd(const swa_fwd_params *p, void *workspace, size_t workspace_bytes,
                   swa_stream_t stream);

/*
 * swa_decode parameters (all contiguous).
 *   q          bf16 [B, H_q, d_h]    the current token's queries
 *   k_cache    bf16 [B, H_kv, W, d_h] the W cache slots (the current token already stored)
 *   v_cache    bf16 [B, H_kv, W, d_h]
 *   slot_pos   int32 [B, W]  true token position held by each slot (< 0: never written)
 *   q_pos      int32 [B]     position t_b of the current token
 *   o          bf16 [B, H_q, d_h]
 *   lse        fp32 [B, H_q]
 *   row_counts optional int32 [B, H_q]
 *   window     the window in positions, >= 0 (0: W)            (ABI version 2)
 *   n_sink     positions 0 .. n_sink-1 are attended whatever the window, >= 0
 *              (0: none); a cache with sinks keeps them in slots of their own
 *              (see swa_cache_append)                          (ABI version 2)
 * Requirements: d_h in {64, 128, 256}; H_q % H_kv == 0 and H_q / H_kv <= 16; W >= 1;
 * pointers 16-byte aligned.
 */
typedef struct swa_decode_params {
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *slot_pos;
    const int32_t *q_pos;
    int32_t B, H_q, H_kv, d_h, W;
    float scale;
    void *o;
    float *lse;
    int32_t *row_counts;
    int32_t window;
    int32_t n_sink;
} swa_decode_params;

/* Bytes of device workspace swa_decode needs (split partials); 0 for invalid params. */
SWA_API size_t swa_decode_workspace_size(const swa_decode_params *p);

/*
 * Split-K decode: the W slots are cut into splits scored in parallel, each split
 * keeps a running (max, sum, weighted values) triple, and a second kernel merges
 * the splits by log-sum-exp.  workspace: >= swa_decode_workspace_size(p) bytes,
 * 256-byte aligned.  Errors as for swa_fwd.
 */
SWA_API swa_status swa_decode(const swa_decode_params *p, void *workspace, size_t workspace_bytes,
                      swa_stream_t stream);

/*
 * A ring-buffer KV cache (lizeman page, KV cache paragraph, after Mistral 7B section
 * 2: the keys and values of token p are stored in slot p mod W, overwriting older
 * ones).  A cache with n_sink pinned attention sinks keeps position p < n_sink in
 * slot p and rings the other positions through the remaining slots:
 *     slot(p) = p                                          if p < n_sink
 *             = n_sink + (p - n_sink) mod (n_slots - n_sink) otherwise.
 *   k_cache, v_cache  bf16 [B, H_kv, n_slots, d_h], contiguous
 *   slot_pos          int32 [B, n_slots]: the position each slot holds (< 0: never written)
 * This is the layout swa_decode reads (its W is n_slots).
 */
typedef struct swa_cache_params {
    void *k_cache;
    void *v_cache;
    int32_t *slot_pos;
    int32_t B, H_kv, d_h, n_slots, n_sink;
} swa_cache_params;

/*
 * Appends n_new tokens to every sequence: token i of sequence b has position
 * p0[b] + i and its rows k_new[b, i], v_new[b, i] (bf16 [B, n_new, H_kv, d_h],
 * contiguous) go to slot(p) of every kv head, with slot_pos set to p.  Tokens are
 * applied in order, so of two tokens mapping to one ring slot the later one stays.
 * p0: device int32 [B], each >= 0 (a negative entry skips that sequence and is
 * reported by swa_check_device_error as SWA_ERR_INVALID_ARG).
 * Requirements: d_h in {64, 128, 256}; 0 <= n_sink < n_slots; pointers 16-byte
 * aligned (slot_pos, p0: 4-byte); B * n_new * H_kv < 2^31 rows, else
 * SWA_ERR_UNSUPPORTED.  n_new = 0 is a no-op.
 */
SWA_API swa_status swa_cache_append(const swa_cache_params *c, const void *k_new, const void *v_new, int32_t n_new,
                            const int32_t *p0, swa_stream_t stream);

/*
 * Decode with the current token appended in the same pass: k_new, v_new (bf16
 * [B, H_kv, d_h], contiguous) are written to slot(q_pos[b]) of p->k_cache and
 * p->v_cache -- the slot rule of swa_cache_append with n_slots = p->W and n_sink =
 * p->n_sink -- slot_pos there is set to q_pos[b], and the query attends exactly as
 * swa_decode would after a separate swa_cache_append.  The caches and slot_pos are
 * written: they must be writable device memory.  Workspace as swa_decode.
 */
SWA_API swa_status swa_decode_append(const swa_decode_params *p, const void *k_new, const void *v_new,
                             void *workspace, size_t workspace_bytes, swa_stream_t stream);

/*
 * Chunked prefill against a ring cache: C new tokens per sequence, at positions
 * p0[b] .. p0[b] + C - 1, attend to the cached history and to the chunk itself; the
 * query at position t keeps the keys at positions t - window < p <= t (lizeman page,
 * section 2 window; the cache convention above) and, for a cache with n_sink pinned
 * sinks, the sink positions p < n_sink with p <= t (the rule of swa_decode).
 *   q            bf16 [B, C, H_q, d_h], contiguous
 *   k_new, v_new bf16 [B, C, H_kv, d_h], contiguous: the chunk's keys and values
 *   p0           device int32 [B]: position of each sequence's first chunk token
 *   o            bf16 [B, C, H_q, d_h]; lse fp32 [B, H_q, C]; row_counts optional [B, H_q, C]
 *   append       nonzero: afterwards append the chunk to the cache (swa_cache_append)
 * The cache must hold, for every sequence, every position in
 * [max(0, p0 - n_slots), p0) (with sinks: the sinks and the last n_slots - n_sink
 * positions) -- the tokens appended before the chunk; a slot found holding another
 * position is reported by swa_check_device_error as SWA_ERR_INVALID_ARG.
 * Requirements: the cache's B, H_kv, d_h match; window >= 1; H_q / H_kv <= 16; with
 * sinks, n_sink <= 128 and a ring of at least window - 1 slots (n_slots - n_sink);
 * B * (window - 1 + C + n_sink) * H_kv < 2^31 gathered rows; else SWA_ERR_UNSUPPORTED.  Workspace: swa_prefill_chunk_workspace_size bytes, 256-byte
 * aligned (the chunk's key/value rows and the window history gathered in position
 * order, and the sinks' rows).
 */
typedef struct swa_chunk_params {
    const void *q;
    const void *k_new;
    const void *v_new;
    const int32_t *p0;
    int32_t B, C, H_q, H_kv, d_h;
    int32_t window;
    float scale;
    void *o;
    float *lse;
    int32_t *row_counts;
    int32_t append;
} swa_chunk_params;

SWA_API size_t swa_prefill_chunk_workspace_size(const swa_chunk_params *p, const swa_cache_params *c);
SWA_API swa_status swa_prefill_chunk(const swa_chunk_params *p, const swa_cache_params *c, void *workspace,
                             size_t workspace_bytes, swa_stream_t stream);

/* Bytes of the built-in scratch array used by swa_decode_noalloc (16 MiB per device). */
#define SWA_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * swa_decode without a caller-provided workspace, for callers that cannot allocate
 * device memory where they call this: for example a serving loop that must not
 * allocate once it is running (cudaMalloc can synchronise the device and can fail
 * under memory pressure), or a plugin interface that hands the kernel only its
 * inputs and outputs.  The paper has no counterpart; this is a library convenience.
 *
 * The split partials go to one fixed scratch array of SWA_DECODE_NOALLOC_SCRATCH_BYTES
 * compiled into the library; every GPU that loads the library holds that array until
 * the process exits.  Nothing is allocated: no cudaMalloc, cudaFree or allocating
 * library routine is called.  The first call on each device looks up the array's
 * device address (with that device current) and caches it for the current CUDA
 * context, so make that first call before any stream capture -- and again first after
 * a device reset, whose new context holds the array at a new address.  All calls on a device share the array and it keeps the
 * previous call's contents (no part of it needs to start at zero); calls that overlap
 * on the GPU -- on different streams or host threads -- race on it and must be
 * serialised by the caller.  Parameters, layouts and results are those of swa_decode.
 * Errors: as swa_decode; SWA_ERR_WORKSPACE when the problem needs more scratch than
 * SWA_DECODE_NOALLOC_SCRATCH_BYTES (swa_decode_workspace_size(p) tells how much).
 */
SWA_API swa_status swa_decode_noalloc(const swa_decode_params *p, swa_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the library's device error words.
 * Returns SWA_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last
 * call, SWA_ERR_INVALID_ARG if a kernel found device data breaking its contract
 * (a global_idx list that is not strictly increasing within [0, T), a negative
 * append position, a cache slot not holding a position a chunked prefill needs),
 * SWA_ERR_CUDA if the synchronisation failed, else SWA_OK.
 * The words are per device and shared by every stream: this call synchronises only
 * `stream`, then reads and clears them for all work on the current device.  Work
 * still running on another stream may set them afterwards (a later call reports it),
 * and an error raised by another stream's work is reported to whichever call reads
 * first.  A caller that drives several streams should synchronise them all first.
 */
SWA_API swa_status swa_check_device_error(swa_stream_t stream);

/* Bits of the device error words (swa_device_errors). */
#define SWA_DEVERR_WAIT_TIMEOUT 1u  /* prefill, split: a bounded wait expired */
#define SWA_DEVERR_DRAIN_TIMEOUT 2u /* prefill, split: the exit path could not drain its copies in time */
#define SWA_DEVERR_GLOBAL_LIST 4u   /* prefill: global_idx not strictly increasing within [0, T) */
#define SWA_DEVERR_BAD_POSITION 1u  /* cache: a negative (or overflowing) append position */
#define SWA_DEVERR_CACHE_MISMATCH 2u /* cache: a slot not holding a position a chunked prefill needs */
#define SWA_DEVERR_BOUNDS 8u         /* any word, debug library only: an index outside its tensor (access skipped) */

/* The device error words, one per group of kernels. */
typedef struct swa_device_errors {
    uint32_t prefill; /* the band kernel of swa_fwd / swa_prefill_chunk */
    uint32_t split;   /* decode and the global-row pass of swa_fwd (split-K and merge) */
    uint32_t cache;   /* swa_cache_append, the history gather of swa_prefill_chunk */
} swa_device_errors;

/*
 * As swa_check_device_error (same synchronisation, same status), and also returns the
 * raw words it read and cleared in *out (may be NULL), for diagnosis: which group of
 * kernels failed and how.  SWA_DEVERR_BOUNDS is set only by the debug build of the
 * library (libswa_debug.so, compiled with -DSWA_DEBUG), whose kernels check every
 * computed gather, store and copy index against its tensor before the access and skip
 * the access when the check fails; it is reported as SWA_ERR_INVALID_ARG.  A wait that expired sets SWA_DEVERR_WAIT_TIMEOUT in the
 * CTA that gave up; the other roles of that CTA then stop without a timeout of their
 * own, and SWA_DEVERR_DRAIN_TIMEOUT means a copy or MMA was still outstanding when the
 * CTA left (a second fault, not a consequence of the first).
 */
SWA_API swa_status swa_read_device_errors(swa_stream_t stream, swa_device_errors *out);

/*
 * Failure detection without a GPU fault (test hook; the pages have no counterpart).
 * Makes the bounded-wait path above run on purpose: a producer that stops issuing
 * copies, so that the waits of the kernel's other roles run out (after the fixed bound
 * of about 2.1 s).  Nothing faults, traps or hangs: the kernel drains the copies it did
 * issue, frees its tensor memory, returns, and the next call works normally.
 *   band_stop_fill    the prefill kernel's K/V producer of every CTA issues no ring
 *                     fill numbered at or past this (fills are numbered 0, 1, ... per
 *                     CTA: K_0, V_0, K_1, V_1, ... of its units in order); -1 = off.
 *   split_stop_stage  the producer of every CTA of the decode / global-row split pass
 *                     emits no stage numbered at or past this (one stage per 64-slot
 *                     chunk streamed, numbered per CTA); -1 = off.
 * The plan is process-wide and read by every launch that follows; NULL (or -1, -1)
 * restores normal operation.  Outputs of a call that hit a planted stop are undefined.
 * Returns SWA_ERR_INVALID_ARG for a stop below -1.
 */
typedef struct swa_debug_faults {
    int32_t band_stop_fill;
    int32_t split_stop_stage;
} swa_debug_faults;
SWA_API swa_status swa_debug_set_faults(const swa_debug_faults *f);

/*
 * Description of the CUDA error behind the most recent SWA_ERR_CUDA returned to the
 * calling host thread ("no error" if none).  The string is static.
 */
SWA_API const char *swa_last_error_string(void);

/* Static description of a status code. */
SWA_API const char *swa_status_string(swa_status s);

/* ABI version of this header (incremented on any layout change). */
SWA_API int32_t swa_abi_version(void);

#define SWA_ABI_VERSION 2

#ifdef __cplusplus
}
#endif

#endif /* SWA_H */
