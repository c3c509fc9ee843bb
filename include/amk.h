/*
 * amk.h — C ABI of the single-launch decode MegaKernel for GB300 (sm_103a).
 *
 * One call of amk_decode_step runs one autoregressive decode step of a
 * Llama-style decoder stack plus LM head (RMSNorm, QKV GEMV, RoPE, KV-cache
 * attention, O projection + residual, RMSNorm, SwiGLU gate/up/down + residual,
 * final norm, LM-head logits) as ONE persistent kernel launch, with no
 * inter-operator kernel boundary.  This is the MegaKernel of the Ada-MK
 * technical summary (gist.science, "Problem Statement": fuse operators into a
 * single persistent kernel to remove launch overhead and inter-operator HBM
 * round trips; "Methodology", Phase I: the fused scope is the Transformer
 * decoder and the LM head; Phase II: the engine switches to the MegaKernel for
 * the decode phase only, so prefill and the KV cache belong to the caller).
 *
 * amk_create also runs the offline part of that method once per fixed
 * configuration: it decomposes the step into a tile-task DAG with RAW/WAR
 * dependencies, searches task order, context split, K split and pipeline
 * depth against a shared-memory model of the device (Ada-MK summary,
 * Methodology, "Adaptive Shared Memory Modeling" and "Offline Search and Path
 * Solidification"), solidifies the result into a static per-SM task table,
 * and checks it for deadlock- and race-freedom before it is ever launched
 * (the schedule validator of the AutoMegaKernel abstract).
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" must point to device memory of the current
 *    CUDA device; "host" pointers are read during the call only.
 *  - No call throws; every call returns an amk_status.
 *  - A handle is used from one host thread / one stream at a time.
 *  - Nothing here falls back to the CPU: without a usable sm_103a device,
 *    amk_create fails with AMK_ERR_CUDA or AMK_ERR_UNSUPPORTED.
 */
#ifndef AMK_H
#define AMK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *amk_stream_t; /* the same type as cudaStream_t; NULL = legacy default stream */

typedef enum amk_status {
    AMK_OK = 0,
    AMK_ERR_INVALID_ARG = 1,  /* a NULL, misaligned or out-of-range argument */
    AMK_ERR_UNSUPPORTED = 2,  /* a shape or device this build does not handle */
    AMK_ERR_CUDA = 3,         /* a CUDA runtime call failed */
    AMK_ERR_OOM = 4,          /* device or host allocation failed */
    AMK_ERR_SCHEDULE = 5,     /* the validator rejected the solidified schedule */
    AMK_ERR_COOPERATIVE = 6,  /* one CTA per SM cannot be co-resident; nothing was launched */
    AMK_ERR_TIMEOUT = 7       /* a device-side wait gave up; see amk_last_error */
} amk_status;

typedef enum amk_weight_dtype {
    AMK_WEIGHT_BF16 = 0, /* bf16 matrices */
    AMK_WEIGHT_INT8 = 1, /* W8A16: int8 matrices, one fp32 scale per output row, bf16 activations */
    AMK_WEIGHT_INT4 = 2  /* W4A16 (Ada-MK summary, Key Contributions): 4-bit codes u in 0..15, value
                            scale * (u - 8), two codes per byte with element 2j in the low nibble of byte j;
                            one fp32 scale per group_size weights along K ([out][in / group_size]); bf16
                            activations; batch 1 only (max_batch = 1) */
} amk_weight_dtype;

/* Model and capacity.  head_dim must be 64 or 128 and even; n_heads a
 * multiple of n_kv_heads; hidden, n_heads*head_dim and intermediate multiples
 * of 16 (so that every weight row is a whole number of 16-byte units). */
typedef struct amk_config {
    int32_t n_layers;
    int32_t hidden;        /* H */
    int32_t n_heads;       /* query heads */
    int32_t n_kv_heads;    /* key/value heads (GQA groups) */
    int32_t head_dim;      /* d */
    int32_t intermediate;  /* I (SwiGLU) */
    int32_t vocab;         /* V */
    float rms_eps;
    float rope_theta;      /* RoPE base; rotate-half pairs (i, i + d/2) */
    int32_t max_batch;     /* 1..16 sequences per step */
    int32_t max_seq;       /* KV-cache capacity per sequence (Smax) */
    int32_t weight_dtype;  /* amk_weight_dtype */
    int32_t tied_embeddings; /* 1: the LM head is the bf16 embedding matrix */
    int32_t group_size;    /* AMK_WEIGHT_INT4: weights per scale along K, a multiple of 32 dividing hidden,
                              n_heads*head_dim and intermediate; 0: 128.  Ignored for other formats. */
} amk_config;

/* Device pointers of one layer, each matrix [out, in] row-major, rows
 * 16-byte aligned.  The s_* scales (fp32) are read only for the scaled
 * formats: one per output row for AMK_WEIGHT_INT8, [out][in / group_size]
 * for AMK_WEIGHT_INT4.  Norm gains are bf16 [H]. */
typedef struct amk_layer_weights {
    const void *attn_norm, *mlp_norm;
    const void *wq;     /* [n_heads*d, H]    */
    const void *wk;     /* [n_kv_heads*d, H] */
    const void *wv;     /* [n_kv_heads*d, H] */
    const void *wo;     /* [H, n_heads*d]    */
    const void *w_gate; /* [I, H] */
    const void *w_up;   /* [I, H] */
    const void *w_down; /* [H, I] */
    const float *s_q, *s_k, *s_v, *s_o, *s_gate, *s_up, *s_down;
} amk_layer_weights;

/* Whole-model weights.  `layers` is a HOST array of n_layers entries whose
 * members are device pointers.  embed is bf16 [V, H]; lm_head is [V, H] in
 * the weight dtype (ignored when tied_embeddings); s_lm its scales (int8: [V];
 * int4: [V][H / group_size]).
 * The caller keeps every weight allocated and unchanged while the handle
 * lives; the handle copies only the pointers. */
typedef struct amk_weights {
    const void *embed;
    const void *final_norm;
    const void *lm_head;
    const float *s_lm;
    const amk_layer_weights *layers;
} amk_weights;

/* Overrides for the offline search; 0 in a field means "search chooses".
 * Offline profiling can pin a measured-best point here (Ada-MK summary,
 * Contribution 2: offline profiling solidifies the path). */
typedef struct amk_schedule_options {
    int32_t n_sm;            /* persistent CTAs (<= SM count); 0: every SM */
    int32_t att_chunks;      /* context chunks per (sequence, kv head) */
    int32_t slot_bytes;      /* bytes per shared-memory ring slot (multiple of 1024) */
    int32_t n_slots;         /* ring depth (pipeline stages) */
    int32_t ksplit;          /* K-dimension split of GEMV tiles (1, 2, 4) */
    int32_t scratch_depth;   /* layers of activation scratch kept before reuse (>= 1) */
    int32_t l2_prefetch_kb;  /* KB each CTA's loader prefetches into L2 ahead of its ring fills, only while
                                the ring is full; 0 or -1: none (the default; it measured slower).  Only a
                                library built with AMK_L2_PREFETCH=1 accepts a positive value; the default
                                build leaves the code out and returns AMK_ERR_UNSUPPORTED. */
    int32_t trace;           /* 1: record per-task timestamps of every step (amk_debug_read_trace).  Only a
                                library built with the timing code (AMK_TRACE=1 at build time) accepts it;
                                the default build returns AMK_ERR_UNSUPPORTED. */
    int64_t wait_timeout_ns; /* bound on every device-side wait; 0: 1 s */
    int32_t l2_evict_first;  /* 1 or 0 (the default): ring fills carry an L2 evict-first hint, so that the
                                once-per-step weight and KV stream does not push code and activation scratch
                                out of L2; -1: no hint.  Results are identical either way. */
    int32_t task_order;      /* placement of attention chunks and merges: 0 the search chooses (by the
                                task-level simulation), 1 both spread over all CTAs in step, 2 merges on the
                                CTAs that run no attention chunk (chunks filled from the top) */
} amk_schedule_options;

typedef struct amk_handle amk_handle;

/* Builds, validates and uploads the schedule; copies the weight pointers.
 * options may be NULL.  On success *out owns device memory for the task
 * table, the epoch and error words, the RoPE table and the activation
 * scratch (released by amk_destroy).  Errors: INVALID_ARG (NULL/misaligned/inconsistent),
 * UNSUPPORTED (shape or device), SCHEDULE (validator), COOPERATIVE, CUDA, OOM. */
amk_status amk_create(const amk_config *config, const amk_weights *weights,
                      const amk_schedule_options *options, amk_handle **out);

/* One decode step for `batch` (1..max_batch) sequences, enqueued on `stream`
 * as a single cooperative kernel launch; returns without synchronising.
 *   tokens    device int32 [batch]: the token each sequence consumes;
 *   positions device int32 [batch]: its position p (0 <= p < max_seq);
 *             the step writes K/V at p and attends over positions 0..p;
 *   kv_cache  device bf16, the K cache followed by the V cache, each laid out
 *             [n_layers][max_batch][n_kv_heads][max_seq][head_dim];
 *             positions < p of every sequence must hold its prefix;
 *   logits    device fp32 [batch][vocab], written by the step.
 * Argument errors are returned at once; a device-side timeout is reported by
 * the next amk_sync_status, and steps launched after it do no work.
 * The step's epoch (the tag that tells this step's activation words from
 * older ones) lives in handle-owned device memory and is advanced by the
 * kernel itself, so launches of this call may be captured in a CUDA graph
 * and the graph replayed: every replay is a new step.  The steps of one
 * handle must still run one after another (one stream, or a graph whose
 * steps are chained). */
amk_status amk_decode_step(amk_handle *h, int32_t batch, const int32_t *tokens,
                           const int32_t *positions, void *kv_cache, float *logits,
                           amk_stream_t stream);

/* Greedy decoding on the device: one decode step as amk_decode_step which,
 * in the same launch, also reduces each sequence's logits to its greedy
 * token, the argmax over the vocabulary with the lowest index winning ties
 * (the AutoMegaKernel abstract reproduces greedy decode token for token),
 * and writes the inputs of the next step:
 *   next_tokens    device int32 [batch]: argmax of row b of `logits`;
 *   next_positions device int32 [batch]: positions[b] + 1.
 * They must not alias tokens / positions (the step reads those throughout);
 * ping-pong two pairs of buffers, e.g. in a CUDA graph of two steps, and the
 * host is needed only to read tokens back.  Errors as amk_decode_step, plus
 * AMK_ERR_INVALID_ARG for NULL, misaligned or aliasing next_* pointers. */
amk_status amk_decode_step_greedy(amk_handle *h, int32_t batch, const int32_t *tokens,
                                  const int32_t *positions, void *kv_cache, float *logits,
                                  int32_t *next_tokens, int32_t *next_positions,
                                  amk_stream_t stream);

/* A decode step that allocates nothing, for callers that cannot allocate
 * device memory (an external allocator owns the device, or allocation is
 * forbidden after start-up).  The method's pages have no counterpart: it is a
 * deployment variant of amk_decode_step.  Instead of a handle, every call
 * takes the configuration and the weights (as in amk_create, with default
 * schedule options) and keeps the schedule, RoPE table, error word and
 * activation scratch in one static device array of 16 MiB per device.
 *   - The first call on a device, with that device current, looks up the
 *     array's address (cudaGetSymbolAddress) and clears it; make that first
 *     call before any stream capture.  A call whose configuration or weight
 *     pointers differ from the previous call's re-plans and re-uploads.
 *   - A configuration whose state does not fit in 16 MiB is refused with
 *     AMK_ERR_UNSUPPORTED (the needed size is printed to stderr).
 *   - tokens, positions, kv_cache, logits and stream are as in
 *     amk_decode_step.  The call waits for the step to finish and returns
 *     AMK_ERR_TIMEOUT or AMK_ERR_INVALID_ARG for a device-side failure
 *     (AMK_ERR_CUDA if the error word then cannot be cleared).  It runs the
 *     same kernel on the same default schedule as a handle created with
 *     options = NULL, so its logits and K/V slots are bit-identical to
 *     amk_decode_step's on the same inputs.
 *   - All calls share the array: calls are serialised by a process-wide lock;
 *     calls that overlapped on the GPU would race.  A call blocks on `stream`
 *     (cudaStreamSynchronize) while it holds that lock, so it must not be
 *     made from a stream callback or host function, nor while `stream` waits
 *     on work that another thread's call would enqueue. */
amk_status amk_decode_step_noalloc(const amk_config *config, const amk_weights *weights,
                                   int32_t batch, const int32_t *tokens,
                                   const int32_t *positions, void *kv_cache,
                                   float *logits, amk_stream_t stream);

/* Synchronises the stream of the last step and reads the device error word.
 * Returns AMK_ERR_TIMEOUT if any wait of any step since the last call gave up
 * (then the error word is cleared, so the next step runs normally: the
 * failed step still advanced the device epoch, so none of its words can pass
 * for the next step's). */
amk_status amk_sync_status(amk_handle *h);

/* Frees everything the handle owns (synchronises first).  NULL is accepted. */
amk_status amk_destroy(amk_handle *h);

/* Static description of a status code. */
const char *amk_status_string(amk_status s);

/* What the last failed wait saw (filled by amk_sync_status on a timeout). */
typedef struct amk_error_info {
    int32_t code;        /* 1 dependency (an activation word never became current), 2 ring full barrier,
                            3 ring empty barrier, 4 out-of-range token or position */
    int32_t sm;          /* CTA that gave up */
    int32_t task;        /* index of its task in that CTA's list (-1: none) */
    int32_t counter;     /* code 1: which activation buffer the wait polled: 0 residual at a layer's input,
                            1 residual after attention, 2 q/k/v, 3 attention chunk partials, 4 attention
                            output, 5 SwiGLU output, 6 LM-head partial argmaxes; else -1 */
    uint32_t observed;   /* code 1: the epoch flag the stale word carried; codes 2, 3: 0 */
    uint32_t target;     /* code 1: the flag awaited (epoch * (n_layers + 1) + layer); codes 2, 3: the
                            barrier phase parity awaited */
} amk_error_info;
amk_status amk_last_error(const amk_handle *h, amk_error_info *info);

/* Summary of the solidified schedule of a handle or a plan. */
typedef struct amk_plan_info {
    int32_t n_sm, n_tasks;
    int32_t n_counters;       /* dependency ids of the schedule graph (what the validator checks; the
                                 kernel keeps no counters: it polls epoch-tagged words) */
    int32_t n_levels;
    int32_t att_chunks, slot_bytes, n_slots, ksplit, scratch_depth, att_tile;
    int32_t smem_bytes;       /* dynamic shared memory per CTA */
    int32_t max_tasks_per_sm;
    int64_t weight_bytes;     /* linear-weight bytes streamed per step (incl. int8 scales) */
    int64_t scratch_bytes;    /* device activation scratch */
    double modeled_us;        /* the analytic per-level model's estimate for one step */
    double search_ms;         /* host time of DAG build + search + solidify + validate */
    int32_t candidates;       /* schedule points the search evaluated (analytic + simulated) */
    int32_t l2_evict_first;   /* 1 if ring fills carry the L2 evict-first hint */
    double simulated_us;      /* the task-level simulation's step time for the chosen plan */
    int32_t task_order;       /* the chosen placement (task_order values of amk_schedule_options) */
} amk_plan_info;
amk_status amk_get_plan_info(const amk_handle *h, amk_plan_info *info);

/* Test support: make task `task` of CTA `sm` skip its completion signal, so
 * that the waits depending on it run into their timeout.  sm = -1 clears. */
amk_status amk_debug_drop_signal(amk_handle *h, int32_t sm, int32_t task);

/* Test support: copy the residual stream of the last step to host memory.
 * Needs a handle created with scratch_depth = n_layers + 1, so that no layer's
 * scratch is reused within a step (else AMK_ERR_UNSUPPORTED).  x_in receives
 * [n_layers + 1][max_batch][hidden] fp32: entry l is the input of layer l
 * (entry 0 is not written by the kernel: layer 0 reads the token's embedding
 * row) and entry n_layers the input of the final norm; x_mid receives
 * [n_layers][max_batch][hidden], the residual after each layer's attention.
 * Synchronises the device first. */
amk_status amk_debug_read_residuals(const amk_handle *h, float *x_in, float *x_mid);

/* Test and tuning support: per-task timings of the last step of a handle
 * created with options.trace = 1 (else AMK_ERR_UNSUPPORTED).  For every task
 * of every CTA, in CTA order then task order, sixteen uint64 entries:
 * globaltimer times (ns) [0] task start ([1] repeats it), [2] first tile
 * arrived, [3] end (after the completion signal), [6] inputs met and
 * prologue done, [7] last tile consumed, [8] epilogue written; durations (ns)
 * [4] consumer warp 0 waiting for tiles, [5] consumer warp 0 computing tiles,
 * [9] the loader waiting for free ring slots while issuing the task's tiles;
 * other entries are unused (0).  `out` holds n_tasks * 16 entries (n_tasks
 * from amk_get_plan_info); synchronises the device first. */
amk_status amk_debug_read_trace(const amk_handle *h, uint64_t *out, size_t n_entries);

#ifdef __cplusplus
}
#endif
#endif /* AMK_H */
