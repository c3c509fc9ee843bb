/*
 * amk_unfused.h — the decode step as one kernel launch per operator, for
 * comparison with amk_decode_step on the same device and data.
 *
 * The Ada-MK abstract counts kernel launches and inter-operator HBM round
 * trips among the costs of per-operator decode that the MegaKernel removes,
 * and the AutoMegaKernel abstract measures its fused kernel against
 * CUDA-graphed per-operator kernels.  This entry point is that per-operator
 * form: embedding, then per layer RMSNorm, the QKV GEMV, RoPE with the K/V
 * store, attention (split over the context into about two blocks per SM,
 * then a merge launch), the O projection, the residual add, RMSNorm, the
 * gate/up GEMV, SwiGLU, the down projection and the residual add, then the
 * final RMSNorm and the LM head; each a separate launch reading its inputs
 * from and writing its outputs to global memory (13 launches per layer plus
 * 3).  Its arithmetic follows the same definition as amk_decode_step (bf16 or
 * int8-with-row-scale weights, bf16 GEMV inputs and KV cache, fp32 sums,
 * residual and logits), so its logits meet the same tolerance against the
 * reference; they are not bit-identical to amk_decode_step's.
 *
 * Argument meanings, layouts and ownership are those of amk_create and
 * amk_decode_step (include/amk.h); max_batch may be 1..16.  The step only
 * launches kernels on `stream`, so it may be captured in a CUDA graph.
 */
#ifndef AMK_UNFUSED_H
#define AMK_UNFUSED_H

#include "amk.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct amk_unfused amk_unfused;

/* Allocates the handle's activation buffers, attention partials and RoPE
 * table (device);
 * copies the weight pointers.  Errors: INVALID_ARG, UNSUPPORTED, OOM, CUDA. */
amk_status amk_unfused_create(const amk_config *config, const amk_weights *weights, amk_unfused **out);

/* Enqueues one decode step (13 launches per layer plus 3) on `stream`;
 * arguments as amk_decode_step.  Launch errors come back as AMK_ERR_CUDA. */
amk_status amk_unfused_decode_step(amk_unfused *u, int32_t batch, const int32_t *tokens, const int32_t *positions,
                                   void *kv_cache, float *logits, amk_stream_t stream);

/* Frees the handle (NULL accepted). */
amk_status amk_unfused_destroy(amk_unfused *u);

#ifdef __cplusplus
}
#endif
#endif /* AMK_UNFUSED_H */
