/*
 * amk_plan.h — the offline half of the decode MegaKernel, callable without a
 * GPU: build the tile-task DAG of one decode step, search its schedule
 * knobs, solidify it into per-SM task lists, and validate the result.
 *
 * Ada-MK technical summary (gist.science), Methodology, Phase I:
 *  - the step is decomposed into a fine-grained DAG that records RAW and WAR
 *    dependencies and resource constraints ("MLIR-Based Fine-Grained DAG
 *    Construction"; here the nodes are tile tasks built directly from the
 *    model configuration);
 *  - a shared-memory constraint model over hardware, model and workload
 *    bounds the feasible ring depth, and splitting the K dimension of a tile
 *    trades tile size against pipeline stages ("Adaptive Shared Memory
 *    Modeling");
 *  - an exhaustive search over the feasible space picks the execution trace,
 *    which is then solidified so that the kernel takes no runtime scheduling
 *    decisions ("Offline Search and Path Solidification").
 * AutoMegaKernel abstract: a schedule validator statically certifies
 * deadlock- and race-freedom and rejects unsafe schedules before launch; it
 * was evaluated on adversarial schedules.  amk_plan_mutate produces such
 * adversarial variants of a real plan for the same purpose.
 *
 * amk_create (amk.h) runs exactly this pipeline for the device it creates on.
 */
#ifndef AMK_PLAN_H
#define AMK_PLAN_H

#include "amk.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct amk_plan amk_plan;

/* Build, search and solidify the schedule for `batch` sequences on `n_sm`
 * persistent CTAs with `smem_per_cta` bytes of dynamic shared memory each
 * (sm_103a: 232448).  The plan is validated before it is returned; an
 * invalid plan is an AMK_ERR_SCHEDULE, with the reason in amk_plan_last_message.
 * options may be NULL. */
amk_status amk_plan_build(const amk_config *config, int32_t batch, int32_t n_sm, int32_t smem_per_cta,
                          const amk_schedule_options *options, amk_plan **out);

/* Re-run the validator (after amk_plan_mutate).  AMK_OK or AMK_ERR_SCHEDULE;
 * the reason is written to msg (NUL-terminated, truncated to msg_len). */
amk_status amk_plan_validate(const amk_plan *plan, char *msg, size_t msg_len);

amk_status amk_plan_get_info(const amk_plan *plan, amk_plan_info *info);

/* Number of tasks of CTA `sm`, and one task's fields:
 * out[0] op (0 QKV, 1 ATT, 2 OPR, 3 GUP, 4 DWN, 5 LMH, 6 MRG, 7 ARG), [1] layer, [2] r0, [3] r1,
 * [4] batch row, [5] kv head (MRG: query head), [6] the dependency the task waits on
 * (-1 none), [7] its number of producer tasks, [8] number of dependencies the task
 * produces for, [9..14] those dependencies, [15] QKV matrix (0 q, 1 k, 2 v).
 * A dependency is an id of the schedule graph that the validator checks: its
 * producers write a region of one activation buffer and its waiters read it.
 * The kernel keeps no counter for it: every word of the region carries the
 * epoch flag of the step and layer that wrote it, and a waiter polls the words
 * it reads until they carry the flag it expects. */
int32_t amk_plan_num_tasks(const amk_plan *plan, int32_t sm);
amk_status amk_plan_get_task(const amk_plan *plan, int32_t sm, int32_t idx, int32_t out[16]);

/* Adversarial mutation for validator tests.  kind:
 *   0 drop one signal (a dependency loses a producer)
 *   1 lower one wait count (a consumer may start before all producers)
 *   2 remove one wait (a consumer ignores its producers)
 *   3 move a consumer task in front of a producer on the same CTA (deadlock)
 *   4 redirect a wait to an unrelated dependency
 *   5 raise one wait count (a wait that can never be met)
 * `seed` picks the victim deterministically.  AMK_OK if a mutation was applied. */
amk_status amk_plan_mutate(amk_plan *plan, int32_t kind, uint64_t seed);

/* The search's task-level simulation of one decode step of a solidified
 * plan (Ada-MK summary, Methodology, Phase I: the offline search scores
 * candidate execution traces).  Every CTA's consumers run its tasks in order;
 * a task starts when its CTA is free and every producer of what it waits on
 * has finished, plus the hand-off latency; its tiles cannot finish before
 * the CTA's loader has streamed their bytes, in task order, at the CTA's
 * share of HBM and at most one ring ahead of what the consumers released.
 * consts: NULL for the built-in constants (fitted to GB300), or n_consts = 15
 * values in this order: [0] hand-off s, [1] RMSNorm prologue s, [2] copy
 * prologue s, [3] GEMV epilogue s, [4] batch-1 bf16 consumer bytes/s per
 * CTA, [5] int8 consumer bytes/s per CTA, [6] HBM bytes/s, [7] attention
 * prologue s, [8] attention s per (position, head, element), [9] attention
 * epilogue s, [10] merge s, [11] s per ring stage, [12] s of prologue per
 * further sequence at batch > 1, [13] most bytes/s one CTA's loader pulls,
 * [14] bf16 consumer bytes/s per CTA at batch > 1 (the tensor-core tile;
 * half of it above batch 8).  Any other n_consts is AMK_ERR_INVALID_ARG.
 * Writes the step time in microseconds to *step_us. */
amk_status amk_plan_simulate(const amk_plan *plan, const double *consts, int32_t n_consts, double *step_us);

/* Message of the last build/validate failure on this thread. */
const char *amk_plan_last_message(void);

void amk_plan_destroy(amk_plan *plan);

#ifdef __cplusplus
}
#endif
#endif /* AMK_PLAN_H */
