/*
 * amk_plan_impl.h — host-side representation of a solidified schedule.
 */
#pragma once
#include <stdint.h>

#include <string>
#include <vector>

#include "amk.h"
#include "amk_internal.h"

namespace amk {

/* Activation buffers whose accesses the validator tracks.  A buffer has
 * `depth` slots; the data of layer l lives in slot l % depth ("version" l). */
enum : uint8_t { BUF_XIN = 0, BUF_XMID, BUF_QKV, BUF_PART, BUF_AOUT, BUF_ACT, BUF_KVNEW, BUF_LOGITS, BUF_ARGP, BUF_NEXT,
                 BUF_COUNT };

/* One read or write of a rectangle [b0, b1) x [e0, e1) of (buffer, slot). */
struct Access {
    uint8_t buf, write;
    uint16_t slot;
    int32_t version;
    int32_t b0, b1;
    int64_t e0, e1;
};

struct Knobs {
    int C = 1;              /* attention context chunks per (sequence, kv head) */
    int slot_bytes = 16384; /* ring slot */
    int n_slots = 8;        /* ring depth */
    int ksplit = 1;         /* K split of GEMV tiles */
    int depth = 2;          /* scratch slots */
    int att_tile = 64;      /* positions per attention tile */
    int l2_prefetch_kb = 0;
    int evict_first = 1;    /* ring fills carry an L2 evict-first hint */
    int order = 0;          /* task placement: 0 attention chunks and merges spread over all CTAs in step;
                               1 merges on the CTAs that run no attention chunk (attention from the top) */
};

/* Constants of the task-level simulation (amk_plan_simulate); see amk_plan.h. */
constexpr int COST_NCONST = 15;
extern const double COST_DEFAULT[COST_NCONST];

/* Model geometry seen by the planner. */
struct Geo {
    int L, H, nq, nkv, d, I, V, G, qkv_rows, B, Smax;
    int wf, lm_wf, group; /* weight formats (WF_*) and the int4 scale group */
    int K(int op) const {
        return op == OP_OPR ? nq * d : op == OP_DWN ? I : H;
    }
    int rows(int op) const {
        return op == OP_QKV ? qkv_rows : op == OP_GUP ? I : op == OP_LMH ? V : H;
    }
    int nmat(int op) const { return op == OP_GUP ? 2 : 1; }
    int wf_of(int op) const { return op == OP_LMH ? lm_wf : wf; }
    /* bytes of k weights of `op` in its format */
    int64_t wbytes(int op, int64_t k) const { return wf_bytes(wf_of(op), k); }
    /* fp32 scales of one output row over k weights: int8 one, int4 one per group */
    int64_t row_scales(int op, int64_t k) const {
        return wf_of(op) == WF_I8 ? 1 : wf_of(op) == WF_I4 ? k / group : 0;
    }
    int64_t row_bytes(int op) const { return wbytes(op, K(op)) + 4 * row_scales(op, K(op)); }
};

Geo make_geo(const amk_config &c, int batch);
int ksplit_for(const Geo &g, int op, int ks);

}  // namespace amk

struct amk_plan {
    amk_config cfg;
    int batch = 0, n_sm = 0, smem_per_cta = 0;
    amk::Knobs k;
    std::vector<std::vector<amk::Task>> sm_tasks;
    std::vector<std::vector<std::vector<amk::Access>>> acc; /* parallel to sm_tasks */
    int n_counters = 0, n_levels = 0;
    int n_lmh = 0; /* LM-head tasks (each publishes one partial argmax per sequence) */
    int act_bytes = 0, result_bytes = 0, scale_bytes = 0, fac_bytes = 0, work_bytes = 0, smem_bytes = 0;
    int64_t weight_bytes = 0, scratch_bytes = 0;
    double modeled_us = 0, search_ms = 0, simulated_us = 0;
    int candidates = 0;
};

namespace amk {
/* Full pipeline: DAG + search + solidify + validate.  Returns AMK_OK or an error with *msg set. */
amk_status plan_build(const amk_config *cfg, int batch, int n_sm, int smem_per_cta,
                      const amk_schedule_options *opt, amk_plan **out, std::string *msg);
/* Deadlock- and race-freedom check; true if the plan is safe. */
bool plan_validate(const amk_plan &p, std::string *msg);
/* Task-level simulation of one step of a solidified plan (µs). */
double plan_simulate(const amk_plan &p, const double *c);
/* Element counts of the scratch buffers described in Params. */
struct ScratchSizes {
    int64_t x_in, x_mid, qkv, part, aout, act; /* 8-byte epoch-tagged words */
    int64_t argp;                              /* [Bmax][n_lmh][2]: LM-head partial argmaxes */
};
ScratchSizes scratch_sizes(const amk_plan &p);
}  // namespace amk
