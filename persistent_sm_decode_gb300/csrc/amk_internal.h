/*
 * amk_internal.h — the solidified schedule as the kernel reads it, and the
 * kernel's launch parameters.  Shared by the host planner (amk_plan.cpp),
 * the C ABI (amk_api.cpp) and the persistent kernel (amk_kernel.cu).
 */
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define AMK_HD __host__ __device__
#else
#define AMK_HD
#endif

namespace amk {

/* Task kinds: one per operator of the decode step.  QKV, OPR, GUP, DWN and
 * LMH are row blocks of a GEMV (each fused with its prologue/epilogue),
 * ATT is one context chunk of one (sequence, kv head). */
enum : uint8_t { OP_QKV = 0, OP_ATT = 1, OP_OPR = 2, OP_GUP = 3, OP_DWN = 4, OP_LMH = 5, OP_COUNT = 6 };

enum : uint8_t {
    TF_SKIP_SIGNAL = 1u, /* debug: do not signal on completion (timeout tests) */
    TF_NEW_TOKEN = 2u    /* ATT: this chunk holds position p; it writes K/V slot p */
};

/* QKV tasks stay inside one of the three matrices; `mat` says which. */
enum : uint8_t { MAT_Q = 0, MAT_K = 1, MAT_V = 2 };

constexpr uint16_t NO_WAIT = 0xFFFFu;
constexpr int MAX_SIG = 6;
constexpr int NCW = 8;                    /* consumer warps per CTA */
constexpr int NTHREADS = (NCW + 1) * 32;  /* + one loader warp */
constexpr int MAXB = 8;                   /* sequences per step */
constexpr int COUNTER_STRIDE = 32;        /* uint32 words per counter: one 128-byte line each */
constexpr int MAX_SLOTS = 32;
constexpr int PART_PAD = 4;               /* attention partial: o[d], m, l, 2 pad floats */
constexpr int ERR_WORDS = 8;

/* One task of a CTA's static list (48 bytes). */
struct Task {
    uint8_t op;
    uint8_t flags;
    uint16_t layer;
    int32_t r0, r1;          /* GEMV: output rows [r0, r1) within matrix `mat` (QKV) or the op;
                                ATT: r0 = chunk index c, r1 = number of chunks C */
    uint16_t b, g;           /* ATT: sequence and kv head */
    uint16_t rows_per_stage; /* GEMV: rows per ring slot; ATT: positions per tile */
    uint8_t ksplit;          /* GEMV: K split (k-outer loop over ksplit slices) */
    uint8_t nsig;            /* number of valid entries of sig[] */
    uint16_t wait_id;        /* counter awaited before the task reads its inputs, or NO_WAIT */
    uint8_t mat;             /* QKV: MAT_Q/K/V */
    uint8_t pad0;
    uint32_t wait_count;     /* producers of wait_id per step (target = epoch * wait_count) */
    uint16_t sig[MAX_SIG];   /* counters incremented once the task's writes are visible */
    uint32_t pad1[2];
};
static_assert(sizeof(Task) == 48, "Task layout");

/* Device pointers of one layer. */
struct LayerPtrs {
    const void *w[7];        /* wq, wk, wv, wo, w_gate, w_up, w_down */
    const float *s[7];       /* int8 row scales, same order */
    const uint16_t *attn_norm, *mlp_norm;
};
enum : int { W_Q = 0, W_K = 1, W_V = 2, W_O = 3, W_GATE = 4, W_UP = 5, W_DOWN = 6 };

/* Everything the persistent kernel needs, passed by value. */
struct Params {
    /* model */
    int L, H, nq, nkv, d, I, V, G, Bmax, Smax, qkv_rows;
    float eps;
    float qk_scale_log2;     /* log2(e) / sqrt(d) */
    int wint8, lm_int8;
    /* schedule */
    const Task *tasks;
    const int32_t *task_start; /* [n_sm + 1] */
    int C, depth, slot_bytes, n_slots, att_tile;
    int act_bytes, result_bytes, scale_bytes;
    int l2_prefetch_bytes;
    /* weights */
    const LayerPtrs *layers;
    const uint16_t *embed, *final_norm;
    const void *lm;
    const float *s_lm;
    /* scratch (device, handle-owned) */
    float *x_in;     /* [depth][Bmax][H]   residual at a layer's input (slot l % depth) */
    float *x_mid;    /* [depth][Bmax][H]   residual after attention */
    float *qkv;      /* [depth][Bmax][qkv_rows] */
    float *part;     /* [depth][Bmax][nkv][C][G][d + PART_PAD] */
    uint16_t *act;   /* [depth][Bmax][I]   SwiGLU output, bf16 */
    uint32_t *counters;
    uint32_t *err;   /* [ERR_WORDS] */
    const float *rope;  /* [Smax][d/2][2]: cos, sin of position * theta^(-2i/d) */
    /* step */
    const int32_t *tokens, *positions;
    uint16_t *kc, *vc;   /* [L][Bmax][nkv][Smax][d] */
    float *logits;       /* [batch][V] */
    int batch;
    uint32_t epoch;
    long long timeout_ns;
};

/* shared-memory layout (bytes), common to host sizing and device carving */
constexpr int SMEM_BARRIERS = 2 * MAX_SLOTS * 8;
constexpr int SMEM_MISC = 1024;

AMK_HD inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

}  // namespace amk
