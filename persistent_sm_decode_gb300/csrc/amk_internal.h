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
 * ATT is one context chunk of one (sequence, kv head), MRG merges the chunks
 * of one (sequence, kv head) into its heads' attention output.  ARG reduces
 * the LM-head tasks' partial argmaxes to each sequence's greedy token (run
 * only by the greedy entry point). */
enum : uint8_t { OP_QKV = 0, OP_ATT = 1, OP_OPR = 2, OP_GUP = 3, OP_DWN = 4, OP_LMH = 5, OP_MRG = 6, OP_ARG = 7,
                 OP_COUNT = 8 };

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
constexpr int MAXB = 16;                  /* sequences per step (the M of one tensor-core tile) */
constexpr int MAX_SLOTS = 32;
constexpr int PART_PAD = 4;               /* attention partial: o[d], m, l, 2 pad floats */
constexpr int ERR_WORDS = 8;

/* One task of a CTA's static list (48 bytes). */
struct Task {
    uint8_t op;
    uint8_t flags;
    uint16_t layer;
    int32_t r0, r1;          /* GEMV: output rows [r0, r1) within matrix `mat` (QKV) or the op;
                                ATT: r0 = chunk index c, r1 = number of chunks C; MRG: r1 = C;
                                ARG: r1 = number of LM-head tasks */
    uint16_t b, g;           /* ATT, MRG: sequence and kv head; LMH: g = index of the LM-head task */
    uint16_t rows_per_stage; /* GEMV: rows per ring slot; ATT: positions per tile */
    uint8_t ksplit;          /* GEMV: K split (k-outer loop over ksplit slices) */
    uint8_t nsig;            /* number of valid entries of sig[] */
    uint16_t wait_id;        /* dependency the task waits on (the producers of the region it reads), or NO_WAIT */
    uint8_t mat;             /* QKV: MAT_Q/K/V */
    uint8_t seg;             /* GEMV: K segments per row (consumer warps per row), 1, 2, 4 or 8 */
    uint32_t wait_count;     /* number of producers of wait_id */
    uint16_t sig[MAX_SIG];   /* dependencies the task's outputs take part in; the kernel realises a
                                dependency as epoch-tagged words that its consumers poll */
    uint32_t pad1[2];
};
static_assert(sizeof(Task) == 48, "Task layout");

/* Device pointers of one layer. */
struct LayerPtrs {
    const void *w[7];        /* wq, wk, wv, wo, w_gate, w_up, w_down */
    const float *s[7];       /* int8 row scales or int4 group scales [rows][K / group], same order */
    const uint16_t *attn_norm, *mlp_norm;
};
enum : int { W_Q = 0, W_K = 1, W_V = 2, W_O = 3, W_GATE = 4, W_UP = 5, W_DOWN = 6 };

/* Everything the persistent kernel needs, passed by value. */
struct Params {
    /* model */
    int L, H, nq, nkv, d, I, V, G, Bmax, Smax, qkv_rows;
    float eps;
    float qk_scale_log2;     /* log2(e) / sqrt(d) */
    int wf, lm_wf;       /* weight format of the layer matrices and of the LM head (WF_*) */
    int group;           /* WF_I4: weights per scale along K */
    /* schedule */
    const Task *tasks;
    const int32_t *task_start; /* [n_sm + 1] */
    int C, depth, slot_bytes, n_slots, att_tile;
    int act_bytes, result_bytes, scale_bytes, fac_bytes;
    int work_bytes; /* the per-task region: GEMV sums + scales + activations, or attention state, or merge sums */
    int l2_prefetch_bytes;
    int evict_first; /* 1: ring fills carry an L2 evict-first hint: weights and the cached prefix are read once
                        per step, while code, scratch and tables are reused every layer */
    /* weights */
    const LayerPtrs *layers;
    const uint16_t *embed, *final_norm;
    const void *lm;
    const float *s_lm;
    /* scratch (device, handle-owned).  Every word is {payload, flag}: the low
     * 32 bits hold an fp32 value or two bf16 values, the high 32 bits the flag
     * epoch * (L + 1) + version, where version is the layer whose data the
     * word holds (x_in: the layer it is the input of).  A consumer polls the
     * words it needs until they carry the flag of the current step and
     * version: the data is its own dependency flag, and neither an older step
     * nor another layer sharing the slot can be mistaken for it. */
    uint64_t *x_in;   /* [depth][Bmax][H]         residual at a layer's input, fp32 */
    uint64_t *x_mid;  /* [depth][Bmax][H]         residual after attention, fp32 */
    uint64_t *qkv;    /* [depth][Bmax][qkv_rows]  fp32 */
    uint64_t *part;   /* [depth][Bmax][nkv][C][G][d + PART_PAD]  chunk partials, fp32 */
    uint64_t *aout;   /* [depth][Bmax][nq * d / 2]  attention output, bf16 pairs */
    uint64_t *act;    /* [depth][Bmax][I / 2]       SwiGLU output, bf16 pairs */
    uint32_t *err;    /* [ERR_WORDS] */
    const float *rope;  /* [Smax][d/2][2]: cos, sin of position * theta^(-2i/d) */
    /* step */
    const int32_t *tokens, *positions;
    uint16_t *kc, *vc;   /* [L][Bmax][nkv][Smax][d] */
    float *logits;       /* [batch][V] */
    int batch;
    uint32_t epoch;      /* the step's epoch when epoch_word is NULL; flags of the step are
                            epoch * (L + 1) + version */
    uint32_t *epoch_word; /* device [2]: the epoch of the next step, and how many CTAs have finished the
                             current one.  Every CTA reads word 0 at start; the last CTA to finish
                             advances it.  Keeping the epoch on the device lets a captured CUDA graph
                             replay steps: a kernel argument would repeat the same epoch. */
    /* greedy feedback (NULL: none): next_tokens[b] = argmax of row b of the logits (lowest index on
     * ties), next_positions[b] = positions[b] + 1 */
    int32_t *next_tokens, *next_positions;
    uint64_t *argp;      /* [Bmax][n_lmh][2] tagged partial argmax (value, index) of each LM-head task */
    int n_lmh;           /* LM-head tasks of the schedule */
    long long timeout_ns;
    unsigned long long *trace; /* NULL, or [n_tasks][16] timings */
};

/* Weight formats: bf16; int8 with one fp32 scale per output row (W8A16);
 * 4-bit codes around the zero point 8, two per byte (element 2j in the low
 * nibble of byte j), with one fp32 scale per `group` weights along K
 * (W4A16).  A 16-byte chunk holds wf_epc weights. */
enum : int { WF_BF16 = 0, WF_I8 = 1, WF_I4 = 2 };
AMK_HD constexpr int wf_epc(int wf) { return wf == WF_BF16 ? 8 : wf == WF_I8 ? 16 : 32; }
AMK_HD constexpr long long wf_bytes(int wf, long long k) { return k * 16 / wf_epc(wf); }

/* Batch-1 GEMV.  A task's prologue writes the bf16 activations of its K
 * slice to shared memory once; then every consumer warp copies the part it
 * multiplies into registers.  A row of the K slice is cut into S segments
 * (1, 2, 4 or 8): warp w owns segment w % S for the whole task, holding its
 * activations as J 16-byte chunks per lane (chunk c of the segment in lane
 * c % 32, slot c / 32), and the 8 / S warps that share a segment take turns
 * over the rows of every tile, RPG1 rows at a time.  A lane carries its sums
 * across the whole segment, so a warp reduces once per row and segment.  J is
 * a loop bound, not a template parameter: the loop is unrolled to JMAX with
 * a warp-uniform guard, so one code instance serves every K (each task type
 * runs once per layer from a cold instruction cache, and its code size is
 * what that costs).  S is the fewest segments that keep J <= JMAX, raised
 * while a tile has too few rows to give every warp work. */
constexpr int JMAX_BF16 = 8;
constexpr int JMAX_INT8 = 2;
constexpr int JMAX_INT4 = 2;
constexpr int RPG1 = 1;
AMK_HD constexpr int wf_jmax(int wf) { return wf == WF_BF16 ? JMAX_BF16 : wf == WF_I8 ? JMAX_INT8 : JMAX_INT4; }

/* chunks per lane J of a batch-1 segment (0: the slice is too long) */
AMK_HD inline int gemv_lane_chunks(int Kc, int S, int wf) {
    const int nch = Kc / wf_epc(wf);
    const int per = (nch + S - 1) / S;
    const int J = (per + 31) / 32;
    return J > wf_jmax(wf) ? 0 : J;
}

/* K segments per row.  Batch 1 as above.  Larger batches read activations
 * from shared memory: bf16 weights go through the tensor cores with each of
 * the 8 warps taking one K segment of every row block (S = 8); int8 weights
 * use the CUDA-core tile with 8 / rows_per_stage segments when a tile has
 * fewer than 8 rows. */
AMK_HD inline int gemv_segments(int batch_max, int Kc, int wf, int rows_per_stage) {
    if (batch_max > 1 && wf == WF_BF16) return NCW;
    if (batch_max == 1) {
        int S = 1;
        while (S < NCW && gemv_lane_chunks(Kc, S, wf) == 0) S *= 2;
        /* every warp gets rows: (8 / S) row groups of RPG1 rows per round */
        while (S < NCW && rows_per_stage < (NCW / S) * RPG1) S *= 2;
        return S;
    }
    return rows_per_stage < NCW ? NCW / rows_per_stage : 1;
}

/* Rows of stage rb of a GEMV task of n rows cut into nst stages: the rows are
 * spread evenly over the stages (the loader and the consumers agree). */
AMK_HD inline void stage_rows(int n, int nst, int rb, int &a, int &e) {
    a = (int)((long long)rb * n / nst);
    e = (int)((long long)(rb + 1) * n / nst);
}

/* Attention: positions per warp block; q heads per kv head rounded up to a
 * power of two; chunk partials one merge thread can hold. */
constexpr int ATT_BP = 16;
constexpr int MRG_MAX_CPT = 2;
AMK_HD inline int att_gp(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8; }
/* most context chunks the merge supports: (threads / (d/4)) * MRG_MAX_CPT */
AMK_HD inline int att_max_chunks(int d) { return (NCW * 32 / (d / 4)) * MRG_MAX_CPT; }

/* shared-memory layout (bytes), common to host sizing and device carving */
constexpr int SMEM_BARRIERS = 2 * MAX_SLOTS * 8;
constexpr int SMEM_MISC = 2048;

/* At batch above 1, every weight row of a ring slot and every activation row
 * of the K slice sits in shared memory at a pitch of its bytes rounded up to
 * 128 plus 64: a tensor-core fragment load gives each row 64 consecutive
 * bytes, and a quarter-warp's two rows then fall on distinct banks. */
AMK_HD inline int smem_pitch(int row_bytes, int batch_max) {
    return batch_max > 1 ? (row_bytes + 127) / 128 * 128 + 64 : row_bytes;
}

AMK_HD inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

}  // namespace amk
