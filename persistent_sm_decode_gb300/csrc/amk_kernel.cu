/*
 * amk_kernel.cu — the decode MegaKernel: one persistent cooperative kernel
 * that runs a whole decode step (decoder stack + LM head) from a static,
 * solidified per-CTA task list.
 *
 * Ada-MK technical summary (gist.science): "Problem Statement" (one
 * persistent kernel instead of per-operator launches and HBM round trips),
 * "Methodology" Phase II "Warp Specialization" (SM resources split into
 * warp roles that cooperate through shared memory to overlap memory traffic
 * with compute) and Phase I "Path Solidification" (no runtime scheduling
 * branches: every CTA walks its task table).  The AutoMegaKernel abstract
 * names cross-SM synchronisation as what limits such kernels on
 * high-bandwidth GPUs; this kernel never uses a grid-wide barrier.
 *
 * GB300 (sm_103a) design:
 *  - grid = one CTA per SM (cooperative launch, so every CTA is resident);
 *  - warp 8 is the LOADER: one thread streams every weight tile and KV tile
 *    of the CTA's task list into a ring of shared-memory slots with
 *    cp.async.bulk (TMA bulk copies) completing on mbarriers.  Weights and
 *    the cached prefix never depend on this step's activations, so the
 *    loader runs ahead across dependency waits and keeps HBM busy;
 *  - warps 0-7 are CONSUMERS.  As CONTROLLER they wait for a task's inputs,
 *    then run its prologue (RMSNorm, merged attention output, SwiGLU output
 *    into shared memory), its tiles from the ring, and as STORER its
 *    epilogue (residual, SwiGLU, attention partials, logits);
 *  - cross-SM dependencies ride on the data: every activation word is
 *    {payload, epoch}, written with one 8-byte store, and a consumer polls
 *    the words it needs until they carry the current step's epoch.  One
 *    cross-SM round trip per dependency, no fences, no counters;
 *  - batch-1 GEMV (about 1 flop per weight byte): CUDA cores, each consumer
 *    warp keeps the activations of a fixed K segment in registers and
 *    streams 16-byte weight chunks (bf16, int8 or int4 codes) from the ring
 *    into mixed-precision FMAs; fp32 accumulation;
 *  - GEMV at batch 2..16: tensor cores (mma.sync m16n8k16, 16 weight rows as
 *    A, the sequences as N), several independent accumulator chains per warp;
 *  - attention: split-context flash decoding per (sequence, kv head) chunk on
 *    the tensor cores (bf16 scores with q split in two, tf32 P.V with P split
 *    in two), online softmax in log2 units; MRG tasks merge the chunks;
 *  - greedy steps: every LM-head task keeps its rows' best logit, one ARG
 *    task reduces them to the next token and position;
 *  - every wait is bounded: on timeout the CTA records the error, stops,
 *    waits for its own bulk copies in flight and returns; later launches see
 *    the error word and do nothing until the host clears it.
 */
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "amk_internal.h"
#include "amk_launch.h"

/* Build switches:
 *  AMK_TRACE_CODE       1 compiles in the per-task timing code that the
 *                       trace option records (a tuning build).  The default
 *                       build leaves it out: every task type runs once per
 *                       layer from a cold instruction cache, and the
 *                       never-taken timing branches inside the hot loops
 *                       alone cost about 7 % of a step.
 *  AMK_L2_PREFETCH_CODE 1 compiles in the loader's L2 prefetch (the
 *                       l2_prefetch_kb option; measured slower at every
 *                       distance, and 24 KB of loader code the default build
 *                       leaves out). */
#ifndef AMK_TRACE_CODE
#define AMK_TRACE_CODE 0
#endif
#ifndef AMK_L2_PREFETCH_CODE
#define AMK_L2_PREFETCH_CODE 0
#endif
#define TRACE(p) (AMK_TRACE_CODE ? (p).trace : (unsigned long long *)nullptr)

namespace amk {

/* ----------------------------------------------------------- PTX wrappers */

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

/* 1-D bulk copy global -> this CTA's shared memory, completing on `bar` */
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

/* the same copy with an L2 cache policy (createpolicy) attached */
__device__ __forceinline__ void bulk_copy_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

/* L2 policy under which the lines a copy brings in are the first to go */
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

/* fill of one ring slot, with or without the evict-first policy */
__device__ __forceinline__ void ring_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar, bool hint,
                                          uint64_t policy) {
    if (hint)
        bulk_copy_hint(dst, src, bytes, bar, policy);
    else
        bulk_copy(dst, src, bytes, bar);
}

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

/* epoch-tagged words: one 8-byte store publishes payload and flag together;
 * a two-word load returns each 8-byte element whole */
/* one 8-byte store or load of each word is single-copy atomic; gpu scope is
 * enough, since every producer and consumer runs on this device */
__device__ __forceinline__ void st_ll(uint64_t *p, uint32_t payload, uint32_t epoch) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(((uint64_t)epoch << 32) | payload) : "memory");
}

__device__ __forceinline__ ulonglong2 ld_ll2(const uint64_t *p) {
    ulonglong2 v;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_ll1(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ll_flag(uint64_t w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ float ll_f(uint64_t w) { return __uint_as_float((uint32_t)w); }

/* Consumer-warps-only barrier; returns the OR of `pred` over all consumers,
 * so that every consumer takes the same abort decision.  The non-.aligned
 * forms count threads, not warps: a warp that arrives diverged (after
 * per-lane waits) is still counted correctly. */
__device__ __forceinline__ bool cbar_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(NCW * 32)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void cbar() { asm volatile("barrier.sync 1, %0;" ::"n"(NCW * 32) : "memory"); }

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&b);
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}
/* the bf16 value nearest to f, as fp32 */
__device__ __forceinline__ float round_bf(float f) { return bf2f(f2bf(f)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

/* ----------------------------------------------------------- shared state */

struct Misc {
    volatile int abort;
    volatile int cons_op; /* op of the task the consumers are running (loader's L2 prefetch window) */
    int issued;
    float red[MAXB][NCW];
    float rnorm[MAXB];
    float argv[NCW * MAXB]; /* greedy feedback: per-warp best value and row */
    int argi[NCW * MAXB];
    uint32_t epoch_base;    /* epoch * (L + 1) of the step this CTA runs */
    unsigned long long t_first;     /* trace: first tile of the current task arrived */
    unsigned long long t_wait_full; /* trace: consumer warp 0 waiting for tiles (ns) */
    unsigned long long t_tiles;     /* trace: consumer warp 0 computing tiles (ns) */
    unsigned long long t_pro;       /* trace: prologue done */
    unsigned long long t_stages;    /* trace: last tile consumed */
    unsigned long long t_epi;       /* trace: epilogue written */
    unsigned long long t_x[3];      /* trace: SM cycles from epilogue start to sums formed, stores issued, closing barrier (thread 0) */
};

static_assert(sizeof(Misc) <= SMEM_MISC, "Misc fits its shared-memory region");

struct Smem {
    uint64_t *full, *empty;
    Misc *misc;
    uint8_t *work;
    float *res;
    float *sc;
    float *fac;
    uint8_t *act;
    uint8_t *ring;
};

/* first error wins; every CTA then stops at its next check */
__device__ __noinline__ void raise_error(const Params &p, Smem &s, int code, int task, int what, uint32_t seen, uint32_t target) {
    if (atomicCAS(&p.err[0], 0u, (uint32_t)code) == 0u) {
        p.err[1] = blockIdx.x;
        p.err[2] = (uint32_t)task;
        p.err[3] = (uint32_t)what;
        p.err[4] = seen;
        p.err[5] = target;
        __threadfence();
    }
    s.misc->abort = 1;
}

/* Bounded wait on an mbarrier phase; false on abort or timeout.  Ring waits
 * only follow from a dependency wait elsewhere, so they get twice the limit:
 * the dependency that is really stuck reports first. */
__device__ bool wait_phase(const Params &p, Smem &s, uint64_t *bar, uint32_t parity, int code, int task) {
    if (mbar_test(bar, parity)) return true;
    uint64_t t0 = now_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_test(bar, parity)) return true;
        if (s.misc->abort) return false;
        if ((n & 255u) == 0u) {
            if (ld_relaxed(p.err) != 0u) {
                s.misc->abort = 1;
                return false;
            }
            if ((long long)(now_ns() - t0) > 2 * p.timeout_ns) {
                raise_error(p, s, code, task, -1, 0, parity);
                return false;
            }
        }
    }
}

/* Warp-uniform gate of one ring stage: false (for every lane) if any lane has
 * seen the abort flag or gave up waiting for the slot.  Lanes must agree:
 * a tile ends in full-warp shuffles, and a lane that skipped it would leave
 * the others waiting. */
__device__ __forceinline__ bool stage_ready(const Params &p, Smem &s, uint64_t *bar, uint32_t parity, int task) {
    bool ok = !__any_sync(0xffffffffu, s.misc->abort != 0);
    if (ok) ok = wait_phase(p, s, bar, parity, 2, task);
    return __all_sync(0xffffffffu, ok);
}

/* Which activation buffer a poll waits on (reported in the error word). */
enum : int { WB_XIN = 0, WB_XMID = 1, WB_QKV = 2, WB_PART = 3, WB_AOUT = 4, WB_ACT = 5, WB_ARGP = 6 };

/* the CTA's dynamic shared memory (barriers first, then Misc) */
extern __shared__ __align__(1024) uint8_t smem[];

/* flag of the current step for data of layer `version`: Misc holds epoch *
 * (L + 1) of the step this CTA runs, set once at kernel start */
__device__ __forceinline__ uint32_t ver(const Params &, int version) {
    return reinterpret_cast<const Misc *>(smem + SMEM_BARRIERS)->epoch_base + (uint32_t)version;
}

__device__ __forceinline__ bool ll_ok(uint32_t f, const ulonglong2 &v) { return ll_flag(v.x) == f && ll_flag(v.y) == f; }

/* wait for one word with flag f */
__device__ __noinline__ float ll_wait1(const Params &p, Smem &s, const uint64_t *src, uint32_t f, int task, int which) {
    const uint64_t t0 = now_ns();
    for (uint32_t n = 0;; ++n) {
        const uint64_t w = ld_ll1(src);
        if (ll_flag(w) == f) return ll_f(w);
        if (s.misc->abort) return 0.f;
        if ((n & 63u) == 63u) {
            if (ld_relaxed(p.err) != 0u) {
                s.misc->abort = 1;
                return 0.f;
            }
            if ((long long)(now_ns() - t0) > p.timeout_ns) {
                raise_error(p, s, 1, task, which, ll_flag(w), f);
                return 0.f;
            }
        }
    }
}

/* Checked every 64 passes of a multi-word wait: stop on another CTA's error,
 * or raise a timeout that reports the flag `seen` of a word still stale. */
__device__ __forceinline__ bool poll_slow(const Params &p, Smem &s, uint64_t t0, int task, int which, uint32_t seen,
                                       uint32_t f) {
    if (ld_relaxed(p.err) != 0u) {
        s.misc->abort = 1;
        return false;
    }
    if ((long long)(now_ns() - t0) > p.timeout_ns) {
        raise_error(p, s, 1, task, which, seen, f);
        return false;
    }
    return true;
}

/* Wait for N tagged words (W = uint64_t) or word pairs (W = ulonglong2) at
 * once.  v[i] holds the caller's first read of the word(s) at addr(i); bit i
 * of `pend` marks it stale (clear for words that are current or not needed).
 * Every pass re-reads all stale words before it checks any, so a wait costs
 * one L2 round trip per pass rather than one per word.  On abort or timeout
 * it returns with words still stale; the caller's next abort check stops the
 * task. */
__device__ __forceinline__ uint64_t ll_load(const uint64_t *a, uint64_t) { return ld_ll1(a); }
__device__ __forceinline__ ulonglong2 ll_load(const uint64_t *a, ulonglong2) { return ld_ll2(a); }
__device__ __forceinline__ bool ll_cur(uint32_t f, uint64_t w) { return ll_flag(w) == f; }
__device__ __forceinline__ bool ll_cur(uint32_t f, const ulonglong2 &v) { return ll_ok(f, v); }
__device__ __forceinline__ uint32_t ll_seen(uint32_t f, uint64_t w) { return ll_flag(w); }
__device__ __forceinline__ uint32_t ll_seen(uint32_t f, const ulonglong2 &v) {
    return ll_flag(v.x) != f ? ll_flag(v.x) : ll_flag(v.y);
}

template <int N, class W, class A>
__device__ __forceinline__ void settle_all(const Params &p, Smem &s, W (&v)[N], uint32_t pend, A addr, uint32_t f,
                                           int task, int which) {
    if (pend == 0u) return;
    const uint64_t t0 = now_ns();
    for (uint32_t n = 1;; ++n) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (pend >> i & 1u) v[i] = ll_load(addr(i), v[i]);
#pragma unroll
        for (int i = 0; i < N; ++i)
            if ((pend >> i & 1u) && ll_cur(f, v[i])) pend &= ~(1u << i);
        if (pend == 0u || s.misc->abort) return;
        if ((n & 63u) == 0u) {
            uint32_t seen = 0u;
#pragma unroll
            for (int i = N - 1; i >= 0; --i)
                if (pend >> i & 1u) seen = ll_seen(f, v[i]);
            if (!poll_slow(p, s, t0, task, which, seen, f)) return;
        }
    }
}

/* ----------------------------------------------------------- task geometry */

__device__ __forceinline__ int op_K(const Params &p, int op) {
    return op == OP_OPR ? p.nq * p.d : op == OP_DWN ? p.I : p.H;
}

__device__ __forceinline__ const uint8_t *op_weights(const Params &p, const Task &t, int m) {
    if (t.op == OP_LMH) return (const uint8_t *)p.lm;
    const LayerPtrs &L = p.layers[t.layer];
    const void *w = t.op == OP_QKV ? L.w[t.mat] : t.op == OP_OPR ? L.w[W_O] : t.op == OP_GUP ? L.w[W_GATE + m] : L.w[W_DOWN];
    return (const uint8_t *)w;
}

__device__ __forceinline__ const float *op_scales(const Params &p, const Task &t, int m) {
    if (t.op == OP_LMH) return p.s_lm;
    const LayerPtrs &L = p.layers[t.layer];
    return t.op == OP_QKV ? L.s[t.mat] : t.op == OP_OPR ? L.s[W_O] : t.op == OP_GUP ? L.s[W_GATE + m] : L.s[W_DOWN];
}

struct GemvGeo {
    int ks, R, nrows, nrb, nmat, K, Kc;
};

__device__ __forceinline__ GemvGeo gemv_geo(const Params &p, const Task &t) {
    GemvGeo g;
    g.ks = t.ksplit;
    g.R = t.rows_per_stage;
    g.nrows = t.r1 - t.r0;
    g.nrb = (g.nrows + g.R - 1) / g.R;
    g.nmat = t.op == OP_GUP ? 2 : 1;
    g.K = op_K(p, t.op);
    g.Kc = g.K / g.ks;
    return g;
}

/* context chunk of an attention task: cached positions [s0, e) and whether it
 * holds the new position p */
struct AttGeo {
    int p, s0, e, ntile;
};

__device__ __forceinline__ AttGeo att_geo(const Params &p, const Task &t) {
    AttGeo a;
    a.p = 0;
    a.s0 = a.e = 0;
    a.ntile = 0;
    if ((int)t.b >= p.batch) return a;
    a.p = p.positions[t.b];
    const int n = a.p + 1, C = t.r1, c = t.r0;
    a.s0 = (int)((long long)c * n / C);
    const int s1 = (int)((long long)(c + 1) * n / C);
    a.e = min(s1, a.p);
    a.ntile = a.e > a.s0 ? (a.e - a.s0 + t.rows_per_stage - 1) / t.rows_per_stage : 0;
    return a;
}

/* The stages of a GEMV task in order: stage rb holds the task's rows
 * [rb·n/nst, (rb+1)·n/nst) (stage_rows), walked by additions, with one
 * division per task instead of two 64-bit ones per stage. */
struct StageWalk {
    int q, r, nst, carry, end;
    __device__ __forceinline__ StageWalk(int n, int nst_) : q(0), r(n), nst(nst_), carry(0), end(0) {
        if (nst > 0) {
            q = n / nst;
            r = n - q * nst;
        }
    }
    /* rows [a, e) of the next stage */
    __device__ __forceinline__ void next(int &a, int &e) {
        a = end;
        end += q;
        carry += r;
        if (carry >= nst) {
            carry -= nst;
            ++end;
        }
        e = end;
    }
};

__device__ __forceinline__ void load_task(const Task *src, Task &t) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
    uint4 *d = reinterpret_cast<uint4 *>(&t);
    d[0] = __ldg(s);
    d[1] = __ldg(s + 1);
    d[2] = __ldg(s + 2);
}

/* Position in the ring: slot and pass (how many times the ring wrapped).  The
 * k-th fill of a slot completes phase k of its full barrier; the k-th release
 * completes phase k of its empty barrier. */
struct Ring {
    int slot;
    uint32_t pass;
    uint32_t count; /* stages so far */
    __device__ __forceinline__ void advance(int NS) {
        ++count;
        if (++slot == NS) {
            slot = 0;
            ++pass;
        }
    }
};

/* ----------------------------------------------------------- loader */

/* L2 prefetch ahead of the ring.  The ring holds a few stages; while the
 * loader waits for a free slot, HBM would idle.  The loader therefore walks a
 * second cursor over the same byte sequence and issues bulk L2 prefetches
 * for the tiles the ring will take next, up to l2_prefetch_bytes ahead of
 * what it has filled, so that later fills come from L2. */
__device__ __forceinline__ void l2_prefetch(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

/* The idx-th contiguous byte range a task streams, in fill order: a GEMV
 * task's row block of one matrix per stage (whole rows when K is split), an
 * attention tile's K then V.  False past the last range. */
__device__ bool task_range(const Params &p, const Task &t, int idx, const uint8_t *&ptr, uint32_t &bytes) {
    if (t.op == OP_MRG || t.op == OP_ARG) return false;
    if (t.op == OP_ATT) {
        const AttGeo a = att_geo(p, t);
        const int k = idx / 2;
        if (k >= a.ntile) return false;
        const int t0 = a.s0 + k * t.rows_per_stage, t1 = min(a.e, t0 + (int)t.rows_per_stage);
        const size_t row = (((size_t)t.layer * p.Bmax + t.b) * p.nkv + t.g) * (size_t)p.Smax + t0;
        ptr = (const uint8_t *)((idx & 1 ? p.vc : p.kc) + row * p.d);
        bytes = (uint32_t)(t1 - t0) * p.d * 2;
        return true;
    }
    const GemvGeo g = gemv_geo(p, t);
    const size_t rowb = (size_t)wf_bytes(t.op == OP_LMH ? p.lm_wf : p.wf, g.K);
    if (g.ks > 1) {
        if (idx >= g.nmat) return false;
        ptr = op_weights(p, t, idx) + (size_t)t.r0 * rowb;
        bytes = (uint32_t)((size_t)g.nrows * rowb);
        return true;
    }
    const int rb = idx / g.nmat, m = idx % g.nmat;
    if (rb >= g.nrb) return false;
    int ra, re;
    stage_rows(g.nrows, g.nrb, rb, ra, re);
    ptr = op_weights(p, t, m) + (size_t)(t.r0 + ra) * rowb;
    bytes = (uint32_t)((size_t)(re - ra) * rowb);
    return true;
}

struct Prefetch {
    int ti, r;               /* task and range of the cursor */
    uint32_t off;            /* offset in the range */
    unsigned long long pos;  /* bytes the cursor has passed (prefetched or skipped) */
    unsigned long long fill; /* bytes the ring has been given so far */
    int cached;              /* task index held in t */
    Task t;
};

/* move the prefetch cursor towards `ahead` bytes past the fill position, at
 * most four prefetches per call so that the loader returns to its ring
 * promptly; ranges the ring has already taken are skipped, not prefetched */
__device__ void prefetch_ahead(const Params &p, Prefetch &pf, int tend) {
    const unsigned long long goal = pf.fill + (unsigned long long)p.l2_prefetch_bytes;
    for (int issued = 0; pf.pos < goal && pf.ti < tend && issued < 4;) {
        if (pf.cached != pf.ti) {
            load_task(p.tasks + pf.ti, pf.t);
            pf.cached = pf.ti;
        }
        const uint8_t *ptr;
        uint32_t bytes;
        if (!task_range(p, pf.t, pf.r, ptr, bytes)) {
            ++pf.ti;
            pf.r = 0;
            pf.off = 0;
            continue;
        }
        uint32_t step = min(bytes - pf.off, 65536u);
        if (pf.pos < pf.fill) {
            step = (uint32_t)min((unsigned long long)step, pf.fill - pf.pos);
        } else {
            l2_prefetch(ptr + pf.off, step);
            ++issued;
        }
        pf.off += step;
        pf.pos += step;
        if (pf.off >= bytes) {
            ++pf.r;
            pf.off = 0;
        }
    }
}

/* claim the next slot (bounded wait for its release) and arm its full barrier */
__device__ __forceinline__ uint8_t *loader_claim(const Params &p, Smem &s, Ring &r, uint32_t bytes, int ti,
                                                 Prefetch &pf, int tend) {
    const unsigned long long t0 = TRACE(p) ? now_ns() : 0;
    /* prefetch only while the ring is full and the consumers run attention
     * (a chain of short, latency-bound tasks that leaves HBM idle): fills of a
     * streaming level come first */
#if AMK_L2_PREFETCH_CODE
    if (p.l2_prefetch_bytes > 0 && r.pass > 0 && (s.misc->cons_op == OP_ATT || s.misc->cons_op == OP_MRG) &&
        !mbar_test(&s.empty[r.slot], (r.pass - 1u) & 1u))
        prefetch_ahead(p, pf, tend);
#endif
    if (r.pass > 0 && !wait_phase(p, s, &s.empty[r.slot], (r.pass - 1u) & 1u, 3, ti)) return nullptr;
    if (TRACE(p)) TRACE(p)[16 * (size_t)ti + 9] += now_ns() - t0;
    if (s.misc->abort) return nullptr;
    mbar_arrive_expect_tx(&s.full[r.slot], bytes);
    pf.fill += bytes;
    return s.ring + (size_t)r.slot * p.slot_bytes;
}

__device__ void loader(const Params &p, Smem &s, int tbeg, int tend) {
    const int NS = p.n_slots;
    /* the weight and KV stream passes through L2 once per step; marking it
     * evict-first keeps the lines that are reused every layer (code, the
     * activation words, RoPE rows, task records) resident */
    const bool hint = p.evict_first != 0;
    const uint64_t pol = hint ? policy_evict_first() : 0ull;
    Ring r{0, 0, 0};
    Prefetch pf;
    pf.ti = tbeg;
    pf.r = 0;
    pf.off = 0u;
    pf.pos = pf.fill = 0ull;
    pf.cached = -1;
    for (int ti = tbeg; ti < tend; ++ti) {
        Task t;
        load_task(p.tasks + ti, t);
        if (TRACE(p)) TRACE(p)[16 * (size_t)ti + 9] = 0;
        if (t.op == OP_MRG || t.op == OP_ARG) continue;
        if (t.op == OP_ATT) {
            const AttGeo a = att_geo(p, t);
            const size_t row = (((size_t)t.layer * p.Bmax + t.b) * p.nkv + t.g) * (size_t)p.Smax;
            const uint8_t *kb = (const uint8_t *)(p.kc + row * p.d), *vb = (const uint8_t *)(p.vc + row * p.d);
            const size_t tb = (size_t)t.rows_per_stage * p.d * 2;
            for (int t0 = a.s0; t0 < a.e; t0 += t.rows_per_stage) {
                const int t1 = min(a.e, t0 + (int)t.rows_per_stage);
                const uint32_t bytes = (uint32_t)(t1 - t0) * p.d * 2;
                uint8_t *dst = loader_claim(p, s, r, 2 * bytes, ti, pf, tend);
                if (!dst) {
                    s.misc->issued = (int)r.count;
                    return;
                }
                ring_copy(dst, kb + (size_t)t0 * p.d * 2, bytes, &s.full[r.slot], hint, pol);
                ring_copy(dst + tb, vb + (size_t)t0 * p.d * 2, bytes, &s.full[r.slot], hint, pol);
                r.advance(NS);
            }
            continue;
        }
        const GemvGeo g = gemv_geo(p, t);
        const int wf = t.op == OP_LMH ? p.lm_wf : p.wf;
        const uint8_t *W[2] = {op_weights(p, t, 0), op_weights(p, t, g.nmat - 1)};
        const size_t rowb = (size_t)wf_bytes(wf, g.K), segb = (size_t)wf_bytes(wf, g.Kc);
        /* batch 1: rows back to back; larger batches: rows at the padded pitch */
        const size_t pitch = (size_t)smem_pitch((int)segb, p.Bmax);
        for (int kp = 0; kp < g.ks; ++kp) {
            StageWalk sw(g.nrows, g.nrb);
            for (int rb = 0; rb < g.nrb; ++rb) {
                int ra, re;
                sw.next(ra, re);
                ra += t.r0;
                re += t.r0;
                const uint32_t bytes = (uint32_t)((re - ra) * segb);
                for (int m = 0; m < g.nmat; ++m) {
                    uint8_t *dst = loader_claim(p, s, r, bytes, ti, pf, tend);
                    if (!dst) {
                        s.misc->issued = (int)r.count;
                        return;
                    }
                    if (g.ks == 1 && pitch == segb) {
                        ring_copy(dst, W[m] + (size_t)ra * rowb, bytes, &s.full[r.slot], hint, pol);
                    } else {
                        const uint8_t *src = W[m] + (size_t)ra * rowb + (size_t)kp * segb;
                        for (int q = 0; q < re - ra; ++q)
                            ring_copy(dst + (size_t)q * pitch, src + (size_t)q * rowb, (uint32_t)segb, &s.full[r.slot],
                                      hint, pol);
                    }
                    r.advance(NS);
                }
            }
        }
    }
    s.misc->issued = (int)r.count;
}

/* ----------------------------------------------------------- prologues */

/* U groups of four consecutive x values, group u starting at element
 * 4 * idx(u) (idx(u) < 0: none, zeros): the token's embedding row (layer 0)
 * or epoch-tagged residual words, every word read before the first wait */
template <int U, class I>
__device__ __forceinline__ void load_x4s(const Params &p, Smem &s, const uint64_t *xs, const uint16_t *emb, I idx,
                                         float4 (&x)[U], uint32_t f, int task, int which) {
    if (emb) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i4 = idx(u);
            const uint2 w = i4 >= 0 ? __ldg(reinterpret_cast<const uint2 *>(emb) + i4) : make_uint2(0u, 0u);
            x[u] = make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
        }
        return;
    }
    ulonglong2 v[2 * U];
    uint32_t pend = 0u;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int i4 = idx(u);
        if (i4 >= 0) {
            v[2 * u] = ld_ll2(xs + 4 * (size_t)i4);
            v[2 * u + 1] = ld_ll2(xs + 4 * (size_t)i4 + 2);
        } else {
            v[2 * u] = v[2 * u + 1] = ulonglong2{0ull, 0ull};
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (idx(u) >= 0) {
            if (!ll_ok(f, v[2 * u])) pend |= 1u << (2 * u);
            if (!ll_ok(f, v[2 * u + 1])) pend |= 2u << (2 * u);
        }
    settle_all(p, s, v, pend, [=](int i) { return xs + 4 * (size_t)idx(i >> 1) + 2 * (i & 1); }, f, task, which);
#pragma unroll
    for (int u = 0; u < U; ++u)
        x[u] = make_float4(ll_f(v[2 * u].x), ll_f(v[2 * u].y), ll_f(v[2 * u + 1].x), ll_f(v[2 * u + 1].y));
}

/* RMSNorm prologue into shared memory (batches above 1, or a K split):
 * act[b][k - k0] = bf16(x[b][k] * r_b * gain[k]) for k in [k0, k1), packed two
 * per word.  r_b is computed once per task (need_r) from the whole of x[b].
 * Reading x waits for its producers, XU groups of four per thread at a time. */
constexpr int XU = 4;
template <int NB>
__device__ void norm_prologue(const Params &p, Smem &s, const uint64_t *xbase, bool from_embed, const uint16_t *gain,
                              int k0, int k1, bool need_r, uint32_t f, int task, int which, int ctid, int warp,
                              int lane) {
    const int H = p.H, H4 = H / 4;
    constexpr int TS = NCW * 32;
    if (p.batch == 1 && need_r && k0 == 0 && k1 == H && H4 <= XU * TS) {
        /* one sequence, the whole row, at most XU groups of four per thread:
         * x is read once and stays in registers; the gains are read before
         * the wait, and every thread adds the warps' sums itself after the
         * one barrier */
        const uint64_t *xs = from_embed ? nullptr : xbase;
        const uint16_t *emb = from_embed ? p.embed + (size_t)__ldg(p.tokens) * H : nullptr;
        uint2 gw[XU];
#pragma unroll
        for (int u = 0; u < XU; ++u) {
            const int i = ctid + u * TS;
            gw[u] = i < H4 ? __ldg(reinterpret_cast<const uint2 *>(gain) + i) : make_uint2(0u, 0u);
        }
        float4 x[XU];
        load_x4s<XU>(p, s, xs, emb, [=](int u) { return ctid + u * TS < H4 ? ctid + u * TS : -1; }, x, f, task,
                     which);
        float ss = 0.f;
#pragma unroll
        for (int u = 0; u < XU; ++u) ss += x[u].x * x[u].x + x[u].y * x[u].y + x[u].z * x[u].z + x[u].w * x[u].w;
        ss = warp_sum(ss);
        if (lane == 0) s.misc->red[0][warp] = ss;
        cbar();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) tot += s.misc->red[0][w];
        const float r = rsqrtf(tot / (float)H + p.eps);
        uint2 *dst = reinterpret_cast<uint2 *>(s.act);
#pragma unroll
        for (int u = 0; u < XU; ++u) {
            const int i = ctid + u * TS;
            if (i < H4) {
                const float4 v = x[u];
                dst[i] = make_uint2(pack_bf2(v.x * r * bf_lo(gw[u].x), v.y * r * bf_hi(gw[u].x)),
                                    pack_bf2(v.z * r * bf_lo(gw[u].y), v.w * r * bf_hi(gw[u].y)));
            }
        }
        return;
    }
    const int kc = k1 - k0, a4 = k0 / 4, n4 = kc / 4, apitch = smem_pitch(kc * 2, p.Bmax);
    if (NB > 1 && !from_embed && H4 % 32 == 0) {
        /* several sequences: the rows of x are contiguous, so both passes run
         * over (sequence, group) pairs, XB groups per thread at a time, and
         * one round trip serves several sequences.  A warp's 32 groups of a
         * round belong to one sequence (H4 is a multiple of 32). */
        constexpr int XB = 4;
        if (need_r) {
            if (lane < p.batch) s.misc->red[lane][warp] = 0.f;
            __syncwarp();
            const int T = p.batch * H4;
            /* group i = b * H4 + g: a thread's groups step by TS, so its
             * sequence b advances without a division per group */
            int b = ctid / H4, g = ctid - b * H4;
            for (int i0 = ctid; i0 < T; i0 += XB * TS) {
                float4 x[XB];
                load_x4s<XB>(p, s, xbase, nullptr, [=](int u) { return i0 + u * TS < T ? i0 + u * TS : -1; }, x, f,
                             task, which);
#pragma unroll
                for (int u = 0; u < XB; ++u) {
                    const int i = i0 + u * TS;
                    if (i - lane >= T) break; /* warp-uniform: the warp's groups are past the end */
                    float v = i < T ? x[u].x * x[u].x + x[u].y * x[u].y + x[u].z * x[u].z + x[u].w * x[u].w : 0.f;
                    v = warp_sum(v);
                    if (lane == 0) s.misc->red[b][warp] += v;
                    for (g += TS; g >= H4; g -= H4) ++b;
                }
            }
            cbar();
            if (ctid < p.batch) {
                float ss = 0.f;
#pragma unroll
                for (int w = 0; w < NCW; ++w) ss += s.misc->red[ctid][w];
                s.misc->rnorm[ctid] = rsqrtf(ss / (float)H + p.eps);
            }
            cbar();
        }
        /* item i = b * n4 + j: group j of sequence b's slice, (b, j) walked
         * as in the first pass; gi holds the round's group indices in x */
        const int T = p.batch * n4, ap2 = apitch / 8;
        int b = ctid / n4, j = ctid - b * n4;
        for (int i0 = ctid; i0 < T; i0 += XB * TS) {
            const int rb = b, rj = j;
            int gi[XB];
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                gi[u] = i0 + u * TS < T ? b * H4 + a4 + j : -1;
                for (j += TS; j >= n4; j -= n4) ++b;
            }
            float4 x[XB];
            load_x4s<XB>(p, s, xbase, nullptr, [=](int u) { return gi[u]; }, x, f, task, which);
            int sb = rb, sj = rj;
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                if (gi[u] >= 0) {
                    const float r = s.misc->rnorm[sb];
                    const float4 v = x[u];
                    const uint2 gw = __ldg(reinterpret_cast<const uint2 *>(gain) + a4 + sj);
                    reinterpret_cast<uint2 *>(s.act)[sb * ap2 + sj] =
                        make_uint2(pack_bf2(v.x * r * bf_lo(gw.x), v.y * r * bf_hi(gw.x)),
                                   pack_bf2(v.z * r * bf_lo(gw.y), v.w * r * bf_hi(gw.y)));
                }
                for (sj += TS; sj >= n4; sj -= n4) ++sb;
            }
        }
        return;
    }
    if (need_r) {
        for (int b = 0; b < p.batch; ++b) {
            const uint64_t *xs = from_embed ? nullptr : xbase + (size_t)b * H;
            const uint16_t *emb = from_embed ? p.embed + (size_t)__ldg(p.tokens + b) * H : nullptr;
            float ss = 0.f;
            for (int i0 = ctid; i0 < H4; i0 += XU * TS) {
                float4 x[XU];
                load_x4s<XU>(p, s, xs, emb, [=](int u) { return i0 + u * TS < H4 ? i0 + u * TS : -1; }, x, f, task,
                             which);
#pragma unroll
                for (int u = 0; u < XU; ++u) ss += x[u].x * x[u].x + x[u].y * x[u].y + x[u].z * x[u].z + x[u].w * x[u].w;
            }
            ss = warp_sum(ss);
            if (lane == 0) s.misc->red[b][warp] = ss;
        }
        cbar();
        if (ctid < p.batch) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) ss += s.misc->red[ctid][w];
            s.misc->rnorm[ctid] = rsqrtf(ss / (float)H + p.eps);
        }
        cbar();
    }
    for (int b = 0; b < p.batch; ++b) {
        const uint64_t *xs = from_embed ? nullptr : xbase + (size_t)b * H;
        const uint16_t *emb = from_embed ? p.embed + (size_t)__ldg(p.tokens + b) * H : nullptr;
        const float r = s.misc->rnorm[b];
        uint2 *dst = reinterpret_cast<uint2 *>(s.act + (size_t)b * apitch);
        for (int i0 = ctid; i0 < n4; i0 += XU * TS) {
            float4 x[XU];
            load_x4s<XU>(p, s, xs, emb, [=](int u) { return i0 + u * TS < n4 ? a4 + i0 + u * TS : -1; }, x, f, task,
                         which);
#pragma unroll
            for (int u = 0; u < XU; ++u) {
                const int i = i0 + u * TS;
                if (i < n4) {
                    const float4 v = x[u];
                    const uint2 gw = __ldg(reinterpret_cast<const uint2 *>(gain) + a4 + i);
                    dst[i] = make_uint2(pack_bf2(v.x * r * bf_lo(gw.x), v.y * r * bf_hi(gw.x)),
                                        pack_bf2(v.z * r * bf_lo(gw.y), v.w * r * bf_hi(gw.y)));
                }
            }
        }
    }
}

/* O-projection and down-projection prologues: bf16 activations [k0, k1) of
 * rows of `len` elements (attention output, SwiGLU output), held two per
 * epoch-tagged word, copied as they are (two per word); waits for their
 * producers, CU word pairs per thread at a time.  Up to 8 sequences, one
 * sequence's slice per run of rounds; above 8, the items (sequence, word
 * pair) of all of them run as one sequence of rounds, so that a round trip
 * serves several sequences (measured on the 1.1B shape at context 64: 17 %
 * faster at 16 sequences, 5 % slower at 2 and 8). */
constexpr int CU = 8;
template <int NB>
__device__ void copy_prologue(const Params &p, Smem &s, const uint64_t *src0, int len, int k0, int k1, uint32_t f,
                              int task, int which, int ctid) {
    constexpr int TS = NCW * 32;
    const int kc = k1 - k0, n4 = kc / 4, apitch = smem_pitch(kc * 2, p.Bmax);
    if (NB > 1 && p.batch > 8) {
        /* item i = b * n4 + j: word pair j of sequence b's slice, elements
         * k0 + 4 j .. k0 + 4 j + 3.  A thread's items step by TS, so (b, j)
         * advance without a division per item. */
        const int T = p.batch * n4, ap2 = apitch / 8;
        uint2 *act = reinterpret_cast<uint2 *>(s.act);
        int b = ctid / n4, j = ctid - b * n4;
        for (int i0 = ctid; i0 < T; i0 += CU * TS) {
            const int rb = b, rj = j; /* the round's first item */
            ulonglong2 v[CU];
            uint32_t pend = 0u;
#pragma unroll
            for (int u = 0; u < CU; ++u) {
                const bool in = i0 + u * TS < T;
                v[u] = in ? ld_ll2(src0 + (b * len + k0) / 2 + 2 * j) : ulonglong2{0ull, 0ull};
                if (in && !ll_ok(f, v[u])) pend |= 1u << u;
                for (j += TS; j >= n4; j -= n4) ++b;
            }
            /* (re-polls only: the item's place found again from the round's start) */
            settle_all(p, s, v, pend, [=](int u) {
                int bb = rb, jj = rj + u * TS;
                for (; jj >= n4; jj -= n4) ++bb;
                return src0 + (bb * len + k0) / 2 + 2 * jj;
            }, f, task, which);
            int sb = rb, sj = rj;
#pragma unroll
            for (int u = 0; u < CU; ++u) {
                if (i0 + u * TS < T) act[sb * ap2 + sj] = make_uint2((uint32_t)v[u].x, (uint32_t)v[u].y);
                for (sj += TS; sj >= n4; sj -= n4) ++sb;
            }
        }
    } else {
        for (int b = 0; b < p.batch; ++b) {
            /* word pair i of the slice holds elements k0 + 4 i .. k0 + 4 i + 3 */
            const uint64_t *sb = src0 + ((size_t)b * len + k0) / 2;
            uint2 *dst = reinterpret_cast<uint2 *>(s.act + (size_t)b * apitch);
            for (int i0 = ctid; i0 < n4; i0 += CU * TS) {
                ulonglong2 v[CU];
                uint32_t pend = 0u;
#pragma unroll
                for (int u = 0; u < CU; ++u) {
                    const int i = i0 + u * TS;
                    v[u] = i < n4 ? ld_ll2(sb + 2 * (size_t)i) : ulonglong2{0ull, 0ull};
                }
#pragma unroll
                for (int u = 0; u < CU; ++u)
                    if (i0 + u * TS < n4 && !ll_ok(f, v[u])) pend |= 1u << u;
                settle_all(p, s, v, pend, [=](int u) { return sb + 2 * (size_t)(i0 + u * TS); }, f, task, which);
#pragma unroll
                for (int u = 0; u < CU; ++u) {
                    const int i = i0 + u * TS;
                    if (i < n4) dst[i] = make_uint2((uint32_t)v[u].x, (uint32_t)v[u].y);
                }
            }
        }
    }
}

/* ----------------------------------------------------------- GEMV tiles */

/* int8 -> fp32, exact: byte b of x becomes (2^23 + 128 + b) by placing b ^ 0x80
 * under the exponent bits of 2^23, then 2^23 + 128 is subtracted. */
__device__ __forceinline__ float i8_to_f(uint32_t xflip, int k) {
    return __uint_as_float(__byte_perm(xflip, 0x4B000000u, 0x7540u | (unsigned)k)) - 8388736.0f;
}

/* a += w * h over one pair of bf16 values (low or high halves): the
 * mixed-precision FMA takes both operands as bf16, forms their product
 * exactly in fp32 and rounds once, as fmaf on the widened values would */
__device__ __forceinline__ void fma_bf16_lo(float &a, uint32_t w, uint32_t h) {
    asm("{\n\t.reg .b16 w0, w1, h0, h1;\n\tmov.b32 {w0, w1}, %1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, w0, h0, %0;\n\t}"
        : "+f"(a)
        : "r"(w), "r"(h));
}
__device__ __forceinline__ void fma_bf16_hi(float &a, uint32_t w, uint32_t h) {
    asm("{\n\t.reg .b16 w0, w1, h0, h1;\n\tmov.b32 {w0, w1}, %1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, w1, h1, %0;\n\t}"
        : "+f"(a)
        : "r"(w), "r"(h));
}

/* Dot product of one 16-byte weight chunk (8 bf16 or 16 int8) with EPC
 * bf16 activations at h, packed two per word in element order. */
template <bool I8>
__device__ __forceinline__ float dot_chunk(const uint4 &w, const uint32_t *h) {
    float s0 = 0.f, s1 = 0.f;
    if constexpr (I8) {
        const uint4 ha = reinterpret_cast<const uint4 *>(h)[0], hb = reinterpret_cast<const uint4 *>(h)[1];
        const uint32_t hw[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
        const uint32_t x[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            s0 = fmaf(i8_to_f(x[q], 0), bf_lo(hw[2 * q]), s0);
            s1 = fmaf(i8_to_f(x[q], 1), bf_hi(hw[2 * q]), s1);
            s0 = fmaf(i8_to_f(x[q], 2), bf_lo(hw[2 * q + 1]), s0);
            s1 = fmaf(i8_to_f(x[q], 3), bf_hi(hw[2 * q + 1]), s1);
        }
    } else {
        const uint4 a = reinterpret_cast<const uint4 *>(h)[0];
        fma_bf16_lo(s0, w.x, a.x);
        fma_bf16_hi(s1, w.x, a.x);
        fma_bf16_lo(s0, w.y, a.y);
        fma_bf16_hi(s1, w.y, a.y);
        fma_bf16_lo(s0, w.z, a.z);
        fma_bf16_hi(s1, w.z, a.z);
        fma_bf16_lo(s0, w.w, a.w);
        fma_bf16_hi(s1, w.w, a.w);
    }
    return s0 + s1;
}

/* Batched CUDA-core tile (int8 weights): activations act[b][0..Kc) at
 * `apitch` bytes per sequence, weight rows at `wpitch` bytes.  With S > 1
 * segments per row warp w takes row w / S, K segment w % S; with S == 1 warp
 * w takes rows w, w + 8, ...  Partial sums go to res[(seg * sstride + row) * Bmax + b]
 * (accumulating over K-split passes); the epilogue adds the S segments in a
 * fixed order, so results do not depend on timing. */
template <bool I8, int NB>
__device__ void gemv_tile(const uint8_t *tile, int nrows, int S, int Kc, int wpitch, const uint8_t *act, int apitch,
                          int batch, float *res, int sstride, int Bmax, bool first, int warp, int lane) {
    constexpr int EPC = I8 ? 16 : 8;
    const int nch = Kc / EPC;
    const int RG = NCW / S, seg = warp % S;
    const int c0 = seg * nch / S, c1 = (seg + 1) * nch / S;
    for (int rr = warp / S; rr < nrows; rr += RG) {
        float a[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) a[b] = 0.f;
        const uint4 *w = reinterpret_cast<const uint4 *>(tile + (size_t)rr * wpitch);
        for (int c = c0 + lane; c < c1; c += 32) {
            const uint4 wv = w[c];
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (b < batch)
                    a[b] += dot_chunk<I8>(wv, reinterpret_cast<const uint32_t *>(act + (size_t)b * apitch) +
                                                  (size_t)c * EPC / 2);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b < batch) {
                const float v = warp_sum(a[b]);
                if (lane == 0) {
                    float *r = res + ((size_t)seg * sstride + rr) * Bmax + b;
                    *r = first ? v : *r + v;
                }
            }
        }
    }
}

/* D += A.B on the tensor cores: m16n8k16, bf16 operands, fp32 accumulators */
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

/* Batched tensor-core tile (bf16 weights, batch 2..16).  One m16n8k16 takes
 * 16 weight rows as A (M = output rows) and the activations of 8 sequences as
 * B (N = sequences; a second n-tile above batch 8), so every weight element
 * loaded feeds all sequences.  The sum over K is the same for any order of
 * K, so each k16 step pairs A and B through one permutation: thread t of a
 * fragment row supplies four consecutive elements where the fragment layout
 * names 2t, 2t + 1, 2t + 8, 2t + 9, and one 16-byte shared load (elements
 * 8t .. 8t + 7 of 32) serves two steps.  Warp w takes K segment w of 8 for every row block of the
 * stage.  A dependent chain of mmas waits out each one's latency, so the
 * warp keeps several independent accumulator sets (four with one n-tile, two
 * with two): NR row blocks times CH interleaved K chains (k16 step kb feeds
 * chain kb % CH), summed at the end.
 * res[(w * sstride + row) * Bmax + b] receives the warp's partial sums
 * (added over K-split passes). */
__device__ __forceinline__ uint4 ld_shared16(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 ld_shared8(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

template <int NT, int NR, int CH>
__device__ __forceinline__ void mma_chains(uint32_t tile, int rb0, int nrows, int wpitch, uint32_t act, int apitch,
                                           int batch, int k0, int k1, float *res, int sstride, int Bmax, bool first,
                                           int warp, int g, int t) {
    float acc[NR * CH][NT][4];
    uint32_t wr[NR][2], xs[NT]; /* shared addresses of this lane's row, at K step 0 */
    bool rok[NR][2], xok[NT];
#pragma unroll
    for (int a = 0; a < NR * CH; ++a)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[a][n][0] = acc[a][n][1] = acc[a][n][2] = acc[a][n][3] = 0.f;
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = rb0 + 16 * r + 8 * h + g;
            rok[r][h] = row < nrows;
            wr[r][h] = tile + (uint32_t)(row * wpitch + 32 * k0 + 16 * t);
        }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        xok[n] = 8 * n + g < batch;
        xs[n] = act + (uint32_t)((8 * n + g) * apitch + 32 * k0 + 16 * t);
    }
    /* pairs of k16 steps: a lane's 16 bytes are elements 8t .. 8t + 7 of 32,
     * the first four for the first step, the last four for the second; CH
     * pairs feed CH independent chains, all loads before the first mma */
    const int np = (k1 - k0) / 2;
    for (int p0 = 0; p0 < np; p0 += CH) {
        uint4 bx[CH][NT], w0[CH][NR], w1[CH][NR];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const bool in = p0 + c < np;
            const uint32_t o = 64u * (uint32_t)(p0 + c);
#pragma unroll
            for (int n = 0; n < NT; ++n) bx[c][n] = in && xok[n] ? ld_shared16(xs[n] + o) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                w0[c][r] = in && rok[r][0] ? ld_shared16(wr[r][0] + o) : make_uint4(0u, 0u, 0u, 0u);
                w1[c][r] = in && rok[r][1] ? ld_shared16(wr[r][1] + o) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int c = 0; c < CH; ++c)
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    mma_bf16_16816(acc[r * CH + c][n], w0[c][r].x, w1[c][r].x, w0[c][r].y, w1[c][r].y, bx[c][n].x,
                                   bx[c][n].y);
                    mma_bf16_16816(acc[r * CH + c][n], w0[c][r].z, w1[c][r].z, w0[c][r].w, w1[c][r].w, bx[c][n].z,
                                   bx[c][n].w);
                }
    }
    if ((k1 - k0) & 1) { /* the last step alone: 8 bytes per lane, elements 4t .. 4t + 3 */
        const uint32_t o = 64u * (uint32_t)np;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint2 a0 = rok[r][0] ? ld_shared8(wr[r][0] + o - 8u * t) : make_uint2(0u, 0u);
            const uint2 a1 = rok[r][1] ? ld_shared8(wr[r][1] + o - 8u * t) : make_uint2(0u, 0u);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint2 b = xok[n] ? ld_shared8(xs[n] + o - 8u * t) : make_uint2(0u, 0u);
                mma_bf16_16816(acc[r * CH][n], a0.x, a1.x, a0.y, a1.y, b.x, b.y);
            }
        }
    }
    /* acc 0, 1: row g, sequences 2t, 2t + 1 of the n-tile; 2, 3: row g + 8 */
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float v = acc[r * CH][n][q];
#pragma unroll
                for (int c = 1; c < CH; ++c) v += acc[r * CH + c][n][q];
                const int rr = rb0 + 16 * r + g + (q >= 2 ? 8 : 0), b = 8 * n + 2 * t + (q & 1);
                if (b < batch && rr < nrows) {
                    float *o = res + ((size_t)warp * sstride + rr) * Bmax + b;
                    *o = first ? v : *o + v;
                }
            }
}

template <int NT>
__device__ void gemv_tile_mma_nt(const uint8_t *tile_p, int nrows, int Kc, int wpitch, const uint8_t *act_p,
                                 int apitch, int batch, float *res, int sstride, int Bmax, bool first, int warp,
                                 int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t tile = smem_addr(tile_p), act = smem_addr(act_p);
    const int nblk = Kc / 16, k0 = warp * nblk / NCW, k1 = (warp + 1) * nblk / NCW;
    /* accumulator sets: four with one n-tile, two with two (registers) */
    constexpr int AS = NT == 1 ? 4 : 2;
    for (int rb0 = 0; rb0 < nrows; rb0 += 16 * AS) {
        const int nrb = min(AS, (nrows - rb0 + 15) / 16); /* warp-uniform: row blocks with rows */
        if (nrb == 1)
            mma_chains<NT, 1, AS>(tile, rb0, nrows, wpitch, act, apitch, batch, k0, k1, res, sstride, Bmax, first,
                                  warp, g, t);
        else if (AS == 4 && nrb == 2)
            mma_chains<NT, 2, AS / 2>(tile, rb0, nrows, wpitch, act, apitch, batch, k0, k1, res, sstride, Bmax,
                                      first, warp, g, t);
        else
            mma_chains<NT, AS, 1>(tile, rb0, nrows, wpitch, act, apitch, batch, k0, k1, res, sstride, Bmax, first,
                                  warp, g, t);
    }
}

template <int NB>
__device__ void gemv_tile_mma(const uint8_t *tile, int nrows, int Kc, int wpitch, const uint8_t *act, int apitch,
                              int batch, float *res, int sstride, int Bmax, bool first, int warp, int lane) {
    if (NB <= 8 || batch <= 8)
        gemv_tile_mma_nt<1>(tile, nrows, Kc, wpitch, act, apitch, batch, res, sstride, Bmax, first, warp, lane);
    else
        gemv_tile_mma_nt<2>(tile, nrows, Kc, wpitch, act, apitch, batch, res, sstride, Bmax, first, warp, lane);
}

/* ------------------------------------------- batch-1 GEMV, activations in registers */

/* Sums of R values over the 32 lanes of a warp at once (R = 1, 2, 4, 8):
 * each butterfly step halves the values a lane holds, sending one half to
 * its partner.  Afterwards lane l holds the full sum of value l / (32 / R). */
template <int N, int O, int R>
__device__ __forceinline__ void xstep(float (&v)[R], int lane) {
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = up ? v[i] : v[i + N / 2];
        const float keep = up ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
}

/* Sums of R values over groups of LP lanes at once (R = 1, 2, 4, 8; LP a
 * power of two >= R): each butterfly step halves the values a lane holds,
 * sending one half to its partner.  Afterwards lane l holds the full group
 * sum of value (l % LP) / (LP / R). */
template <int R, int LP>
__device__ __forceinline__ float xsum_g(float (&v)[R], int lane) {
    static_assert(R == 1 || R == 2 || R == 4 || R == 8, "xsum width");
    static_assert(LP >= R && LP <= 32, "xsum group");
    if constexpr (R >= 2) xstep<R, LP / 2>(v, lane);
    if constexpr (R >= 4) xstep<R / 2, LP / 4>(v, lane);
    if constexpr (R >= 8) xstep<R / 4, LP / 8>(v, lane);
    float t = v[0];
#pragma unroll
    for (int o = LP / (2 * R); o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

template <int R>
__device__ __forceinline__ float xsum(float (&v)[R], int lane) {
    return xsum_g<R, 32>(v, lane);
}

/* packed fp32 pairs (sm_100 and later): (a, b) += (c, d); (s0, s1) += (a, b) * (c, d) */
__device__ __forceinline__ void add_f32x2(float &a, float &b, float c, float d) {
    asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
        "add.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(a), "+f"(b)
        : "f"(c), "f"(d));
}
__device__ __forceinline__ void fma_f32x2(float &s0, float &s1, float a, float b, float c, float d) {
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmov.b64 z, {%0, %1};\n\t"
        "fma.rn.f32x2 z, x, y, z;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "f"(a), "f"(b), "f"(c), "f"(d));
}

/* Activations matching one 16-byte weight chunk, in registers, bf16 packed
 * two per word: eight values for bf16 weights, sixteen for int8, thirty-two
 * for int4 (whose pairs are ordered to match the weight pairs that
 * acc_chunk_i4 forms: see act_regs). */
template <int WF>
struct ActChunk {
    uint32_t w[wf_epc(WF) / 2];
};

/* (s0, s1) += one 16-byte weight chunk . its activations (fp32 sums; the
 * products are exact).  bf16: the mixed-precision FMA takes both operands as
 * bf16.  int8: the byte-permute places b ^ 0x80 under the exponent of 2^23,
 * the packed subtraction removes 2^23 + 128 (exact for every int8), and the
 * packed FMA takes two products at once; `hf` holds the sixteen activations
 * already widened to fp32 (once per chunk, for all rows of a group). */
__device__ __forceinline__ void acc_chunk(float &s0, float &s1, const uint4 &w, const ActChunk<WF_BF16> &h) {
    fma_bf16_lo(s0, w.x, h.w[0]);
    fma_bf16_hi(s1, w.x, h.w[0]);
    fma_bf16_lo(s0, w.y, h.w[1]);
    fma_bf16_hi(s1, w.y, h.w[1]);
    fma_bf16_lo(s0, w.z, h.w[2]);
    fma_bf16_hi(s1, w.z, h.w[2]);
    fma_bf16_lo(s0, w.w, h.w[3]);
    fma_bf16_hi(s1, w.w, h.w[3]);
}
/* fp16 pairs and the mixed-precision FMA with fp16 operands */
__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ void fma_f16_lo(float &a, uint32_t w, uint32_t h) {
    asm("{\n\t.reg .b16 w0, w1, h0, h1;\n\tmov.b32 {w0, w1}, %1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "fma.rn.f32.f16 %0, w0, h0, %0;\n\t}"
        : "+f"(a)
        : "r"(w), "r"(h));
}
__device__ __forceinline__ void fma_f16_hi(float &a, uint32_t w, uint32_t h) {
    asm("{\n\t.reg .b16 w0, w1, h0, h1;\n\tmov.b32 {w0, w1}, %1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "fma.rn.f32.f16 %0, w1, h1, %0;\n\t}"
        : "+f"(a)
        : "r"(w), "r"(h));
}
/* bf16 pair -> fp16 pair (the activations of an int8 task, once per task):
 * exact for magnitudes in [2^-14, 65504]; below that the fp16 subnormals keep
 * multiples of 2^-24 */
__device__ __forceinline__ uint32_t bf2_to_f16x2(uint32_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(bf_hi(v)), "f"(bf_lo(v)));
    return r;
}
/* int8 x fp16 activations: four codes b of one word become two fp16 pairs
 * exactly, the byte b ^ 0x80 = b + 128 under the exponent of 1024 (fp16
 * 1024 + b + 128) minus 1152; the products are exact in fp32 (11-bit by
 * 11-bit significands) and accumulate in fp32 */
__device__ __forceinline__ void acc_chunk_i8(float &s0, float &s1, const uint4 &w, const ActChunk<WF_I8> &h) {
    const uint32_t x[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t p01 = sub_f16x2(__byte_perm(x[q], 0x64646464u, 0x4140u), 0x64806480u);
        const uint32_t p23 = sub_f16x2(__byte_perm(x[q], 0x64646464u, 0x4342u), 0x64806480u);
        fma_f16_lo(s0, p01, h.w[2 * q]);
        fma_f16_hi(s1, p01, h.w[2 * q]);
        fma_f16_lo(s0, p23, h.w[2 * q + 1]);
        fma_f16_hi(s1, p23, h.w[2 * q + 1]);
    }
}

/* bf16 pair (x, y) -= (8, 8)... as a packed bf16 subtraction: (128 + u) - 136
 * is u - 8, exact for every 4-bit code u */
__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

/* int4: one word holds elements 0..7 of its group of eight, byte j holding
 * elements 2j (low nibble) and 2j + 1 (high nibble).  t = the low nibbles
 * (elements 0, 2, 4, 6 in bytes 0..3), u = the high nibbles (1, 3, 5, 7); a
 * byte-permute against 0x43 bytes makes bf16 pairs 128 + code, which the
 * packed subtraction turns into code - 8 exactly.  The pairs come out as
 * (0, 2), (4, 6), (1, 3), (5, 7): act_regs stores the activations in that
 * order, so each pair meets its activations in one mixed-precision FMA. */
__device__ __forceinline__ void acc_chunk_i4(float &s0, float &s1, const uint4 &w, const ActChunk<WF_I4> &h) {
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t t = x[q] & 0x0F0F0F0Fu, u = (x[q] >> 4) & 0x0F0F0F0Fu;
        const uint32_t p02 = sub_bf16x2(__byte_perm(t, 0x43434343u, 0x4140u), 0x43084308u);
        const uint32_t p46 = sub_bf16x2(__byte_perm(t, 0x43434343u, 0x4342u), 0x43084308u);
        const uint32_t p13 = sub_bf16x2(__byte_perm(u, 0x43434343u, 0x4140u), 0x43084308u);
        const uint32_t p57 = sub_bf16x2(__byte_perm(u, 0x43434343u, 0x4342u), 0x43084308u);
        fma_bf16_lo(s0, p02, h.w[4 * q]);
        fma_bf16_hi(s1, p02, h.w[4 * q]);
        fma_bf16_lo(s0, p46, h.w[4 * q + 1]);
        fma_bf16_hi(s1, p46, h.w[4 * q + 1]);
        fma_bf16_lo(s0, p13, h.w[4 * q + 2]);
        fma_bf16_hi(s1, p13, h.w[4 * q + 2]);
        fma_bf16_lo(s0, p57, h.w[4 * q + 3]);
        fma_bf16_hi(s1, p57, h.w[4 * q + 3]);
    }
}

/* This warp's activations from the benchmark's bf16 slice in shared memory:
 * chunk j of the lane is chunk c0 + lane + 32 j of the row (zero past c1).
 * For int4, each group of eight activations (h0 .. h7, four words) is
 * reordered to the pairs (h0, h2), (h4, h6), (h1, h3), (h5, h7). */
template <int WF>
__device__ __forceinline__ void act_regs(const uint8_t *act, int c0, int c1, ActChunk<WF> (&hv)[wf_jmax(WF)],
                                         int lane) {
    constexpr int JM = wf_jmax(WF), NQ = wf_epc(WF) / 8;
    const uint4 *A = reinterpret_cast<const uint4 *>(act);
#pragma unroll
    for (int j = 0; j < JM; ++j) {
        const int c = c0 + lane + 32 * j;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const uint4 v = c < c1 ? A[(size_t)c * NQ + q] : make_uint4(0u, 0u, 0u, 0u);
            if constexpr (WF == WF_I4) {
                hv[j].w[4 * q] = __byte_perm(v.x, v.y, 0x5410u);     /* (h0, h2) */
                hv[j].w[4 * q + 1] = __byte_perm(v.z, v.w, 0x5410u); /* (h4, h6) */
                hv[j].w[4 * q + 2] = __byte_perm(v.x, v.y, 0x7632u); /* (h1, h3) */
                hv[j].w[4 * q + 3] = __byte_perm(v.z, v.w, 0x7632u); /* (h5, h7) */
            } else if constexpr (WF == WF_I8) { /* fp16 pairs for acc_chunk_i8 */
                hv[j].w[4 * q] = bf2_to_f16x2(v.x);
                hv[j].w[4 * q + 1] = bf2_to_f16x2(v.y);
                hv[j].w[4 * q + 2] = bf2_to_f16x2(v.z);
                hv[j].w[4 * q + 3] = bf2_to_f16x2(v.w);
            } else {
                hv[j].w[4 * q] = v.x;
                hv[j].w[4 * q + 1] = v.y;
                hv[j].w[4 * q + 2] = v.z;
                hv[j].w[4 * q + 3] = v.w;
            }
        }
    }
}

/* One ring tile of a batch-1 task: nrows rows of rowc 16-byte chunks.  Warp
 * w multiplies K segment [c0, c1) (its registers hv) of rows g * RPG1 + i +
 * k * RG * RPG1 (g = w / S its row group, RG = 8 / S groups): RPG1 rows at a
 * time, each lane summing its chunks of those rows into two accumulators per
 * row, then one transposing reduction for the group.  res[seg * sstride + row]
 * receives the segment's sum (first K slice) or has it added (later ones).
 * int4: each chunk's sum is multiplied by its group's scale, sc[row * ng +
 * (kbase + 32 c) / group] (the task's scales in shared memory). */
template <int WF>
__device__ __forceinline__ void gemv_stage1(const uint8_t *tile, int nrows, int RG, int rgp, int rowc, int c0, int c1,
                                            const ActChunk<WF> (&hv)[wf_jmax(WF)], float *res, int sstride, int seg,
                                            bool first, int lane, const float *sc = nullptr, int ng = 0,
                                            int kbase = 0, int group = 1) {
    constexpr int JM = wf_jmax(WF), RPG = RPG1;
    const uint4 *W = reinterpret_cast<const uint4 *>(tile);
#pragma unroll 1
    for (int r0 = rgp * RPG; r0 < nrows; r0 += RG * RPG) {
        float a0[RPG], a1[RPG];
#pragma unroll
        for (int i = 0; i < RPG; ++i) a0[i] = a1[i] = 0.f;
        /* every slot j runs, with its loads predicated: a branch per slot
         * would keep the loads of slot j + 1 behind the products of slot j,
         * while this way all of a group's loads are in flight at once (slots
         * past the segment multiply zeros) */
#pragma unroll
        for (int j = 0; j < JM; ++j) {
            const int c = c0 + lane + 32 * j;
            uint4 wv[RPG];
#pragma unroll
            for (int i = 0; i < RPG; ++i)
                wv[i] = (r0 + i < nrows && c < c1) ? W[(size_t)(r0 + i) * rowc + c] : make_uint4(0u, 0u, 0u, 0u);
            if constexpr (WF == WF_I8) {
#pragma unroll
                for (int i = 0; i < RPG; ++i) acc_chunk_i8(a0[i], a1[i], wv[i], hv[j]);
            } else if constexpr (WF == WF_I4) {
                const int gi = (kbase + 32 * c) / group;
#pragma unroll
                for (int i = 0; i < RPG; ++i) {
                    float t0 = 0.f, t1 = 0.f;
                    acc_chunk_i4(t0, t1, wv[i], hv[j]);
                    const float scl = (r0 + i < nrows && c < c1) ? sc[(size_t)(r0 + i) * ng + gi] : 0.f;
                    a0[i] = fmaf(scl, t0, a0[i]);
                    a1[i] = fmaf(scl, t1, a1[i]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < RPG; ++i) acc_chunk(a0[i], a1[i], wv[i], hv[j]);
            }
        }
        float v[RPG];
#pragma unroll
        for (int i = 0; i < RPG; ++i) v[i] = a0[i] + a1[i];
        const float y = xsum<RPG>(v, lane);
        const int rr = r0 + lane / (32 / RPG);
        if ((lane & (32 / RPG - 1)) == 0 && rr < nrows) {
            /* later K slices of a K split add to the first slice's sum */
            float *r = res + seg * sstride + rr;
            *r = first ? y : *r + y;
        }
    }
}

/* Residual inputs of a task's epilogue (O projection: x_in of the layer, or
 * the embedding row at layer 0; down projection: x_mid), one per epilogue
 * item, read at task start; their producers ran levels earlier, so the words
 * are normally current and the epilogue does not wait on L2. */
struct ResidPre {
    uint64_t w[2];
};

__device__ __forceinline__ void resid_prefetch(const Params &p, const Task &t, int ctid, ResidPre &rp) {
    rp.w[0] = rp.w[1] = 0ull;
    if (t.op != OP_OPR && t.op != OP_DWN) return;
    const int n = t.r1 - t.r0, B = p.batch, l = t.layer, slot = l % p.depth;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = ctid + k * NCW * 32;
        if (i >= n * B) break;
        const int row = t.r0 + i / B, b = i % B;
        if (t.op == OP_OPR && l == 0)
            rp.w[k] = (uint64_t)__float_as_uint(bf2f(__ldg(p.embed + (size_t)__ldg(p.tokens + b) * p.H + row))) |
                      ((uint64_t)ver(p, 0) << 32);
        else if (t.op == OP_OPR)
            rp.w[k] = ld_ll1(p.x_in + ((size_t)slot * p.Bmax + b) * p.H + row);
        else
            rp.w[k] = ld_ll1(p.x_mid + ((size_t)slot * p.Bmax + b) * p.H + row);
    }
}

/* the prefetched residual of epilogue item k, or a wait for it */
__device__ __forceinline__ float resid_value(const Params &p, Smem &s, const Task &t, int ti, const ResidPre &rp, int k,
                                             int b, int row) {
    const int l = t.layer, slot = l % p.depth;
    const uint64_t w = k == 0 ? rp.w[0] : k == 1 ? rp.w[1] : 0ull; /* no dynamic index: rp stays in registers */
    if (ll_flag(w) == ver(p, l)) return ll_f(w);
    if (t.op == OP_OPR) {
        if (l == 0) return bf2f(__ldg(p.embed + (size_t)__ldg(p.tokens + b) * p.H + row));
        return ll_wait1(p, s, p.x_in + ((size_t)slot * p.Bmax + b) * p.H + row, ver(p, l), ti, WB_XIN);
    }
    return ll_wait1(p, s, p.x_mid + ((size_t)slot * p.Bmax + b) * p.H + row, ver(p, l), ti, WB_XMID);
}

/* (v, i) becomes the better of (v, i) and (v2, i2): the larger value, the
 * lower index between equal values */
__device__ __forceinline__ void arg_better(float &v, int &i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

/* The LM-head task's argmax of every sequence over its rows, from each
 * thread's best: a warp reduction, then across warps in shared memory; the
 * result goes out as two tagged words (value, row) in argp. */
template <int NB>
__device__ void lmh_argmax(const Params &p, Smem &s, const Task &t, float (&bv)[NB], int (&bi)[NB], int ctid) {
    const int warp = ctid >> 5, lane = ctid & 31;
    float *wv = s.misc->argv; /* [NCW][NB] values */
    int *wi = s.misc->argi;   /* [NCW][NB] rows */
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float v = bv[b];
        int i = bi[b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) arg_better(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
        if (lane == 0) {
            wv[warp * NB + b] = v;
            wi[warp * NB + b] = i;
        }
    }
    cbar();
    const int B = NB == 1 ? 1 : p.batch;
    if (ctid < B) {
        float v = wv[ctid];
        int i = wi[ctid];
        for (int w = 1; w < NCW; ++w) arg_better(v, i, wv[w * NB + ctid], wi[w * NB + ctid]);
        uint64_t *dst = p.argp + ((size_t)ctid * p.n_lmh + t.g) * 2;
        const uint32_t f = ver(p, p.L) - ((t.flags & TF_SKIP_SIGNAL) ? (uint32_t)(p.L + 1) : 0u);
        st_ll(dst, __float_as_uint(v), f);
        st_ll(dst + 1, (uint32_t)i, f);
    }
}

/* Greedy feedback: the argmax of every sequence over all LM-head tasks'
 * partials (the larger value; the lower row between equal values), written
 * as that sequence's next token, with its position advanced by one. */
__device__ bool arg_task(const Params &p, Smem &s, const Task &t, int ti, int ctid) {
    const int nt = t.r1, B = p.batch;
    const uint32_t f = ver(p, p.L);
    float *wv = s.misc->argv;
    int *wi = s.misc->argi;
    const int warp = ctid >> 5, lane = ctid & 31;
    for (int b = 0; b < B; ++b) {
        float v = -INFINITY;
        int i = 0x7fffffff;
        constexpr int AU = 4, TS = NCW * 32;
        for (int j0 = ctid; j0 < nt; j0 += AU * TS) {
            ulonglong2 w[AU];
            uint32_t pend = 0u;
#pragma unroll
            for (int u = 0; u < AU; ++u) {
                const int j = j0 + u * TS;
                w[u] = j < nt ? ld_ll2(p.argp + ((size_t)b * p.n_lmh + j) * 2) : ulonglong2{0ull, 0ull};
                if (j < nt && !ll_ok(f, w[u])) pend |= 1u << u;
            }
            settle_all(p, s, w, pend, [=](int u) { return p.argp + ((size_t)b * p.n_lmh + j0 + u * TS) * 2; }, f, ti,
                       WB_ARGP);
#pragma unroll
            for (int u = 0; u < AU; ++u)
                if (j0 + u * TS < nt) arg_better(v, i, ll_f(w[u].x), (int)(uint32_t)w[u].y);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) arg_better(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
        if (lane == 0) {
            wv[warp] = v;
            wi[warp] = i;
        }
        cbar();
        if (ctid == 0) {
            for (int w = 1; w < NCW; ++w) arg_better(v, i, wv[w], wi[w]);
            p.next_tokens[b] = i;
            p.next_positions[b] = __ldg(p.positions + b) + 1;
        }
        cbar();
    }
    return !cbar_or(s.misc->abort != 0);
}

/* Epilogue: publish the task's rows as epoch-tagged words (a task marked
 * TF_SKIP_SIGNAL publishes them with a stale flag: timeout tests).  Partial
 * sums of the S segments are added in a fixed order. */
template <int WF, int NB>
__device__ bool gemv_epilogue(const Params &p, Smem &s, const Task &t, int ti, int S, const ResidPre &rp, int ctid) {
    if (TRACE(p) && ctid == 0) s.misc->t_stages = now_ns();
    const long long c0 = TRACE(p) ? clock64() : 0;
    const int l = t.layer, slot = l % p.depth;
    const uint32_t stale = (t.flags & TF_SKIP_SIGNAL) ? (uint32_t)(p.L + 1) : 0u;
    const uint32_t ep = ver(p, l) - stale, ep_next = ver(p, l + 1) - stale;
    const int n = t.r1 - t.r0, B = NB == 1 ? 1 : p.batch;
    /* partial sums are segment-major, res[((seg * nmat + m) * n + row) * Bmax + b]:
     * consecutive threads read consecutive words; the segments are added in order */
    const int nmat = t.op == OP_GUP ? 2 : 1;
    const int Bmax = NB == 1 ? 1 : p.Bmax;
    const int sstride = nmat * n * Bmax;
    /* (the epilogue runs once per task, from a cold instruction cache: the
     * segment loop stays rolled) */
    auto y_of = [&](int m, int rr, int b) {
        const float *r = s.res + ((size_t)m * n + rr) * Bmax + b;
        float y = 0.f;
#pragma unroll 1
        for (int sg = 0; sg < S; ++sg) y += r[(size_t)sg * sstride];
        return WF == WF_I8 ? y * s.sc[m * n + rr] : y; /* int8: the row scale; int4's are in the sums */
    };
    if (t.op == OP_GUP) {
        /* one SwiGLU output per thread; the thread of the even row packs its
         * neighbour's value (lane + 1) with its own: task rows start at an
         * even row and come in pairs, B items per row */
        const int items = n * B;
        for (int base = 0; base < items; base += NCW * 32) {
            /* item index j = (row) * B + b, laid so that rows 2r and 2r+1 of
             * sequence b sit in lanes that differ by one: j = ((r2 * B + b) * 2 + q) */
            const int j = base + ctid;
            float a = 0.f;
            int pr = 0, b = 0, q = 0;
            if (j < items) {
                q = j & 1;
                b = (j >> 1) % B;
                pr = (j >> 1) / B;
                const int rr = 2 * pr + q;
                const float gte = y_of(0, rr, b), up = y_of(1, rr, b);
                a = gte / (1.f + __expf(-gte)) * up;
            }
            if (TRACE(p) && ctid == 0) s.misc->t_x[0] = clock64() - c0;
            const float other = __shfl_down_sync(0xffffffffu, a, 1);
            if (j < items && q == 0)
                st_ll(p.act + (((size_t)slot * p.Bmax + b) * p.I + t.r0 + 2 * pr) / 2, pack_bf2(a, other), ep);
        }
    } else {
        /* where row `row` of sequence b goes: dst + b * bstride + row, flag fl
         * (logits: a plain fp32 store) */
        uint64_t *dst = nullptr;
        size_t bstride = 0;
        uint32_t fl = ep;
        if (t.op == OP_QKV) {
            const int base = t.mat == MAT_Q ? 0 : t.mat == MAT_K ? p.nq * p.d : (p.nq + p.nkv) * p.d;
            dst = p.qkv + (size_t)slot * p.Bmax * p.qkv_rows + base;
            bstride = p.qkv_rows;
        } else if (t.op == OP_OPR) {
            dst = p.x_mid + (size_t)slot * p.Bmax * p.H;
            bstride = p.H;
        } else if (t.op == OP_DWN) {
            dst = p.x_in + (size_t)((l + 1) % p.depth) * p.Bmax * p.H;
            bstride = p.H;
            fl = ep_next;
        }
        const bool resid = t.op == OP_OPR || t.op == OP_DWN;
        /* greedy feedback: each thread keeps the best (value, row) of every
         * sequence over its items; rows rise along a thread's items, so a
         * strict comparison keeps the lowest row among equal values */
        const bool arg = t.op == OP_LMH && p.next_tokens != nullptr;
        float bv[NB];
        int bi[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            bv[b] = -INFINITY;
            bi[b] = 0x7fffffff;
        }
        int k = 0;
        for (int i = ctid; i < n * B; i += NCW * 32, ++k) {
            const int rr = i / B, b = i % B, row = t.r0 + rr;
            float y = y_of(0, rr, b);
            if (TRACE(p) && ctid == 0 && k == 0) s.misc->t_x[0] = clock64() - c0;
            if (t.op == OP_LMH) {
                p.logits[(size_t)b * p.V + row] = y;
                if (arg) {
#pragma unroll
                    for (int bb = 0; bb < NB; ++bb)
                        if (bb == b && (y > bv[bb] || (y == bv[bb] && row < bi[bb]))) {
                            bv[bb] = y;
                            bi[bb] = row;
                        }
                }
                continue;
            }
            if (resid) y += resid_value(p, s, t, ti, rp, k, b, row);
            st_ll(dst + (size_t)b * bstride + row, __float_as_uint(y), fl);
        }
        if (arg) lmh_argmax<NB>(p, s, t, bv, bi, ctid);
    }
    if (TRACE(p) && ctid == 0) s.misc->t_x[1] = clock64() - c0;
    const bool ok = !cbar_or(s.misc->abort != 0);
    if (TRACE(p) && ctid == 0) s.misc->t_x[2] = clock64() - c0;
    if (TRACE(p) && ctid == 0) s.misc->t_epi = now_ns();
    return ok;
}

/* A GEMV task: for each K slice (ksplit of them), the prologue writes the
 * slice's bf16 activations to shared memory (the RMSNorm of the residual for
 * QKV, gate/up and the LM head; the attention or SwiGLU output for the O and
 * down projections), then the tiles stream through the ring; the epilogue
 * adds the segments' partial sums and publishes the rows. */
template <int WF, int NB>
__device__ bool gemv_task(const Params &p, Smem &s, const Task &t, int ti, Ring &rg, const ResidPre &rp, int ctid,
                          int warp, int lane) {
    constexpr bool I8 = WF == WF_I8;
    const GemvGeo g = gemv_geo(p, t);
    const int NS = p.n_slots;
    const int l = t.layer, slot = l % p.depth;
    const int S = t.seg;
    /* one call site per prologue kind: the op only picks the pointers */
    const bool norm = t.op == OP_QKV || t.op == OP_GUP || t.op == OP_LMH;
    const uint64_t *src;
    const uint16_t *gain = nullptr;
    int which, ver_l = l, len = 0;
    bool emb = false;
    if (t.op == OP_QKV) {
        emb = l == 0;
        src = p.x_in + (size_t)slot * p.Bmax * p.H;
        gain = p.layers[l].attn_norm;
        which = WB_XIN;
    } else if (t.op == OP_GUP) {
        src = p.x_mid + (size_t)slot * p.Bmax * p.H;
        gain = p.layers[l].mlp_norm;
        which = WB_XMID;
    } else if (t.op == OP_LMH) {
        src = p.x_in + (size_t)(p.L % p.depth) * p.Bmax * p.H;
        gain = p.final_norm;
        which = WB_XIN;
        ver_l = p.L;
    } else if (t.op == OP_OPR) {
        src = p.aout + (size_t)slot * p.Bmax * p.nq * p.d / 2;
        len = p.nq * p.d;
        which = WB_AOUT;
    } else {
        src = p.act + (size_t)slot * p.Bmax * p.I / 2;
        len = p.I;
        which = WB_ACT;
    }
    const uint32_t f = ver(p, ver_l);
    /* batch 1: this warp's K segment and row group */
    constexpr int EPC = wf_epc(WF);
    const int rowc = g.Kc / EPC, seg = warp % S, RG = NCW / S, rgp = warp / S;
    const int ng = WF == WF_I4 ? g.K / p.group : 0; /* int4 scale groups per row */
    const int c0 = seg * rowc / S, c1 = (seg + 1) * rowc / S;
    for (int kp = 0; kp < g.ks; ++kp) {
        const int k0 = kp * g.Kc, k1 = k0 + g.Kc;
        if (norm)
            norm_prologue<NB>(p, s, src, emb, gain, k0, k1, kp == 0, f, ti, which, ctid, warp, lane);
        else
            copy_prologue<NB>(p, s, src, len, k0, k1, f, ti, which, ctid);
        if (cbar_or(s.misc->abort != 0)) return false;
        if (TRACE(p) && kp == 0 && ctid == 0) s.misc->t_pro = now_ns();
        ActChunk<WF> hv[wf_jmax(WF)];
        if constexpr (NB == 1) act_regs<WF>(s.act, c0, c1, hv, lane);
        StageWalk sw(g.nrows, g.nrb);
        for (int rb = 0; rb < g.nrb; ++rb) {
            int ra, re;
            sw.next(ra, re);
            for (int m = 0; m < g.nmat; ++m, rg.advance(NS)) {
                const int sl = rg.slot;
                const unsigned long long tw0 = TRACE(p) ? now_ns() : 0;
                if (!stage_ready(p, s, &s.full[sl], rg.pass & 1u, ti)) continue;
                const unsigned long long tw1 = TRACE(p) ? now_ns() : 0;
                if (TRACE(p) && kp == 0 && rb == 0 && m == 0 && warp == 0 && lane == 0) s.misc->t_first = tw1;
                const uint8_t *tile = s.ring + (size_t)sl * p.slot_bytes;
                if constexpr (NB == 1) {
                    gemv_stage1<WF>(tile, re - ra, RG, rgp, rowc, c0, c1, hv, s.res + (size_t)m * g.nrows + ra,
                                    g.nmat * g.nrows, seg, kp == 0, lane, s.sc + ((size_t)m * g.nrows + ra) * ng, ng,
                                    k0, p.group);
                } else {
                    float *res = s.res + ((size_t)m * g.nrows + ra) * p.Bmax;
                    const int wpitch = smem_pitch((int)wf_bytes(WF, g.Kc), NB), apitch = smem_pitch(g.Kc * 2, NB);
                    if constexpr (I8)
                        gemv_tile<I8, NB>(tile, re - ra, S, g.Kc, wpitch, s.act, apitch, p.batch, res, g.nmat * g.nrows,
                                          p.Bmax, kp == 0, warp, lane);
                    else
                        gemv_tile_mma<NB>(tile, re - ra, g.Kc, wpitch, s.act, apitch, p.batch, res, g.nmat * g.nrows,
                                          p.Bmax, kp == 0, warp, lane);
                }
                if (TRACE(p) && warp == 0 && lane == 0) {
                    s.misc->t_wait_full += tw1 - tw0;
                    s.misc->t_tiles += now_ns() - tw1;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.empty[sl]);
            }
        }
        if (cbar_or(s.misc->abort != 0)) return false;
    }
    return gemv_epilogue<WF, NB>(p, s, t, ti, S, rp, ctid);
}

/* ----------------------------------------------------------- attention */

/* Shared memory of an attention task, carved from the activation region. */
struct AttSmem {
    float *q;        /* [GP][d]: rotated q of the group's heads, pre-scaled by log2(e)/sqrt(d) */
    uint16_t *knew;  /* [d] bf16(rope(k)) of position p */
    uint16_t *vnew;  /* [d] */
    float *wst;      /* [NCW][GP][d + PART_PAD]: per-warp (o, m, l) of each head */
    float *sbuf;     /* [NCW][GP] merge factors, then [GP] head maxima */
    uint4 *qf;       /* [d / 16][32]: the q fragment of every k16 step and lane */
};

__device__ __forceinline__ AttSmem att_smem(const Params &p, Smem &s, int GP) {
    AttSmem a;
    uint8_t *base = s.work;
    a.q = reinterpret_cast<float *>(base);
    base += align_up(GP * p.d * 4, 16);
    a.knew = reinterpret_cast<uint16_t *>(base);
    a.vnew = a.knew + p.d;
    base += align_up(2 * p.d * 2, 16);
    a.wst = reinterpret_cast<float *>(base);
    a.sbuf = a.wst + NCW * GP * (p.d + PART_PAD);
    /* 16-byte aligned: q, k/v and wst are whole multiples of 16 bytes
     * (NCW GP (d + PART_PAD) floats with d + PART_PAD a multiple of 4), and so
     * is the block-score area of NCW ATT_BP GP floats */
    a.qf = reinterpret_cast<uint4 *>(a.sbuf + NCW * ATT_BP * GP);
    return a;
}

/* Tensor-core attention.  A warp takes blocks of up to 16 positions of a K/V
 * tile in shared memory and keeps the online-softmax state of every head of
 * the kv group (at most 8) over the positions it has seen.
 *
 * Scores S = Q K^T: one m16n8k16 bf16 mma per 8 positions and 16 dims.  A is
 * the group's rotated, pre-scaled q split in two: row h holds bf16(q) of head
 * h and row h + 8 the bf16 rounding of what is left, so S = D[h] + D[h + 8]
 * carries q to about 16 bits at no extra mma; B is K, exact in bf16.  The
 * sum over dims may take any order, so one lane reads 16 consecutive bytes of
 * a K row per load: in k16 step (c, e) the fragment's dims 2t, 2t + 1, 2t + 8,
 * 2t + 9 are the row's dims 32c + 8t + 4e + 0, 1, 2, 3.
 *
 * P.V as O^T += V^T P^T: m16n8k8 tf32 mmas per 16 dims and 8 positions, M =
 * dims, N = heads, K = positions.  bf16 V is exact in tf32; P goes in twice,
 * as its tf32 rounding and the tf32 rounding of the remainder, so it carries
 * about 22 bits (one tf32 pass alone, 2^-11 relative, measurably widened the
 * deep-stack deviation from the oracle).  Step j
 * takes positions 8j .. 8j + 7 of the block with fragment slot t at position
 * 8j + 2t and slot t + 4 at 8j + 2t + 1: exactly where the score fragment left
 * P of head g in lane (g, t), so P needs no shuffle.  Row g of m-tile i is dim
 * 2 w and row g + 8 dim 2 w + 1, w = 32 (i / 4) + 4g + i % 4, so a lane's V
 * loads are 16 consecutive bytes and each load fills whole wavefronts.
 *
 * The q fragments are the same in every warp: they are made once per task
 * into shared memory.  Lane (g, t) holds the O^T accumulators of heads 2t and
 * 2t + 1 at those dims; the running maximum m of head g (equal in the four
 * lanes of a quad); and its own part of the sum l of head g. */
template <int D>
struct AttState {
    static constexpr int KS = D / 16; /* k16 steps of the scores = m-tiles of P.V */
    float o[KS][4];
    float m, l;
};

/* D += A.B on the tensor cores: m16n8k8, tf32 operands, fp32 accumulators */
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f2tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

/* q fragment of k16 step s for lane (g, t), from q ([G][D] fp32 in shared
 * memory; heads g >= G are zero): rows g and g + 8 of A */
template <int D>
__device__ __forceinline__ uint4 att_qfrag(const float *q, int G, int s, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (g < G) v = *reinterpret_cast<const float4 *>(q + g * D + 32 * (s >> 1) + 8 * t + 4 * (s & 1));
    const float h0 = round_bf(v.x), h1 = round_bf(v.y), h2 = round_bf(v.z), h3 = round_bf(v.w);
    return make_uint4(pack_bf2(h0, h1), pack_bf2(v.x - h0, v.y - h1), pack_bf2(h2, h3), pack_bf2(v.z - h2, v.w - h3));
}

template <int D>
__device__ __forceinline__ void att_init(AttState<D> &st) {
#pragma unroll
    for (int s = 0; s < AttState<D>::KS; ++s) st.o[s][0] = st.o[s][1] = st.o[s][2] = st.o[s][3] = 0.f;
    st.m = -INFINITY;
    st.l = 0.f;
}

/* positions j0 .. j0 + nb - 1 (1 <= nb <= 16) of a K/V tile in shared memory
 * (rows of D bf16); rows past nb are not read */
template <int D>
__device__ __forceinline__ void att_block(AttState<D> &st, const uint4 *qf, const uint16_t *Kt, const uint16_t *Vt,
                                          int j0, int nb, int lane) {
    constexpr int KS = AttState<D>::KS;
    const int g = lane >> 2, t = lane & 3;
    float sc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
    const bool ok0 = g < nb, ok1 = 8 + g < nb;
    const uint4 *kr0 = reinterpret_cast<const uint4 *>(Kt + (size_t)(j0 + g) * D) + t;
    const uint4 *kr1 = reinterpret_cast<const uint4 *>(Kt + (size_t)(j0 + 8 + g) * D) + t;
#pragma unroll
    for (int c = 0; c < KS / 2; ++c) {
        const uint4 k0 = ok0 ? kr0[4 * c] : make_uint4(0u, 0u, 0u, 0u);
        const uint4 k1 = ok1 ? kr1[4 * c] : make_uint4(0u, 0u, 0u, 0u);
        const uint4 qa = qf[2 * c * 32 + lane], qb = qf[(2 * c + 1) * 32 + lane];
        mma_bf16_16816(sc[0], qa.x, qa.y, qa.z, qa.w, k0.x, k0.y);
        mma_bf16_16816(sc[1], qa.x, qa.y, qa.z, qa.w, k1.x, k1.y);
        mma_bf16_16816(sc[0], qb.x, qb.y, qb.z, qb.w, k0.z, k0.w);
        mma_bf16_16816(sc[1], qb.x, qb.y, qb.z, qb.w, k1.z, k1.w);
    }
    /* head g at positions 8j + 2t + e */
    float sv[2][2];
    float mb = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            sv[j][e] = 8 * j + 2 * t + e < nb ? sc[j][e] + sc[j][2 + e] : -INFINITY;
            mb = fmaxf(mb, sv[j][e]);
        }
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float mnew = fmaxf(st.m, mb); /* finite: position 0 is in the block */
    const float alpha = exp2f(st.m - mnew);
    uint32_t pb[2][2], pl[2][2];
    float ps = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float pv = exp2f(sv[j][e] - mnew);
            ps += pv;
            pb[j][e] = f2tf32(pv);
            pl[j][e] = f2tf32(pv - __uint_as_float(pb[j][e]));
        }
    st.l = st.l * alpha + ps;
    st.m = mnew;
    const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);     /* head 2t */
    const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4); /* head 2t + 1 */
#pragma unroll
    for (int i = 0; i < KS; ++i) {
        st.o[i][0] *= a0;
        st.o[i][1] *= a1;
        st.o[i][2] *= a0;
        st.o[i][3] *= a1;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int r0 = 8 * j + 2 * t;
        const uint4 *v0 = reinterpret_cast<const uint4 *>(Vt + (size_t)(j0 + r0) * D) + g;
        const uint4 *v1 = reinterpret_cast<const uint4 *>(Vt + (size_t)(j0 + r0 + 1) * D) + g;
#pragma unroll
        for (int hq = 0; hq < KS / 4; ++hq) {
            const uint4 x0 = r0 < nb ? v0[8 * hq] : make_uint4(0u, 0u, 0u, 0u);
            const uint4 x1 = r0 + 1 < nb ? v1[8 * hq] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w}, w1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
                const uint32_t a0 = w0[i4] << 16, a1 = w0[i4] & 0xffff0000u;
                const uint32_t a2 = w1[i4] << 16, a3 = w1[i4] & 0xffff0000u;
                mma_tf32_1688(st.o[4 * hq + i4], a0, a1, a2, a3, pb[j][0], pb[j][1]);
                mma_tf32_1688(st.o[4 * hq + i4], a0, a1, a2, a3, pl[j][0], pl[j][1]);
            }
        }
    }
}

/* the warp's state into w = [GP][D + PART_PAD]: o of every head, then m and
 * the full l of head g (its quad's parts added) */
template <int D>
__device__ __forceinline__ void att_store(const AttState<D> &st, float *w, int GP, int lane) {
    const int g = lane >> 2, t = lane & 3;
    constexpr int RS = D + PART_PAD;
#pragma unroll
    for (int i = 0; i < AttState<D>::KS; ++i) {
        const int dm = 2 * (32 * (i >> 2) + 4 * g + (i & 3));
        if (2 * t < GP) {
            w[2 * t * RS + dm] = st.o[i][0];
            w[2 * t * RS + dm + 1] = st.o[i][2];
        }
        if (2 * t + 1 < GP) {
            w[(2 * t + 1) * RS + dm] = st.o[i][1];
            w[(2 * t + 1) * RS + dm + 1] = st.o[i][3];
        }
    }
    float l = st.l + __shfl_xor_sync(0xffffffffu, st.l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (t == 0 && g < GP) {
        w[g * RS + D] = st.m;
        w[g * RS + D + 1] = l;
    }
}

template <int D>
__device__ bool att_task(const Params &p, Smem &s, const Task &t, int ti, Ring &rg, int ctid, int warp, int lane) {
    constexpr int d = D;
    const int G = p.G, GP = att_gp(G), NS = p.n_slots;
    const int l = t.layer, slot = l % p.depth, b = t.b, grp = t.g;
    const AttGeo ag = att_geo(p, t);
    const bool active_seq = b < p.batch;
    AttSmem as = att_smem(p, s, GP);

    /* prologue: wait for q, k, v of this kv head, rotate q and the new k,
     * round k and v to bf16 */
    if (active_seq) {
        const uint64_t *qkv = p.qkv + ((size_t)slot * p.Bmax + b) * p.qkv_rows;
        const float *rope = p.rope + (size_t)ag.p * d; /* [d/2][2] */
        const int half = d / 2, tot = (G + 2) * half;
        const uint32_t f = ver(p, l);
        /* item i = (h, e): element e of q head h (h < G), of k (h == G) or of
         * v (h == G + 1), with its partner e + half; AU items per thread are
         * read before the first wait ((G + 2) d / 2 <= 640 <= AU * 256) */
        constexpr int AU = 3, TS = NCW * 32;
        auto src = [=](int i) {
            const int h = i / half, e = i % half;
            const uint64_t *r = h < G ? qkv + (size_t)(grp * G + h) * d
                                : h == G ? qkv + (size_t)p.nq * d + grp * d
                                         : qkv + (size_t)(p.nq + p.nkv) * d + grp * d;
            return r + e;
        };
        for (int i0 = ctid; i0 < tot; i0 += AU * TS) {
            uint64_t w[2 * AU];
            uint32_t pend = 0u;
#pragma unroll
            for (int u = 0; u < AU; ++u) {
                const int i = i0 + u * TS;
                w[2 * u] = i < tot ? ld_ll1(src(i)) : 0ull;
                w[2 * u + 1] = i < tot ? ld_ll1(src(i) + half) : 0ull;
            }

#pragma unroll
            for (int u = 0; u < AU; ++u)
                if (i0 + u * TS < tot) {
                    if (ll_flag(w[2 * u]) != f) pend |= 1u << (2 * u);
                    if (ll_flag(w[2 * u + 1]) != f) pend |= 2u << (2 * u);
                }
            settle_all(p, s, w, pend, [=](int k) { return src(i0 + (k >> 1) * TS) + (k & 1) * half; }, f, ti, WB_QKV);
#pragma unroll
            for (int u = 0; u < AU; ++u) {
                const int i = i0 + u * TS;
                if (i >= tot) continue;
                const int h = i / half, e = i % half;
                const float c = __ldg(rope + 2 * e), sn = __ldg(rope + 2 * e + 1);
                const float a = ll_f(w[2 * u]), bb = ll_f(w[2 * u + 1]);
                if (h < G) {
                    as.q[h * d + e] = (a * c - bb * sn) * p.qk_scale_log2;
                    as.q[h * d + e + half] = (bb * c + a * sn) * p.qk_scale_log2;
                } else if (h == G) {
                    as.knew[e] = f2bf(a * c - bb * sn);
                    as.knew[e + half] = f2bf(bb * c + a * sn);
                } else {
                    as.vnew[e] = f2bf(a);
                    as.vnew[e + half] = f2bf(bb);
                }
            }
        }
    }
    if (cbar_or(s.misc->abort != 0)) return false;
    if (TRACE(p) && ctid == 0) s.misc->t_pro = now_ns();
    if (active_seq && (t.flags & TF_NEW_TOKEN)) {
        const size_t row = ((((size_t)l * p.Bmax + b) * p.nkv + grp) * p.Smax + ag.p) * d;
        for (int i = ctid; i < d; i += NCW * 32) {
            p.kc[row + i] = as.knew[i];
            p.vc[row + i] = as.vnew[i];
        }
    }

    /* the q fragments, once for all warps */
    if (ctid < AttState<D>::KS * 32) as.qf[ctid] = att_qfrag<D>(as.q, active_seq ? G : 0, ctid >> 5, ctid & 31);
    cbar();
    AttState<D> st;
    att_init<D>(st);

    const bool with_new = active_seq && (t.flags & TF_NEW_TOKEN);
    bool new_done = false; /* warp-uniform */
    int gb = 0;            /* blocks of 16 positions dealt so far, round-robin over the warps */
    for (int k = 0; k < ag.ntile; ++k, rg.advance(NS)) {
        const int sl = rg.slot;
        const unsigned long long tw0 = TRACE(p) ? now_ns() : 0;
        if (!stage_ready(p, s, &s.full[sl], rg.pass & 1u, ti)) continue;
        const unsigned long long tw1 = TRACE(p) ? now_ns() : 0;
        if (TRACE(p) && k == 0 && warp == 0 && lane == 0) s.misc->t_first = tw1;
        const int t0 = ag.s0 + k * t.rows_per_stage;
        const int nt = min(ag.e, t0 + (int)t.rows_per_stage) - t0;
        uint16_t *Kt = reinterpret_cast<uint16_t *>(s.ring + (size_t)sl * p.slot_bytes);
        uint16_t *Vt = Kt + (size_t)t.rows_per_stage * d;
        /* the new position joins the last tile of the last chunk when the slot
         * has a free row after the cached positions: the warp whose share
         * covers it copies its K and V into that row first */
        const bool add_new = with_new && k == ag.ntile - 1 && nt < (int)t.rows_per_stage;
        const int ntot = nt + (add_new ? 1 : 0);
        const int nblk = (ntot + ATT_BP - 1) / ATT_BP;
        for (int bi = (warp - gb % NCW + NCW) % NCW; bi < nblk; bi += NCW) {
            const int j0 = bi * ATT_BP, nb = min(ATT_BP, ntot - j0);
            if (add_new && j0 <= nt && nt < j0 + nb) {
                for (int i = lane; i < d / 8; i += 32) {
                    reinterpret_cast<uint4 *>(Kt + (size_t)nt * d)[i] = reinterpret_cast<const uint4 *>(as.knew)[i];
                    reinterpret_cast<uint4 *>(Vt + (size_t)nt * d)[i] = reinterpret_cast<const uint4 *>(as.vnew)[i];
                }
                __syncwarp();
            }
            att_block<D>(st, as.qf, Kt, Vt, j0, nb, lane);
        }
        gb += nblk;
        if (add_new) new_done = true;
        if (TRACE(p) && warp == 0 && lane == 0) {
            s.misc->t_wait_full += tw1 - tw0;
            s.misc->t_tiles += now_ns() - tw1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.empty[sl]);
    }
    /* otherwise the new position on its own, from shared memory, on the next warp in turn */
    if (with_new && !new_done && warp == gb % NCW) att_block<D>(st, as.qf, as.knew, as.vnew, 0, 1, lane);
    if (TRACE(p) && ctid == 0) s.misc->t_stages = now_ns();

    /* the warp's state: o of every head, m and l of each head */
    att_store<D>(st, as.wst + (size_t)warp * GP * (d + PART_PAD), GP, lane);
    if (cbar_or(s.misc->abort != 0)) return false;

    /* merge the warps of each head.  First the per-(warp, head) factors
     * 2^(m_w - M) with M the head's maximum over warps, once each, into the
     * block-score buffer (free after the tiles); then every output element is
     * a weighted sum over the warps.  Publish the chunk's partial (o
     * unnormalised, m, l), head-major: part[b][kv head][head][chunk]. */
    float *fw = as.sbuf;          /* [NCW][GP] factors */
    float *mh = as.sbuf + NCW * GP; /* [GP] head maxima */
    if (ctid < NCW * GP) {
        const int w2 = ctid / GP, hh = ctid % GP;
        float M = -INFINITY;
        for (int w3 = 0; w3 < NCW; ++w3) M = fmaxf(M, as.wst[((size_t)w3 * GP + hh) * (d + PART_PAD) + d]);
        const float mw = as.wst[((size_t)w2 * GP + hh) * (d + PART_PAD) + d];
        fw[ctid] = (mw == -INFINITY || M == -INFINITY) ? 0.f : exp2f(mw - M);
        if (w2 == 0) mh[hh] = M;
    }
    cbar();
    if (active_seq) {
        const uint32_t ep = ver(p, l) - ((t.flags & TF_SKIP_SIGNAL) ? (uint32_t)(p.L + 1) : 0u);
        uint64_t *part = p.part + (((size_t)slot * p.Bmax + b) * p.nkv + grp) * G * p.C * (d + PART_PAD);
        for (int i = ctid; i < G * (d + 2); i += NCW * 32) {
            const int hh = i / (d + 2), e = i % (d + 2);
            float v = 0.f;
            if (e == d) {
                v = mh[hh];
            } else {
                const int ee = e == d + 1 ? d + 1 : e;
#pragma unroll 2
                for (int w2 = 0; w2 < NCW; ++w2)
                    v = fmaf(fw[w2 * GP + hh], as.wst[((size_t)w2 * GP + hh) * (d + PART_PAD) + ee], v);
            }
            st_ll(part + ((size_t)hh * p.C + t.r0) * (d + PART_PAD) + e, __float_as_uint(v), ep);
        }
    }
    if (TRACE(p) && ctid == 0) s.misc->t_epi = now_ns();
    return !cbar_or(s.misc->abort != 0);
}


/* Merge the C chunk partials of one query head of one sequence into its bf16
 * attention output: o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c (the
 * log-sum-exp combination of split softmax).  Every partial word is loaded
 * before the first wait; thread t takes four output elements (t % (d/4)) of
 * the chunks c = t / (d/4) (mod NCL); the NCL sums of each element are added
 * in a fixed order. */
template <int D>
__device__ bool mrg_task(const Params &p, Smem &s, const Task &t, int ti, int ctid) {
    constexpr int d = D;
    const int G = p.G, C = t.r1, slot = t.layer % p.depth, b = t.b, h = t.g;
    const int grp = h / G, hh = h % G;
    constexpr int Q4 = d / 4, NCL = NCW * 32 / Q4;
    const int e4 = ctid % Q4, cl = ctid / Q4;
    constexpr int MAXCPT = MRG_MAX_CPT;
    float *num = s.fac;                  /* [NCL][d] */
    float *den = s.fac + NCL * d;        /* [NCL] */
    float *mx = den + NCL;               /* [NCL] */
    if (b < p.batch) {
        const uint32_t f = ver(p, t.layer);
        const uint64_t *base = p.part + ((((size_t)slot * p.Bmax + b) * p.nkv + grp) * G + hh) * C * (d + PART_PAD);
        /* word pairs 3k, 3k+1, 3k+2: (m, l), o[4 e4 ..], o[4 e4 + 2 ..] of chunk cl + k NCL */
        auto addr = [=](int i) {
            const uint64_t *r = base + (size_t)(cl + (i / 3) * NCL) * (d + PART_PAD);
            return i % 3 == 0 ? r + d : r + 4 * e4 + 2 * (i % 3 - 1);
        };
        ulonglong2 v[3 * MAXCPT];
        uint32_t pend = 0u;
#pragma unroll
        for (int i = 0; i < 3 * MAXCPT; ++i) v[i] = cl + (i / 3) * NCL < C ? ld_ll2(addr(i)) : ulonglong2{0ull, 0ull};
#pragma unroll
        for (int i = 0; i < 3 * MAXCPT; ++i)
            if (cl + (i / 3) * NCL < C && !ll_ok(f, v[i])) pend |= 1u << i;
        settle_all(p, s, v, pend, addr, f, ti, WB_PART);
        ulonglong2 ml[MAXCPT], o0[MAXCPT], o1[MAXCPT];
        float mloc = -INFINITY;
#pragma unroll
        for (int k = 0; k < MAXCPT; ++k) {
            ml[k] = v[3 * k];
            o0[k] = v[3 * k + 1];
            o1[k] = v[3 * k + 2];
            if (cl + k * NCL < C) mloc = fmaxf(mloc, ll_f(ml[k].x));
        }
        if (e4 == 0) mx[cl] = mloc;
        if (TRACE(p) && ctid == 0) s.misc->t_pro = now_ns();
        cbar();
        float M = -INFINITY;
        for (int i = 0; i < NCL; ++i) M = fmaxf(M, mx[i]);
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, dl = 0.f;
#pragma unroll
        for (int k = 0; k < MAXCPT; ++k) {
            const int c = cl + k * NCL;
            if (c < C) {
                const float mc = ll_f(ml[k].x);
                const float w = mc == -INFINITY ? 0.f : exp2f(mc - M);
                dl = fmaf(w, ll_f(ml[k].y), dl);
                acc[0] = fmaf(w, ll_f(o0[k].x), acc[0]);
                acc[1] = fmaf(w, ll_f(o0[k].y), acc[1]);
                acc[2] = fmaf(w, ll_f(o1[k].x), acc[2]);
                acc[3] = fmaf(w, ll_f(o1[k].y), acc[3]);
            }
        }
        *reinterpret_cast<float4 *>(num + (size_t)cl * d + 4 * e4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        if (e4 == 0) den[cl] = dl;
        cbar();
        if (TRACE(p) && ctid == 0) s.misc->t_stages = now_ns();
        if (ctid < Q4) {
            float o[4] = {0.f, 0.f, 0.f, 0.f}, dd = 0.f;
            for (int i = 0; i < NCL; ++i) {
                const float4 v = *reinterpret_cast<const float4 *>(num + (size_t)i * d + 4 * ctid);
                o[0] += v.x;
                o[1] += v.y;
                o[2] += v.z;
                o[3] += v.w;
                dd += den[i];
            }
            const float inv = 1.f / dd;
            const uint32_t ep = f - ((t.flags & TF_SKIP_SIGNAL) ? (uint32_t)(p.L + 1) : 0u);
            uint64_t *out = p.aout + (((size_t)slot * p.Bmax + b) * p.nq * d + (size_t)h * d + 4 * ctid) / 2;
            st_ll(out, pack_bf2(o[0] * inv, o[1] * inv), ep);
            st_ll(out + 1, pack_bf2(o[2] * inv, o[3] * inv), ep);
        }
    }
    if (TRACE(p) && ctid == 0) s.misc->t_epi = now_ns();
    return !cbar_or(s.misc->abort != 0);
}

/* ----------------------------------------------------------- the kernel */

template <int WF, int NB>
__device__ __forceinline__ void run_tasks(const Params &p, Smem &s, int tbeg, int tend, int tid, int warp, int lane) {
    if (warp == NCW) {
        if (lane == 0) loader(p, s, tbeg, tend);
        __syncwarp();
    } else {
        const int ctid = tid;
        Ring rg{0, 0, 0};
        for (int ti = tbeg; ti < tend; ++ti) {
            Task t;
            load_task(p.tasks + ti, t);
            /* weights-only inputs are fetched before the task's inputs are ready */
            if (WF != WF_BF16 && t.op != OP_ATT && t.op != OP_MRG && t.op != OP_ARG) {
                /* int8: one scale per row, [m][row]; int4: [m][row][group] */
                const int n = t.r1 - t.r0, nm = t.op == OP_GUP ? 2 : 1;
                const int per = WF == WF_I4 ? op_K(p, t.op) / p.group : 1;
                for (int i = ctid; i < n * nm * per; i += NCW * 32) {
                    const int m = i / (n * per), r = i % (n * per);
                    s.sc[i] = __ldg(op_scales(p, t, m) + (size_t)t.r0 * per + r);
                }
            }
#if AMK_L2_PREFETCH_CODE
            if (ctid == 0) s.misc->cons_op = t.op;
#endif
            ResidPre rp;
            resid_prefetch(p, t, ctid, rp);
            unsigned long long *tr = TRACE(p) ? TRACE(p) + 16 * (size_t)ti : nullptr;
            if (tr && ctid == 0) {
                tr[0] = tr[1] = now_ns();
                s.misc->t_first = 0;
                s.misc->t_wait_full = 0;
                s.misc->t_tiles = 0;
                s.misc->t_pro = s.misc->t_stages = s.misc->t_epi = 0;
                s.misc->t_x[0] = s.misc->t_x[1] = s.misc->t_x[2] = 0;
            }
            bool ok;
            if (t.op == OP_ATT)
                ok = p.d == 64 ? att_task<64>(p, s, t, ti, rg, ctid, warp, lane)
                               : att_task<128>(p, s, t, ti, rg, ctid, warp, lane);
            else if (t.op == OP_MRG)
                ok = p.d == 64 ? mrg_task<64>(p, s, t, ti, ctid) : mrg_task<128>(p, s, t, ti, ctid);
            else if (t.op == OP_ARG)
                ok = p.next_tokens ? arg_task(p, s, t, ti, ctid) : true;
            else
                ok = gemv_task<WF, NB>(p, s, t, ti, rg, rp, ctid, warp, lane);
            if (!ok) break;
            if (tr && ctid == 0) {
                tr[2] = s.misc->t_first;
                tr[3] = now_ns();
                tr[4] = s.misc->t_wait_full;
                tr[5] = s.misc->t_tiles;
                tr[6] = s.misc->t_pro;
                tr[7] = s.misc->t_stages;
                tr[8] = s.misc->t_epi;
                tr[10] = s.misc->t_x[0];
                tr[11] = s.misc->t_x[1];
                tr[12] = s.misc->t_x[2];
            }
        }
    }
    __syncthreads();
    /* never leave with bulk copies in flight into this CTA's shared memory */
    if (warp == NCW && lane == 0) {
        const int issued = s.misc->issued, NS = p.n_slots;
        for (int u = max(0, issued - NS); u < issued; ++u) {
            uint64_t t0 = now_ns();
            while (!mbar_test(&s.full[u % NS], (uint32_t)(u / NS) & 1u))
                if ((long long)(now_ns() - t0) > p.timeout_ns) break;
        }
    }
}

template <int WF, int NB>
__global__ void __launch_bounds__(NTHREADS, 1) amk_decode_kernel(const Params p) {
    Smem s;
    s.full = reinterpret_cast<uint64_t *>(smem);
    s.empty = s.full + MAX_SLOTS;
    s.misc = reinterpret_cast<Misc *>(smem + SMEM_BARRIERS);
    /* one region per task: GEMV [sums | scales | activations], attention
     * state, or merge sums (tasks of a CTA never overlap) */
    s.work = smem + SMEM_BARRIERS + SMEM_MISC;
    s.res = reinterpret_cast<float *>(s.work);
    s.sc = reinterpret_cast<float *>(s.work + p.result_bytes);
    s.act = s.work + p.result_bytes + p.scale_bytes;
    s.fac = reinterpret_cast<float *>(s.work);
    s.ring = s.work + p.work_bytes;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tbeg = p.task_start[blockIdx.x], tend = p.task_start[blockIdx.x + 1];

    if (tid == 0) {
        s.misc->abort = 0;
        s.misc->cons_op = OP_COUNT;
        s.misc->issued = 0;
        for (int i = 0; i < p.n_slots; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], NCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    /* a previous step's error stops every later step until the host clears it;
     * out-of-range tokens or positions stop this one before any memory access */
    bool bad_input = false;
    if (tid == 0) {
        for (int b = 0; b < p.batch; ++b) {
            const int tok = __ldg(p.tokens + b), pos = __ldg(p.positions + b);
            if (tok < 0 || tok >= p.V || pos < 0 || pos >= p.Smax) bad_input = true;
        }
        if (bad_input && blockIdx.x == 0) raise_error(p, s, 4, -1, -1, 0, 0);
    }
    uint32_t epoch = p.epoch;
    if (tid == 0) {
        if (p.epoch_word) epoch = ld_relaxed(p.epoch_word);
        s.misc->epoch_base = epoch * (uint32_t)(p.L + 1);
    }
    const bool stale = __syncthreads_or(tid == 0 && (bad_input || ld_relaxed(p.err) != 0u));
    if (!stale) run_tasks<WF, NB>(p, s, tbeg, tend, tid, warp, lane);
    /* the last CTA to finish advances the device epoch for the next step (a
     * CTA reads it only at its start, so every CTA of this step has) */
    if (tid == 0 && p.epoch_word) {
        __threadfence();
        if (atomicAdd(p.epoch_word + 1, 1u) == gridDim.x - 1) {
            p.epoch_word[1] = 0u;
            p.epoch_word[0] = epoch + 1u;
        }
    }
}

/* ----------------------------------------------------------- host entry */

bool kernel_has_trace() { return AMK_TRACE_CODE != 0; }
bool kernel_has_l2_prefetch() { return AMK_L2_PREFETCH_CODE != 0; }

KernelFn select_kernel(int weight_dtype, int max_batch) {
    if (weight_dtype == 2) return amk_decode_kernel<WF_I4, 1>; /* 4-bit weights: batch 1 only */
    if (weight_dtype == 1) return max_batch == 1 ? amk_decode_kernel<WF_I8, 1> : amk_decode_kernel<WF_I8, MAXB>;
    return max_batch == 1 ? amk_decode_kernel<WF_BF16, 1> : amk_decode_kernel<WF_BF16, MAXB>;
}

cudaError_t prepare_kernel(KernelFn fn, int smem_bytes) {
    return cudaFuncSetAttribute((const void *)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t occupancy(KernelFn fn, int smem_bytes, int *blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, (const void *)fn, NTHREADS, smem_bytes);
}

cudaError_t launch_decode(KernelFn fn, const Params &p, int n_sm, int smem_bytes, cudaStream_t stream) {
    void *args[] = {const_cast<Params *>(&p)};
    return cudaLaunchCooperativeKernel((const void *)fn, dim3(n_sm), dim3(NTHREADS), args, (size_t)smem_bytes, stream);
}

}  // namespace amk
