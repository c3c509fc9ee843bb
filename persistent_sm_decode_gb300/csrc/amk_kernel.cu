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
 *  - batch-1 GEMV: CUDA cores, each consumer warp keeps the activations of a
 *    fixed K segment in registers and streams 16-byte weight chunks from the
 *    ring with short independent FMA chains; fp32 accumulation;
 *  - attention: split-context flash decoding per (sequence, kv head) chunk
 *    with an online softmax in log2 units; MRG tasks merge the chunks;
 *  - every wait is bounded: on timeout the CTA records the error, stops,
 *    waits for its own bulk copies in flight and returns; later launches see
 *    the error word and do nothing until the host clears it.
 */
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "amk_internal.h"
#include "amk_launch.h"

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
__device__ __forceinline__ void st_ll(uint64_t *p, uint32_t payload, uint32_t epoch) {
    asm volatile("st.volatile.global.u64 [%0], %1;" ::"l"(p), "l"(((uint64_t)epoch << 32) | payload) : "memory");
}

__device__ __forceinline__ ulonglong2 ld_ll2(const uint64_t *p) {
    ulonglong2 v;
    asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_ll1(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ll_flag(uint64_t w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ float ll_f(uint64_t w) { return __uint_as_float((uint32_t)w); }

/* consumer-warps-only barrier; returns the OR of `pred` over all consumers,
 * so that every consumer takes the same abort decision */
__device__ __forceinline__ bool cbar_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(NCW * 32)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory"); }

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
    int issued;
    float red[MAXB][NCW];
    float rnorm[MAXB];
    unsigned long long t_first;     /* trace: first tile of the current task arrived */
    unsigned long long t_wait_full; /* trace: consumer warp 0 waiting for tiles (ns) */
    unsigned long long t_tiles;     /* trace: consumer warp 0 computing tiles (ns) */
    unsigned long long t_pro;       /* trace: prologue done */
    unsigned long long t_stages;    /* trace: last tile consumed */
    unsigned long long t_epi;       /* trace: epilogue written */
};

struct Smem {
    uint64_t *full, *empty;
    Misc *misc;
    float *res;
    float *sc;
    float *fac;
    uint8_t *act;
    uint8_t *ring;
};

/* first error wins; every CTA then stops at its next check */
__device__ void raise_error(const Params &p, Smem &s, int code, int task, int what, uint32_t seen, uint32_t target) {
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

/* Which activation buffer a poll waits on (reported in the error word). */
enum : int { WB_XIN = 0, WB_XMID = 1, WB_QKV = 2, WB_PART = 3, WB_AOUT = 4, WB_ACT = 5 };

/* flag of the current step for data of layer `version` */
__device__ __forceinline__ uint32_t ver(const Params &p, int version) { return p.epoch_base + (uint32_t)version; }

__device__ __forceinline__ bool ll_ok(uint32_t f, const ulonglong2 &v) { return ll_flag(v.x) == f && ll_flag(v.y) == f; }

/* Re-read two tagged words until both carry flag f (the first read was
 * issued by the caller).  False on abort or timeout. */
__device__ __noinline__ bool ll_settle(const Params &p, Smem &s, const uint64_t *src, ulonglong2 &v, uint32_t f,
                                       int task, int which) {
    const uint64_t t0 = now_ns();
    for (uint32_t n = 0;; ++n) {
        if (ll_ok(f, v)) return true;
        if (s.misc->abort) return false;
        if ((n & 63u) == 63u) {
            if (ld_relaxed(p.err) != 0u) {
                s.misc->abort = 1;
                return false;
            }
            if ((long long)(now_ns() - t0) > p.timeout_ns) {
                raise_error(p, s, 1, task, which, ll_flag(v.x) != f ? ll_flag(v.x) : ll_flag(v.y), f);
                return false;
            }
        }
        v = ld_ll2(src);
    }
}

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

/* claim the next slot (bounded wait for its release) and arm its full barrier */
__device__ __forceinline__ uint8_t *loader_claim(const Params &p, Smem &s, Ring &r, uint32_t bytes, int ti) {
    const unsigned long long t0 = p.trace ? now_ns() : 0;
    if (r.pass > 0 && !wait_phase(p, s, &s.empty[r.slot], (r.pass - 1u) & 1u, 3, ti)) return nullptr;
    if (p.trace) p.trace[16 * (size_t)ti + 9] += now_ns() - t0;
    if (s.misc->abort) return nullptr;
    mbar_arrive_expect_tx(&s.full[r.slot], bytes);
    return s.ring + (size_t)r.slot * p.slot_bytes;
}

__device__ void loader(const Params &p, Smem &s, int tbeg, int tend) {
    const int NS = p.n_slots;
    Ring r{0, 0, 0};
    for (int ti = tbeg; ti < tend; ++ti) {
        Task t;
        load_task(p.tasks + ti, t);
        if (p.trace) p.trace[16 * (size_t)ti + 9] = 0;
        if (t.op == OP_MRG) continue;
        if (t.op == OP_ATT) {
            const AttGeo a = att_geo(p, t);
            const size_t row = (((size_t)t.layer * p.Bmax + t.b) * p.nkv + t.g) * (size_t)p.Smax;
            const uint8_t *kb = (const uint8_t *)(p.kc + row * p.d), *vb = (const uint8_t *)(p.vc + row * p.d);
            const size_t tb = (size_t)t.rows_per_stage * p.d * 2;
            for (int t0 = a.s0; t0 < a.e; t0 += t.rows_per_stage) {
                const int t1 = min(a.e, t0 + (int)t.rows_per_stage);
                const uint32_t bytes = (uint32_t)(t1 - t0) * p.d * 2;
                uint8_t *dst = loader_claim(p, s, r, 2 * bytes, ti);
                if (!dst) {
                    s.misc->issued = (int)r.count;
                    return;
                }
                bulk_copy(dst, kb + (size_t)t0 * p.d * 2, bytes, &s.full[r.slot]);
                bulk_copy(dst + tb, vb + (size_t)t0 * p.d * 2, bytes, &s.full[r.slot]);
                r.advance(NS);
            }
            continue;
        }
        const GemvGeo g = gemv_geo(p, t);
        const int web = (t.op == OP_LMH ? p.lm_int8 : p.wint8) ? 1 : 2;
        const uint8_t *W[2] = {op_weights(p, t, 0), op_weights(p, t, g.nmat - 1)};
        const size_t rowb = (size_t)g.K * web, segb = (size_t)g.Kc * web;
        for (int kp = 0; kp < g.ks; ++kp) {
            for (int ra = t.r0; ra < t.r1; ra += g.R) {
                const int re = min(t.r1, ra + g.R);
                const uint32_t bytes = (uint32_t)((re - ra) * segb);
                for (int m = 0; m < g.nmat; ++m) {
                    uint8_t *dst = loader_claim(p, s, r, bytes, ti);
                    if (!dst) {
                        s.misc->issued = (int)r.count;
                        return;
                    }
                    if (g.ks == 1) {
                        bulk_copy(dst, W[m] + (size_t)ra * rowb, bytes, &s.full[r.slot]);
                    } else {
                        const uint8_t *src = W[m] + (size_t)ra * rowb + (size_t)kp * segb;
                        for (int q = 0; q < re - ra; ++q)
                            bulk_copy(dst + (size_t)q * segb, src + (size_t)q * rowb, (uint32_t)segb, &s.full[r.slot]);
                    }
                    r.advance(NS);
                }
            }
        }
    }
    s.misc->issued = (int)r.count;
}

/* ----------------------------------------------------------- prologues */

constexpr int MAXG = 4; /* float4 of x (and of the gain) per consumer thread kept in registers: H <= 4096 */

/* batch 1 with the whole row in one K slice: x and the gain stay in registers */
template <int NB>
__device__ __forceinline__ bool norm_keeps_x(const Params &p, int k0, int k1) {
    return NB == 1 && p.H / 4 <= MAXG * NCW * 32 && k0 == 0 && k1 == p.H;
}

/* four consecutive x values: the token's embedding row (layer 0) or epoch-
 * tagged residual words (waited for) */
__device__ __forceinline__ float4 load_x4(const Params &p, Smem &s, const uint64_t *xs, const uint16_t *emb, int i4,
                                          uint32_t f, int task, int which) {
    if (emb) {
        uint2 w = __ldg(reinterpret_cast<const uint2 *>(emb) + i4);
        return make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
    }
    const uint64_t *src = xs + 4 * (size_t)i4;
    ulonglong2 a = ld_ll2(src), b = ld_ll2(src + 2);
    if (!ll_ok(f, a)) ll_settle(p, s, src, a, f, task, which);
    if (!ll_ok(f, b)) ll_settle(p, s, src + 2, b, f, task, which);
    return make_float4(ll_f(a.x), ll_f(a.y), ll_f(b.x), ll_f(b.y));
}

/* RMSNorm prologue: act[b][k - k0] = bf16(x[b][k] * r_b * gain[k]) for k in
 * [k0, k1), stored as fp32 (the bf16 value exactly).  r_b is computed once per
 * task (need_r) from the whole of x[b].  Reading x waits for its producers. */
template <int NB>
__device__ void norm_prologue(const Params &p, Smem &s, const uint64_t *xbase, bool from_embed, const uint16_t *gain,
                              int k0, int k1, bool need_r, const uint2 *gpre, uint32_t f, int task, int which, int ctid,
                              int warp, int lane) {
    const int H = p.H, H4 = H / 4;
    const bool keep = norm_keeps_x<NB>(p, k0, k1);
    float4 xr[MAXG];
    if (need_r) {
        for (int b = 0; b < p.batch; ++b) {
            const uint64_t *xs = from_embed ? nullptr : xbase + (size_t)b * H;
            const uint16_t *emb = from_embed ? p.embed + (size_t)__ldg(p.tokens + b) * H : nullptr;
            float ss = 0.f;
            if (keep) {
#pragma unroll
                for (int g = 0; g < MAXG; ++g) {
                    const int i4 = ctid + g * NCW * 32;
                    xr[g] = i4 < H4 ? load_x4(p, s, xs, emb, i4, f, task, which) : make_float4(0.f, 0.f, 0.f, 0.f);
                    ss += xr[g].x * xr[g].x + xr[g].y * xr[g].y + xr[g].z * xr[g].z + xr[g].w * xr[g].w;
                }
            } else {
                for (int i4 = ctid; i4 < H4; i4 += NCW * 32) {
                    float4 v = load_x4(p, s, xs, emb, i4, f, task, which);
                    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                }
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
        if (keep) {
            /* every thread derives r itself: no second barrier */
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) ss += s.misc->red[0][w];
            const float r = rsqrtf(ss / (float)H + p.eps);
            float4 *dst = reinterpret_cast<float4 *>(s.act);
#pragma unroll
            for (int g = 0; g < MAXG; ++g) {
                const int i4 = ctid + g * NCW * 32;
                if (i4 < H4) {
                    const uint2 gw = gpre[g];
                    dst[i4] = make_float4(round_bf(xr[g].x * r * bf_lo(gw.x)), round_bf(xr[g].y * r * bf_hi(gw.x)),
                                          round_bf(xr[g].z * r * bf_lo(gw.y)), round_bf(xr[g].w * r * bf_hi(gw.y)));
                }
            }
            return;
        }
        cbar();
    }
    const int kc = k1 - k0;
    for (int b = 0; b < p.batch; ++b) {
        const uint64_t *xs = from_embed ? nullptr : xbase + (size_t)b * H;
        const uint16_t *emb = from_embed ? p.embed + (size_t)__ldg(p.tokens + b) * H : nullptr;
        const float r = s.misc->rnorm[b];
        float4 *dst = reinterpret_cast<float4 *>(s.act + (size_t)b * kc * 4);
        for (int i4 = k0 / 4 + ctid; i4 < k1 / 4; i4 += NCW * 32) {
            float4 v = load_x4(p, s, xs, emb, i4, f, task, which);
            uint2 gw = __ldg(reinterpret_cast<const uint2 *>(gain) + i4);
            dst[i4 - k0 / 4] = make_float4(round_bf(v.x * r * bf_lo(gw.x)), round_bf(v.y * r * bf_hi(gw.x)),
                                           round_bf(v.z * r * bf_lo(gw.y)), round_bf(v.w * r * bf_hi(gw.y)));
        }
    }
}

/* O-projection and down-projection prologues: bf16 activations [k0, k1) of
 * rows of `len` elements (attention output, SwiGLU output), held two per
 * epoch-tagged word, as fp32; waits for their producers */
__device__ void copy_prologue(const Params &p, Smem &s, const uint64_t *src0, int len, int k0, int k1, uint32_t f,
                              int task, int which, int ctid) {
    const int kc = k1 - k0;
    for (int b = 0; b < p.batch; ++b) {
        const uint64_t *src = src0 + ((size_t)b * len + k0) / 2;
        float4 *dst = reinterpret_cast<float4 *>(s.act + (size_t)b * kc * 4);
        for (int i = ctid; i < kc / 4; i += NCW * 32) {
            ulonglong2 v = ld_ll2(src + 2 * i);
            if (!ll_ok(f, v)) ll_settle(p, s, src + 2 * i, v, f, task, which);
            const uint32_t a = (uint32_t)v.x, c = (uint32_t)v.y;
            dst[i] = make_float4(bf_lo(a), bf_hi(a), bf_lo(c), bf_hi(c));
        }
    }
}

/* ----------------------------------------------------------- GEMV tiles */

/* int8 -> fp32, exact: byte b of x becomes (2^23 + 128 + b) by placing b ^ 0x80
 * under the exponent bits of 2^23, then 2^23 + 128 is subtracted. */
__device__ __forceinline__ float i8_to_f(uint32_t xflip, int k) {
    return __uint_as_float(__byte_perm(xflip, 0x4B000000u, 0x7540u | (unsigned)k)) - 8388736.0f;
}

/* Dot product of one 16-byte weight chunk (8 bf16 or 16 int8) with EPC fp32
 * activations at h. */
template <bool I8>
__device__ __forceinline__ float dot_chunk(const uint4 &w, const float *h) {
    const float4 *h4 = reinterpret_cast<const float4 *>(h);
    float s0 = 0.f, s1 = 0.f;
    if constexpr (I8) {
        const uint32_t x[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 a = h4[q];
            s0 = fmaf(i8_to_f(x[q], 0), a.x, s0);
            s1 = fmaf(i8_to_f(x[q], 1), a.y, s1);
            s0 = fmaf(i8_to_f(x[q], 2), a.z, s0);
            s1 = fmaf(i8_to_f(x[q], 3), a.w, s1);
        }
    } else {
        const float4 a = h4[0], c = h4[1];
        s0 = fmaf(bf_lo(w.x), a.x, s0);
        s1 = fmaf(bf_hi(w.x), a.y, s1);
        s0 = fmaf(bf_lo(w.y), a.z, s0);
        s1 = fmaf(bf_hi(w.y), a.w, s1);
        s0 = fmaf(bf_lo(w.z), c.x, s0);
        s1 = fmaf(bf_hi(w.z), c.y, s1);
        s0 = fmaf(bf_lo(w.w), c.z, s0);
        s1 = fmaf(bf_hi(w.w), c.w, s1);
    }
    return s0 + s1;
}

/* Batch-1 tile with the activations in registers: warp w owns K segment
 * w % S (chunks [c0, c1)) and rows w / S, w / S + 8 / S, ...; hv holds this
 * lane's chunks c0 + lane + 32 j of the activation slice.  All of a row's
 * 16-byte shared loads are issued first, then the products go into eight
 * independent accumulators (short dependency chains). */
template <bool I8>
__device__ __forceinline__ void gemv_tile_b1(const uint8_t *tile, int nrows, int S, int Kc, const float4 (*hv)[I8 ? 4 : 2],
                                             int c0, int c1, float *res, bool first, int warp, int lane) {
    constexpr int EPC = I8 ? 16 : 8;
    constexpr int MAXJ = (I8 ? SEGMAX_INT8 : SEGMAX_BF16) / (32 * EPC);
    const int RG = NCW / S, seg = warp % S;
    const size_t rowb = (size_t)Kc * (I8 ? 1 : 2);
    for (int rr = warp / S; rr < nrows; rr += RG) {
        const uint4 *w = reinterpret_cast<const uint4 *>(tile + rr * rowb);
        uint4 wv[MAXJ];
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) {
            const int c = c0 + lane + 32 * j;
            wv[j] = c < c1 ? w[c] : make_uint4(0u, 0u, 0u, 0u);
        }
        float a[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = 0.f;
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) {
            if constexpr (I8) {
                const uint32_t x[4] = {wv[j].x ^ 0x80808080u, wv[j].y ^ 0x80808080u, wv[j].z ^ 0x80808080u,
                                       wv[j].w ^ 0x80808080u};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 h = hv[j][q];
                    a[2 * q] = fmaf(i8_to_f(x[q], 0), h.x, a[2 * q]);
                    a[2 * q + 1] = fmaf(i8_to_f(x[q], 1), h.y, a[2 * q + 1]);
                    a[2 * q] = fmaf(i8_to_f(x[q], 2), h.z, a[2 * q]);
                    a[2 * q + 1] = fmaf(i8_to_f(x[q], 3), h.w, a[2 * q + 1]);
                }
            } else {
                const float4 x = hv[j][0], y = hv[j][1];
                a[0] = fmaf(bf_lo(wv[j].x), x.x, a[0]);
                a[1] = fmaf(bf_hi(wv[j].x), x.y, a[1]);
                a[2] = fmaf(bf_lo(wv[j].y), x.z, a[2]);
                a[3] = fmaf(bf_hi(wv[j].y), x.w, a[3]);
                a[4] = fmaf(bf_lo(wv[j].z), y.x, a[4]);
                a[5] = fmaf(bf_hi(wv[j].z), y.y, a[5]);
                a[6] = fmaf(bf_lo(wv[j].w), y.z, a[6]);
                a[7] = fmaf(bf_hi(wv[j].w), y.w, a[7]);
            }
        }
        const float v = warp_sum(((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7])));
        if (lane == 0) {
            float *r = res + (size_t)rr * S + seg;
            *r = first ? v : *r + v;
        }
    }
}

/* Batched tile: activations act[b][0..Kc) in shared memory.  With S > 1
 * segments per row warp w takes row w / S, K segment w % S; with S == 1 warp
 * w takes rows w, w + 8, ...  Partial sums go to res[(row * S + seg) * Bmax + b]
 * (accumulating over K-split passes); the epilogue adds the S segments in a
 * fixed order, so results do not depend on timing. */
template <bool I8, int NB>
__device__ void gemv_tile(const uint8_t *tile, int nrows, int S, int Kc, const float *act, int batch, float *res,
                          int Bmax, bool first, int warp, int lane) {
    constexpr int EPC = I8 ? 16 : 8;
    const int nch = Kc / EPC;
    const size_t rowb = (size_t)Kc * (I8 ? 1 : 2);
    const int RG = NCW / S, seg = warp % S;
    const int c0 = seg * nch / S, c1 = (seg + 1) * nch / S;
    for (int rr = warp / S; rr < nrows; rr += RG) {
        float a[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) a[b] = 0.f;
        const uint4 *w = reinterpret_cast<const uint4 *>(tile + rr * rowb);
        for (int c = c0 + lane; c < c1; c += 32) {
            const uint4 wv = w[c];
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (b < batch) a[b] += dot_chunk<I8>(wv, act + (size_t)b * Kc + (size_t)c * EPC);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b < batch) {
                const float v = warp_sum(a[b]);
                if (lane == 0) {
                    float *r = res + ((size_t)rr * S + seg) * Bmax + b;
                    *r = first ? v : *r + v;
                }
            }
        }
    }
}

/* residual value x[b][row] of a layer's input: the embedding row at layer 0 */
__device__ __forceinline__ float x_in_value(const Params &p, Smem &s, int l, int b, int row, int task) {
    if (l == 0) return bf2f(__ldg(p.embed + (size_t)__ldg(p.tokens + b) * p.H + row));
    return ll_wait1(p, s, p.x_in + ((size_t)(l % p.depth) * p.Bmax + b) * p.H + row, ver(p, l), task, WB_XIN);
}

template <bool I8, int NB>
__device__ bool gemv_task(const Params &p, Smem &s, const Task &t, int ti, Ring &rg, const uint2 *gpre, int ctid,
                          int warp, int lane) {
    const GemvGeo g = gemv_geo(p, t);
    const int NS = p.n_slots;
    const int l = t.layer, slot = l % p.depth;
    const int S = t.seg;
    for (int kp = 0; kp < g.ks; ++kp) {
        const int k0 = kp * g.Kc, k1 = k0 + g.Kc;
        if (t.op == OP_QKV) {
            const bool emb = l == 0;
            norm_prologue<NB>(p, s, emb ? nullptr : p.x_in + (size_t)slot * p.Bmax * p.H, emb, p.layers[l].attn_norm, k0,
                              k1, kp == 0, gpre, ver(p, l), ti, WB_XIN, ctid, warp, lane);
        } else if (t.op == OP_GUP) {
            norm_prologue<NB>(p, s, p.x_mid + (size_t)slot * p.Bmax * p.H, false, p.layers[l].mlp_norm, k0, k1, kp == 0,
                              gpre, ver(p, l), ti, WB_XMID, ctid, warp, lane);
        } else if (t.op == OP_LMH) {
            norm_prologue<NB>(p, s, p.x_in + (size_t)(p.L % p.depth) * p.Bmax * p.H, false, p.final_norm, k0, k1,
                              kp == 0, gpre, ver(p, p.L), ti, WB_XIN, ctid, warp, lane);
        } else if (t.op == OP_OPR) {
            copy_prologue(p, s, p.aout + (size_t)slot * p.Bmax * p.nq * p.d / 2, p.nq * p.d, k0, k1, ver(p, l), ti,
                          WB_AOUT, ctid);
        } else {
            copy_prologue(p, s, p.act + (size_t)slot * p.Bmax * p.I / 2, p.I, k0, k1, ver(p, l), ti, WB_ACT, ctid);
        }
        if (cbar_or(s.misc->abort != 0)) return false;
        if (p.trace && kp == 0 && ctid == 0) s.misc->t_pro = now_ns();
        /* batch 1: this warp's K segment of the activations into registers */
        constexpr int EPC = I8 ? 16 : 8;
        constexpr int MAXJ = (I8 ? SEGMAX_INT8 : SEGMAX_BF16) / (32 * EPC);
        float4 hv[NB == 1 ? MAXJ : 1][I8 ? 4 : 2];
        const int nch = g.Kc / EPC, seg = warp % S;
        const int c0 = seg * nch / S, c1 = (seg + 1) * nch / S;
        if constexpr (NB == 1) {
            const float4 *a4 = reinterpret_cast<const float4 *>(s.act);
#pragma unroll
            for (int j = 0; j < MAXJ; ++j) {
                const int c = c0 + lane + 32 * j;
#pragma unroll
                for (int q = 0; q < EPC / 4; ++q)
                    hv[j][q] = c < c1 ? a4[(size_t)c * (EPC / 4) + q] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        for (int rb = 0; rb < g.nrb; ++rb) {
            const int ra = t.r0 + rb * g.R, re = min(t.r1, ra + g.R);
            for (int m = 0; m < g.nmat; ++m, rg.advance(NS)) {
                const int sl = rg.slot;
                if (s.misc->abort) continue;
                const unsigned long long tw0 = p.trace ? now_ns() : 0;
                if (!wait_phase(p, s, &s.full[sl], rg.pass & 1u, 2, ti)) continue;
                const unsigned long long tw1 = p.trace ? now_ns() : 0;
                if (p.trace && kp == 0 && rb == 0 && m == 0 && warp == 0 && lane == 0) s.misc->t_first = tw1;
                float *res = s.res + ((size_t)m * g.nrows + (ra - t.r0)) * S * p.Bmax;
                const uint8_t *tile = s.ring + (size_t)sl * p.slot_bytes;
                if constexpr (NB == 1)
                    gemv_tile_b1<I8>(tile, re - ra, S, g.Kc, hv, c0, c1, res, kp == 0, warp, lane);
                else
                    gemv_tile<I8, NB>(tile, re - ra, S, g.Kc, reinterpret_cast<const float *>(s.act), p.batch, res,
                                      p.Bmax, kp == 0, warp, lane);
                if (p.trace && warp == 0 && lane == 0) {
                    s.misc->t_wait_full += tw1 - tw0;
                    s.misc->t_tiles += now_ns() - tw1;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.empty[sl]);
            }
        }
        if (cbar_or(s.misc->abort != 0)) return false;
    }

    /* epilogue: publish the task's rows as epoch-tagged words; a task marked
     * TF_SKIP_SIGNAL publishes them with a stale epoch (timeout tests) */
    if (p.trace && ctid == 0) s.misc->t_stages = now_ns();
    const uint32_t stale = (t.flags & TF_SKIP_SIGNAL) ? (uint32_t)(p.L + 1) : 0u;
    const uint32_t ep = ver(p, l) - stale, ep_next = ver(p, l + 1) - stale;
    const int n = g.nrows, B = p.batch;
    auto y_of = [&](int m, int rr, int b) {
        float y = 0.f;
        for (int sg = 0; sg < S; ++sg) y += s.res[(((size_t)m * n + rr) * S + sg) * p.Bmax + b];
        return I8 ? y * s.sc[m * n + rr] : y;
    };
    if (t.op == OP_GUP) {
        /* two SwiGLU outputs per word: task rows start at an even row and come in pairs */
        for (int i = ctid; i < (n / 2) * B; i += NCW * 32) {
            const int pr = i / B, b = i % B, rr = 2 * pr;
            float a2[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float gte = y_of(0, rr + q, b), up = y_of(1, rr + q, b);
                a2[q] = gte / (1.f + __expf(-gte)) * up;
            }
            st_ll(p.act + (((size_t)slot * p.Bmax + b) * p.I + t.r0 + rr) / 2, pack_bf2(a2[0], a2[1]), ep);
        }
    } else {
        for (int i = ctid; i < n * B; i += NCW * 32) {
            const int rr = i / B, b = i % B, row = t.r0 + rr;
            const float y0 = y_of(0, rr, b);
            switch (t.op) {
            case OP_QKV: {
                const int base = t.mat == MAT_Q ? 0 : t.mat == MAT_K ? p.nq * p.d : (p.nq + p.nkv) * p.d;
                st_ll(p.qkv + ((size_t)slot * p.Bmax + b) * p.qkv_rows + base + row, __float_as_uint(y0), ep);
                break;
            }
            case OP_OPR: {
                const float xr = x_in_value(p, s, l, b, row, ti);
                st_ll(p.x_mid + ((size_t)slot * p.Bmax + b) * p.H + row, __float_as_uint(xr + y0), ep);
                break;
            }
            case OP_DWN: {
                const float xm =
                    ll_wait1(p, s, p.x_mid + ((size_t)slot * p.Bmax + b) * p.H + row, ver(p, l), ti, WB_XMID);
                st_ll(p.x_in + ((size_t)((l + 1) % p.depth) * p.Bmax + b) * p.H + row, __float_as_uint(xm + y0),
                      ep_next);
                break;
            }
            default:
                p.logits[(size_t)b * p.V + row] = y0;
            }
        }
    }
    const bool ok = !cbar_or(s.misc->abort != 0);
    if (p.trace && ctid == 0) s.misc->t_epi = now_ns();
    return ok;
}

/* ----------------------------------------------------------- attention */

struct AttSmem {
    float *q;        /* [G][d], pre-scaled by log2(e)/sqrt(d) */
    uint16_t *knew;  /* [d] bf16(rope(k)) of position p */
    uint16_t *vnew;  /* [d] */
    float *wst;      /* [NCW][d + PART_PAD]: per-warp (o, m, l) */
    float *sbuf;     /* [NCW][32]: per-warp scores, then probabilities, of a block */
};

__device__ __forceinline__ AttSmem att_smem(const Params &p, Smem &s) {
    AttSmem a;
    uint8_t *base = s.act;
    a.q = reinterpret_cast<float *>(base);
    base += align_up(p.G * p.d * 4, 16);
    a.knew = reinterpret_cast<uint16_t *>(base);
    a.vnew = a.knew + p.d;
    base += align_up(2 * p.d * 2, 16);
    a.wst = reinterpret_cast<float *>(base);
    a.sbuf = a.wst + NCW * (p.d + PART_PAD);
    return a;
}

/* Online-softmax state of one warp, which owns one head and a subset of the
 * positions.  LP = d / 8 lanes share a position when scoring (8 elements
 * each); for the P.V product every lane owns d / 32 output elements. */
template <int LP>
struct AttState {
    float q[8];
    float o[LP / 4];
    float m;  /* running max, warp-uniform (log2 units) */
    float l;  /* this lane's share of the running sum */
};

/* positions j0 .. j0 + nb - 1 (nb <= 32) of a K/V tile in shared memory */
template <int LP>
__device__ __forceinline__ void att_block(AttState<LP> &st, const uint16_t *Kt, const uint16_t *Vt, int j0, int nb,
                                          int d, float *sb, int lane) {
    constexpr int PW = 32 / LP, EL = LP / 4;
    const int pg = lane / LP, ch = lane % LP;
#pragma unroll
    for (int it = 0; it < LP; ++it) {
        const int jj = it * PW + pg;
        float sc = -INFINITY;
        if (jj < nb) {
            const uint4 kv = reinterpret_cast<const uint4 *>(Kt + (size_t)(j0 + jj) * d)[ch];
            const float s0 = st.q[0] * bf_lo(kv.x) + st.q[1] * bf_hi(kv.x) + st.q[2] * bf_lo(kv.y) + st.q[3] * bf_hi(kv.y);
            const float s1 = st.q[4] * bf_lo(kv.z) + st.q[5] * bf_hi(kv.z) + st.q[6] * bf_lo(kv.w) + st.q[7] * bf_hi(kv.w);
            sc = s0 + s1;
        }
#pragma unroll
        for (int o = LP / 2; o > 0; o >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
        if (ch == 0) sb[jj] = sc;
    }
    __syncwarp();
    const float si = sb[lane];
    float mb = si;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const float mnew = fmaxf(st.m, mb);
    const float alpha = exp2f(st.m - mnew);
    const float pi = lane < nb ? exp2f(si - mnew) : 0.f;
    st.l = st.l * alpha + pi;
    st.m = mnew;
#pragma unroll
    for (int e = 0; e < EL; ++e) st.o[e] *= alpha;
    __syncwarp();
    sb[lane] = pi;
    __syncwarp();
    const uint16_t *vcol = Vt + (size_t)j0 * d + lane * EL;
    for (int i = 0; i < nb; ++i) {
        const float w = sb[i];
        if constexpr (EL == 2) {
            const uint32_t v = *reinterpret_cast<const uint32_t *>(vcol + (size_t)i * d);
            st.o[0] = fmaf(w, bf_lo(v), st.o[0]);
            st.o[1] = fmaf(w, bf_hi(v), st.o[1]);
        } else {
            const uint2 v = *reinterpret_cast<const uint2 *>(vcol + (size_t)i * d);
            st.o[0] = fmaf(w, bf_lo(v.x), st.o[0]);
            st.o[1] = fmaf(w, bf_hi(v.x), st.o[1]);
            st.o[2] = fmaf(w, bf_lo(v.y), st.o[2]);
            st.o[3] = fmaf(w, bf_hi(v.y), st.o[3]);
        }
    }
    __syncwarp();
}

template <int LP>
__device__ __forceinline__ void att_tile(AttState<LP> &st, const uint16_t *Kt, const uint16_t *Vt, int nt, int d,
                                         int sub, int wph, float *sb, int lane) {
    for (int j0 = sub * 32; j0 < nt; j0 += wph * 32) att_block<LP>(st, Kt, Vt, j0, min(32, nt - j0), d, sb, lane);
}

template <int LP>
__device__ bool att_task_impl(const Params &p, Smem &s, const Task &t, int ti, Ring &rg, int ctid, int warp, int lane) {
    const int d = p.d, G = p.G, NS = p.n_slots;
    const int l = t.layer, slot = l % p.depth, b = t.b, grp = t.g;
    const AttGeo ag = att_geo(p, t);
    const bool active_seq = b < p.batch;
    AttSmem as = att_smem(p, s);

    /* prologue: wait for q, k, v of this kv head, rotate q and the new k,
     * round k and v to bf16 */
    if (active_seq) {
        const uint64_t *qkv = p.qkv + ((size_t)slot * p.Bmax + b) * p.qkv_rows;
        const float *rope = p.rope + (size_t)ag.p * d; /* [d/2][2] */
        const int half = d / 2;
        for (int i = ctid; i < (G + 2) * half; i += NCW * 32) {
            const int h = i / half, e = i % half;
            const float c = __ldg(rope + 2 * e), sn = __ldg(rope + 2 * e + 1);
            const uint64_t *src = h < G ? qkv + (size_t)(grp * G + h) * d
                                 : h == G ? qkv + (size_t)p.nq * d + grp * d
                                          : qkv + (size_t)(p.nq + p.nkv) * d + grp * d;
            const uint32_t f = ver(p, l);
            uint64_t wa = ld_ll1(src + e), wb = ld_ll1(src + e + half);
            const float a = ll_flag(wa) == f ? ll_f(wa) : ll_wait1(p, s, src + e, f, ti, WB_QKV);
            const float bb = ll_flag(wb) == f ? ll_f(wb) : ll_wait1(p, s, src + e + half, f, ti, WB_QKV);
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
    if (cbar_or(s.misc->abort != 0)) return false;
    if (active_seq && (t.flags & TF_NEW_TOKEN)) {
        const size_t row = ((((size_t)l * p.Bmax + b) * p.nkv + grp) * p.Smax + ag.p) * d;
        for (int i = ctid; i < d; i += NCW * 32) {
            p.kc[row + i] = as.knew[i];
            p.vc[row + i] = as.vnew[i];
        }
    }

    const int wph = NCW / G;
    const bool wactive = warp < wph * G;
    const int h = warp % G, sub = warp / G;
    const int ch = lane % LP;
    constexpr int EL = LP / 4;
    float *sb = as.sbuf + warp * 32;
    AttState<LP> st;
    st.m = -INFINITY;
    st.l = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) st.q[e] = wactive ? as.q[h * d + ch * 8 + e] : 0.f;
#pragma unroll
    for (int e = 0; e < EL; ++e) st.o[e] = 0.f;

    for (int k = 0; k < ag.ntile; ++k, rg.advance(NS)) {
        const int sl = rg.slot;
        if (s.misc->abort) continue;
        const unsigned long long tw0 = p.trace ? now_ns() : 0;
        if (!wait_phase(p, s, &s.full[sl], rg.pass & 1u, 2, ti)) continue;
        const unsigned long long tw1 = p.trace ? now_ns() : 0;
        if (p.trace && k == 0 && warp == 0 && lane == 0) s.misc->t_first = tw1;
        const int t0 = ag.s0 + k * t.rows_per_stage;
        const int nt = min(ag.e, t0 + (int)t.rows_per_stage) - t0;
        const uint16_t *Kt = reinterpret_cast<const uint16_t *>(s.ring + (size_t)sl * p.slot_bytes);
        const uint16_t *Vt = Kt + (size_t)t.rows_per_stage * d;
        if (wactive) att_tile<LP>(st, Kt, Vt, nt, d, sub, wph, sb, lane);
        if (p.trace && warp == 0 && lane == 0) {
            s.misc->t_wait_full += tw1 - tw0;
            s.misc->t_tiles += now_ns() - tw1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.empty[sl]);
    }
    if (active_seq && (t.flags & TF_NEW_TOKEN) && wactive) att_tile<LP>(st, as.knew, as.vnew, 1, d, sub, wph, sb, lane);

    /* the warp's state: l summed over lanes, o spread EL elements per lane */
    st.l = warp_sum(st.l);
    if (wactive) {
        float *w = as.wst + (size_t)warp * (d + PART_PAD);
#pragma unroll
        for (int e = 0; e < EL; ++e) w[lane * EL + e] = st.o[e];
        if (lane == 0) {
            w[d] = st.m;
            w[d + 1] = st.l;
        }
    }
    if (cbar_or(s.misc->abort != 0)) return false;

    /* merge the warps of each head; publish the chunk's partial (o unnormalised, m, l) */
    if (active_seq) {
        const uint32_t ep = ver(p, l) - ((t.flags & TF_SKIP_SIGNAL) ? (uint32_t)(p.L + 1) : 0u);
        uint64_t *part = p.part + ((((size_t)slot * p.Bmax + b) * p.nkv + grp) * p.C + t.r0) * G * (d + PART_PAD);
        for (int i = ctid; i < G * (d + 2); i += NCW * 32) {
            const int hh = i / (d + 2), e = i % (d + 2);
            float M = -INFINITY;
            for (int w2 = 0; w2 < wph; ++w2) M = fmaxf(M, as.wst[(size_t)(w2 * G + hh) * (d + PART_PAD) + d]);
            float v = 0.f;
            if (e == d) {
                v = M;
            } else if (M != -INFINITY) {
                for (int w2 = 0; w2 < wph; ++w2) {
                    const float *w = as.wst + (size_t)(w2 * G + hh) * (d + PART_PAD);
                    const float mw = w[d];
                    if (mw == -INFINITY) continue;
                    v += exp2f(mw - M) * (e == d + 1 ? w[d + 1] : w[e]);
                }
            }
            st_ll(part + (size_t)hh * (d + PART_PAD) + e, __float_as_uint(v), ep);
        }
    }
    return !cbar_or(s.misc->abort != 0);
}

/* Merge the C chunk partials of one (sequence, kv head) into bf16 attention
 * outputs of its G heads: o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c
 * (the log-sum-exp combination of split softmax), in chunk order. */
__device__ bool mrg_task(const Params &p, Smem &s, const Task &t, int ti, int ctid) {
    const int d = p.d, G = p.G, C = t.r1, slot = t.layer % p.depth, b = t.b, grp = t.g;
    if (b < p.batch) {
        const uint32_t f = ver(p, t.layer);
        const uint32_t ep = f - ((t.flags & TF_SKIP_SIGNAL) ? (uint32_t)(p.L + 1) : 0u);
        const uint64_t *base = p.part + (((size_t)slot * p.Bmax + b) * p.nkv + grp) * C * G * (d + PART_PAD);
        float *ml = s.fac;         /* [G][C] m, then factors */
        float *lv = s.fac + G * C; /* [G][C] l */
        for (int i = ctid; i < G * C; i += NCW * 32) {
            const int h = i / C, c = i % C;
            const uint64_t *pc = base + ((size_t)c * G + h) * (d + PART_PAD) + d;
            ulonglong2 v = ld_ll2(pc);
            if (!ll_ok(f, v)) ll_settle(p, s, pc, v, f, ti, WB_PART);
            ml[i] = ll_f(v.x);
            lv[i] = ll_f(v.y);
        }
        if (cbar_or(s.misc->abort != 0)) return false;
        if (ctid < G) {
            float M = -INFINITY;
            for (int c = 0; c < C; ++c) M = fmaxf(M, ml[ctid * C + c]);
            float den = 0.f;
            for (int c = 0; c < C; ++c) {
                const float mc = ml[ctid * C + c];
                const float f = mc == -INFINITY ? 0.f : exp2f(mc - M);
                ml[ctid * C + c] = f;
                den += f * lv[ctid * C + c];
            }
            const float inv = 1.f / den;
            for (int c = 0; c < C; ++c) ml[ctid * C + c] *= inv;
        }
        cbar();
        uint64_t *out = p.aout + (((size_t)slot * p.Bmax + b) * p.nq * d + (size_t)grp * G * d) / 2;
        const int q4 = d / 4;
        for (int i = ctid; i < G * q4; i += NCW * 32) {
            const int h = i / q4, e4 = i % q4;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int c = 0; c < C; ++c) {
                const float w = ml[h * C + c];
                const uint64_t *src = base + ((size_t)c * G + h) * (d + PART_PAD) + 4 * e4;
                ulonglong2 u = ld_ll2(src), v = ld_ll2(src + 2);
                if (!ll_ok(f, u)) ll_settle(p, s, src, u, f, ti, WB_PART);
                if (!ll_ok(f, v)) ll_settle(p, s, src + 2, v, f, ti, WB_PART);
                o.x = fmaf(w, ll_f(u.x), o.x);
                o.y = fmaf(w, ll_f(u.y), o.y);
                o.z = fmaf(w, ll_f(v.x), o.z);
                o.w = fmaf(w, ll_f(v.y), o.w);
            }
            st_ll(out + ((size_t)h * d + 4 * e4) / 2, pack_bf2(o.x, o.y), ep);
            st_ll(out + ((size_t)h * d + 4 * e4) / 2 + 1, pack_bf2(o.z, o.w), ep);
        }
    }
    return !cbar_or(s.misc->abort != 0);
}

/* ----------------------------------------------------------- the kernel */

template <bool I8, int NB>
__global__ void __launch_bounds__(NTHREADS, 1) amk_decode_kernel(const Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Smem s;
    s.full = reinterpret_cast<uint64_t *>(smem);
    s.empty = s.full + MAX_SLOTS;
    s.misc = reinterpret_cast<Misc *>(smem + SMEM_BARRIERS);
    s.res = reinterpret_cast<float *>(smem + SMEM_BARRIERS + SMEM_MISC);
    s.sc = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(s.res) + p.result_bytes);
    s.fac = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(s.sc) + p.scale_bytes);
    s.act = reinterpret_cast<uint8_t *>(s.fac) + p.fac_bytes;
    s.ring = s.act + p.act_bytes;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tbeg = p.task_start[blockIdx.x], tend = p.task_start[blockIdx.x + 1];

    if (tid == 0) {
        s.misc->abort = 0;
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
    const bool stale = __syncthreads_or(tid == 0 && (bad_input || ld_relaxed(p.err) != 0u));
    if (stale) return;

    if (warp == NCW) {
        if (lane == 0) loader(p, s, tbeg, tend);
    } else {
        const int ctid = tid;
        Ring rg{0, 0, 0};
        for (int ti = tbeg; ti < tend; ++ti) {
            Task t;
            load_task(p.tasks + ti, t);
            /* weights-only inputs are fetched before the task's inputs are ready */
            if (I8 && t.op != OP_ATT && t.op != OP_MRG) {
                const int n = t.r1 - t.r0, nm = t.op == OP_GUP ? 2 : 1;
                for (int i = ctid; i < n * nm; i += NCW * 32) {
                    const int m = i / n, rr = i % n;
                    s.sc[i] = __ldg(op_scales(p, t, m) + t.r0 + rr);
                }
            }
            uint2 gpre[MAXG];
            if (NB == 1 && (t.op == OP_QKV || t.op == OP_GUP || t.op == OP_LMH) && t.ksplit == 1) {
                const uint16_t *gain = t.op == OP_QKV   ? p.layers[t.layer].attn_norm
                                       : t.op == OP_GUP ? p.layers[t.layer].mlp_norm
                                                        : p.final_norm;
#pragma unroll
                for (int g = 0; g < MAXG; ++g) {
                    const int i4 = ctid + g * NCW * 32;
                    gpre[g] = i4 < p.H / 4 ? __ldg(reinterpret_cast<const uint2 *>(gain) + i4) : make_uint2(0, 0);
                }
            }
            unsigned long long *tr = p.trace ? p.trace + 16 * (size_t)ti : nullptr;
            if (tr && ctid == 0) {
                tr[0] = tr[1] = now_ns();
                s.misc->t_first = 0;
                s.misc->t_wait_full = 0;
                s.misc->t_tiles = 0;
                s.misc->t_pro = s.misc->t_stages = s.misc->t_epi = 0;
            }
            bool ok;
            if (t.op == OP_ATT)
                ok = p.d == 64 ? att_task_impl<8>(p, s, t, ti, rg, ctid, warp, lane)
                               : att_task_impl<16>(p, s, t, ti, rg, ctid, warp, lane);
            else if (t.op == OP_MRG)
                ok = mrg_task(p, s, t, ti, ctid);
            else
                ok = gemv_task<I8, NB>(p, s, t, ti, rg, gpre, ctid, warp, lane);
            if (!ok) break;
            if (tr && ctid == 0) {
                tr[2] = s.misc->t_first;
                tr[3] = now_ns();
                tr[4] = s.misc->t_wait_full;
                tr[5] = s.misc->t_tiles;
                tr[6] = s.misc->t_pro;
                tr[7] = s.misc->t_stages;
                tr[8] = s.misc->t_epi;
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

/* ----------------------------------------------------------- host entry */

KernelFn select_kernel(bool int8, int max_batch) {
    if (int8) return max_batch == 1 ? amk_decode_kernel<true, 1> : amk_decode_kernel<true, MAXB>;
    return max_batch == 1 ? amk_decode_kernel<false, 1> : amk_decode_kernel<false, MAXB>;
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
