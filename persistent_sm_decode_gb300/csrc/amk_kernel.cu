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
 * high-bandwidth GPUs; this kernel synchronises only through per-dependency
 * counters and never through a grid-wide barrier.
 *
 * GB300 (sm_103a) design:
 *  - grid = one CTA per SM (cooperative launch, so every CTA is resident);
 *  - warp 8 is the LOADER: one thread streams every weight tile and KV tile
 *    of the CTA's task list into a ring of shared-memory slots with
 *    cp.async.bulk (TMA bulk copies) completing on mbarriers.  Weights and
 *    the cached prefix never depend on this step's activations, so the
 *    loader runs ahead across dependency waits and keeps HBM busy;
 *  - warps 0-7 are CONSUMERS: per task, thread 0 acts as CONTROLLER (waits
 *    on the task's dependency counter with ld.acquire, bounded by a
 *    globaltimer limit), all consumers run the prologue (RMSNorm, attention
 *    partial merge, or activation copy into shared memory), the GEMV or
 *    attention tiles from the ring, and the epilogue (residual, SwiGLU,
 *    partials, logits); thread 0 then acts as STORER (fence + counter
 *    increment) so that consumers of the result may start;
 *  - GEMV: CUDA-core dot products with fp32 accumulation, warp-shuffle
 *    reductions, 16-byte shared-memory reads;
 *  - attention: split-context flash-decoding; each chunk keeps an online
 *    softmax (log2 domain) and writes (m, l, o) partials that the O
 *    projection's prologue merges;
 *  - every wait is bounded: on timeout the CTA records the error, stops, waits
 *    for its own bulk copies in flight and returns; later launches see the
 *    error word and do nothing until the host clears it.
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

__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

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
};

struct Smem {
    uint64_t *full, *empty;
    Misc *misc;
    float *res;
    float *sc;
    uint8_t *act;
    uint8_t *ring;
};

/* first error wins; every CTA then stops at its next check */
__device__ void raise_error(const Params &p, Smem &s, int code, int task, int counter, uint32_t seen,
                            uint32_t target) {
    if (atomicCAS(&p.err[0], 0u, (uint32_t)code) == 0u) {
        p.err[1] = blockIdx.x;
        p.err[2] = (uint32_t)task;
        p.err[3] = (uint32_t)counter;
        p.err[4] = seen;
        p.err[5] = target;
        __threadfence();
    }
    s.misc->abort = 1;
}

/* bounded wait on an mbarrier phase; false on abort or timeout */
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
            if ((long long)(now_ns() - t0) > p.timeout_ns) {
                raise_error(p, s, code, task, -1, 0, parity);
                return false;
            }
        }
    }
}

/* controller: wait until counter `id` reaches epoch * count; false on abort or timeout */
__device__ bool wait_counter(const Params &p, Smem &s, int id, uint32_t count, int task) {
    const uint32_t *c = p.counters + (size_t)id * COUNTER_STRIDE;
    const uint32_t target = p.epoch * count;
    uint32_t v = ld_acquire(c);
    if ((int32_t)(v - target) >= 0) return true;
    uint64_t t0 = now_ns();
    for (uint32_t n = 1;; ++n) {
        v = ld_acquire(c);
        if ((int32_t)(v - target) >= 0) return true;
        if ((n & 15u) == 0u) {
            if (ld_relaxed(p.err) != 0u) {
                s.misc->abort = 1;
                return false;
            }
            if ((long long)(now_ns() - t0) > p.timeout_ns) {
                raise_error(p, s, 1, task, id, v, target);
                return false;
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

__device__ __forceinline__ int num_stages(const Params &p, const Task &t) {
    if (t.op == OP_ATT) return att_geo(p, t).ntile;
    GemvGeo g = gemv_geo(p, t);
    return g.ks * g.nrb * g.nmat;
}

__device__ __forceinline__ void load_task(const Task *src, Task &t) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
    uint4 *d = reinterpret_cast<uint4 *>(&t);
    d[0] = __ldg(s);
    d[1] = __ldg(s + 1);
    d[2] = __ldg(s + 2);
}

/* ----------------------------------------------------------- loader */

__device__ void loader(const Params &p, Smem &s, int tbeg, int tend) {
    const int NS = p.n_slots;
    uint32_t it = 0;
    for (int ti = tbeg; ti < tend; ++ti) {
        Task t;
        load_task(p.tasks + ti, t);
        const int ns = num_stages(p, t);
        GemvGeo g;
        AttGeo a;
        const uint8_t *kbase = nullptr, *vbase = nullptr;
        if (t.op == OP_ATT) {
            a = att_geo(p, t);
            size_t row = (((size_t)t.layer * p.Bmax + t.b) * p.nkv + t.g) * (size_t)p.Smax;
            kbase = (const uint8_t *)(p.kc + row * p.d);
            vbase = (const uint8_t *)(p.vc + row * p.d);
        } else {
            g = gemv_geo(p, t);
        }
        for (int st = 0; st < ns; ++st, ++it) {
            const int slot = (int)(it % (uint32_t)NS);
            if (it >= (uint32_t)NS && !wait_phase(p, s, &s.empty[slot], ((it / NS) - 1u) & 1u, 3, ti)) {
                s.misc->issued = (int)it;
                return;
            }
            if (s.misc->abort) {
                s.misc->issued = (int)it;
                return;
            }
            uint8_t *dst = s.ring + (size_t)slot * p.slot_bytes;
            uint64_t *bar = &s.full[slot];
            if (t.op == OP_ATT) {
                const int t0 = a.s0 + st * t.rows_per_stage;
                const int t1 = min(a.e, t0 + (int)t.rows_per_stage);
                const uint32_t bytes = (uint32_t)(t1 - t0) * p.d * 2;
                mbar_arrive_expect_tx(bar, 2 * bytes);
                bulk_copy(dst, kbase + (size_t)t0 * p.d * 2, bytes, bar);
                bulk_copy(dst + (size_t)t.rows_per_stage * p.d * 2, vbase + (size_t)t0 * p.d * 2, bytes, bar);
            } else {
                const int kp = st / (g.nrb * g.nmat), rem = st % (g.nrb * g.nmat);
                const int rb = rem / g.nmat, m = rem % g.nmat;
                const int ra = t.r0 + rb * g.R, re = min(t.r1, ra + g.R);
                const int web = (t.op == OP_LMH ? p.lm_int8 : p.wint8) ? 1 : 2;
                const uint8_t *W = op_weights(p, t, m);
                const size_t rowb = (size_t)g.K * web, segb = (size_t)g.Kc * web;
                const uint32_t bytes = (uint32_t)((re - ra) * segb);
                mbar_arrive_expect_tx(bar, bytes);
                if (g.ks == 1) {
                    bulk_copy(dst, W + (size_t)ra * rowb, bytes, bar);
                } else {
                    for (int r = ra; r < re; ++r)
                        bulk_copy(dst + (size_t)(r - ra) * segb, W + (size_t)r * rowb + (size_t)kp * segb, (uint32_t)segb, bar);
                }
            }
        }
    }
    s.misc->issued = (int)it;
}

/* ----------------------------------------------------------- prologues */

/* x (fp32 residual) that a norm or residual reads: layer-0 input is the
 * token's embedding row */
__device__ __forceinline__ float4 load_x4(const Params &p, const float *xs, const uint16_t *emb, int i4) {
    if (emb) {
        uint2 w = __ldg(reinterpret_cast<const uint2 *>(emb) + i4);
        return make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
    }
    return __ldcg(reinterpret_cast<const float4 *>(xs) + i4);
}

/* RMSNorm prologue: act[b][k - k0] = bf16(x[b][k] * r_b * gain[k]) for k in [k0, k1) */
__device__ void norm_prologue(const Params &p, Smem &s, const float *xbase, bool from_embed, const uint16_t *gain,
                              int k0, int k1, bool need_r, int ctid, int warp, int lane) {
    const int H = p.H, H4 = H / 4;
    if (need_r) {
        for (int b = 0; b < p.batch; ++b) {
            const float *xs = from_embed ? nullptr : xbase + (size_t)b * H;
            const uint16_t *emb = from_embed ? p.embed + (size_t)__ldg(p.tokens + b) * H : nullptr;
            float ss = 0.f;
            for (int i4 = ctid; i4 < H4; i4 += NCW * 32) {
                float4 v = load_x4(p, xs, emb, i4);
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
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
    const int kc = k1 - k0;
    for (int b = 0; b < p.batch; ++b) {
        const float *xs = from_embed ? nullptr : xbase + (size_t)b * H;
        const uint16_t *emb = from_embed ? p.embed + (size_t)__ldg(p.tokens + b) * H : nullptr;
        const float r = s.misc->rnorm[b];
        uint2 *dst = reinterpret_cast<uint2 *>(s.act + (size_t)b * kc * 2);
        for (int i4 = k0 / 4 + ctid; i4 < k1 / 4; i4 += NCW * 32) {
            float4 v = load_x4(p, xs, emb, i4);
            uint2 gw = __ldg(reinterpret_cast<const uint2 *>(gain) + i4);
            uint2 o;
            o.x = pack_bf2(v.x * r * bf_lo(gw.x), v.y * r * bf_hi(gw.x));
            o.y = pack_bf2(v.z * r * bf_lo(gw.y), v.w * r * bf_hi(gw.y));
            dst[i4 - k0 / 4] = o;
        }
    }
}

/* O-projection prologue: merge the attention partials of every chunk into
 * bf16(o) for k in [k0, k1) of the concatenated heads */
__device__ void merge_prologue(const Params &p, Smem &s, int layer, int k0, int k1, int ctid) {
    const int d = p.d, dq = d / 4, C = p.C, G = p.G, slot = layer % p.depth;
    const int kc = k1 - k0;
    const int items = p.batch * (kc / 4);
    for (int it = ctid; it < items; it += NCW * 32) {
        const int b = it / (kc / 4);
        const int k = k0 + (it % (kc / 4)) * 4;
        const int j = k / d, e4 = (k % d) / 4, grp = j / G, h = j % G;
        const float *base = p.part + ((((size_t)slot * p.Bmax + b) * p.nkv + grp) * C * G + h) * (d + PART_PAD);
        const size_t cstride = (size_t)G * (d + PART_PAD);
        float M = -INFINITY;
        for (int c = 0; c < C; ++c) M = fmaxf(M, __ldcg(base + c * cstride + d));
        float den = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < C; ++c) {
            const float *pc = base + c * cstride;
            const float mc = __ldcg(pc + d);
            if (mc == -INFINITY) continue;
            const float f = exp2f(mc - M);
            den += f * __ldcg(pc + d + 1);
            float4 oc = __ldcg(reinterpret_cast<const float4 *>(pc) + e4);
            o.x += f * oc.x;
            o.y += f * oc.y;
            o.z += f * oc.z;
            o.w += f * oc.w;
        }
        const float inv = 1.f / den;
        uint2 w;
        w.x = pack_bf2(o.x * inv, o.y * inv);
        w.y = pack_bf2(o.z * inv, o.w * inv);
        reinterpret_cast<uint2 *>(s.act + (size_t)b * kc * 2)[(k - k0) / 4] = w;
        (void)dq;
    }
}

/* down-projection prologue: copy bf16 SwiGLU activations [k0, k1) */
__device__ void copy_prologue(const Params &p, Smem &s, int layer, int k0, int k1, int ctid) {
    const int slot = layer % p.depth, kc = k1 - k0;
    for (int b = 0; b < p.batch; ++b) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.act + ((size_t)slot * p.Bmax + b) * p.I + k0);
        uint4 *dst = reinterpret_cast<uint4 *>(s.act + (size_t)b * kc * 2);
        for (int i = ctid; i < kc / 8; i += NCW * 32) dst[i] = __ldcg(src + i);
    }
}

/* ----------------------------------------------------------- GEMV tile */

template <bool I8>
__device__ __forceinline__ void unpack16(const uint4 &w, float *f) {
    if constexpr (I8) {
        const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int k = 0; k < 4; ++k) f[4 * q + k] = (float)(int8_t)(x[q] >> (8 * k));
        }
    } else {
        f[0] = bf_lo(w.x);
        f[1] = bf_hi(w.x);
        f[2] = bf_lo(w.y);
        f[3] = bf_hi(w.y);
        f[4] = bf_lo(w.z);
        f[5] = bf_hi(w.z);
        f[6] = bf_lo(w.w);
        f[7] = bf_hi(w.w);
    }
}

/* rows [0, nrows) of a tile of width Kc in shared memory, times the bf16
 * activation slice act[b][0..Kc); warp-per-row, two rows per pass sharing the
 * activation loads; results (or partial sums for K split) into res[rr][b] */
template <bool I8, int NB>
__device__ void gemv_tile(const uint8_t *tile, int nrows, int Kc, const uint8_t *act, int batch, float *res, int Bmax,
                          bool first, int warp, int lane) {
    constexpr int EPC = I8 ? 16 : 8;
    const int nch = Kc / EPC;
    const size_t rowb = (size_t)Kc * (I8 ? 1 : 2);
    for (int rr = warp; rr < nrows; rr += 2 * NCW) {
        const int rr2 = rr + NCW;
        const bool two = rr2 < nrows;
        float a0[NB], a1[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) a0[b] = a1[b] = 0.f;
        const uint4 *w0 = reinterpret_cast<const uint4 *>(tile + rr * rowb);
        const uint4 *w1 = reinterpret_cast<const uint4 *>(tile + (two ? rr2 : rr) * rowb);
        for (int c = lane; c < nch; c += 32) {
            float f0[EPC], f1[EPC];
            unpack16<I8>(w0[c], f0);
            if (two) unpack16<I8>(w1[c], f1);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b < batch) {
                    const uint4 *hp = reinterpret_cast<const uint4 *>(act + ((size_t)b * Kc + (size_t)c * EPC) * 2);
                    float h[EPC];
                    unpack16<false>(hp[0], h);
                    if constexpr (I8) unpack16<false>(hp[1], h + 8);
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int e = 0; e < EPC; ++e) s0 = fmaf(f0[e], h[e], s0);
                    a0[b] += s0;
                    if (two) {
#pragma unroll
                        for (int e = 0; e < EPC; ++e) s1 = fmaf(f1[e], h[e], s1);
                        a1[b] += s1;
                    }
                }
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b < batch) {
                float v0 = warp_sum(a0[b]);
                float v1 = two ? warp_sum(a1[b]) : 0.f;
                if (lane == 0) {
                    float *r0 = res + (size_t)rr * Bmax + b;
                    *r0 = first ? v0 : *r0 + v0;
                    if (two) {
                        float *r1 = res + (size_t)rr2 * Bmax + b;
                        *r1 = first ? v1 : *r1 + v1;
                    }
                }
            }
        }
    }
}

template <bool I8, int NB>
__device__ bool gemv_task(const Params &p, Smem &s, const Task &t, int ti, uint32_t &it, int ctid, int warp, int lane) {
    const GemvGeo g = gemv_geo(p, t);
    const int NS = p.n_slots;
    const int l = t.layer, slot = l % p.depth;
    constexpr bool i8 = I8; /* the LM head has the layers' weight type (tied heads are bf16) */
    for (int kp = 0; kp < g.ks; ++kp) {
        const int k0 = kp * g.Kc, k1 = k0 + g.Kc;
        if (t.op == OP_QKV) {
            const bool emb = l == 0;
            norm_prologue(p, s, emb ? nullptr : p.x_in + (size_t)slot * p.Bmax * p.H, emb, p.layers[l].attn_norm, k0, k1,
                          kp == 0, ctid, warp, lane);
        } else if (t.op == OP_GUP) {
            norm_prologue(p, s, p.x_mid + (size_t)slot * p.Bmax * p.H, false, p.layers[l].mlp_norm, k0, k1, kp == 0, ctid,
                          warp, lane);
        } else if (t.op == OP_LMH) {
            norm_prologue(p, s, p.x_in + (size_t)(p.L % p.depth) * p.Bmax * p.H, false, p.final_norm, k0, k1, kp == 0,
                          ctid, warp, lane);
        } else if (t.op == OP_OPR) {
            merge_prologue(p, s, l, k0, k1, ctid);
        } else {
            copy_prologue(p, s, l, k0, k1, ctid);
        }
        if (cbar_or(s.misc->abort != 0)) return false;
        for (int rb = 0; rb < g.nrb; ++rb) {
            const int ra = t.r0 + rb * g.R, re = min(t.r1, ra + g.R);
            for (int m = 0; m < g.nmat; ++m, ++it) {
                const int sl = (int)(it % (uint32_t)NS);
                if (s.misc->abort) continue;
                if (!wait_phase(p, s, &s.full[sl], (it / NS) & 1u, 2, ti)) continue;
                float *res = s.res + ((size_t)m * g.nrows + (ra - t.r0)) * p.Bmax;
                const uint8_t *tile = s.ring + (size_t)sl * p.slot_bytes;
                gemv_tile<I8, NB>(tile, re - ra, g.Kc, s.act, p.batch, res, p.Bmax, kp == 0, warp, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.empty[sl]);
            }
        }
        if (cbar_or(s.misc->abort != 0)) return false;
    }

    /* epilogue */
    const int n = g.nrows, B = p.batch;
    for (int i = ctid; i < n * B; i += NCW * 32) {
        const int rr = i / B, b = i % B, row = t.r0 + rr;
        float y0 = s.res[(size_t)rr * p.Bmax + b];
        if (i8) y0 *= s.sc[rr];
        switch (t.op) {
        case OP_QKV: {
            const int base = t.mat == MAT_Q ? 0 : t.mat == MAT_K ? p.nq * p.d : (p.nq + p.nkv) * p.d;
            p.qkv[((size_t)slot * p.Bmax + b) * p.qkv_rows + base + row] = y0;
            break;
        }
        case OP_OPR: {
            const float xr = l == 0 ? bf2f(__ldg(p.embed + (size_t)__ldg(p.tokens + b) * p.H + row))
                                    : __ldcg(p.x_in + ((size_t)slot * p.Bmax + b) * p.H + row);
            p.x_mid[((size_t)slot * p.Bmax + b) * p.H + row] = xr + y0;
            break;
        }
        case OP_GUP: {
            float y1 = s.res[((size_t)n + rr) * p.Bmax + b];
            if (i8) y1 *= s.sc[n + rr];
            const float a = y0 / (1.f + __expf(-y0)) * y1;
            p.act[((size_t)slot * p.Bmax + b) * p.I + row] = f2bf(a);
            break;
        }
        case OP_DWN: {
            const float xm = __ldcg(p.x_mid + ((size_t)slot * p.Bmax + b) * p.H + row);
            p.x_in[((size_t)((l + 1) % p.depth) * p.Bmax + b) * p.H + row] = xm + y0;
            break;
        }
        default:
            p.logits[(size_t)b * p.V + row] = y0;
        }
    }
    return !cbar_or(s.misc->abort != 0);
}

/* ----------------------------------------------------------- attention */

struct AttSmem {
    float *q;        /* [G][d], pre-scaled by log2(e)/sqrt(d) */
    uint16_t *knew;  /* [d] bf16(rope(k)) of position p */
    uint16_t *vnew;  /* [d] */
    float *wst;      /* [NCW][d + PART_PAD]: per-warp (o, m, l) */
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
    return a;
}

/* per-warp online-softmax state; a warp owns one head and a subset of positions */
template <int LP>
struct AttState {
    float q[8];
    float o[8];
    float m, l;
};

template <int LP>
__device__ __forceinline__ void att_tile(AttState<LP> &st, const uint16_t *Kt, const uint16_t *Vt, int nt, int d,
                                         int sub, int wph, int lane) {
    constexpr int PW = 32 / LP;
    const int pg = lane / LP, ch = lane % LP;
    for (int j0 = sub * PW; j0 < nt; j0 += wph * PW) {
        const int j = j0 + pg;
        const bool valid = j < nt;
        float sc = -INFINITY;
        uint4 vv = make_uint4(0, 0, 0, 0);
        if (valid) {
            const uint4 kv = reinterpret_cast<const uint4 *>(Kt + (size_t)j * d)[ch];
            vv = reinterpret_cast<const uint4 *>(Vt + (size_t)j * d)[ch];
            sc = st.q[0] * bf_lo(kv.x) + st.q[1] * bf_hi(kv.x) + st.q[2] * bf_lo(kv.y) + st.q[3] * bf_hi(kv.y) +
                 st.q[4] * bf_lo(kv.z) + st.q[5] * bf_hi(kv.z) + st.q[6] * bf_lo(kv.w) + st.q[7] * bf_hi(kv.w);
        }
#pragma unroll
        for (int o = LP / 2; o > 0; o >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
        float mit = sc;
#pragma unroll
        for (int o = LP; o < 32; o <<= 1) mit = fmaxf(mit, __shfl_xor_sync(0xffffffffu, mit, o));
        const float mnew = fmaxf(st.m, mit);
        if (mnew == -INFINITY) continue;
        const float alpha = exp2f(st.m - mnew);
        const float pj = valid ? exp2f(sc - mnew) : 0.f;
        st.l = st.l * alpha + pj;
        const float v[8] = {bf_lo(vv.x), bf_hi(vv.x), bf_lo(vv.y), bf_hi(vv.y),
                            bf_lo(vv.z), bf_hi(vv.z), bf_lo(vv.w), bf_hi(vv.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) st.o[e] = st.o[e] * alpha + pj * v[e];
        st.m = mnew;
    }
}

template <int LP>
__device__ bool att_task_impl(const Params &p, Smem &s, const Task &t, int ti, uint32_t &it, int ctid, int warp,
                              int lane) {
    constexpr int PW = 32 / LP;
    const int d = p.d, G = p.G, NS = p.n_slots;
    const int l = t.layer, slot = l % p.depth, b = t.b, grp = t.g;
    const AttGeo ag = att_geo(p, t);
    const bool active_seq = b < p.batch;
    AttSmem as = att_smem(p, s);

    /* prologue: rotate q and the new k, round k and v to bf16 */
    if (active_seq) {
        const float *qkv = p.qkv + ((size_t)slot * p.Bmax + b) * p.qkv_rows;
        const float *rope = p.rope + (size_t)ag.p * d;  /* [d/2][2] */
        const int half = d / 2;
        for (int i = ctid; i < (G + 2) * half; i += NCW * 32) {
            const int h = i / half, e = i % half;
            const float c = __ldg(rope + 2 * e), sn = __ldg(rope + 2 * e + 1);
            if (h < G) {
                const float *src = qkv + (size_t)(grp * G + h) * d;
                const float a = __ldcg(src + e), bb = __ldcg(src + e + half);
                as.q[h * d + e] = (a * c - bb * sn) * p.qk_scale_log2;
                as.q[h * d + e + half] = (bb * c + a * sn) * p.qk_scale_log2;
            } else if (h == G) {
                const float *src = qkv + (size_t)p.nq * d + grp * d;
                const float a = __ldcg(src + e), bb = __ldcg(src + e + half);
                as.knew[e] = f2bf(a * c - bb * sn);
                as.knew[e + half] = f2bf(bb * c + a * sn);
            } else {
                const float *src = qkv + (size_t)(p.nq + p.nkv) * d + grp * d;
                as.vnew[e] = f2bf(__ldcg(src + e));
                as.vnew[e + half] = f2bf(__ldcg(src + e + half));
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
    AttState<LP> st;
    st.m = -INFINITY;
    st.l = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        st.o[e] = 0.f;
        st.q[e] = wactive ? as.q[h * d + ch * 8 + e] : 0.f;
    }

    for (int k = 0; k < ag.ntile; ++k, ++it) {
        const int sl = (int)(it % (uint32_t)NS);
        if (s.misc->abort) continue;
        if (!wait_phase(p, s, &s.full[sl], (it / NS) & 1u, 2, ti)) continue;
        const int t0 = ag.s0 + k * t.rows_per_stage;
        const int nt = min(ag.e, t0 + (int)t.rows_per_stage) - t0;
        const uint16_t *Kt = reinterpret_cast<const uint16_t *>(s.ring + (size_t)sl * p.slot_bytes);
        const uint16_t *Vt = Kt + (size_t)t.rows_per_stage * d;
        if (wactive) att_tile<LP>(st, Kt, Vt, nt, d, sub, wph, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.empty[sl]);
    }
    if (active_seq && (t.flags & TF_NEW_TOKEN) && wactive) att_tile<LP>(st, as.knew, as.vnew, 1, d, sub, wph, lane);

    /* reduce l and o over the position groups of the warp */
#pragma unroll
    for (int o = LP; o < 32; o <<= 1) {
        st.l += __shfl_xor_sync(0xffffffffu, st.l, o);
#pragma unroll
        for (int e = 0; e < 8; ++e) st.o[e] += __shfl_xor_sync(0xffffffffu, st.o[e], o);
    }
    if (wactive && lane < LP) {
        float *w = as.wst + (size_t)warp * (d + PART_PAD);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[ch * 8 + e] = st.o[e];
        if (lane == 0) {
            w[d] = st.m;
            w[d + 1] = st.l;
        }
    }
    if (cbar_or(s.misc->abort != 0)) return false;

    /* merge the warps of each head; write the chunk's partial (o unnormalised, m, l) */
    if (active_seq) {
        float *part = p.part + ((((size_t)slot * p.Bmax + b) * p.nkv + grp) * p.C + t.r0) * G * (d + PART_PAD);
        for (int i = ctid; i < G * (d + 2); i += NCW * 32) {
            const int hh = i / (d + 2), e = i % (d + 2);
            float M = -INFINITY;
            for (int sb = 0; sb < wph; ++sb) M = fmaxf(M, as.wst[(size_t)(sb * G + hh) * (d + PART_PAD) + d]);
            float v = 0.f;
            if (e == d) {
                v = M;
            } else if (M != -INFINITY) {
                for (int sb = 0; sb < wph; ++sb) {
                    const float *w = as.wst + (size_t)(sb * G + hh) * (d + PART_PAD);
                    const float mw = w[d];
                    if (mw == -INFINITY) continue;
                    v += exp2f(mw - M) * (e == d + 1 ? w[d + 1] : w[e]);
                }
            }
            part[(size_t)hh * (d + PART_PAD) + e] = v;
        }
    }
    (void)PW;
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
    s.act = reinterpret_cast<uint8_t *>(s.sc) + p.scale_bytes;
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
        uint32_t it = 0;
        for (int ti = tbeg; ti < tend; ++ti) {
            Task t;
            load_task(p.tasks + ti, t);
            /* weights-only inputs can be fetched before the dependency is met */
            if (I8 && t.op != OP_ATT) {
                const int n = t.r1 - t.r0, nm = t.op == OP_GUP ? 2 : 1;
                for (int i = ctid; i < n * nm; i += NCW * 32) {
                    const int m = i / n, rr = i % n;
                    s.sc[i] = __ldg(op_scales(p, t, m) + t.r0 + rr);
                }
            }
            if (ctid == 0 && t.wait_id != NO_WAIT) wait_counter(p, s, t.wait_id, t.wait_count, ti);
            if (cbar_or(s.misc->abort != 0)) break;
            bool ok;
            if (t.op == OP_ATT)
                ok = p.d == 64 ? att_task_impl<8>(p, s, t, ti, it, ctid, warp, lane)
                               : att_task_impl<16>(p, s, t, ti, it, ctid, warp, lane);
            else
                ok = gemv_task<I8, NB>(p, s, t, ti, it, ctid, warp, lane);
            if (!ok) break;
            if (ctid == 0 && !(t.flags & TF_SKIP_SIGNAL)) {
                __threadfence();
                for (int k = 0; k < t.nsig; ++k) atomicAdd(p.counters + (size_t)t.sig[k] * COUNTER_STRIDE, 1u);
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

typedef void (*KernelFn)(const Params);

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
