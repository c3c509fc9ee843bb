/*
 * amk_unfused.cu — the same decode step as one kernel launch per operator,
 * for comparison with the single-launch MegaKernel on the same GB300 and the
 * same data.
 *
 * The Ada-MK abstract attributes a measurable share of end-to-end decode time
 * to kernel launches and puts inter-operator HBM round trips among the costs
 * the MegaKernel removes; the AutoMegaKernel abstract compares its fused
 * kernel against CUDA-graphed per-operator library kernels.  This file is
 * that per-operator form: every operator of the step is its own launch and
 * hands its output to the next one through global memory.  Each launch is
 * written to keep HBM busy on its own (GEMV rows with several loads in
 * flight per lane, attention split over the context into about two blocks
 * per SM and merged by a second launch), so the comparison measures the
 * launches and round trips rather than slow kernels.  Callers capture a step
 * in a CUDA graph to take the host's launch cost out.
 *
 * Arithmetic follows the same definition as the MegaKernel (bf16 weights or
 * int8 weights with row scales, bf16 activations at the GEMV inputs and in
 * the KV cache, fp32 sums, fp32 residual and logits); results agree with the
 * oracle within the same tolerance, not bit for bit with the MegaKernel.
 */
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <vector>

#include "amk.h"
#include "amk_unfused.h"

namespace {

constexpr int TB = 256;

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&b);
}

__device__ __forceinline__ float block_sum(float v, float *sh) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < (int)blockDim.x / 32; ++i) t += sh[i];
    return t;
}

__device__ __forceinline__ float block_max(float v, float *sh) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = v;
    __syncthreads();
    float t = -INFINITY;
    for (int i = 0; i < (int)blockDim.x / 32; ++i) t = fmaxf(t, sh[i]);
    return t;
}

/* x[b] = E[tokens[b]] */
__global__ void k_embed(float *x, const uint16_t *embed, const int32_t *tokens, int H) {
    const int b = blockIdx.x;
    const uint16_t *e = embed + (size_t)tokens[b] * H;
    for (int i = threadIdx.x; i < H; i += blockDim.x) x[(size_t)b * H + i] = bf2f(e[i]);
}

/* h[b] = bf16(x[b] * gain / sqrt(mean(x[b]^2) + eps)); groups of four, the
 * loop unrolled so that a thread's loads are in flight together */
__global__ void k_rmsnorm(uint16_t *h, const float *x, const uint16_t *gain, int H, float eps) {
    __shared__ float sh[32];
    const int b = blockIdx.x, H4 = H / 4;
    const float4 *xb = reinterpret_cast<const float4 *>(x + (size_t)b * H);
    float ss = 0.f;
#pragma unroll 4
    for (int i = threadIdx.x; i < H4; i += blockDim.x) {
        const float4 v = xb[i];
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    const float r = rsqrtf(block_sum(ss, sh) / (float)H + eps);
#pragma unroll 4
    for (int i = threadIdx.x; i < H4; i += blockDim.x) {
        const float4 v = xb[i];
        const uint2 gw = reinterpret_cast<const uint2 *>(gain)[i];
        const float g0 = bf2f((uint16_t)gw.x), g1 = bf2f((uint16_t)(gw.x >> 16));
        const float g2 = bf2f((uint16_t)gw.y), g3 = bf2f((uint16_t)(gw.y >> 16));
        reinterpret_cast<uint2 *>(h + (size_t)b * H)[i] =
            make_uint2((uint32_t)f2bf(v.x * r * g0) | ((uint32_t)f2bf(v.y * r * g1) << 16),
                       (uint32_t)f2bf(v.z * r * g2) | ((uint32_t)f2bf(v.w * r * g3) << 16));
    }
}

/* y[b][row0 + r] = (s[r]) * sum_k W[r][k] h[b][k] for up to three matrices
 * stacked in rows (QKV; gate and up): one warp per output row, the weights
 * read once for every sequence */
struct Mats {
    const void *w[3];
    const float *s[3];
    int rows[3];
    int n;
};

template <bool I8>
__global__ void k_gemv(float *y, int ystride, Mats m, const uint16_t *h, int K, int B) {
    const int warp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    int r = warp, mi = 0, base = 0;
    while (mi < m.n && r >= m.rows[mi]) {
        r -= m.rows[mi];
        base += m.rows[mi];
        ++mi;
    }
    if (mi >= m.n) return;
    constexpr int MB = 16;
    float acc[MB];
    for (int b = 0; b < MB; ++b) acc[b] = 0.f;
    if (I8) {
        const int8_t *w = (const int8_t *)m.w[mi] + (size_t)r * K;
#pragma unroll 4
        for (int k = lane * 4; k < K; k += 128) {
            const char4 q = *reinterpret_cast<const char4 *>(w + k);
            for (int b = 0; b < B && b < MB; ++b) {
                const uint16_t *hb = h + (size_t)b * K + k;
                acc[b] += (float)q.x * bf2f(hb[0]) + (float)q.y * bf2f(hb[1]) + (float)q.z * bf2f(hb[2]) +
                          (float)q.w * bf2f(hb[3]);
            }
        }
    } else {
        /* eight 16-byte weight loads per lane in flight before any product */
        constexpr int U = 8;
        const uint16_t *w = (const uint16_t *)m.w[mi] + (size_t)r * K;
        for (int k0 = lane * 8; k0 < K; k0 += 256 * U) {
            uint4 wv[U];
#pragma unroll
            for (int u2 = 0; u2 < U; ++u2) {
                const int k = k0 + 256 * u2;
                wv[u2] = k < K ? *reinterpret_cast<const uint4 *>(w + k) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u2 = 0; u2 < U; ++u2) {
                const int k = k0 + 256 * u2;
                if (k >= K) break;
                const uint16_t *wp = reinterpret_cast<const uint16_t *>(&wv[u2]);
                for (int b = 0; b < B && b < MB; ++b) {
                    const uint4 hv = *reinterpret_cast<const uint4 *>(h + (size_t)b * K + k);
                    const uint16_t *hp = reinterpret_cast<const uint16_t *>(&hv);
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) a = fmaf(bf2f(wp[e]), bf2f(hp[e]), a);
                    acc[b] += a;
                }
            }
        }
    }
    for (int b = 0; b < B && b < MB; ++b) {
        float v = acc[b];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) y[(size_t)b * ystride + base + r] = I8 ? v * m.s[mi][r] : v;
    }
}

/* RoPE on the q and k heads of qkv[b] (in place, rotate-half pairs), then the
 * bf16 K and V of position p into the cache */
__global__ void k_rope_kv(float *qkv, int qkv_rows, uint16_t *kc, uint16_t *vc, const int32_t *positions,
                          const float *rope, int l, int Bmax, int nq, int nkv, int d, int Smax) {
    const int b = blockIdx.x, p = positions[b], half = d / 2;
    float *q = qkv + (size_t)b * qkv_rows;
    const float *cs = rope + (size_t)p * d;
    for (int i = threadIdx.x; i < (nq + nkv) * half; i += blockDim.x) {
        const int hh = i / half, e = i % half;
        float *u = q + (size_t)hh * d;
        const float c = cs[2 * e], s = cs[2 * e + 1], a = u[e], bb = u[e + half];
        u[e] = a * c - bb * s;
        u[e + half] = bb * c + a * s;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nkv * d; i += blockDim.x) {
        const int g = i / d, e = i % d;
        const size_t row = ((((size_t)l * Bmax + b) * nkv + g) * Smax + p) * d + e;
        kc[row] = f2bf(q[(size_t)nq * d + i]);
        vc[row] = f2bf(q[(size_t)(nq + nkv) * d + i]);
    }
}

/* Split-context attention of one (query head, split, sequence): over
 * positions [m0, m1) of 0..p (split sp of S), the softmax partial m = max
 * score, l = sum exp(s - m), o = sum exp(s - m) v (unnormalised) into
 * part[((b nq + j) S + sp) (d + 2)].  Scores: 8 lanes per position, each a
 * 16-byte piece of the K row, kept in shared memory; P.V: (256 / d) thread
 * groups split the positions, each thread one output element, the groups'
 * sums added in order. */
__global__ void k_attn_split(float *part, const float *qkv, int qkv_rows, const uint16_t *kc, const uint16_t *vc,
                             const int32_t *positions, int l, int Bmax, int nq, int nkv, int d, int Smax, int S) {
    extern __shared__ float sc[];
    __shared__ float sh[32];
    __shared__ float pp[TB];
    const int j = blockIdx.x, sp = blockIdx.y, b = blockIdx.z, g = j / (nq / nkv), n = positions[b] + 1;
    const int m0 = (int)((long long)sp * n / S), m1 = (int)((long long)(sp + 1) * n / S);
    float *out = part + ((size_t)(b * nq + j) * S + sp) * (d + 2);
    const float *q = qkv + (size_t)b * qkv_rows + (size_t)j * d;
    const size_t base = (((size_t)l * Bmax + b) * nkv + g) * Smax * d;
    const float scale = rsqrtf((float)d);
    const int lane = threadIdx.x & 31, sub = lane & 7, grp = threadIdx.x >> 3, ngrp = blockDim.x >> 3;
    float mx = -INFINITY;
    for (int a0 = m0; a0 < m1; a0 += ngrp) {
        const int m = a0 + grp;
        float s = 0.f;
        if (m < m1)
            for (int e0 = sub * 8; e0 < d; e0 += 64) {
                const uint4 kv = *reinterpret_cast<const uint4 *>(kc + base + (size_t)m * d + e0);
                const uint16_t *kp = reinterpret_cast<const uint16_t *>(&kv);
                for (int e = 0; e < 8; ++e) s = fmaf(q[e0 + e], bf2f(kp[e]), s);
            }
        for (int o = 4; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (m < m1) {
            s *= scale;
            if (sub == 0) sc[m - m0] = s;
            mx = fmaxf(mx, s);
        }
    }
    mx = block_max(mx, sh);
    float sum = 0.f;
    for (int m = m0 + threadIdx.x; m < m1; m += blockDim.x) {
        const float e = __expf(sc[m - m0] - mx);
        sc[m - m0] = e;
        sum += e;
    }
    sum = block_sum(sum, sh);
    __syncthreads();
    const int e = threadIdx.x % d, gi = threadIdx.x / d, ng = blockDim.x / d;
    float o = 0.f;
    for (int m = m0 + gi; m < m1; m += ng) o = fmaf(sc[m - m0], bf2f(vc[base + (size_t)m * d + e]), o);
    pp[threadIdx.x] = o;
    __syncthreads();
    if (threadIdx.x < d) {
        float t = 0.f;
        for (int i2 = 0; i2 < ng; ++i2) t += pp[i2 * d + threadIdx.x];
        out[threadIdx.x] = t;
    }
    if (threadIdx.x == 0) {
        out[d] = mx;
        out[d + 1] = sum;
    }
}

/* out[b][j] = bf16(sum_s 2^... ) : the S partials of one (query head,
 * sequence) combined by their log-sum-exp weights: o = sum_s e^(m_s - M) o_s /
 * sum_s e^(m_s - M) l_s; one thread per output element */
__global__ void k_attn_merge(uint16_t *out, const float *part, int nq, int d, int S) {
    const int j = blockIdx.x, b = blockIdx.y, e = threadIdx.x;
    if (e >= d) return;
    const float *pj = part + (size_t)(b * nq + j) * S * (d + 2);
    float M = -INFINITY, L = 0.f, O = 0.f;
    /* rounds of eight splits, every load of a round in flight together */
    for (int s0 = 0; s0 < S; s0 += 8) {
        float mv[8], lv[8], ov[8];
#pragma unroll
        for (int u2 = 0; u2 < 8; ++u2) {
            const bool in = s0 + u2 < S;
            const float *q = pj + (size_t)(s0 + u2) * (d + 2);
            mv[u2] = in ? q[d] : -INFINITY;
            lv[u2] = in ? q[d + 1] : 0.f;
            ov[u2] = in ? q[e] : 0.f;
        }
        float Mn = M;
#pragma unroll
        for (int u2 = 0; u2 < 8; ++u2) Mn = fmaxf(Mn, mv[u2]);
        if (Mn == -INFINITY) continue;
        const float c = M == -INFINITY ? 0.f : __expf(M - Mn);
        L *= c;
        O *= c;
#pragma unroll
        for (int u2 = 0; u2 < 8; ++u2) {
            if (mv[u2] == -INFINITY) continue;
            const float f = __expf(mv[u2] - Mn);
            L = fmaf(f, lv[u2], L);
            O = fmaf(f, ov[u2], O);
        }
        M = Mn;
    }
    out[(size_t)b * nq * d + (size_t)j * d + e] = f2bf(O / L);
}

__global__ void k_residual(float *x, const float *y, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) x[i] += y[i];
}

/* a[b][i] = bf16(silu(gate) * up), gu[b] = [gate rows | up rows] */
__global__ void k_swiglu(uint16_t *a, const float *gu, int I, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int b = i / I, r = i % I;
    const float gt = gu[(size_t)b * 2 * I + r], up = gu[(size_t)b * 2 * I + I + r];
    a[i] = f2bf(gt / (1.f + __expf(-gt)) * up);
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

struct amk_unfused {
    amk_config cfg;
    std::vector<amk_layer_weights> layers;
    const void *embed, *final_norm, *lm;
    const float *s_lm;
    float *x = nullptr, *y = nullptr, *qkv = nullptr, *gu = nullptr, *rope = nullptr, *part = nullptr;
    int splits = 1; /* context splits of the attention: about two blocks per SM at batch 1 */
    uint16_t *h = nullptr; /* the bf16 input of the next GEMV: norm, attention or SwiGLU output */
};

extern "C" {

amk_status amk_unfused_create(const amk_config *c, const amk_weights *w, amk_unfused **out) {
    if (!c || !w || !out || !w->layers || !w->embed || !w->final_norm) return AMK_ERR_INVALID_ARG;
    *out = nullptr;
    if (c->head_dim % 2 || c->n_heads % c->n_kv_heads || c->max_batch < 1 || c->max_batch > 16 ||
        c->hidden % 8 || c->intermediate % 8 || (c->n_heads * c->head_dim) % 8)
        return AMK_ERR_UNSUPPORTED;
    if (!c->tied_embeddings && !w->lm_head) return AMK_ERR_INVALID_ARG;
    amk_unfused *u = new amk_unfused;
    u->cfg = *c;
    u->layers.assign(w->layers, w->layers + c->n_layers);
    u->embed = w->embed;
    u->final_norm = w->final_norm;
    u->lm = c->tied_embeddings ? w->embed : w->lm_head;
    u->s_lm = c->tied_embeddings ? nullptr : w->s_lm;
    const int B = c->max_batch, H = c->hidden, I = c->intermediate, d = c->head_dim;
    const int qkv_rows = (c->n_heads + 2 * c->n_kv_heads) * d, KM = std::max(std::max(H, I), c->n_heads * d);
    std::vector<float> rope((size_t)c->max_seq * d);
    for (int p = 0; p < c->max_seq; ++p)
        for (int i = 0; i < d / 2; ++i) {
            const double th = (double)p * std::pow((double)c->rope_theta, -2.0 * i / d);
            rope[(size_t)p * d + 2 * i] = (float)std::cos(th);
            rope[(size_t)p * d + 2 * i + 1] = (float)std::sin(th);
        }
    cudaError_t e = cudaSuccess;
    auto chk = [&](cudaError_t x) {
        if (e == cudaSuccess) e = x;
    };
    chk(cudaMalloc(&u->x, sizeof(float) * B * H));
    chk(cudaMalloc(&u->y, sizeof(float) * B * std::max(H, c->vocab)));
    chk(cudaMalloc(&u->qkv, sizeof(float) * B * qkv_rows));
    chk(cudaMalloc(&u->gu, sizeof(float) * B * 2 * I));
    chk(cudaMalloc(&u->rope, sizeof(float) * rope.size()));
    chk(cudaMalloc(&u->h, sizeof(uint16_t) * B * KM));
    int dev = 0, n_sm = 0;
    chk(cudaGetDevice(&dev));
    chk(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
    u->splits = std::max(1, std::min(32, ceil_div(2 * std::max(1, n_sm), c->n_heads)));
    chk(cudaMalloc(&u->part, sizeof(float) * B * c->n_heads * u->splits * (d + 2)));
    if (e == cudaSuccess) chk(cudaMemcpy(u->rope, rope.data(), sizeof(float) * rope.size(), cudaMemcpyHostToDevice));
    if (e != cudaSuccess) {
        cudaGetLastError();
        amk_unfused_destroy(u);
        return e == cudaErrorMemoryAllocation ? AMK_ERR_OOM : AMK_ERR_CUDA;
    }
    *out = u;
    return AMK_OK;
}

amk_status amk_unfused_decode_step(amk_unfused *u, int32_t batch, const int32_t *tokens, const int32_t *positions,
                                   void *kv_cache, float *logits, amk_stream_t stream) {
    if (!u || !tokens || !positions || !kv_cache || !logits || batch < 1 || batch > u->cfg.max_batch)
        return AMK_ERR_INVALID_ARG;
    const amk_config &c = u->cfg;
    const int B = batch, H = c.hidden, I = c.intermediate, d = c.head_dim, nq = c.n_heads, nkv = c.n_kv_heads;
    const int qkv_rows = (nq + 2 * nkv) * d;
    const bool i8 = c.weight_dtype == AMK_WEIGHT_INT8, lm8 = i8 && !c.tied_embeddings;
    cudaStream_t s = (cudaStream_t)stream;
    uint16_t *kc = (uint16_t *)kv_cache;
    uint16_t *vc = kc + (size_t)c.n_layers * c.max_batch * nkv * c.max_seq * d;
    auto gemv = [&](float *y, int ystride, Mats m, int K, bool int8) {
        int rows = 0;
        for (int i = 0; i < m.n; ++i) rows += m.rows[i];
        if (int8)
            k_gemv<true><<<ceil_div(rows, TB / 32), TB, 0, s>>>(y, ystride, m, u->h, K, B);
        else
            k_gemv<false><<<ceil_div(rows, TB / 32), TB, 0, s>>>(y, ystride, m, u->h, K, B);
    };
    k_embed<<<B, TB, 0, s>>>(u->x, (const uint16_t *)u->embed, tokens, H);
    for (int l = 0; l < c.n_layers; ++l) {
        const amk_layer_weights &L = u->layers[l];
        k_rmsnorm<<<B, TB, 0, s>>>(u->h, u->x, (const uint16_t *)L.attn_norm, H, c.rms_eps);
        gemv(u->qkv, qkv_rows, Mats{{L.wq, L.wk, L.wv}, {L.s_q, L.s_k, L.s_v}, {nq * d, nkv * d, nkv * d}, 3}, H, i8);
        k_rope_kv<<<B, TB, 0, s>>>(u->qkv, qkv_rows, kc, vc, positions, u->rope, l, c.max_batch, nq, nkv, d,
                                   c.max_seq);
        const int S = u->splits;
        k_attn_split<<<dim3(nq, S, B), TB, sizeof(float) * (c.max_seq / S + 2), s>>>(
            u->part, u->qkv, qkv_rows, kc, vc, positions, l, c.max_batch, nq, nkv, d, c.max_seq, S);
        k_attn_merge<<<dim3(nq, B), d, 0, s>>>(u->h, u->part, nq, d, S);
        gemv(u->y, H, Mats{{L.wo}, {L.s_o}, {H}, 1}, nq * d, i8);
        k_residual<<<ceil_div(B * H, TB), TB, 0, s>>>(u->x, u->y, B * H);
        k_rmsnorm<<<B, TB, 0, s>>>(u->h, u->x, (const uint16_t *)L.mlp_norm, H, c.rms_eps);
        gemv(u->gu, 2 * I, Mats{{L.w_gate, L.w_up}, {L.s_gate, L.s_up}, {I, I}, 2}, H, i8);
        k_swiglu<<<ceil_div(B * I, TB), TB, 0, s>>>(u->h, u->gu, I, B * I);
        gemv(u->y, H, Mats{{L.w_down}, {L.s_down}, {H}, 1}, I, i8);
        k_residual<<<ceil_div(B * H, TB), TB, 0, s>>>(u->x, u->y, B * H);
    }
    k_rmsnorm<<<B, TB, 0, s>>>(u->h, u->x, (const uint16_t *)u->final_norm, H, c.rms_eps);
    gemv(logits, c.vocab, Mats{{u->lm}, {u->s_lm}, {c.vocab}, 1}, H, lm8);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? AMK_OK : AMK_ERR_CUDA;
}

amk_status amk_unfused_destroy(amk_unfused *u) {
    if (!u) return AMK_OK;
    cudaFree(u->x);
    cudaFree(u->y);
    cudaFree(u->qkv);
    cudaFree(u->gu);
    cudaFree(u->rope);
    cudaFree(u->h);
    cudaFree(u->part);
    delete u;
    return AMK_OK;
}

}  // extern "C"
