/*
 * amk_unfused.cu — the same decode step as one kernel launch per operator,
 * for comparison with the single-launch MegaKernel on the same GB300 and the
 * same data.
 *
 * The Ada-MK abstract attributes a measurable share of end-to-end decode time
 * to kernel launches and puts inter-operator HBM round trips among the costs
 * the MegaKernel removes; the AutoMegaKernel abstract compares its fused
 * kernel against CUDA-graphed per-operator library kernels.  This file is
 * that per-operator form, written plainly: every operator of the step is its
 * own launch and hands its output to the next one through global memory.
 * Callers capture a step in a CUDA graph to take the host's launch cost out.
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

/* h[b] = bf16(x[b] * gain / sqrt(mean(x[b]^2) + eps)) */
__global__ void k_rmsnorm(uint16_t *h, const float *x, const uint16_t *gain, int H, float eps) {
    __shared__ float sh[32];
    const int b = blockIdx.x;
    const float *xb = x + (size_t)b * H;
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) ss += xb[i] * xb[i];
    const float r = rsqrtf(block_sum(ss, sh) / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x) h[(size_t)b * H + i] = f2bf(xb[i] * r * bf2f(gain[i]));
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
        for (int k = lane * 4; k < K; k += 128) {
            const char4 q = *reinterpret_cast<const char4 *>(w + k);
            for (int b = 0; b < B && b < MB; ++b) {
                const uint16_t *hb = h + (size_t)b * K + k;
                acc[b] += (float)q.x * bf2f(hb[0]) + (float)q.y * bf2f(hb[1]) + (float)q.z * bf2f(hb[2]) +
                          (float)q.w * bf2f(hb[3]);
            }
        }
    } else {
        const uint16_t *w = (const uint16_t *)m.w[mi] + (size_t)r * K;
        for (int k = lane * 8; k < K; k += 256) {
            const uint4 wv = *reinterpret_cast<const uint4 *>(w + k);
            const uint16_t *wp = reinterpret_cast<const uint16_t *>(&wv);
            for (int b = 0; b < B && b < MB; ++b) {
                const uint4 hv = *reinterpret_cast<const uint4 *>(h + (size_t)b * K + k);
                const uint16_t *hp = reinterpret_cast<const uint16_t *>(&hv);
                float a = 0.f;
                for (int e = 0; e < 8; ++e) a = fmaf(bf2f(wp[e]), bf2f(hp[e]), a);
                acc[b] += a;
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

/* softmax(q K^T / sqrt(d)) V over positions 0..p of one (sequence, query
 * head); the scores sit in shared memory.  Scores: 8 lanes per position, each
 * a 16-byte piece of the K row; P.V: (256 / d) thread groups split the
 * positions, each thread one output element, the groups' sums added in order. */
__global__ void k_attention(uint16_t *out, const float *qkv, int qkv_rows, const uint16_t *kc, const uint16_t *vc,
                            const int32_t *positions, int l, int Bmax, int nq, int nkv, int d, int Smax) {
    extern __shared__ float sc[];
    __shared__ float sh[32];
    __shared__ float part[TB];
    const int j = blockIdx.x, b = blockIdx.y, g = j / (nq / nkv), p = positions[b];
    const float *q = qkv + (size_t)b * qkv_rows + (size_t)j * d;
    const size_t base = (((size_t)l * Bmax + b) * nkv + g) * Smax * d;
    const float scale = rsqrtf((float)d);
    const int lane = threadIdx.x & 31, sub = lane & 7, grp = threadIdx.x >> 3, ngrp = blockDim.x >> 3;
    float mx = -INFINITY;
    for (int m0 = 0; m0 <= p; m0 += ngrp) {
        const int m = m0 + grp;
        float s = 0.f;
        if (m <= p)
            for (int e0 = sub * 8; e0 < d; e0 += 64) {
                const uint4 kv = *reinterpret_cast<const uint4 *>(kc + base + (size_t)m * d + e0);
                const uint16_t *kp = reinterpret_cast<const uint16_t *>(&kv);
                for (int e = 0; e < 8; ++e) s = fmaf(q[e0 + e], bf2f(kp[e]), s);
            }
        for (int o = 4; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (m <= p) {
            s *= scale;
            if (sub == 0) sc[m] = s;
            mx = fmaxf(mx, s);
        }
    }
    mx = block_max(mx, sh);
    float sum = 0.f;
    for (int m = threadIdx.x; m <= p; m += blockDim.x) {
        const float e = __expf(sc[m] - mx);
        sc[m] = e;
        sum += e;
    }
    sum = block_sum(sum, sh);
    __syncthreads();
    const int e = threadIdx.x % d, gi = threadIdx.x / d, ng = blockDim.x / d;
    float o = 0.f;
    for (int m = gi; m <= p; m += ng) o = fmaf(sc[m], bf2f(vc[base + (size_t)m * d + e]), o);
    part[threadIdx.x] = o;
    __syncthreads();
    if (threadIdx.x < d) {
        float t = 0.f;
        for (int i2 = 0; i2 < ng; ++i2) t += part[i2 * d + threadIdx.x];
        out[(size_t)b * nq * d + (size_t)j * d + threadIdx.x] = f2bf(t / sum);
    }
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
    float *x = nullptr, *y = nullptr, *qkv = nullptr, *gu = nullptr, *rope = nullptr;
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
        k_attention<<<dim3(nq, B), TB, sizeof(float) * c.max_seq, s>>>(u->h, u->qkv, qkv_rows, kc, vc, positions,
                                                                      l, c.max_batch, nq, nkv, d, c.max_seq);
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
    delete u;
    return AMK_OK;
}

}  // extern "C"
