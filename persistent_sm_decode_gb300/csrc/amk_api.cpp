/*
 * amk_api.cpp — the C ABI of amk.h: handle lifetime, schedule upload,
 * argument checks, the per-step launch and error reporting.
 */
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "amk.h"
#include "amk_launch.h"
#include "amk_plan.h"
#include "amk_plan_impl.h"

using namespace amk;

struct amk_handle {
    amk_config cfg;
    amk_plan *plan = nullptr;
    int device = 0, n_sm = 0;
    KernelFn fn = nullptr;
    std::vector<Task> h_tasks;
    std::vector<int32_t> h_start;
    /* device memory owned by the handle */
    Task *d_tasks = nullptr;
    int32_t *d_start = nullptr;
    LayerPtrs *d_layers = nullptr;
    uint32_t *d_err = nullptr;
    uint32_t *d_epoch = nullptr; /* [2]: epoch of the next step, CTAs done with the current one */
    float *d_rope = nullptr;
    uint8_t *d_scratch = nullptr;
    size_t scratch_bytes = 0;
    unsigned long long *d_trace = nullptr;
    Params params;
    uint32_t epoch = 0;
    cudaStream_t last_stream = nullptr;
    bool launched = false;
    amk_error_info last_err;
};

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

amk_status cuda_fail(cudaError_t e) {
    if (e == cudaSuccess) return AMK_OK;
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? AMK_ERR_OOM : AMK_ERR_CUDA;
}

void free_handle(amk_handle *h) {
    if (!h) return;
    cudaFree(h->d_tasks);
    cudaFree(h->d_start);
    cudaFree(h->d_layers);
    cudaFree(h->d_err);
    cudaFree(h->d_epoch);
    cudaFree(h->d_rope);
    cudaFree(h->d_scratch);
    cudaFree(h->d_trace);
    if (h->plan) amk_plan_destroy(h->plan);
    delete h;
}

amk_status check_weights(const amk_config &c, const amk_weights *w) {
    if (!w || !w->embed || !w->final_norm || !w->layers) return AMK_ERR_INVALID_ARG;
    const bool i8 = c.weight_dtype == AMK_WEIGHT_INT8 || c.weight_dtype == AMK_WEIGHT_INT4; /* scaled formats */
    if (!aligned16(w->embed) || !aligned16(w->final_norm)) return AMK_ERR_INVALID_ARG;
    if (!c.tied_embeddings) {
        if (!w->lm_head || !aligned16(w->lm_head)) return AMK_ERR_INVALID_ARG;
        if (i8 && !w->s_lm) return AMK_ERR_INVALID_ARG;
    }
    for (int l = 0; l < c.n_layers; ++l) {
        const amk_layer_weights &L = w->layers[l];
        const void *m[] = {L.wq, L.wk, L.wv, L.wo, L.w_gate, L.w_up, L.w_down, L.attn_norm, L.mlp_norm};
        for (const void *p : m)
            if (!p || !aligned16(p)) return AMK_ERR_INVALID_ARG;
        if (i8) {
            const float *s[] = {L.s_q, L.s_k, L.s_v, L.s_o, L.s_gate, L.s_up, L.s_down};
            for (const float *p : s)
                if (!p || ((uintptr_t)p & 3u)) return AMK_ERR_INVALID_ARG;
        }
    }
    return AMK_OK;
}

}  // namespace

extern "C" {

const char *amk_status_string(amk_status s) {
    switch (s) {
    case AMK_OK: return "ok";
    case AMK_ERR_INVALID_ARG: return "invalid argument";
    case AMK_ERR_UNSUPPORTED: return "unsupported shape or device";
    case AMK_ERR_CUDA: return "CUDA runtime error";
    case AMK_ERR_OOM: return "out of memory";
    case AMK_ERR_SCHEDULE: return "schedule rejected by the validator";
    case AMK_ERR_COOPERATIVE: return "one CTA per SM cannot be co-resident";
    case AMK_ERR_TIMEOUT: return "a device-side wait timed out";
    }
    return "unknown status";
}

amk_status amk_create(const amk_config *config, const amk_weights *weights, const amk_schedule_options *options,
                      amk_handle **out) {
    if (!config || !out) return AMK_ERR_INVALID_ARG;
    *out = nullptr;
    /* the timing code and the loader's L2 prefetch exist only in builds
     * that compile them in */
    if (options && options->trace && !kernel_has_trace()) return AMK_ERR_UNSUPPORTED;
    if (options && options->l2_prefetch_kb > 0 && !kernel_has_l2_prefetch()) return AMK_ERR_UNSUPPORTED;
    amk_status st = check_weights(*config, weights);
    if (st != AMK_OK) return st;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaErrorNoDevice);
    int n_sm = 0, smem_optin = 0, coop = 0;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
        cudaGetLastError();
        return AMK_ERR_CUDA;
    }
    if (!coop) return AMK_ERR_COOPERATIVE;
    if (options && options->n_sm > 0) n_sm = std::min(n_sm, (int)options->n_sm);

    amk_handle *h = new amk_handle;
    h->cfg = *config;
    h->device = dev;
    h->n_sm = n_sm;
    std::memset(&h->last_err, 0, sizeof h->last_err);
    std::string msg;
    st = plan_build(config, config->max_batch, n_sm, smem_optin, options, &h->plan, &msg);
    if (st != AMK_OK) {
        std::fprintf(stderr, "amk_create: %s\n", msg.c_str());
        free_handle(h);
        return st;
    }
    const amk_plan &P = *h->plan;

    /* the sm_103a image must exist for this device; no other path is built */
    h->fn = select_kernel(config->weight_dtype, config->max_batch);
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, (const void *)h->fn) != cudaSuccess) {
        cudaGetLastError();
        free_handle(h);
        return AMK_ERR_UNSUPPORTED;
    }
    if (prepare_kernel(h->fn, P.smem_bytes) != cudaSuccess) {
        cudaGetLastError();
        free_handle(h);
        return AMK_ERR_UNSUPPORTED;
    }
    int per_sm = 0;
    if (occupancy(h->fn, P.smem_bytes, &per_sm) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        free_handle(h);
        return AMK_ERR_COOPERATIVE;
    }

    /* flatten and upload the solidified task table */
    h->h_start.assign(n_sm + 1, 0);
    for (int s = 0; s < n_sm; ++s) {
        h->h_start[s + 1] = h->h_start[s] + (int)P.sm_tasks[s].size();
        h->h_tasks.insert(h->h_tasks.end(), P.sm_tasks[s].begin(), P.sm_tasks[s].end());
    }
    const Geo g = make_geo(*config, config->max_batch);
    const int L = config->n_layers, d = config->head_dim;
    std::vector<LayerPtrs> lp(L);
    for (int l = 0; l < L; ++l) {
        const amk_layer_weights &w = weights->layers[l];
        const void *m[7] = {w.wq, w.wk, w.wv, w.wo, w.w_gate, w.w_up, w.w_down};
        const float *sc[7] = {w.s_q, w.s_k, w.s_v, w.s_o, w.s_gate, w.s_up, w.s_down};
        for (int i = 0; i < 7; ++i) {
            lp[l].w[i] = m[i];
            lp[l].s[i] = sc[i];
        }
        lp[l].attn_norm = (const uint16_t *)w.attn_norm;
        lp[l].mlp_norm = (const uint16_t *)w.mlp_norm;
    }
    /* RoPE table: angle p * theta^(-2i/d) in double, stored as fp32 cos, sin */
    std::vector<float> rope((size_t)config->max_seq * d);
    for (int p = 0; p < config->max_seq; ++p)
        for (int i = 0; i < d / 2; ++i) {
            double th = (double)p * std::pow((double)config->rope_theta, -2.0 * i / d);
            rope[(size_t)p * d + 2 * i] = (float)std::cos(th);
            rope[(size_t)p * d + 2 * i + 1] = (float)std::sin(th);
        }
    /* activation scratch: epoch-tagged 8-byte words, zero (epoch 0) at start */
    ScratchSizes ss = scratch_sizes(P);
    const size_t w8 = 8;
    size_t off_xin = 0, off_xmid = off_xin + ss.x_in * w8, off_qkv = off_xmid + ss.x_mid * w8;
    size_t off_part = off_qkv + ss.qkv * w8, off_aout = off_part + ss.part * w8;
    size_t off_act = off_aout + ss.aout * w8;
    size_t off_argp = off_act + ss.act * w8;
    size_t scratch_bytes = ((off_argp + ss.argp * w8) + 255) / 256 * 256;
    h->scratch_bytes = scratch_bytes;
    cudaError_t e = cudaSuccess;
    auto chk = [&](cudaError_t x) {
        if (e == cudaSuccess) e = x;
    };
    chk(cudaMalloc(&h->d_tasks, sizeof(Task) * std::max<size_t>(1, h->h_tasks.size())));
    chk(cudaMalloc(&h->d_start, sizeof(int32_t) * (n_sm + 1)));
    chk(cudaMalloc(&h->d_layers, sizeof(LayerPtrs) * L));
    chk(cudaMalloc(&h->d_err, sizeof(uint32_t) * ERR_WORDS));
    chk(cudaMalloc(&h->d_epoch, sizeof(uint32_t) * 2));
    chk(cudaMalloc(&h->d_rope, sizeof(float) * rope.size()));
    chk(cudaMalloc(&h->d_scratch, scratch_bytes));
    if (options && options->trace)
        chk(cudaMalloc(&h->d_trace, sizeof(unsigned long long) * 16 * std::max<size_t>(1, h->h_tasks.size())));
    if (e == cudaSuccess) {
        chk(cudaMemcpy(h->d_tasks, h->h_tasks.data(), sizeof(Task) * h->h_tasks.size(), cudaMemcpyHostToDevice));
        chk(cudaMemcpy(h->d_start, h->h_start.data(), sizeof(int32_t) * (n_sm + 1), cudaMemcpyHostToDevice));
        chk(cudaMemcpy(h->d_layers, lp.data(), sizeof(LayerPtrs) * L, cudaMemcpyHostToDevice));
        chk(cudaMemcpy(h->d_rope, rope.data(), sizeof(float) * rope.size(), cudaMemcpyHostToDevice));
        chk(cudaMemset(h->d_err, 0, sizeof(uint32_t) * ERR_WORDS));
        /* epoch 1 first: the zeroed scratch carries flags of epoch 0 */
        const uint32_t ep0[2] = {1u, 0u};
        chk(cudaMemcpy(h->d_epoch, ep0, sizeof ep0, cudaMemcpyHostToDevice));
        chk(cudaMemset(h->d_scratch, 0, scratch_bytes));
        chk(cudaDeviceSynchronize());
    }
    if (e != cudaSuccess) {
        st = cuda_fail(e);
        free_handle(h);
        return st;
    }

    Params &p = h->params;
    std::memset(&p, 0, sizeof p);
    p.L = L;
    p.H = g.H;
    p.nq = g.nq;
    p.nkv = g.nkv;
    p.d = d;
    p.I = g.I;
    p.V = g.V;
    p.G = g.G;
    p.Bmax = config->max_batch;
    p.Smax = config->max_seq;
    p.qkv_rows = g.qkv_rows;
    p.eps = config->rms_eps;
    p.qk_scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
    p.wf = g.wf;
    p.lm_wf = g.lm_wf;
    p.group = g.group;
    p.tasks = h->d_tasks;
    p.task_start = h->d_start;
    p.C = P.k.C;
    p.depth = P.k.depth;
    p.slot_bytes = P.k.slot_bytes;
    p.n_slots = P.k.n_slots;
    p.att_tile = P.k.att_tile;
    p.act_bytes = P.act_bytes;
    p.result_bytes = P.result_bytes;
    p.scale_bytes = P.scale_bytes;
    p.fac_bytes = P.fac_bytes;
    p.work_bytes = P.work_bytes;
    p.l2_prefetch_bytes = P.k.l2_prefetch_kb > 0 ? P.k.l2_prefetch_kb * 1024 : 0;
    p.evict_first = P.k.evict_first;
    p.layers = h->d_layers;
    p.embed = (const uint16_t *)weights->embed;
    p.final_norm = (const uint16_t *)weights->final_norm;
    p.lm = config->tied_embeddings ? weights->embed : weights->lm_head;
    p.s_lm = config->tied_embeddings ? nullptr : weights->s_lm;
    p.x_in = (uint64_t *)(h->d_scratch + off_xin);
    p.x_mid = (uint64_t *)(h->d_scratch + off_xmid);
    p.qkv = (uint64_t *)(h->d_scratch + off_qkv);
    p.part = (uint64_t *)(h->d_scratch + off_part);
    p.aout = (uint64_t *)(h->d_scratch + off_aout);
    p.act = (uint64_t *)(h->d_scratch + off_act);
    p.argp = (uint64_t *)(h->d_scratch + off_argp);
    p.n_lmh = P.n_lmh;
    p.epoch_word = h->d_epoch;
    p.err = h->d_err;
    p.rope = h->d_rope;
    p.timeout_ns = (options && options->wait_timeout_ns > 0) ? options->wait_timeout_ns : 1000000000LL;
    p.trace = h->d_trace;
    *out = h;
    return AMK_OK;
}

namespace {

/* one launch of the step; the epoch comes from the handle's device word */
amk_status launch_step(amk_handle *h, int32_t batch, const int32_t *tokens, const int32_t *positions,
                       void *kv_cache, float *logits, int32_t *next_tokens, int32_t *next_positions,
                       amk_stream_t stream) {
    if (!h || !tokens || !positions || !kv_cache || !logits) return AMK_ERR_INVALID_ARG;
    if (batch < 1 || batch > h->cfg.max_batch) return AMK_ERR_INVALID_ARG;
    if (!aligned16(kv_cache) || ((uintptr_t)tokens & 3u) || ((uintptr_t)positions & 3u) || ((uintptr_t)logits & 3u))
        return AMK_ERR_INVALID_ARG;
    Params p = h->params;
    const size_t per_cache = (size_t)h->cfg.n_layers * h->cfg.max_batch * h->cfg.n_kv_heads * h->cfg.max_seq *
                             h->cfg.head_dim;
    p.kc = (uint16_t *)kv_cache;
    p.vc = p.kc + per_cache;
    p.tokens = tokens;
    p.positions = positions;
    p.logits = logits;
    p.next_tokens = next_tokens;
    p.next_positions = next_positions;
    p.batch = batch;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_decode(h->fn, p, h->n_sm, h->plan->smem_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e);
    ++h->epoch;
    h->last_stream = s;
    h->launched = true;
    return AMK_OK;
}

}  // namespace

amk_status amk_decode_step(amk_handle *h, int32_t batch, const int32_t *tokens, const int32_t *positions,
                           void *kv_cache, float *logits, amk_stream_t stream) {
    return launch_step(h, batch, tokens, positions, kv_cache, logits, nullptr, nullptr, stream);
}

amk_status amk_decode_step_greedy(amk_handle *h, int32_t batch, const int32_t *tokens, const int32_t *positions,
                                  void *kv_cache, float *logits, int32_t *next_tokens, int32_t *next_positions,
                                  amk_stream_t stream) {
    if (!next_tokens || !next_positions || ((uintptr_t)next_tokens & 3u) || ((uintptr_t)next_positions & 3u))
        return AMK_ERR_INVALID_ARG;
    if (next_tokens == tokens || next_positions == positions) return AMK_ERR_INVALID_ARG;
    return launch_step(h, batch, tokens, positions, kv_cache, logits, next_tokens, next_positions, stream);
}

amk_status amk_sync_status(amk_handle *h) {
    if (!h) return AMK_ERR_INVALID_ARG;
    if (h->launched && cudaStreamSynchronize(h->last_stream) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    uint32_t err[ERR_WORDS];
    if (cudaMemcpy(err, h->d_err, sizeof err, cudaMemcpyDeviceToHost) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    if (err[0] == 0) return AMK_OK;
    h->last_err.code = (int32_t)err[0];
    h->last_err.sm = (int32_t)err[1];
    h->last_err.task = (int32_t)err[2];
    h->last_err.counter = (int32_t)err[3];
    h->last_err.observed = err[4];
    h->last_err.target = err[5];
    /* Words an aborted step published carry its epoch; later steps use larger
     * epochs, so none of them can be taken for current data.  Only the error
     * word needs clearing. */
    cudaError_t e = cudaMemset(h->d_err, 0, sizeof(uint32_t) * ERR_WORDS);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    return err[0] == 4 ? AMK_ERR_INVALID_ARG : AMK_ERR_TIMEOUT;
}

amk_status amk_destroy(amk_handle *h) {
    if (!h) return AMK_OK;
    cudaDeviceSynchronize();
    free_handle(h);
    return AMK_OK;
}

amk_status amk_last_error(const amk_handle *h, amk_error_info *info) {
    if (!h || !info) return AMK_ERR_INVALID_ARG;
    *info = h->last_err;
    return AMK_OK;
}

amk_status amk_get_plan_info(const amk_handle *h, amk_plan_info *info) {
    if (!h) return AMK_ERR_INVALID_ARG;
    return amk_plan_get_info(h->plan, info);
}

amk_status amk_debug_drop_signal(amk_handle *h, int32_t sm, int32_t task) {
    if (!h) return AMK_ERR_INVALID_ARG;
    for (Task &t : h->h_tasks) t.flags &= (uint8_t)~TF_SKIP_SIGNAL;
    if (sm >= 0) {
        if (sm >= h->n_sm || task < 0 || task >= h->h_start[sm + 1] - h->h_start[sm]) return AMK_ERR_INVALID_ARG;
        h->h_tasks[h->h_start[sm] + task].flags |= TF_SKIP_SIGNAL;
    }
    cudaError_t e = cudaMemcpy(h->d_tasks, h->h_tasks.data(), sizeof(Task) * h->h_tasks.size(), cudaMemcpyHostToDevice);
    return cuda_fail(e);
}

amk_status amk_debug_read_residuals(const amk_handle *h, float *x_in, float *x_mid) {
    if (!h || !x_in || !x_mid) return AMK_ERR_INVALID_ARG;
    const int L = h->cfg.n_layers;
    if (h->params.depth != L + 1) return AMK_ERR_UNSUPPORTED;
    const size_t per = (size_t)h->cfg.max_batch * h->cfg.hidden;
    if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    std::vector<uint64_t> w(per * (L + 1));
    cudaError_t e = cudaMemcpy(w.data(), h->params.x_in, sizeof(uint64_t) * per * (L + 1), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    for (size_t i = 0; i < w.size(); ++i) {
        const uint32_t u = (uint32_t)w[i];
        std::memcpy(&x_in[i], &u, 4);
    }
    e = cudaMemcpy(w.data(), h->params.x_mid, sizeof(uint64_t) * per * L, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    for (size_t i = 0; i < per * L; ++i) {
        const uint32_t u = (uint32_t)w[i];
        std::memcpy(&x_mid[i], &u, 4);
    }
    return AMK_OK;
}

amk_status amk_debug_read_trace(const amk_handle *h, uint64_t *out, size_t n_entries) {
    if (!h || !out) return AMK_ERR_INVALID_ARG;
    if (!h->d_trace) return AMK_ERR_UNSUPPORTED;
    if (n_entries < 16 * h->h_tasks.size()) return AMK_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    return cuda_fail(cudaMemcpy(out, h->d_trace, sizeof(uint64_t) * 16 * h->h_tasks.size(), cudaMemcpyDeviceToHost));
}

}  // extern "C"
