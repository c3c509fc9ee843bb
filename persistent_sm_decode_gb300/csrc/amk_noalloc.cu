/*
 * amk_noalloc.cu — a decode step for callers that cannot allocate device
 * memory.
 *
 * amk_create allocates the task table, RoPE table, error word and activation
 * scratch with cudaMalloc.  Some callers cannot do that at all: code running
 * under an external memory manager that owns every device allocation, or in
 * an environment where cudaMalloc is forbidden after start-up.  For them,
 * amk_decode_step_noalloc runs the same persistent kernel with all of that
 * state in one file-scope device array (g_noalloc_state below, 16 MiB), which
 * every GPU that loads this library holds until the process exits.
 *
 * On its first call on a device (with that device current) the entry point
 * takes the array's device address with cudaGetSymbolAddress and clears it;
 * make that first call before any stream capture.  A call with a new
 * configuration or new weight pointers plans the schedule on the host and
 * copies it into the array (clearing the epoch-tagged scratch, which must
 * start at zero).  No call makes cudaMalloc, cudaFree or any other allocating
 * routine; the state only moves by cudaMemset and cudaMemcpy.
 *
 * All calls on a device share the array, so two calls that overlapped on the
 * GPU would race on it.  To keep that from happening inside one process, each
 * call holds a process-wide lock and waits for its own step to finish before
 * it returns (which is also how it reports a device-side timeout).  The wait
 * is a cudaStreamSynchronize on the caller's stream made while the lock is
 * held: do not call this from a stream callback or host function, nor while
 * the caller's stream waits on work that another thread's call enqueues.
 */
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "amk.h"
#include "amk_launch.h"
#include "amk_plan.h"
#include "amk_plan_impl.h"

using namespace amk;

namespace {

constexpr size_t NOALLOC_BYTES = (size_t)16 << 20; /* the stated maximum of the shared state */
constexpr int MAX_DEVICES = 64;

static __device__ __align__(256) uint8_t g_noalloc_state[NOALLOC_BYTES];

struct DeviceState {
    bool ready = false;
    uint8_t *base = nullptr; /* device address of g_noalloc_state on this device */
    uint32_t epoch = 0;      /* keeps growing across calls and configurations */
    std::vector<uint8_t> key; /* configuration + weight pointers of the uploaded schedule */
    amk_plan *plan = nullptr;
    KernelFn fn = nullptr;
    Params params;
};

std::mutex g_mu;
DeviceState g_dev[MAX_DEVICES];

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

amk_status fail(cudaError_t e) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? AMK_ERR_OOM : AMK_ERR_CUDA;
}

amk_status check_args(const amk_config *c, const amk_weights *w) {
    if (!c || !w || !w->embed || !w->final_norm || !w->layers) return AMK_ERR_INVALID_ARG;
    if (!aligned16(w->embed) || !aligned16(w->final_norm)) return AMK_ERR_INVALID_ARG;
    const bool i8 = c->weight_dtype == AMK_WEIGHT_INT8 || c->weight_dtype == AMK_WEIGHT_INT4; /* scaled formats */
    if (!c->tied_embeddings && (!w->lm_head || !aligned16(w->lm_head) || (i8 && !w->s_lm))) return AMK_ERR_INVALID_ARG;
    if (c->n_layers < 1 || c->n_layers > 4096) return AMK_ERR_INVALID_ARG;
    for (int l = 0; l < c->n_layers; ++l) {
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

/* Plan the configuration and lay its state out in the array: error word,
 * task table, CTA offsets, layer pointers, RoPE table, activation scratch. */
amk_status upload(DeviceState &ds, const amk_config *c, const amk_weights *w, int dev) {
    int n_sm = 0, smem_optin = 0, coop = 0;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
        return fail(cudaErrorUnknown);
    if (!coop) return AMK_ERR_COOPERATIVE;
    if (ds.plan) {
        amk_plan_destroy(ds.plan);
        ds.plan = nullptr;
    }
    ds.key.clear();
    std::string msg;
    amk_status st = plan_build(c, c->max_batch, n_sm, smem_optin, nullptr, &ds.plan, &msg);
    if (st != AMK_OK) {
        std::fprintf(stderr, "amk_decode_step_noalloc: %s\n", msg.c_str());
        return st;
    }
    const amk_plan &P = *ds.plan;
    std::vector<Task> tasks;
    std::vector<int32_t> start(n_sm + 1, 0);
    for (int s = 0; s < n_sm; ++s) {
        start[s + 1] = start[s] + (int)P.sm_tasks[s].size();
        tasks.insert(tasks.end(), P.sm_tasks[s].begin(), P.sm_tasks[s].end());
    }
    const Geo g = make_geo(*c, c->max_batch);
    const int L = c->n_layers, d = c->head_dim;
    std::vector<LayerPtrs> lp(L);
    for (int l = 0; l < L; ++l) {
        const amk_layer_weights &x = w->layers[l];
        const void *m[7] = {x.wq, x.wk, x.wv, x.wo, x.w_gate, x.w_up, x.w_down};
        const float *sc[7] = {x.s_q, x.s_k, x.s_v, x.s_o, x.s_gate, x.s_up, x.s_down};
        for (int i = 0; i < 7; ++i) {
            lp[l].w[i] = m[i];
            lp[l].s[i] = sc[i];
        }
        lp[l].attn_norm = (const uint16_t *)x.attn_norm;
        lp[l].mlp_norm = (const uint16_t *)x.mlp_norm;
    }
    std::vector<float> rope((size_t)c->max_seq * d);
    for (int p = 0; p < c->max_seq; ++p)
        for (int i = 0; i < d / 2; ++i) {
            const double th = (double)p * std::pow((double)c->rope_theta, -2.0 * i / d);
            rope[(size_t)p * d + 2 * i] = (float)std::cos(th);
            rope[(size_t)p * d + 2 * i + 1] = (float)std::sin(th);
        }
    const ScratchSizes ss = scratch_sizes(P);
    size_t off = 0;
    const size_t o_err = off;
    off += up256(sizeof(uint32_t) * ERR_WORDS);
    const size_t o_tasks = off;
    off += up256(sizeof(Task) * tasks.size());
    const size_t o_start = off;
    off += up256(sizeof(int32_t) * start.size());
    const size_t o_layers = off;
    off += up256(sizeof(LayerPtrs) * L);
    const size_t o_rope = off;
    off += up256(sizeof(float) * rope.size());
    const size_t o_xin = off;
    off += up256(8 * ss.x_in);
    const size_t o_xmid = off;
    off += up256(8 * ss.x_mid);
    const size_t o_qkv = off;
    off += up256(8 * ss.qkv);
    const size_t o_part = off;
    off += up256(8 * ss.part);
    const size_t o_aout = off;
    off += up256(8 * ss.aout);
    const size_t o_act = off;
    off += up256(8 * ss.act);
    const size_t o_argp = off;
    off += up256(8 * ss.argp);
    if (off > NOALLOC_BYTES) {
        std::fprintf(stderr,
                     "amk_decode_step_noalloc: this configuration needs %zu bytes of static device state; "
                     "the maximum is %zu\n",
                     off, NOALLOC_BYTES);
        amk_plan_destroy(ds.plan);
        ds.plan = nullptr;
        return AMK_ERR_UNSUPPORTED;
    }
    /* from here on every failure also drops the plan, so that a later call
     * plans again instead of running a half-uploaded schedule */
    auto drop = [&](amk_status why) {
        amk_plan_destroy(ds.plan);
        ds.plan = nullptr;
        return why;
    };
    ds.fn = select_kernel(c->weight_dtype, c->max_batch);
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, (const void *)ds.fn) != cudaSuccess ||
        prepare_kernel(ds.fn, P.smem_bytes) != cudaSuccess) {
        cudaGetLastError();
        return drop(AMK_ERR_UNSUPPORTED);
    }
    int per_sm = 0;
    if (occupancy(ds.fn, P.smem_bytes, &per_sm) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        return drop(AMK_ERR_COOPERATIVE);
    }
    cudaError_t e = cudaMemset(ds.base, 0, off);
    if (e == cudaSuccess) e = cudaMemcpy(ds.base + o_tasks, tasks.data(), sizeof(Task) * tasks.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(ds.base + o_start, start.data(), sizeof(int32_t) * start.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(ds.base + o_layers, lp.data(), sizeof(LayerPtrs) * L, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(ds.base + o_rope, rope.data(), sizeof(float) * rope.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return drop(fail(e));

    Params &p = ds.params;
    std::memset(&p, 0, sizeof p);
    p.L = L;
    p.H = g.H;
    p.nq = g.nq;
    p.nkv = g.nkv;
    p.d = d;
    p.I = g.I;
    p.V = g.V;
    p.G = g.G;
    p.Bmax = c->max_batch;
    p.Smax = c->max_seq;
    p.qkv_rows = g.qkv_rows;
    p.eps = c->rms_eps;
    p.qk_scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
    p.wf = g.wf;
    p.lm_wf = g.lm_wf;
    p.group = g.group;
    p.tasks = (const Task *)(ds.base + o_tasks);
    p.task_start = (const int32_t *)(ds.base + o_start);
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
    p.layers = (const LayerPtrs *)(ds.base + o_layers);
    p.embed = (const uint16_t *)w->embed;
    p.final_norm = (const uint16_t *)w->final_norm;
    p.lm = c->tied_embeddings ? w->embed : w->lm_head;
    p.s_lm = c->tied_embeddings ? nullptr : w->s_lm;
    p.x_in = (uint64_t *)(ds.base + o_xin);
    p.x_mid = (uint64_t *)(ds.base + o_xmid);
    p.qkv = (uint64_t *)(ds.base + o_qkv);
    p.part = (uint64_t *)(ds.base + o_part);
    p.aout = (uint64_t *)(ds.base + o_aout);
    p.act = (uint64_t *)(ds.base + o_act);
    p.argp = (uint64_t *)(ds.base + o_argp);
    p.n_lmh = P.n_lmh;
    p.epoch_word = nullptr; /* the epoch is passed with each launch */
    p.err = (uint32_t *)(ds.base + o_err);
    p.rope = (const float *)(ds.base + o_rope);
    p.timeout_ns = 1000000000LL;
    p.trace = nullptr;
    return AMK_OK;
}

std::vector<uint8_t> make_key(const amk_config *c, const amk_weights *w) {
    std::vector<uint8_t> k(sizeof(amk_config) + sizeof(void *) * 4 + sizeof(amk_layer_weights) * c->n_layers);
    uint8_t *q = k.data();
    std::memcpy(q, c, sizeof(amk_config));
    q += sizeof(amk_config);
    const void *top[4] = {w->embed, w->final_norm, w->lm_head, w->s_lm};
    std::memcpy(q, top, sizeof top);
    q += sizeof top;
    std::memcpy(q, w->layers, sizeof(amk_layer_weights) * c->n_layers);
    return k;
}

}  // namespace

extern "C" amk_status amk_decode_step_noalloc(const amk_config *config, const amk_weights *weights, int32_t batch,
                                              const int32_t *tokens, const int32_t *positions, void *kv_cache,
                                              float *logits, amk_stream_t stream) {
    amk_status st = check_args(config, weights);
    if (st != AMK_OK) return st;
    if (!tokens || !positions || !kv_cache || !logits || batch < 1 || batch > config->max_batch) return AMK_ERR_INVALID_ARG;
    if (!aligned16(kv_cache) || ((uintptr_t)tokens & 3u) || ((uintptr_t)positions & 3u) || ((uintptr_t)logits & 3u))
        return AMK_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(cudaErrorNoDevice);
    if (dev < 0 || dev >= MAX_DEVICES) return AMK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &ds = g_dev[dev];
    if (!ds.ready) {
        /* set-up, once per device with that device current: the host-side
         * name of the array is not a device address */
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_state);
        if (e != cudaSuccess) return fail(e);
        e = cudaMemset(ptr, 0, NOALLOC_BYTES);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return fail(e);
        ds.base = (uint8_t *)ptr;
        ds.ready = true;
    }
    std::vector<uint8_t> key = make_key(config, weights);
    if (key != ds.key) {
        st = upload(ds, config, weights, dev);
        if (st != AMK_OK) return st;
        ds.key = std::move(key);
    }
    Params p = ds.params;
    const size_t per_cache =
        (size_t)config->n_layers * config->max_batch * config->n_kv_heads * config->max_seq * config->head_dim;
    p.kc = (uint16_t *)kv_cache;
    p.vc = p.kc + per_cache;
    p.tokens = tokens;
    p.positions = positions;
    p.logits = logits;
    p.batch = batch;
    p.epoch = ++ds.epoch;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_decode(ds.fn, p, ds.plan->n_sm, ds.plan->smem_bytes, s);
    if (e != cudaSuccess) {
        --ds.epoch; /* nothing ran under this epoch */
        return fail(e);
    }
    /* synchronous: report a device-side timeout or bad input of this step */
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(e);
    uint32_t err[ERR_WORDS];
    e = cudaMemcpy(err, p.err, sizeof err, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(e);
    if (err[0] != 0) {
        /* a step that sees a set error word does nothing, so the word must be
         * clear before the next call; if clearing fails, say so */
        e = cudaMemset(p.err, 0, sizeof err);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return fail(e);
        return err[0] == 4 ? AMK_ERR_INVALID_ARG : AMK_ERR_TIMEOUT;
    }
    return AMK_OK;
}
