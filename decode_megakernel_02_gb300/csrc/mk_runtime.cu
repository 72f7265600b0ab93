// Runtime half of the C ABI: contract + schedule checks at create, then one
// cooperative launch per prefill/decode call on the caller's stream.
//
// Netra Kernel summary (section details): the runtime binds persistent and
// boundary buffers and replays a fixed launch on a caller-owned stream; the
// AutoMegaKernel explainer ("Methodology", safety gate): a schedule that fails
// validation is rejected before any GPU launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "mk_host.h"
#include "mk_prefill.h"

namespace mk {
const void* vm_kernel_for(int wdtype, int base, int hd, bool sel);
size_t vm_shared_bytes(int wdtype, int xs_floats, int tab_cap);
cudaError_t launch_dequant(int wdtype, const uint8_t* rows, int64_t stride, int first, int step, int nrows,
                           int K, float* out, cudaStream_t st);
cudaError_t launch_watchdog(uint32_t* ctr, uint32_t* status, int64_t limit_ns, cudaStream_t st);
cudaError_t static_scratch_address(void** ptr);
}  // namespace mk

using namespace mk;

struct mk_handle {
    mk_model_desc d;
    Config c;
    WsLayout ws;
    BlobLayout bl;
    int32_t n_tasks = 0, n_counters = 0;
    const uint8_t* w = nullptr;
    uint16_t* kv = nullptr;
    uint8_t* wsp = nullptr;
    cudaStream_t st = nullptr;
    int device = 0;
    const void* kfn = nullptr;      // greedy instance
    const void* kfn_sel = nullptr;  // token-selection instance (sampling, EOS, token-select task)
    size_t smem = 0;
    int32_t pos = 0, pending = -1;
    bool has_seq = false;
    uint32_t epoch = 0;
    bool dirty = false;
    int64_t launches = 0;
    int32_t xs_floats = 0;
    int32_t tab_cap = 0;                 // longest per-CTA queue (shared-memory task table)
    const int32_t* queue = nullptr;      // task id of each queue index (host copy, for errors)
    std::vector<int32_t> queue_store;    // owns `queue` for handles made by mk_create
    unsigned long long* trace = nullptr;
    int32_t trace_cap = 0;
    // token selection (mk_set_sampling)
    float temperature = 0.f;
    int32_t top_k = 0;
    uint64_t seed = 0;
    int32_t eos = -1;
    int32_t ctr_tok = 0, n_tok = 0;      // the counter after which a step's token is final, its producers
    int32_t lm_rows_max = 0;
    int32_t launched = 0;                // steps of the last launch
    int32_t last_steps = 0;              // steps it ran (fewer after an EOS stop)
    bool unsettled = false;              // an async launch with EOS whose step count is not read yet
    // tensor-core prefill: weight maps per layer (QKV, O, gate/up, down) and the
    // chunk activations' maps (normed x, attention output, SwiGLU output)
    std::vector<CUtensorMap> pf_w;
    CUtensorMap pf_a[6]{};               // normed x, attention output, SwiGLU output: hi, lo each
    std::string err;
};

static mk_status prefill_maps(mk_handle* h);

namespace {

mk_status herr(mk_handle* h, mk_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (h) h->err = buf;
    set_error("%s", buf);
    return st;
}

mk_status cuda_fail(mk_handle* h, cudaError_t e, const char* what) {
    return herr(h, MK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CK(h, call)                                   \
    do {                                              \
        cudaError_t e_ = (call);                      \
        if (e_ != cudaSuccess) return cuda_fail(h, e_, #call); \
    } while (0)

mk_status reset_sync_state(mk_handle* h) {
    CK(h, cudaMemsetAsync(h->wsp + h->ws.status, 0, 32, h->st));
    CK(h, cudaMemsetAsync(h->wsp + h->ws.counters, 0, (size_t)h->n_counters * CTR_STRIDE * 4, h->st));
    CK(h, cudaMemsetAsync(h->wsp + h->ws.key, 0, 8, h->st));
    CK(h, cudaMemsetAsync(h->wsp + h->ws.tokw, 0, 8, h->st));
    CK(h, cudaMemsetAsync(h->wsp + h->ws.cand, 0, (size_t)h->c.sms * MAX_TOP_K * 8, h->st));
    // tagged values: tags restart with the epoch, so no stale word may match
    CK(h, cudaMemsetAsync(h->wsp + h->ws.qkv, 0, (size_t)(h->ws.part_ml - h->ws.qkv), h->st));
    h->epoch = 0;
    h->dirty = false;
    return MK_OK;
}

// Let the kernel take up to the device's opt-in shared memory per block
// (minus its static shared memory).  The attribute is per kernel function, so
// every handle and static call sets the same value.
cudaError_t raise_smem_limit(const void* kfn, int smem_optin) {
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kfn);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_optin - (int)fa.sharedSizeBytes);
}

mk_status launch(mk_handle* h, int n_steps, const int32_t* forced, int32_t* out_ids, float* logits,
                 int skip_lm) {
    if (h->unsettled)
        return herr(h, MK_ERR_INVALID_ARG, "an earlier launch with an EOS id is not finished: call mk_finish first");
    if (h->dirty || h->epoch + (uint32_t)n_steps >= (uint32_t)KEY_TAG_MAX - 1u) {
        mk_status st = reset_sync_state(h);
        if (st) return st;
    }
    VmParams p{};
    p.w = h->w;
    p.kv = h->kv;
    p.status = (uint32_t*)(h->wsp + h->ws.status);
    p.counters = (uint32_t*)(h->wsp + h->ws.counters);
    p.key = (unsigned long long*)(h->wsp + h->ws.key);
    p.recs = (const TaskRec*)(h->wsp + h->ws.recs);
    p.queue_off = (const int32_t*)(h->wsp + h->ws.queue_off);
    p.inv_freq = (const float*)(h->wsp + h->ws.inv_freq);
    p.x = (float*)(h->wsp + h->ws.x);
    p.qkv = (unsigned long long*)(h->wsp + h->ws.qkv);
    p.part_ml = (float*)(h->wsp + h->ws.part_ml);
    p.part_acc = (uint16_t*)(h->wsp + h->ws.part_acc);
    p.att = (float*)(h->wsp + h->ws.att);
    p.merge_tasks = merge_tasks(&h->d, h->c) ? 1 : 0;
    p.h = (float*)(h->wsp + h->ws.h);
    p.forced = forced;
    p.out_ids = out_ids;
    p.logits = logits;
    const mk_model_desc& d = h->d;
    p.L = d.n_layers;
    p.d = d.d_model;
    p.Hq = d.n_q_heads;
    p.Hkv = d.n_kv_heads;
    p.hd = d.head_dim;
    p.F = d.d_ffn;
    p.V = d.vocab;
    p.max_seq = d.max_seq;
    p.wdtype = d.wdtype;
    p.base_dtype = d.base_dtype;
    p.q_dim = d.n_q_heads * d.head_dim;
    p.kv_dim = d.n_kv_heads * d.head_dim;
    p.C = h->c.C;
    p.fused = h->bl.down_cols ? 1 : 0;
    p.eps = d.rms_eps;
    p.layer_bytes = h->bl.layer_bytes;
    p.l_attn_norm = h->bl.l_attn_norm;
    p.l_ffn_norm = h->bl.l_ffn_norm;
    p.l_down = h->bl.l_down;
    p.final_norm = h->bl.final_norm;
    p.embed = h->bl.embed;
    p.n_steps = n_steps;
    p.pos0 = h->pos;
    p.epoch0 = (int32_t)h->epoch;
    p.skip_lm = skip_lm;
    p.pending = h->pending;
    p.xs_floats = h->xs_floats;
    p.tab_cap = h->tab_cap;
    p.watchdog_ns = h->c.watchdog_ns;
    const bool sampling = h->temperature > 0.f && !skip_lm;
    p.inv_temp = sampling ? 1.f / h->temperature : 0.f;
    p.top_k = sampling ? h->top_k : 0;
    p.seed_lo = (uint32_t)h->seed;
    p.seed_hi = (uint32_t)(h->seed >> 32);
    p.eos = skip_lm ? -1 : h->eos;
    p.ctr_tok = h->ctr_tok;
    p.n_tok = h->n_tok;
    p.cand = (unsigned long long*)(h->wsp + h->ws.cand);
    p.tokw = h->c.token_select ? (unsigned long long*)(h->wsp + h->ws.tokw) : nullptr;
    p.trace = h->trace;
    p.trace_cap = h->trace_cap;
    void* args[] = {&p};
    const bool sel = p.inv_temp > 0.f || p.eos >= 0 || p.tokw != nullptr;
    CK(h, cudaLaunchCooperativeKernel(sel ? h->kfn_sel : h->kfn, dim3(h->c.sms), dim3(THREADS), args, h->smem, h->st));
    h->epoch += (uint32_t)n_steps;
    h->launches++;
    h->launched = n_steps;
    h->last_steps = n_steps;
    return MK_OK;
}

// Steps the last decode launch ran, from the status word the FIN / select task
// writes (s[4]); with an EOS id it may be fewer than launched, and the
// synchronisation epoch advances only by the steps that ran.
int32_t steps_run(mk_handle* h, const uint32_t* s) {
    if (h->eos < 0) return h->launched;
    const int32_t ran = (int32_t)s[4];
    const int32_t steps = ran >= 1 && ran <= h->launched ? ran : h->launched;
    h->epoch -= (uint32_t)(h->launched - steps);
    h->last_steps = steps;
    return steps;
}

mk_status read_status(mk_handle* h, uint32_t* out5 = nullptr) {
    uint32_t s[5] = {0, 0, 0, 0, 0};
    CK(h, cudaMemcpyAsync(s, h->wsp + h->ws.status, sizeof s, cudaMemcpyDeviceToHost, h->st));
    CK(h, cudaStreamSynchronize(h->st));
    if (out5) std::memcpy(out5, s, sizeof s);
    if (s[0] == DEV_OK) return MK_OK;
    h->dirty = true;
    h->unsettled = false;
    const int task = h->queue && s[1] < (uint32_t)h->n_tasks ? h->queue[s[1]] : -1;
    if (s[0] == DEV_TIMEOUT)
        return herr(h, MK_ERR_TIMEOUT, "device wait gave up (task %d, step %u); counters are reset on the next launch",
                    task, s[2]);
    return herr(h, MK_ERR_DEVICE, "device reported error %u (task %d, step %u)", s[0], task, s[2]);
}

}  // namespace

extern "C" {

mk_status mk_workspace_size(const mk_model_desc* desc, const mk_schedule_config* cfg, int32_t n_sms,
                            size_t* bytes) {
    mk_status st = check_desc(desc);
    if (st) return st;
    if (!bytes) {
        set_error("bytes is NULL");
        return MK_ERR_INVALID_ARG;
    }
    if (n_sms <= 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) {
            set_error("no CUDA device to take the SM count from: %s", cudaGetErrorString(e));
            return MK_ERR_CUDA;
        }
    }
    Config c;
    if ((st = resolve_config(desc, cfg, n_sms, &c))) return st;
    Lowering lw;
    if ((st = lower(desc, c, &lw))) return st;
    *bytes = (size_t)ws_layout(desc, c, (int64_t)lw.tasks.size(), lw.n_counters).total;
    return MK_OK;
}

mk_status mk_create(const mk_model_desc* desc, const mk_schedule_config* cfg, const void* weights_dev,
                    size_t weights_bytes, void* kv_dev, size_t kv_bytes, void* workspace_dev,
                    size_t workspace_bytes, mk_stream_t stream, mk_handle** out) {
    mk_status st = check_desc(desc);
    if (st) return st;
    if (!out || !weights_dev || !kv_dev || !workspace_dev) {
        set_error("NULL argument");
        return MK_ERR_INVALID_ARG;
    }
    *out = nullptr;
    if (((uintptr_t)weights_dev & 255) || ((uintptr_t)workspace_dev & 255) || ((uintptr_t)kv_dev & 15)) {
        set_error("misaligned buffer: weights and workspace need 256-byte, the KV cache 16-byte alignment");
        return MK_ERR_INVALID_ARG;
    }
    int dev = 0, n_sms = 0, smem_optin = 0, coop = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (e != cudaSuccess) {
        set_error("CUDA device query failed: %s", cudaGetErrorString(e));
        return MK_ERR_CUDA;
    }
    if (!coop) {
        set_error("device %d does not support cooperative launches", dev);
        return MK_ERR_UNSUPPORTED;
    }
    Config c;
    if ((st = resolve_config(desc, cfg, n_sms, &c))) return st;
    const int xs_floats = std::max(desc->d_model, desc->n_q_heads * desc->head_dim);
    Lowering lw;
    if ((st = lower(desc, c, &lw))) return st;
    std::vector<TaskRec> recs;
    std::vector<int32_t> queue, qoff;
    int32_t tab_cap = 0;
    if ((st = device_tables(lw, c.sms, &recs, &queue, &qoff, &tab_cap))) return st;
    if (vm_shared_bytes(desc->wdtype, xs_floats, tab_cap) > (size_t)smem_optin) {
        set_error("shared memory need %zu > %d (%d tasks per CTA)", vm_shared_bytes(desc->wdtype, xs_floats, tab_cap),
                  smem_optin, tab_cap);
        return MK_ERR_UNSUPPORTED;
    }
    {
        mk_ir* ir = to_ir(lw, c.sms);
        std::string why;
        st = validate_ir(ir, &why);
        mk_free_ir(ir);
        if (st) {
            set_error("schedule rejected before launch: %s", why.c_str());
            return MK_ERR_SCHEDULE_INVALID;
        }
    }
    size_t need_w = 0, need_kv = 0;
    mk_packed_size(desc, &need_w);
    mk_kv_cache_size(desc, &need_kv);
    WsLayout ws = ws_layout(desc, c, (int64_t)lw.tasks.size(), lw.n_counters);
    if (weights_bytes < need_w || kv_bytes < need_kv || workspace_bytes < (size_t)ws.total) {
        set_error("buffer too small: weights %zu/%zu, kv %zu/%zu, workspace %zu/%lld", weights_bytes, need_w,
                  kv_bytes, need_kv, workspace_bytes, (long long)ws.total);
        return MK_ERR_CAPACITY;
    }
    mk_handle* h = new mk_handle();
    h->d = *desc;
    h->c = c;
    h->ws = ws;
    h->bl = blob_layout(desc);
    h->n_tasks = (int32_t)lw.tasks.size();
    h->n_counters = lw.n_counters;
    h->w = (const uint8_t*)weights_dev;
    h->kv = (uint16_t*)kv_dev;
    h->wsp = (uint8_t*)workspace_dev;
    h->st = (cudaStream_t)stream;
    h->device = dev;
    h->kfn = vm_kernel_for(desc->wdtype, desc->base_dtype, desc->head_dim, false);
    h->kfn_sel = vm_kernel_for(desc->wdtype, desc->base_dtype, desc->head_dim, true);
    h->smem = vm_shared_bytes(desc->wdtype, xs_floats, tab_cap);
    h->xs_floats = xs_floats;
    h->tab_cap = tab_cap;
    h->queue_store = queue;
    h->queue = h->queue_store.data();
    h->ctr_tok = lw.ctr_tok;
    h->n_tok = lw.n_tok;
    h->lm_rows_max = lw.lm_rows_max;
    if (!h->kfn || !h->kfn_sel) {
        delete h;
        set_error("no kernel for wdtype %d / base %d", desc->wdtype, desc->base_dtype);
        return MK_ERR_UNSUPPORTED;
    }
    auto fail = [&](mk_status s) {
        set_error("%s", h->err.c_str());
        delete h;
        return s;
    };
    // The attribute belongs to the kernel function, not to this handle: other
    // handles launch the same instantiation with their own (possibly larger)
    // shared memory, so it is raised to the device's opt-in limit instead of
    // this handle's need, and no handle can lower it under another.
    for (const void* fn : {h->kfn, h->kfn_sel}) {
        e = raise_smem_limit(fn, smem_optin);
        if (e != cudaSuccess) return fail(cuda_fail(h, e, "cudaFuncSetAttribute"));
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, THREADS, h->smem);
        if (e != cudaSuccess) return fail(cuda_fail(h, e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor"));
        if (per_sm < 1 || (int64_t)per_sm * n_sms < c.sms)
            return fail(herr(h, MK_ERR_UNSUPPORTED, "%d CTAs cannot be co-resident (%d per SM)", c.sms, per_sm));
    }

    // device tables: task records, queue offsets, RoPE inverse frequencies
    std::vector<float> inv(desc->head_dim / 2);
    for (int i = 0; i < desc->head_dim / 2; ++i)
        inv[i] = (float)std::pow((double)desc->rope_theta, -2.0 * i / (double)desc->head_dim);
    e = cudaMemcpyAsync(h->wsp + ws.recs, recs.data(), recs.size() * sizeof(TaskRec), cudaMemcpyHostToDevice, h->st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->wsp + ws.queue_off, qoff.data(), qoff.size() * 4, cudaMemcpyHostToDevice, h->st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->wsp + ws.inv_freq, inv.data(), inv.size() * 4, cudaMemcpyHostToDevice, h->st);
    if (e != cudaSuccess) return fail(cuda_fail(h, e, "uploading the schedule"));
    if ((st = reset_sync_state(h))) return fail(st);
    if (c.pf_chunk > 0 && (st = prefill_maps(h))) return fail(st);
    e = cudaStreamSynchronize(h->st);
    if (e != cudaSuccess) return fail(cuda_fail(h, e, "cudaStreamSynchronize"));
    *out = h;
    return MK_OK;
}

}  // extern "C"

// Tensor maps of the tensor-core prefill (mk_create, prefill_chunk > 0).
static mk_status prefill_maps(mk_handle* h) {
    const mk_model_desc& d = h->d;
    const BlobLayout& bl = h->bl;
    const bool f16 = d.base_dtype == MK_W_FP16;
    const int64_t qd = (int64_t)d.n_q_heads * d.head_dim, kd = (int64_t)d.n_kv_heads * d.head_dim;
    if (d.wdtype != d.base_dtype || kd % 128 != 0)
        return herr(h, MK_ERR_UNSUPPORTED, "tensor-core prefill needs 16-bit weights and n_kv_heads * head_dim %% 128 == 0");
    if (!pf::tensor_map_encoder_ready())
        return herr(h, MK_ERR_UNSUPPORTED, "the driver offers no tensor-map encoder");
    const int64_t mc = h->c.pf_chunk;
    bool ok = pf::make_map_rows(&h->pf_a[0], h->wsp + h->ws.pf_h, mc, d.d_model, d.d_model * 2, pf::BM, f16) &&
              pf::make_map_rows(&h->pf_a[1], h->wsp + h->ws.pf_hl, mc, d.d_model, d.d_model * 2, pf::BM, f16) &&
              pf::make_map_rows(&h->pf_a[2], h->wsp + h->ws.pf_ao, mc, qd, qd * 2, pf::BM, f16) &&
              pf::make_map_rows(&h->pf_a[3], h->wsp + h->ws.pf_aol, mc, qd, qd * 2, pf::BM, f16) &&
              pf::make_map_rows(&h->pf_a[4], h->wsp + h->ws.pf_gu, mc, d.d_ffn, (int64_t)d.d_ffn * 2, pf::BM, f16) &&
              pf::make_map_rows(&h->pf_a[5], h->wsp + h->ws.pf_gul, mc, d.d_ffn, (int64_t)d.d_ffn * 2, pf::BM, f16);
    h->pf_w.assign((size_t)d.n_layers * 4, CUtensorMap{});
    for (int l = 0; l < d.n_layers && ok; ++l) {
        const uint8_t* lb = h->w + bl.layer_bytes * l;
        CUtensorMap* m = &h->pf_w[(size_t)l * 4];
        ok = pf::make_map_rows(&m[0], lb + bl.l_qkv, qd + 2 * kd, d.d_model, bl.row_qkv, pf::BN, f16) &&
             pf::make_map_rows(&m[1], lb + bl.l_o, d.d_model, qd, bl.row_o, pf::BN, f16) &&
             pf::make_map_rows(&m[2], lb + bl.l_gu, 2 * (int64_t)d.d_ffn, d.d_model, bl.row_gu, pf::BN, f16) &&
             (bl.down_cols ? pf::make_map_blocks(&m[3], lb + bl.l_down, d.d_model, d.d_ffn, pf::BN, f16)
                           : pf::make_map_rows(&m[3], lb + bl.l_down, d.d_model, d.d_ffn, bl.row_down, pf::BN, f16));
    }
    if (!ok) return herr(h, MK_ERR_CUDA, "cuTensorMapEncodeTiled rejected a prefill tensor map");
    return MK_OK;
}

// Positions 0 .. n-2 through the layers, pf_chunk tokens at a time (the
// tokens are already in the workspace).  The last layer stops after its KV
// append: nothing after it reaches the cache.
static mk_status prefill_tensor_cores(mk_handle* h, int32_t n) {
    const mk_model_desc& d = h->d;
    const BlobLayout& bl = h->bl;
    const bool f16 = d.base_dtype == MK_W_FP16;
    const int qd = d.n_q_heads * d.head_dim, kd = d.n_kv_heads * d.head_dim;
    float* x = (float*)(h->wsp + h->ws.pf_x);
    uint16_t* hb = (uint16_t*)(h->wsp + h->ws.pf_h);
    uint16_t* hbl = (uint16_t*)(h->wsp + h->ws.pf_hl);
    float* q = (float*)(h->wsp + h->ws.pf_q);
    uint16_t* ao = (uint16_t*)(h->wsp + h->ws.pf_ao);
    uint16_t* aol = (uint16_t*)(h->wsp + h->ws.pf_aol);
    uint16_t* gu = (uint16_t*)(h->wsp + h->ws.pf_gu);
    uint16_t* gul = (uint16_t*)(h->wsp + h->ws.pf_gul);
    uint32_t* err = (uint32_t*)(h->wsp + h->ws.pf_err);
    const int32_t* tok = (const int32_t*)(h->wsp + h->ws.tok);
    CK(h, cudaMemsetAsync(err, 0, 4, h->st));
    for (int c0 = 0; c0 < n - 1; c0 += h->c.pf_chunk) {
        const int mv = std::min(h->c.pf_chunk, n - 1 - c0), mr = (mv + pf::BM - 1) / pf::BM * pf::BM;
        CK(h, pf::launch_embed((const uint16_t*)(h->w + bl.embed), tok + c0, mv, d.d_model, f16, x, h->st));
        for (int l = 0; l < d.n_layers; ++l) {
            const uint8_t* lb = h->w + bl.layer_bytes * l;
            const CUtensorMap* m = &h->pf_w[(size_t)l * 4];
            pf::GemmArgs g{};
            g.M = mr;
            g.m_valid = mv;
            g.f16 = f16 ? 1 : 0;
            g.err = err;
            CK(h, pf::launch_rmsnorm(x, (const uint16_t*)(lb + bl.l_attn_norm), mv, d.d_model, d.rms_eps, f16, hb, hbl,
                                     h->st));
            pf::GemmArgs gq = g;
            gq.N = qd + 2 * kd;
            gq.K = d.d_model;
            gq.epi = pf::EPI_QKV;
            gq.out_f32 = q;
            gq.ldo = qd;
            gq.q_dim = qd;
            gq.kv_dim = kd;
            gq.hd = d.head_dim;
            gq.max_seq = d.max_seq;
            gq.pos0 = c0;
            gq.layer = l;
            gq.n_kv_heads = d.n_kv_heads;
            gq.inv_freq = (const float*)(h->wsp + h->ws.inv_freq);
            gq.kv = h->kv;
            CK(h, pf::launch_gemm(h->pf_a[0], h->pf_a[1], m[0], gq, h->st));
            if (l == d.n_layers - 1) break;
            CK(h, pf::launch_attention(q, h->kv, l, c0, mv, d.n_q_heads, d.n_kv_heads, d.head_dim, d.max_seq, f16, ao,
                                       aol, h->st));
            pf::GemmArgs go = g;
            go.N = d.d_model;
            go.K = qd;
            go.epi = pf::EPI_RESID;
            go.out_f32 = x;
            go.ldo = d.d_model;
            CK(h, pf::launch_gemm(h->pf_a[2], h->pf_a[3], m[1], go, h->st));
            CK(h, pf::launch_rmsnorm(x, (const uint16_t*)(lb + bl.l_ffn_norm), mv, d.d_model, d.rms_eps, f16, hb, hbl,
                                     h->st));
            pf::GemmArgs gg = g;
            gg.N = 2 * d.d_ffn;
            gg.K = d.d_model;
            gg.epi = pf::EPI_SWIGLU;
            gg.out16 = gu;
            gg.out16_lo = gul;
            gg.ld16 = d.d_ffn;
            CK(h, pf::launch_gemm(h->pf_a[0], h->pf_a[1], m[2], gg, h->st));
            pf::GemmArgs gd = g;
            gd.N = d.d_model;
            gd.K = d.d_ffn;
            gd.epi = pf::EPI_RESID;
            gd.out_f32 = x;
            gd.ldo = d.d_model;
            gd.b_blocks = bl.down_cols ? 1 : 0;
            CK(h, pf::launch_gemm(h->pf_a[4], h->pf_a[5], m[3], gd, h->st));
        }
    }
    uint32_t e = 0;
    CK(h, cudaMemcpyAsync(&e, err, 4, cudaMemcpyDeviceToHost, h->st));
    CK(h, cudaStreamSynchronize(h->st));
    if (e) return herr(h, MK_ERR_TIMEOUT, "a prefill GEMM wait gave up (code %u)", e);
    return MK_OK;
}

extern "C" {

mk_status mk_prefill(mk_handle* h, const int32_t* tokens_host, int32_t n) {
    if (!h || !tokens_host) {
        set_error("NULL argument");
        return MK_ERR_INVALID_ARG;
    }
    if (n < 1) return herr(h, MK_ERR_INVALID_ARG, "prefill needs at least one token");
    if (n > h->d.max_seq) return herr(h, MK_ERR_CAPACITY, "prompt of %d tokens > max_seq %d", n, h->d.max_seq);
    for (int i = 0; i < n; ++i)
        if (tokens_host[i] < 0 || tokens_host[i] >= h->d.vocab)
            return herr(h, MK_ERR_INVALID_ARG, "token %d at %d out of range", tokens_host[i], i);
    h->pos = 0;
    h->has_seq = false;
    if (n > 1) {
        CK(h, cudaMemcpyAsync(h->wsp + h->ws.tok, tokens_host, (size_t)(n - 1) * 4, cudaMemcpyHostToDevice, h->st));
        mk_status st;
        if (h->c.pf_chunk > 0) {
            if ((st = prefill_tensor_cores(h, n))) return st;
        } else {
            if ((st = launch(h, n - 1, (const int32_t*)(h->wsp + h->ws.tok), nullptr, nullptr, 1))) return st;
            if ((st = read_status(h))) return st;
        }
    }
    h->pos = n - 1;
    h->pending = tokens_host[n - 1];
    h->has_seq = true;
    return MK_OK;
}

static mk_status check_decode(mk_handle* h, int32_t n_steps) {
    if (!h) {
        set_error("NULL handle");
        return MK_ERR_INVALID_ARG;
    }
    if (!h->has_seq) return herr(h, MK_ERR_INVALID_ARG, "no sequence: call mk_prefill first");
    if (n_steps < 1 || n_steps >= KEY_TAG_MAX - 1) return herr(h, MK_ERR_INVALID_ARG, "n_steps %d out of range", n_steps);
    if ((int64_t)h->pos + n_steps > h->d.max_seq)
        return herr(h, MK_ERR_CAPACITY, "pos %d + %d steps > max_seq %d", h->pos, n_steps, h->d.max_seq);
    return MK_OK;
}

mk_status mk_decode(mk_handle* h, int32_t n_steps, int32_t* out_ids_host) {
    mk_status st = check_decode(h, n_steps);
    if (st) return st;
    if (!out_ids_host) return herr(h, MK_ERR_INVALID_ARG, "out_ids_host is NULL");
    int32_t* ids_dev = (int32_t*)(h->wsp + h->ws.out_ids);
    if ((st = launch(h, n_steps, nullptr, ids_dev, nullptr, 0))) return st;
    CK(h, cudaMemcpyAsync(out_ids_host, ids_dev, (size_t)n_steps * 4, cudaMemcpyDeviceToHost, h->st));
    uint32_t s[5];
    if ((st = read_status(h, s))) return st;
    const int32_t steps = steps_run(h, s);
    for (int32_t i = steps; i < n_steps; ++i) out_ids_host[i] = -1;  // after an EOS stop
    h->pos += steps;
    h->pending = out_ids_host[steps - 1];
    return MK_OK;
}

mk_status mk_decode_async(mk_handle* h, int32_t n_steps, const int32_t* forced_dev, int32_t* out_ids_dev,
                          float* logits_dev) {
    mk_status st = check_decode(h, n_steps);
    if (st) return st;
    if ((st = launch(h, n_steps, forced_dev, out_ids_dev, logits_dev, 0))) return st;
    h->pos += n_steps;
    h->pending = -1;  // the last argmax stays on the device
    h->unsettled = h->eos >= 0;  // pos is provisional until mk_finish reads the steps that ran
    return MK_OK;
}

mk_status mk_finish(mk_handle* h) {
    if (!h) {
        set_error("NULL handle");
        return MK_ERR_INVALID_ARG;
    }
    uint32_t s[5];
    const bool unsettled = h->unsettled;
    mk_status st = read_status(h, s);
    if (st) return st;
    if (unsettled) {
        const int32_t launched = h->launched;
        h->pos -= launched - steps_run(h, s);
        h->unsettled = false;
    }
    return MK_OK;
}

mk_status mk_set_sampling(mk_handle* h, const mk_sampling* smp) {
    if (!h || !smp) {
        set_error("NULL argument");
        return MK_ERR_INVALID_ARG;
    }
    if (!(smp->temperature >= 0.f) || !std::isfinite(smp->temperature))
        return herr(h, MK_ERR_INVALID_ARG, "temperature %g: need a finite value >= 0", (double)smp->temperature);
    if (smp->top_k < 0 || smp->top_k > MAX_TOP_K || smp->top_k > h->d.vocab)
        return herr(h, MK_ERR_INVALID_ARG, "top_k %d: need 0 .. %d (and <= vocab)", smp->top_k, MAX_TOP_K);
    if (smp->eos_id < -1 || smp->eos_id >= h->d.vocab)
        return herr(h, MK_ERR_INVALID_ARG, "eos_id %d out of range", smp->eos_id);
    if (smp->top_k > 0 && smp->temperature > 0.f) {
        if (!h->c.token_select)
            return herr(h, MK_ERR_UNSUPPORTED, "top-k sampling needs a handle created with token_select = 1");
        if (h->lm_rows_max > LM_MAX_ROWS)
            return herr(h, MK_ERR_UNSUPPORTED, "top-k sampling: %d LM-head rows on one CTA > %d", h->lm_rows_max,
                        LM_MAX_ROWS);
    }
    if (h->unsettled) return herr(h, MK_ERR_INVALID_ARG, "call mk_finish first");
    h->temperature = smp->temperature;
    h->top_k = smp->top_k;
    h->seed = smp->seed;
    h->eos = smp->eos_id;
    return MK_OK;
}

int32_t mk_last_steps(const mk_handle* h) { return h ? h->last_steps : 0; }

mk_status mk_get_state(const mk_handle* h, int32_t* pos, int32_t* pending) {
    if (!h) {
        set_error("NULL handle");
        return MK_ERR_INVALID_ARG;
    }
    if (pos) *pos = h->pos;
    if (pending) *pending = h->pending;
    return MK_OK;
}

mk_status mk_set_state(mk_handle* h, int32_t pos, int32_t pending) {
    if (!h) {
        set_error("NULL handle");
        return MK_ERR_INVALID_ARG;
    }
    if (!h->has_seq || pos < 0 || pos > h->pos) return herr(h, MK_ERR_INVALID_ARG, "can only rewind to 0..%d", h->pos);
    if (pending < 0 || pending >= h->d.vocab) return herr(h, MK_ERR_INVALID_ARG, "pending token %d out of range", pending);
    h->pos = pos;
    h->pending = pending;
    return MK_OK;
}

mk_status mk_get_launch_info(const mk_handle* h, int32_t* ctas, int32_t* threads, int32_t* smem_bytes,
                             int32_t* rows_in_flight, int32_t* n_tasks) {
    if (!h) {
        set_error("NULL handle");
        return MK_ERR_INVALID_ARG;
    }
    if (ctas) *ctas = h->c.sms;
    if (threads) *threads = THREADS;
    if (smem_bytes) *smem_bytes = (int32_t)h->smem;
    if (rows_in_flight) *rows_in_flight = h->c.rw;
    if (n_tasks) *n_tasks = h->n_tasks;
    return MK_OK;
}

int64_t mk_launch_count(const mk_handle* h) { return h ? h->launches : 0; }

const char* mk_last_error(const mk_handle* h) { return h ? h->err.c_str() : thread_error(); }

void mk_destroy(mk_handle* h) { delete h; }

}  // extern "C"

namespace {

// Per-device state of mk_decode_static: the scratch array's address and the
// schedule currently uploaded into it.
struct StaticSlot {
    uint8_t* base = nullptr;  // set once per device context
    unsigned long long ctx_id = 0;  // the context `base` belongs to
    bool ready = false;       // tables below match the uploaded schedule
    mk_model_desc d{};
    Config c{};
    WsLayout ws{};
    int32_t n_tasks = 0, n_counters = 0;
    const void* kfn = nullptr, *kfn_sel = nullptr;
    size_t smem = 0;
    int32_t xs_floats = 0, tab_cap = 0;
    int32_t ctr_tok = 0, n_tok = 0;
    std::vector<int32_t> queue;
};
constexpr int MAX_STATIC_DEVICES = 64;
std::mutex g_static_mu;
StaticSlot g_static[MAX_STATIC_DEVICES];

// Unique id of the device's current context, through the driver entry points
// that the runtime hands out (no link against the driver library).  The
// device is made current first, which also creates its primary context.
mk_status context_id(int dev, unsigned long long* id) {
    using GetCurrent = int (*)(void**);
    using GetId = int (*)(void*, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    cudaError_t e = cudaSetDevice(dev);
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
    if (e == cudaSuccess && !get_current)
        e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", (void**)&get_current, 12000, cudaEnableDefault, &q1);
    if (e == cudaSuccess && !get_id)
        e = cudaGetDriverEntryPointByVersion("cuCtxGetId", (void**)&get_id, 12000, cudaEnableDefault, &q2);
    if (e != cudaSuccess || !get_current || !get_id) {
        get_current = nullptr;
        get_id = nullptr;
        set_error("context query: %s", e != cudaSuccess ? cudaGetErrorString(e) : "driver entry point not found");
        return MK_ERR_CUDA;
    }
    void* ctx = nullptr;
    if (get_current(&ctx) != 0 || !ctx || get_id(ctx, id) != 0) {
        set_error("no current CUDA context on device %d", dev);
        return MK_ERR_CUDA;
    }
    return MK_OK;
}

bool same_config(const Config& a, const Config& b) {
    return a.sms == b.sms && a.rw == b.rw && a.C == b.C && a.watchdog_ns == b.watchdog_ns &&
           a.token_select == b.token_select;
}

// Lower, validate and upload the schedule for (desc, c) into the slot's scratch.
mk_status static_setup(StaticSlot& s, const mk_model_desc* desc, const Config& c, int n_sms, int smem_optin,
                       cudaStream_t stream) {
    s.ready = false;
    Lowering lw;
    mk_status st = lower(desc, c, &lw);
    if (st) return st;
    const WsLayout ws = ws_layout(desc, c, (int64_t)lw.tasks.size(), lw.n_counters);
    if ((uint64_t)ws.total > (uint64_t)MK_STATIC_SCRATCH_BYTES) {
        set_error("this model needs %lld bytes of scratch; the static scratch holds %u (MK_STATIC_SCRATCH_BYTES)",
                  (long long)ws.total, (unsigned)MK_STATIC_SCRATCH_BYTES);
        return MK_ERR_CAPACITY;
    }
    {
        mk_ir* ir = to_ir(lw, c.sms);
        std::string why;
        st = validate_ir(ir, &why);
        mk_free_ir(ir);
        if (st) {
            set_error("schedule rejected before launch: %s", why.c_str());
            return MK_ERR_SCHEDULE_INVALID;
        }
    }
    std::vector<TaskRec> recs;
    std::vector<int32_t> queue, qoff;
    int32_t tab_cap = 0;
    if ((st = device_tables(lw, c.sms, &recs, &queue, &qoff, &tab_cap))) return st;
    const int xs_floats = std::max(desc->d_model, desc->n_q_heads * desc->head_dim);
    const size_t smem = vm_shared_bytes(desc->wdtype, xs_floats, tab_cap);
    const void* kfn = vm_kernel_for(desc->wdtype, desc->base_dtype, desc->head_dim, false);
    const void* kfn_sel = vm_kernel_for(desc->wdtype, desc->base_dtype, desc->head_dim, true);
    if (!kfn || !kfn_sel) {
        set_error("no kernel for wdtype %d / base %d", desc->wdtype, desc->base_dtype);
        return MK_ERR_UNSUPPORTED;
    }
    if (smem > (size_t)smem_optin) {
        set_error("shared memory need %zu > %d", smem, smem_optin);
        return MK_ERR_UNSUPPORTED;
    }
    // the kernel-wide limit, as in mk_create (shared with every handle)
    cudaError_t e = raise_smem_limit(kfn, smem_optin);
    if (e == cudaSuccess) e = raise_smem_limit(kfn_sel, smem_optin);
    int per_sm = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, THREADS, smem);
    if (e != cudaSuccess) {
        set_error("kernel set-up: %s", cudaGetErrorString(e));
        return MK_ERR_CUDA;
    }
    if (per_sm < 1 || (int64_t)per_sm * n_sms < c.sms) {
        set_error("%d CTAs cannot be co-resident (%d per SM)", c.sms, per_sm);
        return MK_ERR_UNSUPPORTED;
    }
    std::vector<float> inv(desc->head_dim / 2);
    for (int i = 0; i < desc->head_dim / 2; ++i)
        inv[i] = (float)std::pow((double)desc->rope_theta, -2.0 * i / (double)desc->head_dim);
    e = cudaMemcpyAsync(s.base + ws.recs, recs.data(), recs.size() * sizeof(TaskRec), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(s.base + ws.queue_off, qoff.data(), qoff.size() * 4, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(s.base + ws.inv_freq, inv.data(), inv.size() * 4, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);  // the host vectors die on return
    if (e != cudaSuccess) {
        set_error("uploading the schedule: %s", cudaGetErrorString(e));
        return MK_ERR_CUDA;
    }
    s.d = *desc;
    s.c = c;
    s.ws = ws;
    s.n_tasks = (int32_t)lw.tasks.size();
    s.n_counters = lw.n_counters;
    s.kfn = kfn;
    s.kfn_sel = kfn_sel;
    s.smem = smem;
    s.xs_floats = xs_floats;
    s.tab_cap = tab_cap;
    s.queue = std::move(queue);
    s.ctr_tok = lw.ctr_tok;
    s.n_tok = lw.n_tok;
    s.ready = true;
    return MK_OK;
}

}  // namespace

extern "C" {

mk_status mk_decode_static(const mk_model_desc* desc, const mk_schedule_config* cfg, const void* weights_dev,
                           size_t weights_bytes, void* kv_dev, size_t kv_bytes, int32_t pos, int32_t token,
                           int32_t n_steps, int32_t* out_ids_host, float* logits_dev, mk_stream_t stream) {
    mk_status st = check_desc(desc);
    if (st) return st;
    if (!weights_dev || !kv_dev || !out_ids_host) {
        set_error("NULL argument");
        return MK_ERR_INVALID_ARG;
    }
    if (((uintptr_t)weights_dev & 255) || ((uintptr_t)kv_dev & 15)) {
        set_error("misaligned buffer: weights need 256-byte, the KV cache 16-byte alignment");
        return MK_ERR_INVALID_ARG;
    }
    if (token < 0 || token >= desc->vocab) {
        set_error("token %d out of range", token);
        return MK_ERR_INVALID_ARG;
    }
    if (pos < 0 || n_steps < 1 || n_steps >= KEY_TAG_MAX - 1) {
        set_error("pos %d / n_steps %d out of range", pos, n_steps);
        return MK_ERR_INVALID_ARG;
    }
    std::lock_guard<std::mutex> lock(g_static_mu);
    int dev = 0, n_sms = 0, smem_optin = 0, coop = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (e != cudaSuccess) {
        set_error("CUDA device query failed: %s", cudaGetErrorString(e));
        return MK_ERR_CUDA;
    }
    if (!coop || dev >= MAX_STATIC_DEVICES) {
        set_error("device %d: no cooperative launch or index above %d", dev, MAX_STATIC_DEVICES - 1);
        return MK_ERR_UNSUPPORTED;
    }
    StaticSlot& s = g_static[dev];
    // A reset of the device's primary context (cudaDeviceReset) re-creates the
    // array, zeroed, at a possibly new address: a context with a new id gets
    // the symbol lookup and the schedule upload again.
    unsigned long long ctx = 0;
    if ((st = context_id(dev, &ctx))) return st;
    if (!s.base || s.ctx_id != ctx) {
        void* p = nullptr;
        e = static_scratch_address(&p);
        if (e != cudaSuccess || !p) {
            set_error("cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
            return MK_ERR_CUDA;
        }
        s.base = (uint8_t*)p;
        s.ctx_id = ctx;
        s.ready = false;
    }
    Config c;
    if ((st = resolve_config(desc, cfg, n_sms, &c))) return st;
    c.pf_chunk = 0;  // this entry point decodes only: no prefill buffers in the scratch
    const cudaStream_t cs = (cudaStream_t)stream;
    if (!s.ready || std::memcmp(&s.d, desc, sizeof s.d) != 0 || !same_config(s.c, c)) {
        if ((st = static_setup(s, desc, c, n_sms, smem_optin, cs))) return st;
    }
    size_t need_w = 0, need_kv = 0;
    mk_packed_size(desc, &need_w);
    mk_kv_cache_size(desc, &need_kv);
    if (weights_bytes < need_w || kv_bytes < need_kv) {
        set_error("buffer too small: weights %zu/%zu, kv %zu/%zu", weights_bytes, need_w, kv_bytes, need_kv);
        return MK_ERR_CAPACITY;
    }
    if ((int64_t)pos + n_steps > desc->max_seq) {
        set_error("pos %d + %d steps > max_seq %d", pos, n_steps, desc->max_seq);
        return MK_ERR_CAPACITY;
    }
    // A handle on the stack over the static scratch: nothing is allocated.
    mk_handle h;
    h.d = *desc;
    h.c = c;
    h.ws = s.ws;
    h.bl = blob_layout(desc);
    h.n_tasks = s.n_tasks;
    h.n_counters = s.n_counters;
    h.w = (const uint8_t*)weights_dev;
    h.kv = (uint16_t*)kv_dev;
    h.wsp = s.base;
    h.st = cs;
    h.device = dev;
    h.kfn = s.kfn;
    h.kfn_sel = s.kfn_sel;
    h.smem = s.smem;
    h.xs_floats = s.xs_floats;
    h.tab_cap = s.tab_cap;
    h.queue = s.queue.data();
    h.ctr_tok = s.ctr_tok;
    h.n_tok = s.n_tok;
    h.pos = pos;
    h.pending = token;
    h.has_seq = true;
    // status words, sync counters and the argmax key must start at zero
    if ((st = reset_sync_state(&h))) return st;
    int32_t* ids_dev = (int32_t*)(s.base + s.ws.out_ids);
    if ((st = launch(&h, n_steps, nullptr, ids_dev, logits_dev, 0))) return st;
    e = cudaMemcpyAsync(out_ids_host, ids_dev, (size_t)n_steps * 4, cudaMemcpyDeviceToHost, cs);
    if (e != cudaSuccess) {
        set_error("reading the ids: %s", cudaGetErrorString(e));
        return MK_ERR_CUDA;
    }
    return read_status(&h);
}

mk_status mk_debug_dequant(const mk_model_desc* desc, const void* weights_dev, int32_t tensor, int32_t layer,
                           float* out_dev, mk_stream_t stream) {
    size_t off = 0, stride = 0;
    int32_t first = 0, step = 1, rows = 0;
    mk_status st = mk_tensor_layout(desc, tensor, layer, &off, &stride, &first, &step, &rows);
    if (st) return st;
    const bool cols = stride == 0 && tensor == MK_T_WDOWN &&
                      (desc->wdtype == MK_W_INT8_ROW || desc->wdtype == MK_W_INT4_G128 ||
                       desc->wdtype == MK_W_FP8_E4M3);  // column blocks
    if (!weights_dev || !out_dev || (stride == 0 && !cols)) {
        set_error("NULL pointer or not a quantisable GEMV tensor");
        return MK_ERR_INVALID_ARG;
    }
    int K = 0;
    switch (tensor) {
        case MK_T_WO: K = desc->n_q_heads * desc->head_dim; break;
        case MK_T_WDOWN: K = desc->d_ffn; break;
        default: K = desc->d_model; break;
    }
    cudaError_t e = launch_dequant(desc->wdtype, (const uint8_t*)weights_dev + off, (int64_t)stride, first, step,
                                   rows, K, out_dev, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) {
        set_error("dequant kernel: %s", cudaGetErrorString(e));
        return MK_ERR_CUDA;
    }
    return MK_OK;
}

mk_status mk_debug_set_trace(mk_handle* h, void* trace_dev, int32_t records_per_cta) {
    if (!h) {
        set_error("NULL handle");
        return MK_ERR_INVALID_ARG;
    }
    if (trace_dev && records_per_cta < 1) return herr(h, MK_ERR_INVALID_ARG, "records_per_cta must be >= 1");
    h->trace = (unsigned long long*)trace_dev;
    h->trace_cap = trace_dev ? records_per_cta : 0;
    return MK_OK;
}

mk_status mk_debug_watchdog(int32_t timeout_us, void* counter_dev, mk_stream_t stream) {
    if (!counter_dev || timeout_us < 1) {
        set_error("bad arguments");
        return MK_ERR_INVALID_ARG;
    }
    uint32_t* base = (uint32_t*)counter_dev;
    cudaError_t e = launch_watchdog(base, base + 16, (int64_t)timeout_us * 1000, (cudaStream_t)stream);
    uint32_t s = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&s, base + 16, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) {
        set_error("watchdog kernel: %s", cudaGetErrorString(e));
        return MK_ERR_CUDA;
    }
    if (s == DEV_TIMEOUT) {
        set_error("wait gave up after %d us", timeout_us);
        return MK_ERR_TIMEOUT;
    }
    return MK_OK;
}

}  // extern "C"
