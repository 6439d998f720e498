// rpa_host.cu -- host runtime behind the C ABI of include/rpa.h.
//
// Validates configurations and arguments, owns the workspace (plan buffers
// and split-KV partials sized for the worst case of a configuration), and
// enqueues the planner, the attention kernels and the combine kernel on the
// caller's stream.  No call synchronises except rpa_get_status,
// rpa_read_plan and rpa_destroy.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cmath>
#include <new>

#include "rpa_internal.cuh"

using namespace rpa;

struct RpaHandle {
    RpaCfg cfg;
    int device;
    KernelSet ks;         // kernels, tiles, occupancy and capacities of cfg
    MapCache maps;        // tensor maps of the last call
    void* ws;             // the workspace (one allocation, worst case of cfg)
    size_t ws_bytes;
    Workspace w;          // its parts
    // staging for rpa_forward_host
    uint8_t* stage;
    size_t stage_bytes;
    // per-kernel timing (rpa_profile_begin / rpa_profile_read)
    cudaEvent_t* prof_ev;   // [prof_cap][kProfEvents]
    int prof_cap;
    int prof_used;
    // decode and prefill may run concurrently (tensor-memory prefill of 2-byte K/V): on the caller's
    // stream, or with the profile events on, decode on a second stream forked after the planner
    int can_concurrent;   // and the side stream and events exist
    int serial;           // RPA_OPT_SERIAL: run the two one after the other on the caller's stream
    int concurrent;       // the mode of the last call
    cudaStream_t side;
    cudaEvent_t ev_plan, ev_dec;
    int debug_stall;                // RPA_OPT_TEST_STALL_PRODUCER
    unsigned long long timeout_ns;  // RPA_OPT_WAIT_TIMEOUT_MS
    int force_pf_sms, force_dec_sms;  // RPA_OPT_PREFILL_SMS / RPA_OPT_DECODE_SMS
    int plan_early;                   // RPA_OPT_PLAN_EARLY
    int epoch;                        // calls so far (the planner publishes each call's number)
};

namespace {

bool is_finite(float x) { return std::isfinite(x); }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t q_elt_bytes(int32_t dt) { return dt == RPA_DT_F32 ? 4 : 2; }

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

void prof_free(RpaHandle* h) {
    if (!h->prof_ev) return;
    for (int i = 0; i < h->prof_cap * kProfEvents; ++i)
        if (h->prof_ev[i]) cudaEventDestroy(h->prof_ev[i]);
    free(h->prof_ev);
    h->prof_ev = nullptr;
    h->prof_cap = h->prof_used = 0;
}

}  // namespace

extern "C" {

int rpa_version(void) { return 200; }

const char* rpa_strerror(int code) {
    switch (code) {
        case RPA_OK: return "ok";
        case RPA_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer or bad configuration value)";
        case RPA_ERR_UNSUPPORTED: return "unsupported configuration (dtype, head_dim, or head grouping)";
        case RPA_ERR_CUDA: return "CUDA runtime error";
        case RPA_ERR_BAD_PAGE_INDEX: return "page index outside [0, total_num_pages)";
        case RPA_ERR_BAD_LENGTHS: return "bad lengths (kv_len > capacity, q_len > kv_len, or cu_q_lens not monotone / past num_q_tokens)";
        case RPA_ERR_TIMEOUT: return "a bounded device wait timed out";
        case RPA_ERR_NO_ALLOC_LIMIT: return "workspace exceeds the fixed 32 MiB scratch array of rpa_forward_noalloc";
        default: return "unknown status code";
    }
}

void rpa_cfg_init(RpaCfg* c) {
    if (!c) return;
    RpaCfg z;
    memset(&z, 0, sizeof z);
    z.num_q_tokens = c->num_q_tokens;
    z.num_q_heads = c->num_q_heads;
    z.num_kv_heads = c->num_kv_heads;
    z.head_dim = c->head_dim;
    z.total_num_pages = c->total_num_pages;
    z.page_size = c->page_size;
    z.max_num_seqs = c->max_num_seqs;
    z.pages_per_seq = c->pages_per_seq;
    z.q_dtype = RPA_DT_BF16;
    z.kv_dtype = RPA_DT_BF16;
    z.sm_scale = c->head_dim > 0 ? (float)(1.0 / sqrt((double)c->head_dim)) : 1.0f;
    z.mask_value = -2.38197633e38f;
    z.soft_cap = 0.f;
    z.k_scale = 1.f;
    z.v_scale = 1.f;
    z.is_causal = 1;
    *c = z;
}

int rpa_validate_cfg(const RpaCfg* c) {
    if (!c) return RPA_ERR_INVALID_ARG;
    const int64_t lim = (int64_t)1 << 31;
    if (c->num_q_tokens < 0 || c->num_q_tokens >= lim) return RPA_ERR_INVALID_ARG;
    if (c->num_q_heads < 1 || c->num_kv_heads < 1 || c->num_q_heads >= 65536) return RPA_ERR_INVALID_ARG;
    if (c->total_num_pages < 1 || c->total_num_pages >= lim) return RPA_ERR_INVALID_ARG;
    if (c->page_size < 1 || c->pages_per_seq < 1 || c->max_num_seqs < 1) return RPA_ERR_INVALID_ARG;
    if (c->max_num_seqs >= ((int64_t)1 << 28)) return RPA_ERR_INVALID_ARG;
    if (c->pages_per_seq * c->page_size >= lim || c->pages_per_seq >= lim) return RPA_ERR_INVALID_ARG;
    if (!is_finite(c->sm_scale)) return RPA_ERR_INVALID_ARG;
    if (c->has_soft_cap && !(is_finite(c->soft_cap) && c->soft_cap > 0.f)) return RPA_ERR_INVALID_ARG;
    if (c->has_k_scale && !is_finite(c->k_scale)) return RPA_ERR_INVALID_ARG;
    if (c->has_v_scale && !is_finite(c->v_scale)) return RPA_ERR_INVALID_ARG;
    if (c->has_sliding_window && c->sliding_window < 1) return RPA_ERR_INVALID_ARG;
    if (c->has_sinks && (!c->sinks || !aligned(c->sinks, 4))) return RPA_ERR_INVALID_ARG;
    if (c->reserved != 0) return RPA_ERR_INVALID_ARG;
    if (c->num_q_heads % c->num_kv_heads) return RPA_ERR_UNSUPPORTED;
    const int64_t G = c->num_q_heads / c->num_kv_heads;
    if (c->kv_layout == RPA_KV_LATENT) {
        // latent rows of 576 with 512-wide values; 2-byte rows; page runs of >= 8 slots (so that
        // every run lands on a 1 KB boundary); blocks of <= 16 query heads
        if (c->head_dim != kMlaDqk || c->v_head_dim != kMlaDv) return RPA_ERR_UNSUPPORTED;
        if (c->kv_dtype != RPA_DT_BF16 && c->kv_dtype != RPA_DT_F16) return RPA_ERR_UNSUPPORTED;
        if (c->page_size % 8) return RPA_ERR_UNSUPPORTED;
        if (G > kMlaRows && G % kMlaRows) return RPA_ERR_UNSUPPORTED;
    } else {
        if (c->kv_layout != RPA_KV_SPLIT) return RPA_ERR_UNSUPPORTED;
        if (c->v_head_dim != 0 && c->v_head_dim != c->head_dim) return RPA_ERR_UNSUPPORTED;
        if (G > kMaxGroup) return RPA_ERR_UNSUPPORTED;
        if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return RPA_ERR_UNSUPPORTED;
        if (c->page_size % 4) return RPA_ERR_UNSUPPORTED;  // page runs of the gather are >= 4 slots
    }
    if (c->q_dtype != RPA_DT_BF16 && c->q_dtype != RPA_DT_F16 && c->q_dtype != RPA_DT_F32) return RPA_ERR_UNSUPPORTED;
    if (c->kv_dtype != RPA_DT_BF16 && c->kv_dtype != RPA_DT_F16 && c->kv_dtype != RPA_DT_FP8_E4M3 &&
        c->kv_dtype != RPA_DT_FP8_E5M2 && c->kv_dtype != RPA_DT_INT8)
        return RPA_ERR_UNSUPPORTED;
    // masked keys get weight exactly 0 only if the additive mask value is huge and negative
    if (!(c->mask_value <= -1e30f)) return RPA_ERR_UNSUPPORTED;
    return RPA_OK;
}

int rpa_create(const RpaCfg* cfg, RpaHandle** out) {
    if (!out) return RPA_ERR_INVALID_ARG;
    *out = nullptr;
    int v = rpa_validate_cfg(cfg);
    if (v != RPA_OK) return v;
    RpaHandle* h = new (std::nothrow) RpaHandle;
    if (!h) return RPA_ERR_CUDA;
    memset(h, 0, sizeof *h);
    h->cfg = *cfg;
    const RpaCfg& c = h->cfg;
    h->timeout_ns = 1000000000ull;  // bound of every device wait (RPA_OPT_WAIT_TIMEOUT_MS)
    int sms = 0;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return RPA_ERR_CUDA;
    }
    kernels_choose(c, sms, &h->ks);
    // the SM-split model is calibrated for the tensor-memory prefill of 2-byte K/V only
    h->can_concurrent = h->ks.tc;
    if (kernels_prepare(c, &h->ks) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return RPA_ERR_CUDA;
    }
    h->ws_bytes = workspace_bytes(c, h->ks);
    if (cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return RPA_ERR_CUDA;
    }
    if (h->can_concurrent && (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
                              cudaEventCreateWithFlags(&h->ev_plan, cudaEventDisableTiming) != cudaSuccess ||
                              cudaEventCreateWithFlags(&h->ev_dec, cudaEventDisableTiming) != cudaSuccess)) {
        cudaGetLastError();
        if (h->ev_plan) cudaEventDestroy(h->ev_plan);
        if (h->side) cudaStreamDestroy(h->side);
        cudaFree(h->ws);
        delete h;
        return RPA_ERR_CUDA;
    }
    h->w = workspace_carve(c, h->ks, h->ws);
    if (cudaMemset(h->w.ctrl, 0, kCtrlWords * sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        if (h->can_concurrent) {
            cudaEventDestroy(h->ev_dec);
            cudaEventDestroy(h->ev_plan);
            cudaStreamDestroy(h->side);
        }
        cudaFree(h->ws);
        delete h;
        return RPA_ERR_CUDA;
    }
    *out = h;
    return RPA_OK;
}

int rpa_forward(RpaHandle* h, const void* q, const void* kv_pages, const int32_t* kv_lens,
                const int32_t* page_indices, const int32_t* cu_q_lens, int32_t num_seqs, void* o,
                void* stream) {
    if (!h) return RPA_ERR_INVALID_ARG;
    const RpaCfg& c = h->cfg;
    if (num_seqs < 0 || num_seqs > c.max_num_seqs) return RPA_ERR_INVALID_ARG;
    if (!kv_pages || !kv_lens || !page_indices || !cu_q_lens) return RPA_ERR_INVALID_ARG;
    if (c.num_q_tokens > 0 && (!q || !o)) return RPA_ERR_INVALID_ARG;
    if ((q && !aligned(q, 16)) || (o && !aligned(o, 16)) || !aligned(kv_pages, 16) ||
        !aligned(kv_lens, 4) || !aligned(page_indices, 4) || !aligned(cu_q_lens, 4))
        return RPA_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return RPA_ERR_CUDA;
    EnqueueOpts eo;
    memset(&eo, 0, sizeof eo);
    eo.st = static_cast<cudaStream_t>(stream);
    eo.conc = h->can_concurrent && !h->serial;
    eo.side = h->side;
    eo.ev_plan = h->ev_plan;
    eo.ev_dec = h->ev_dec;
    const bool prof = h->prof_ev && h->prof_used < h->prof_cap;
    for (int k = 0; k < kProfEvents; ++k) eo.ev[k] = prof ? h->prof_ev[h->prof_used * kProfEvents + k] : nullptr;
    eo.debug_stall = h->debug_stall;
    eo.timeout_ns = h->timeout_ns;
    eo.force_pf_sms = h->force_pf_sms;
    eo.force_dec_sms = h->force_dec_sms;
    eo.plan_early = h->plan_early;
    eo.epoch = h->epoch = (h->epoch + 1) & 0x7FFFFFFF;
    h->concurrent = eo.conc;
    const int r = enqueue_forward(c, h->ks, h->w, &h->maps, q, kv_pages, kv_lens, page_indices, cu_q_lens, num_seqs,
                                  o, eo);
    if (r == RPA_OK && prof) ++h->prof_used;
    return r;
}

int rpa_profile_begin(RpaHandle* h, int32_t max_calls) {
    if (!h || max_calls < 0) return RPA_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return RPA_ERR_CUDA;
    prof_free(h);
    if (max_calls == 0) return RPA_OK;
    h->prof_ev = static_cast<cudaEvent_t*>(calloc((size_t)max_calls * kProfEvents, sizeof(cudaEvent_t)));
    if (!h->prof_ev) return RPA_ERR_INVALID_ARG;
    h->prof_cap = max_calls;
    for (int i = 0; i < max_calls * kProfEvents; ++i) {
        if (cudaEventCreate(&h->prof_ev[i]) != cudaSuccess) {
            cudaGetLastError();
            prof_free(h);
            return RPA_ERR_CUDA;
        }
    }
    return RPA_OK;
}

int rpa_profile_read(RpaHandle* h, float* ms, int32_t max_calls, int32_t* n_calls) {
    if (!h || !ms || !n_calls) return RPA_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return RPA_ERR_CUDA;
    const int n = h->prof_used < max_calls ? h->prof_used : max_calls;
    // kernel k runs between events from[k] and to[k] of its call, both on the kernel's own stream
    static const int from[4] = {kEvStart, kEvDecStart, kEvPfStart, kEvCombStart};
    static const int to[4] = {kEvPlanEnd, kEvDecEnd, kEvPfEnd, kEvCombEnd};
    for (int c = 0; c < n; ++c) {
        cudaEvent_t* e = h->prof_ev + (size_t)c * kProfEvents;
        if (cudaEventSynchronize(e[kEvCombEnd]) != cudaSuccess || cudaEventSynchronize(e[kEvPfEnd]) != cudaSuccess)
            return RPA_ERR_CUDA;
        for (int k = 0; k < 4; ++k) {
            float t = 0.f;
            if (cudaEventElapsedTime(&t, e[from[k]], e[to[k]]) != cudaSuccess) return RPA_ERR_CUDA;
            ms[c * 4 + k] = t;
        }
    }
    *n_calls = n;
    return RPA_OK;
}

int rpa_set_option(RpaHandle* h, int32_t option, int64_t value) {
    if (!h) return RPA_ERR_INVALID_ARG;
    switch (option) {
        case RPA_OPT_WAIT_TIMEOUT_MS:
            if (value < 1 || value > 3600000) return RPA_ERR_INVALID_ARG;
            h->timeout_ns = (unsigned long long)value * 1000000ull;
            return RPA_OK;
        case RPA_OPT_SERIAL:
            if (value != 0 && value != 1) return RPA_ERR_INVALID_ARG;
            h->serial = (int)value;
            return RPA_OK;
        case RPA_OPT_PREFILL_SMS:
        case RPA_OPT_DECODE_SMS:
            if (value < 0 || value > h->ks.sms) return RPA_ERR_INVALID_ARG;
            (option == RPA_OPT_PREFILL_SMS ? h->force_pf_sms : h->force_dec_sms) = (int)value;
            return RPA_OK;
        case RPA_OPT_PLAN_EARLY:
            if (value != 0 && value != 1) return RPA_ERR_INVALID_ARG;
            h->plan_early = (int)value;
            return RPA_OK;
        case RPA_OPT_TEST_STALL_PRODUCER:
            if (value != 0 && value != 1) return RPA_ERR_INVALID_ARG;
            h->debug_stall = (int)value;
            return RPA_OK;
        default:
            return RPA_ERR_INVALID_ARG;
    }
}

int rpa_forward_host(RpaHandle* h, const void* q_host, const void* kv_pages, const int32_t* kv_lens_host,
                     const int32_t* page_indices_host, const int32_t* cu_q_lens_host, int32_t num_seqs,
                     void* o_host, void* stream) {
    if (!h) return RPA_ERR_INVALID_ARG;
    const RpaCfg& c = h->cfg;
    if (!kv_lens_host || !page_indices_host || !cu_q_lens_host || !kv_pages) return RPA_ERR_INVALID_ARG;
    if (c.num_q_tokens > 0 && (!q_host || !o_host)) return RPA_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_seqs > c.max_num_seqs) return RPA_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return RPA_ERR_CUDA;
    const size_t qb = (size_t)c.num_q_tokens * c.num_q_heads * c.head_dim * q_elt_bytes(c.q_dtype);
    const size_t ob = (size_t)c.num_q_tokens * c.num_q_heads * h->ks.Dv * q_elt_bytes(c.q_dtype);
    const size_t kb = (size_t)c.max_num_seqs * sizeof(int32_t);
    const size_t pb = (size_t)c.max_num_seqs * c.pages_per_seq * sizeof(int32_t);
    const size_t cb = (size_t)(c.max_num_seqs + 1) * sizeof(int32_t);
    const size_t o_q = 0, o_o = align256(qb), o_k = o_o + align256(ob), o_p = o_k + align256(kb),
                 o_c = o_p + align256(pb), total = o_c + align256(cb);
    if (!h->stage) {
        if (cudaMalloc(&h->stage, total) != cudaSuccess) {
            cudaGetLastError();
            return RPA_ERR_CUDA;
        }
        h->stage_bytes = total;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* s = h->stage;
    if ((qb && cudaMemcpyAsync(s + o_q, q_host, qb, cudaMemcpyHostToDevice, st) != cudaSuccess) ||
        cudaMemcpyAsync(s + o_k, kv_lens_host, kb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(s + o_p, page_indices_host, pb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(s + o_c, cu_q_lens_host, cb, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return RPA_ERR_CUDA;
    int r = rpa_forward(h, qb ? s + o_q : nullptr, kv_pages, reinterpret_cast<const int32_t*>(s + o_k),
                        reinterpret_cast<const int32_t*>(s + o_p), reinterpret_cast<const int32_t*>(s + o_c),
                        num_seqs, qb ? s + o_o : nullptr, stream);
    if (r != RPA_OK) return r;
    if (ob && cudaMemcpyAsync(o_host, s + o_o, ob, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return RPA_ERR_CUDA;
    return RPA_OK;
}

int rpa_get_status(RpaHandle* h, void* stream) {
    if (!h) return RPA_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return RPA_ERR_CUDA;
    int v = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&v, h->w.ctrl + kStatus, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return RPA_ERR_CUDA;
    return v;
}

int rpa_read_plan(RpaHandle* h, int32_t* info, int32_t* items, int64_t max_items, void* stream) {
    if (!h || !info) return RPA_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return RPA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int ctrl[kCtrlWords];
    if (cudaMemcpyAsync(ctrl, h->w.ctrl, sizeof ctrl, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return RPA_ERR_CUDA;
    for (int i = 0; i < 16; ++i) info[i] = 0;
    info[0] = ctrl[kStatus];
    info[1] = ctrl[kNumDecItems];
    info[2] = ctrl[kNumPfItems];
    info[3] = ctrl[kNumComb];
    info[4] = ctrl[kDecChunk];
    info[5] = h->ks.dec_rows;
    info[6] = h->ks.pf_tokens;
    info[7] = ctrl[kNumPart];
    info[8] = ctrl[kNumUnits];
    info[9] = ctrl[kSorted];
    info[10] = ctrl[kDecCtas];
    info[11] = ctrl[kPfCtas];
    info[12] = h->ks.sms;
    info[13] = h->ks.dec_bps;
    info[14] = h->ks.pf_bps;
    info[15] = h->concurrent | ((h->ks.tc8 | h->ks.mla) << 1);
    if (items && max_items > 0) {
        // the kernels' unit lists, each unit expanded to its items (one per kv head, as item_at)
        const int64_t H = h->ks.Hp;
        const int64_t nd = ctrl[kNumDecItems] < max_items ? ctrl[kNumDecItems] : max_items;
        const int64_t np = ctrl[kNumPfItems] < max_items - nd ? ctrl[kNumPfItems] : max_items - nd;
        const int64_t ud = (nd + H - 1) / H, up = (np + H - 1) / H;
        Unit* u = static_cast<Unit*>(malloc((size_t)(ud + up + 1) * sizeof(Unit)));
        if (!u) return RPA_ERR_INVALID_ARG;
        if ((ud && cudaMemcpy(u, h->w.dec_units, ud * sizeof(Unit), cudaMemcpyDeviceToHost) != cudaSuccess) ||
            (up && cudaMemcpy(u + ud, h->w.pf_units, up * sizeof(Unit), cudaMemcpyDeviceToHost) != cudaSuccess)) {
            free(u);
            return RPA_ERR_CUDA;
        }
        for (int64_t i = 0; i < nd + np; ++i) {
            const int64_t it = i < nd ? i : i - nd;
            const Unit& x = u[(i < nd ? 0 : ud) + it / H];
            const int hd = (int)(it % H);
            int32_t* d = items + i * 8;
            d[0] = x.seq;
            d[1] = hd;
            d[2] = x.tok0;
            d[3] = x.ntok;
            d[4] = x.kv_begin;
            d[5] = x.kv_end;
            d[6] = x.part >= 0 ? x.part + hd * x.pieces + x.piece : -1;
            d[7] = x.piece;
        }
        free(u);
    }
    return RPA_OK;
}

void rpa_destroy(RpaHandle* h) {
    if (!h) return;
    DeviceGuard g(h->device);
    prof_free(h);
    if (h->ev_dec) cudaEventDestroy(h->ev_dec);
    if (h->ev_plan) cudaEventDestroy(h->ev_plan);
    if (h->side) cudaStreamDestroy(h->side);
    if (h->stage) cudaFree(h->stage);
    if (h->ws) cudaFree(h->ws);
    delete h;
}

}  // extern "C"
