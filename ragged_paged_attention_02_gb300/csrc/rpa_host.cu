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
    CUtensorMap kvmap;   // decode gather: one copy per page run (K and V of a head)
    CUtensorMap kvmap_pf;  // tensor-memory prefill gather: one copy per (page run, K/V, column block)
    CUtensorMap qmap;
    CUtensorMap qmap_pf;  // Q tiles of the tensor-memory prefill kernel
    const void* kvmap_ptr;
    const void* qmap_ptr;
    int tc;               // prefill on tcgen05 (bf16 K/V, head_dim 64 or 128)
    int tc8;              // prefill on tcgen05 with fp8 K/V converted in shared memory (head_dim 128 or 256)
    int pf_tokens;        // query tokens of a prefill item (2 x 128 rows for tc, 128 rows for tc8, else 64)
    RpaCfg cfg;
    int device;
    int sms;
    int G, D, fp8;
    int dec_bps, pf_bps;
    int max_dec_units, max_pf_units, max_units, max_part, max_comb;
    float qk_log2, cap_exp, cap_log2, v_scale;
    int window;
    int BR, br_shift, Tt;
    int dec_rows;         // query rows of a decode tile: 8 (bf16, G <= 8) or 16
    int debug_stall;      // RPA_OPT_TEST_STALL_PRODUCER
    unsigned long long timeout_ns;  // RPA_OPT_WAIT_TIMEOUT_MS
    void* ws;
    size_t ws_bytes;
    int* ctrl;
    int* seq_scratch;
    int* units;
    Item* dec_items;
    Item* pf_items;
    Comb* comb;
    float* part_o;
    float* part_ml;
    // staging for rpa_forward_host
    uint8_t* stage;
    size_t stage_bytes;
    // per-kernel timing (rpa_profile_begin / rpa_profile_read)
    cudaEvent_t* prof_ev;   // [prof_cap][kProfEvents]
    int prof_cap;
    int prof_used;
    // decode and prefill may run concurrently: decode on a second stream forked after the planner
    int can_concurrent;   // the side stream and events exist (tensor-memory bf16 prefill)
    int serial;           // RPA_OPT_SERIAL: run the two one after the other on the caller's stream
    int concurrent;       // the mode of the last call
    cudaStream_t side;
    cudaEvent_t ev_plan, ev_dec;
    int force_pf_sms, force_dec_sms;  // RPA_OPT_PREFILL_SMS / RPA_OPT_DECODE_SMS
};

namespace {

const double kLog2e = 1.4426950408889634;

bool is_finite(float x) { return std::isfinite(x); }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

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

// Profile events of one call: each kernel is timed from an event recorded on its own stream
// just before its launch (after any cross-stream wait) to one recorded just after it.
enum ProfEvent : int {
    kEvStart = 0, kEvPlanEnd, kEvDecStart, kEvDecEnd, kEvPfStart, kEvPfEnd, kEvCombStart, kEvCombEnd,
    kProfEvents
};

// event k of the call being profiled, or nullptr when not profiling
cudaEvent_t prof_event(RpaHandle* h, int k) {
    if (!h->prof_ev || h->prof_used >= h->prof_cap) return nullptr;
    return h->prof_ev[h->prof_used * kProfEvents + k];
}

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
    if (c->kv_layout != RPA_KV_SPLIT || c->v_head_dim != 0) return RPA_ERR_UNSUPPORTED;
    if (c->num_q_heads % c->num_kv_heads) return RPA_ERR_UNSUPPORTED;
    if (c->num_q_heads / c->num_kv_heads > kPfRows) return RPA_ERR_UNSUPPORTED;
    if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return RPA_ERR_UNSUPPORTED;
    if (c->page_size % 4) return RPA_ERR_UNSUPPORTED;  // page runs of the gather are >= 4 slots
    if (c->q_dtype != RPA_DT_BF16) return RPA_ERR_UNSUPPORTED;
    if (c->kv_dtype != RPA_DT_BF16 && c->kv_dtype != RPA_DT_FP8_E4M3) return RPA_ERR_UNSUPPORTED;
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
    h->G = (int)(c.num_q_heads / c.num_kv_heads);
    h->D = (int)c.head_dim;
    h->fp8 = c.kv_dtype == RPA_DT_FP8_E4M3;
    const double ks = c.has_k_scale ? c.k_scale : 1.0;
    h->qk_log2 = (float)(c.sm_scale * ks * kLog2e);
    h->cap_exp = c.has_soft_cap ? (float)(2.0 * c.sm_scale * ks / c.soft_cap * kLog2e) : 0.f;
    h->cap_log2 = c.has_soft_cap ? (float)(c.soft_cap * kLog2e) : 0.f;
    h->v_scale = c.has_v_scale ? c.v_scale : 1.f;
    h->window = c.has_sliding_window ? (int)(c.sliding_window > 0x7fffffff ? 0x7fffffff : c.sliding_window) : 0;
    h->BR = 64;
    while ((int)(c.page_size % h->BR)) h->BR >>= 1;
    h->br_shift = 0;
    while ((1 << h->br_shift) < h->BR) ++h->br_shift;
    // 8-row decode tiles (keys on the MMA's M side) whenever a group fits: bf16 K/V, G <= 8
    h->dec_rows = (!h->fp8 && h->G <= 8) ? 8 : kDecRows;
    h->Tt = h->G <= h->dec_rows ? h->dec_rows / h->G : 1;
    h->tc = (!h->fp8 && (h->D == 64 || h->D == 128)) ? 1 : 0;
    h->tc8 = (h->fp8 && (h->D == 128 || h->D == 256)) ? 1 : 0;
    h->pf_tokens = h->tc    ? 2 * (kTcRows / h->G)
                   : h->tc8 ? kTcRows / h->G
                            : (kPfRows / h->G > 0 ? kPfRows / h->G : 1);
    h->timeout_ns = 1000000000ull;  // bound of every device wait (RPA_OPT_WAIT_TIMEOUT_MS)
    // the SM-split model is calibrated for the tensor-memory bf16 prefill kernel only
    h->can_concurrent = h->tc;
    {
        cudaError_t e = cudaSuccess;
        bool failed = false;
        if ((e = cudaGetDevice(&h->device)) != cudaSuccess) failed = true;
        else if ((e = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device)) != cudaSuccess)
            failed = true;
        else if ((e = plan_prepare()) != cudaSuccess) failed = true;
        else if ((e = h->tc    ? prefill_tc_prepare(h->D, &h->pf_bps)
                      : h->tc8 ? prefill_tc8_prepare(h->D, &h->pf_bps)
                               : attn_prepare(h->D, h->fp8, &h->pf_bps)) != cudaSuccess)
            failed = true;
        else if ((e = decode_prepare(h->D, h->fp8, h->dec_rows, &h->dec_bps)) != cudaSuccess) failed = true;
        else if (h->pf_bps < 1 || h->dec_bps < 1) failed = true;  // a kernel cannot be resident
        if (failed) {
            cudaGetLastError();
            delete h;
            return RPA_ERR_CUDA;
        }
    }

    // worst-case capacities (see the planner's chunk rule)
    const int64_t S = c.max_num_seqs, Hkv = c.num_kv_heads;
    const int64_t Tq = h->pf_tokens;
    const int64_t dec_slots = (int64_t)h->sms * h->dec_bps;
    h->max_dec_units = (int)(S + (kDecWaves * dec_slots + Hkv - 1) / Hkv + 1);
    const int pf_only_units = (int)((c.num_q_tokens + Tq - 1) / Tq + S + 1);
    h->max_units = h->max_dec_units + pf_only_units;
    // with fp8 K/V on tensor memory, decode units are items of the prefill kernel too
    h->max_pf_units = h->tc8 ? h->max_units : pf_only_units;
    h->max_part = (int)(h->max_dec_units * Hkv);
    h->max_comb = (int)(S * Hkv);

    size_t off = 0;
    const size_t o_ctrl = off; off = align256(off + kCtrlWords * sizeof(int));
    const size_t o_seq = off; off = align256(off + 6 * (size_t)(S + 1) * sizeof(int));
    const size_t o_units = off; off = align256(off + (size_t)h->max_units * 8 * sizeof(int));
    const size_t o_dec = off; off = align256(off + (size_t)h->max_dec_units * Hkv * sizeof(Item));
    const size_t o_pf = off; off = align256(off + (size_t)h->max_pf_units * Hkv * sizeof(Item));
    const size_t o_comb = off; off = align256(off + (size_t)h->max_comb * sizeof(Comb));
    const size_t o_po = off; off = align256(off + (size_t)h->max_part * kDecRows * h->D * sizeof(float));
    const size_t o_pml = off; off = align256(off + (size_t)h->max_part * kDecRows * 2 * sizeof(float));
    h->ws_bytes = off;
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
    uint8_t* b = static_cast<uint8_t*>(h->ws);
    h->ctrl = reinterpret_cast<int*>(b + o_ctrl);
    h->seq_scratch = reinterpret_cast<int*>(b + o_seq);
    h->units = reinterpret_cast<int*>(b + o_units);
    h->dec_items = reinterpret_cast<Item*>(b + o_dec);
    h->pf_items = reinterpret_cast<Item*>(b + o_pf);
    h->comb = reinterpret_cast<Comb*>(b + o_comb);
    h->part_o = reinterpret_cast<float*>(b + o_po);
    h->part_ml = reinterpret_cast<float*>(b + o_pml);
    if (cudaMemset(h->ctrl, 0, kCtrlWords * sizeof(int)) != cudaSuccess) {
        cudaFree(h->ws);
        cudaGetLastError();
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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int conc = h->can_concurrent && !h->serial;
    h->concurrent = conc;

    PlanParams pp;
    pp.kv_lens = kv_lens;
    pp.cu_q_lens = cu_q_lens;
    pp.num_seqs = num_seqs;
    pp.T = (int)c.num_q_tokens;
    pp.Hkv = (int)c.num_kv_heads;
    pp.G = h->G;
    pp.P = (int)c.pages_per_seq;
    pp.ps = (int)c.page_size;
    pp.causal = c.is_causal ? 1 : 0;
    pp.has_window = c.has_sliding_window ? 1 : 0;
    pp.window = h->window;
    pp.dec_rows = h->dec_rows;
    pp.pf_tokens = h->pf_tokens;
    pp.dec_slots = h->sms * h->dec_bps;
    pp.concurrent = conc;
    pp.n_sms = h->sms;
    pp.dec_bps = h->dec_bps;
    pp.pf_bps = h->pf_bps;
    pp.pf_mma_rows = h->tc ? 2 * kTcRows : h->tc8 ? kTcRows : kPfRows;
    pp.dec_on_pf = h->tc8;
    pp.D = h->D;
    pp.kv_elt = h->fp8 ? 1 : 2;
    pp.pf_sm_gflops = (h->tc || h->tc8) ? kPfSmGflopsTc : kPfSmGflopsMma;
    pp.dec_sm_gbs = kDecSmGBs;
    pp.hbm_gbs = kHbmGBs;
    pp.force_pf_sms = h->force_pf_sms;
    pp.force_dec_sms = h->force_dec_sms;
    pp.max_units = h->max_units;
    pp.max_dec_units = h->max_dec_units;
    pp.max_pf_units = h->max_pf_units;
    pp.max_part = h->max_part;
    pp.max_comb = h->max_comb;
    pp.ctrl = h->ctrl;
    pp.seq_scratch = h->seq_scratch;
    pp.units = h->units;
    pp.keys = nullptr;
    pp.dec_items = h->dec_items;
    pp.pf_items = h->pf_items;
    pp.comb = h->comb;
    cudaEvent_t ev[kProfEvents];
    for (int k = 0; k < kProfEvents; ++k) ev[k] = prof_event(h, k);
    auto rec = [&](int k, cudaStream_t on) { return !ev[k] || cudaEventRecord(ev[k], on) == cudaSuccess; };
    if (!rec(kEvStart, st)) return RPA_ERR_CUDA;
    if (launch_plan(pp, st, plan_smem_bytes()) != cudaSuccess) return RPA_ERR_CUDA;
    if (!rec(kEvPlanEnd, st)) return RPA_ERR_CUDA;

    AttnParams ap;
    ap.q = static_cast<const uint8_t*>(q);
    ap.kv = static_cast<const uint8_t*>(kv_pages);
    ap.o = static_cast<uint8_t*>(o);
    ap.kv_lens = kv_lens;
    ap.page_indices = page_indices;
    ap.cu_q_lens = cu_q_lens;
    ap.T = (int)c.num_q_tokens;
    ap.Hq = (int)c.num_q_heads;
    ap.Hkv = (int)c.num_kv_heads;
    ap.G = h->G;
    ap.D = h->D;
    ap.ps = (int)c.page_size;
    ap.P = (int)c.pages_per_seq;
    ap.N = (int)c.total_num_pages;
    ap.causal = c.is_causal ? 1 : 0;
    ap.has_window = c.has_sliding_window ? 1 : 0;
    ap.window = h->window;
    ap.has_cap = c.has_soft_cap ? 1 : 0;
    ap.qk_log2 = h->qk_log2;
    ap.cap_exp = h->cap_exp;
    ap.cap_log2 = h->cap_log2;
    ap.v_scale = h->v_scale;
    ap.ctrl = h->ctrl;
    ap.part_o = h->part_o;
    ap.part_ml = h->part_ml;
    ap.sinks = c.has_sinks ? c.sinks : nullptr;

    // With concurrent decode / prefill the decode kernel runs on the side stream, forked from st
    // after the planner.  Once forked, every return joins it back (st waits for whatever was
    // enqueued there), so that no kernel of this call is still writing the workspace when the
    // caller's stream moves on.
    cudaStream_t dst = st;  // stream of the decode kernel
    bool forked = false;
    auto join = [&]() -> bool {
        if (!forked) return true;
        forked = false;
        return cudaEventRecord(h->ev_dec, h->side) == cudaSuccess &&
               cudaStreamWaitEvent(st, h->ev_dec, 0) == cudaSuccess;
    };
    auto fail = [&](int code) {
        join();
        return code;
    };
    if (conc) {
        if (cudaEventRecord(h->ev_plan, st) != cudaSuccess || cudaStreamWaitEvent(h->side, h->ev_plan, 0) != cudaSuccess)
            return RPA_ERR_CUDA;
        dst = h->side;
        forked = true;
    }
    if (c.num_q_tokens > 0) {
        if (h->kvmap_ptr != kv_pages) {
            if (encode_kv_map_runs(&h->kvmap, kv_pages, h->fp8, c.total_num_pages, (int)c.page_size,
                                   (int)c.num_kv_heads, h->D, h->BR) != 0 ||
                (h->tc && encode_kv_map(&h->kvmap_pf, kv_pages, h->fp8, c.total_num_pages, (int)c.page_size,
                                        (int)c.num_kv_heads, h->D, h->BR) != 0)) {
                h->kvmap_ptr = nullptr;
                return fail(RPA_ERR_INVALID_ARG);
            }
            h->kvmap_ptr = kv_pages;
        }
        if (h->qmap_ptr != q) {
            if (encode_q_map(&h->qmap, q, c.num_q_tokens, (int)c.num_q_heads, h->D, h->G, h->Tt) != 0 ||
                ((h->tc || h->tc8) && encode_q_map(&h->qmap_pf, q, c.num_q_tokens, (int)c.num_q_heads, h->D,
                                                   h->G, kTcRows / h->G) != 0)) {
                h->qmap_ptr = nullptr;
                return fail(RPA_ERR_INVALID_ARG);
            }
            h->qmap_ptr = q;
        }
    }
    if (!rec(kEvDecStart, dst)) return fail(RPA_ERR_CUDA);
    if (c.num_q_tokens > 0) {
        DecParams dp;
        dp.a = ap;
        dp.a.items = h->dec_items;
        dp.a.item_count_word = kNumDecItems;
        dp.a.counter_word = kDecCounter;
        dp.BR = h->BR;
        dp.br_shift = h->br_shift;
        dp.Tt = h->Tt;
        dp.debug_stall = h->debug_stall;
        dp.timeout_ns = h->timeout_ns;
        if (launch_decode_tma(h->kvmap, h->qmap, dp, h->fp8, h->dec_rows, Launch{h->sms * h->dec_bps, dst}) !=
            cudaSuccess)
            return fail(RPA_ERR_CUDA);
    }
    if (!rec(kEvDecEnd, dst)) return fail(RPA_ERR_CUDA);

    if (!rec(kEvPfStart, st)) return fail(RPA_ERR_CUDA);
    if (c.num_q_tokens > 0) {
        ap.items = h->pf_items;
        ap.item_count_word = kNumPfItems;
        ap.counter_word = kPfCounter;
        cudaError_t e;
        if (h->tc || h->tc8) {
            TcParams tp;
            tp.a = ap;
            tp.BR = h->BR;
            tp.Tq = h->pf_tokens;
            tp.timeout_ns = h->timeout_ns;
            // the fp8 kernel copies whole page runs (K and V of the head) with the decode gather's map
            e = h->tc ? launch_prefill_tc(h->kvmap_pf, h->qmap_pf, tp, Launch{h->sms * h->pf_bps, st})
                      : launch_prefill_tc8(h->kvmap, h->qmap_pf, tp, Launch{h->sms * h->pf_bps, st});
        } else {
            e = launch_prefill(ap, h->fp8, Launch{h->sms * h->pf_bps, st});
        }
        if (e != cudaSuccess) return fail(RPA_ERR_CUDA);
    }
    if (!rec(kEvPfEnd, st)) return fail(RPA_ERR_CUDA);
    if (!join()) return RPA_ERR_CUDA;

    CombParams cp;
    cp.o = static_cast<uint8_t*>(o);
    cp.cu_q_lens = cu_q_lens;
    cp.num_seqs = num_seqs;
    cp.T = (int)c.num_q_tokens;
    cp.Hq = (int)c.num_q_heads;
    cp.G = h->G;
    cp.D = h->D;
    cp.rows_max = h->dec_rows;
    cp.v_scale = h->v_scale;
    cp.sinks = c.has_sinks ? c.sinks : nullptr;
    cp.ctrl = h->ctrl;
    cp.comb = h->comb;
    cp.part_o = h->part_o;
    cp.part_ml = h->part_ml;
    if (!rec(kEvCombStart, st)) return RPA_ERR_CUDA;
    if (launch_combine(cp, Launch{h->sms * 2, st}) != cudaSuccess) return RPA_ERR_CUDA;
    if (ev[kEvCombEnd]) {
        if (cudaEventRecord(ev[kEvCombEnd], st) != cudaSuccess) return RPA_ERR_CUDA;
        ++h->prof_used;
    }
    return RPA_OK;
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
        if (cudaEventSynchronize(e[kEvCombEnd]) != cudaSuccess) return RPA_ERR_CUDA;
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
            if (value < 0 || value > h->sms) return RPA_ERR_INVALID_ARG;
            (option == RPA_OPT_PREFILL_SMS ? h->force_pf_sms : h->force_dec_sms) = (int)value;
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
    const size_t qb = (size_t)c.num_q_tokens * c.num_q_heads * c.head_dim * 2;
    const size_t kb = (size_t)c.max_num_seqs * sizeof(int32_t);
    const size_t pb = (size_t)c.max_num_seqs * c.pages_per_seq * sizeof(int32_t);
    const size_t cb = (size_t)(c.max_num_seqs + 1) * sizeof(int32_t);
    const size_t o_q = 0, o_o = align256(qb), o_k = o_o + align256(qb), o_p = o_k + align256(kb),
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
    if (qb && cudaMemcpyAsync(o_host, s + o_o, qb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return RPA_ERR_CUDA;
    return RPA_OK;
}

int rpa_get_status(RpaHandle* h, void* stream) {
    if (!h) return RPA_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return RPA_ERR_CUDA;
    int v = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&v, h->ctrl + kStatus, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
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
    if (cudaMemcpyAsync(ctrl, h->ctrl, sizeof ctrl, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return RPA_ERR_CUDA;
    for (int i = 0; i < 16; ++i) info[i] = 0;
    info[0] = ctrl[kStatus];
    info[1] = ctrl[kNumDecItems];
    info[2] = ctrl[kNumPfItems];
    info[3] = ctrl[kNumComb];
    info[4] = ctrl[kDecChunk];
    info[5] = h->dec_rows;
    info[6] = h->pf_tokens;
    info[7] = ctrl[kNumPart];
    info[8] = ctrl[kNumUnits];
    info[9] = ctrl[kSorted];
    info[10] = ctrl[kDecCtas];
    info[11] = ctrl[kPfCtas];
    info[12] = h->sms;
    info[13] = h->dec_bps;
    info[14] = h->pf_bps;
    info[15] = h->concurrent | (h->tc8 << 1);
    if (items && max_items > 0) {
        const int64_t nd = ctrl[kNumDecItems] < max_items ? ctrl[kNumDecItems] : max_items;
        const int64_t np = ctrl[kNumPfItems] < max_items - nd ? ctrl[kNumPfItems] : max_items - nd;
        if ((nd && cudaMemcpy(items, h->dec_items, nd * sizeof(Item), cudaMemcpyDeviceToHost) != cudaSuccess) ||
            (np && cudaMemcpy(items + nd * 8, h->pf_items, np * sizeof(Item), cudaMemcpyDeviceToHost) != cudaSuccess))
            return RPA_ERR_CUDA;
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
