// rpa_noalloc.cu -- rpa_forward_noalloc: the forward call without any allocation.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code executing under a custom or arena allocator that owns all of
// the device memory, engines that forbid cudaMalloc/cudaFree on the serving path
// because those calls synchronise the device, and hosts that embed the
// library through a plain C interface with no allocator to hand over.  For
// them this entry point runs the same planner, attention and combine kernels
// as rpa_forward, but its workspace (plan, work items and split-KV partials)
// lives in one fixed-size array in the library's own device memory,
// reserved when the library's module is loaded on each GPU and kept until
// the process exits.  Nothing here calls cudaMalloc, cudaFree or any other
// allocating routine.
#include <mutex>

#include "rpa_internal.cuh"

using namespace rpa;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per GPU
constexpr int kMaxDevices = 64;

// The scratch array itself.  Host code must not take its address directly:
// the symbol's host-side name is only a stand-in for the device object.
static __device__ __align__(256) unsigned char g_rpa_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices];
int g_dec_bps[kMaxDevices][3][2][2];  // [device][D: 64,128,256][fp8][8-row decode tiles]
int g_pf_bps[kMaxDevices][3][2][2];
bool g_ready[kMaxDevices][3][2][2];
bool g_plan_ready[kMaxDevices];

int d_index(int D) { return D == 64 ? 0 : D == 128 ? 1 : 2; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Once per device (and per head size / K/V type for the kernel attributes),
// with that device current: fetch the scratch array's device address and set
// the kernels' shared-memory limits.  None of this allocates.
int setup(int dev, int D, int fp8, int dec_rows, void** scratch, int* dec_bps, int* pf_bps) {
    if (dev < 0 || dev >= kMaxDevices) return RPA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_dev[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_rpa_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return RPA_ERR_CUDA;
        }
        g_scratch_dev[dev] = ptr;
    }
    if (!g_plan_ready[dev]) {
        if (plan_prepare() != cudaSuccess) {
            cudaGetLastError();
            return RPA_ERR_CUDA;
        }
        g_plan_ready[dev] = true;
    }
    const int di = d_index(D), r8 = dec_rows == 8 ? 1 : 0;
    if (!g_ready[dev][di][fp8][r8]) {
        int a = 0, b = 0;
        const bool tc = !fp8 && (D == 64 || D == 128);
        const bool tc8 = fp8 && (D == 128 || D == 256);
        if (decode_prepare(D, fp8, dec_rows, &a) != cudaSuccess ||
            (tc ? prefill_tc_prepare(D, &b) : tc8 ? prefill_tc8_prepare(D, &b) : attn_prepare(D, fp8, &b)) !=
                cudaSuccess) {
            cudaGetLastError();
            return RPA_ERR_CUDA;
        }
        // a kernel that cannot be resident: refuse before anything is enqueued (as rpa_create does)
        if (a < 1 || b < 1) return RPA_ERR_CUDA;
        g_dec_bps[dev][di][fp8][r8] = a;
        g_pf_bps[dev][di][fp8][r8] = b;
        g_ready[dev][di][fp8][r8] = true;
    }
    *scratch = g_scratch_dev[dev];
    *dec_bps = g_dec_bps[dev][di][fp8][r8];
    *pf_bps = g_pf_bps[dev][di][fp8][r8];
    return RPA_OK;
}

}  // namespace

extern "C" int rpa_forward_noalloc(const RpaCfg* cfg, const void* q, const void* kv_pages,
                                   const int32_t* kv_lens, const int32_t* page_indices,
                                   const int32_t* cu_q_lens, int32_t num_seqs, void* o, void* stream) {
    const int v = rpa_validate_cfg(cfg);
    if (v != RPA_OK) return v;
    const RpaCfg& c = *cfg;
    if (num_seqs < 0 || num_seqs > c.max_num_seqs) return RPA_ERR_INVALID_ARG;
    if (!kv_pages || !kv_lens || !page_indices || !cu_q_lens) return RPA_ERR_INVALID_ARG;
    if (c.num_q_tokens > 0 && (!q || !o)) return RPA_ERR_INVALID_ARG;
    auto misaligned = [](const void* p, size_t a) { return ((uintptr_t)p % a) != 0; };
    if ((q && misaligned(q, 16)) || (o && misaligned(o, 16)) || misaligned(kv_pages, 16) ||
        misaligned(kv_lens, 4) || misaligned(page_indices, 4) || misaligned(cu_q_lens, 4))
        return RPA_ERR_INVALID_ARG;

    const int G = (int)(c.num_q_heads / c.num_kv_heads);
    const int D = (int)c.head_dim;
    const int fp8 = c.kv_dtype == RPA_DT_FP8_E4M3;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return RPA_ERR_CUDA;
    }
    void* scratch = nullptr;
    int dec_bps = 1, pf_bps = 1;
    const int dec_rows = (!fp8 && G <= 8) ? 8 : kDecRows;  // the same rule as rpa_create
    const int su = setup(dev, D, fp8, dec_rows, &scratch, &dec_bps, &pf_bps);
    if (su != RPA_OK) return su;

    // worst-case capacities, the same rule as rpa_create's workspace
    const int64_t S = c.max_num_seqs, Hkv = c.num_kv_heads;
    const bool tc = !fp8 && (D == 64 || D == 128);
    const bool tc8 = fp8 && (D == 128 || D == 256);
    const int pf_tokens = tc ? 2 * (kTcRows / G) : tc8 ? kTcRows / G : (kPfRows / G > 0 ? kPfRows / G : 1);
    const int64_t Tq = pf_tokens;
    const int64_t dec_slots = (int64_t)sms * dec_bps;
    const int64_t max_dec_units = S + (kDecWaves * dec_slots + Hkv - 1) / Hkv + 1;
    const int64_t pf_only_units = (c.num_q_tokens + Tq - 1) / Tq + S + 1;
    const int64_t max_units = max_dec_units + pf_only_units;
    const int64_t max_pf_units = tc8 ? max_units : pf_only_units;
    const int64_t max_part = max_dec_units * Hkv;
    const int64_t max_comb = S * Hkv;
    size_t off = 0;
    const size_t o_ctrl = off; off = align256(off + kCtrlWords * sizeof(int));
    const size_t o_seq = off; off = align256(off + 6 * (size_t)(S + 1) * sizeof(int));
    const size_t o_units = off; off = align256(off + (size_t)max_units * 8 * sizeof(int));
    const size_t o_dec = off; off = align256(off + (size_t)max_dec_units * Hkv * sizeof(Item));
    const size_t o_pf = off; off = align256(off + (size_t)max_pf_units * Hkv * sizeof(Item));
    const size_t o_comb = off; off = align256(off + (size_t)max_comb * sizeof(Comb));
    const size_t o_po = off; off = align256(off + (size_t)max_part * kDecRows * D * sizeof(float));
    const size_t o_pml = off; off = align256(off + (size_t)max_part * kDecRows * 2 * sizeof(float));
    if (off > kNoAllocScratchBytes) return RPA_ERR_NO_ALLOC_LIMIT;

    uint8_t* b = static_cast<uint8_t*>(scratch);
    int* ctrl = reinterpret_cast<int*>(b + o_ctrl);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: start the control block at zero
    if (cudaMemsetAsync(ctrl, 0, kCtrlWords * sizeof(int), st) != cudaSuccess) {
        cudaGetLastError();
        return RPA_ERR_CUDA;
    }
    Item* dec_items = reinterpret_cast<Item*>(b + o_dec);
    Item* pf_items = reinterpret_cast<Item*>(b + o_pf);
    Comb* comb = reinterpret_cast<Comb*>(b + o_comb);
    float* part_o = reinterpret_cast<float*>(b + o_po);
    float* part_ml = reinterpret_cast<float*>(b + o_pml);
    const int window =
        c.has_sliding_window ? (int)(c.sliding_window > 0x7fffffff ? 0x7fffffff : c.sliding_window) : 0;
    const double log2e = 1.4426950408889634;
    const double ks = c.has_k_scale ? c.k_scale : 1.0;

    PlanParams pp;
    pp.kv_lens = kv_lens;
    pp.cu_q_lens = cu_q_lens;
    pp.num_seqs = num_seqs;
    pp.T = (int)c.num_q_tokens;
    pp.Hkv = (int)Hkv;
    pp.G = G;
    pp.P = (int)c.pages_per_seq;
    pp.ps = (int)c.page_size;
    pp.causal = c.is_causal ? 1 : 0;
    pp.has_window = c.has_sliding_window ? 1 : 0;
    pp.window = window;
    pp.dec_rows = dec_rows;
    pp.pf_tokens = pf_tokens;
    pp.dec_slots = (int)dec_slots;
    pp.concurrent = 0;  // one stream: decode and prefill run one after the other on all SMs
    pp.n_sms = sms;
    pp.dec_bps = dec_bps;
    pp.pf_bps = pf_bps;
    pp.pf_mma_rows = tc ? 2 * kTcRows : tc8 ? kTcRows : kPfRows;
    pp.dec_on_pf = tc8 ? 1 : 0;
    pp.D = D;
    pp.kv_elt = fp8 ? 1 : 2;
    pp.pf_sm_gflops = (tc || tc8) ? kPfSmGflopsTc : kPfSmGflopsMma;
    pp.dec_sm_gbs = kDecSmGBs;
    pp.hbm_gbs = kHbmGBs;
    pp.force_pf_sms = 0;
    pp.force_dec_sms = 0;
    pp.max_units = (int)max_units;
    pp.max_dec_units = (int)max_dec_units;
    pp.max_pf_units = (int)max_pf_units;
    pp.max_part = (int)max_part;
    pp.max_comb = (int)max_comb;
    pp.ctrl = ctrl;
    pp.seq_scratch = reinterpret_cast<int*>(b + o_seq);
    pp.units = reinterpret_cast<int*>(b + o_units);
    pp.keys = nullptr;
    pp.dec_items = dec_items;
    pp.pf_items = pf_items;
    pp.comb = comb;
    if (launch_plan(pp, st, plan_smem_bytes()) != cudaSuccess) return RPA_ERR_CUDA;

    AttnParams ap;
    ap.q = static_cast<const uint8_t*>(q);
    ap.kv = static_cast<const uint8_t*>(kv_pages);
    ap.o = static_cast<uint8_t*>(o);
    ap.kv_lens = kv_lens;
    ap.page_indices = page_indices;
    ap.cu_q_lens = cu_q_lens;
    ap.T = (int)c.num_q_tokens;
    ap.Hq = (int)c.num_q_heads;
    ap.Hkv = (int)Hkv;
    ap.G = G;
    ap.D = D;
    ap.ps = (int)c.page_size;
    ap.P = (int)c.pages_per_seq;
    ap.N = (int)c.total_num_pages;
    ap.causal = pp.causal;
    ap.has_window = pp.has_window;
    ap.window = window;
    ap.has_cap = c.has_soft_cap ? 1 : 0;
    ap.qk_log2 = (float)(c.sm_scale * ks * log2e);
    ap.cap_exp = c.has_soft_cap ? (float)(2.0 * c.sm_scale * ks / c.soft_cap * log2e) : 0.f;
    ap.cap_log2 = c.has_soft_cap ? (float)(c.soft_cap * log2e) : 0.f;
    ap.v_scale = c.has_v_scale ? c.v_scale : 1.f;
    ap.ctrl = ctrl;
    ap.part_o = part_o;
    ap.part_ml = part_ml;
    ap.sinks = c.has_sinks ? c.sinks : nullptr;
    if (c.num_q_tokens > 0) {
        int BR = 64, br_shift = 0;
        while ((int)(c.page_size % BR)) BR >>= 1;
        while ((1 << br_shift) < BR) ++br_shift;
        const int Tt = G <= dec_rows ? dec_rows / G : 1;
        CUtensorMap kvm, kvm_pf, qm, qm_pf;  // descriptors are encoded on the host stack
        if (encode_kv_map_runs(&kvm, kv_pages, fp8, c.total_num_pages, (int)c.page_size, (int)Hkv, D, BR) != 0 ||
            (tc && encode_kv_map(&kvm_pf, kv_pages, fp8, c.total_num_pages, (int)c.page_size, (int)Hkv, D, BR) != 0) ||
            encode_q_map(&qm, q, c.num_q_tokens, (int)c.num_q_heads, D, G, Tt) != 0 ||
            ((tc || tc8) && encode_q_map(&qm_pf, q, c.num_q_tokens, (int)c.num_q_heads, D, G, kTcRows / G) != 0))
            return RPA_ERR_INVALID_ARG;
        DecParams dp;
        dp.a = ap;
        dp.a.items = dec_items;
        dp.a.item_count_word = kNumDecItems;
        dp.a.counter_word = kDecCounter;
        dp.BR = BR;
        dp.br_shift = br_shift;
        dp.Tt = Tt;
        dp.debug_stall = 0;
        dp.timeout_ns = 1000000000ull;
        if (launch_decode_tma(kvm, qm, dp, fp8, dec_rows, Launch{(int)dec_slots, st}) != cudaSuccess)
            return RPA_ERR_CUDA;
        ap.items = pf_items;
        ap.item_count_word = kNumPfItems;
        ap.counter_word = kPfCounter;
        if (tc) {
            TcParams tp;
            tp.a = ap;
            tp.BR = BR;
            tp.Tq = pf_tokens;
            tp.timeout_ns = 1000000000ull;
            if (launch_prefill_tc(kvm_pf, qm_pf, tp, Launch{sms * pf_bps, st}) != cudaSuccess) return RPA_ERR_CUDA;
        } else if (tc8) {
            TcParams tp;
            tp.a = ap;
            tp.BR = BR;
            tp.Tq = pf_tokens;
            tp.timeout_ns = 1000000000ull;
            if (launch_prefill_tc8(kvm, qm_pf, tp, Launch{sms * pf_bps, st}) != cudaSuccess) return RPA_ERR_CUDA;
        } else if (launch_prefill(ap, fp8, Launch{sms * pf_bps, st}) != cudaSuccess) {
            return RPA_ERR_CUDA;
        }
    }

    CombParams cp;
    cp.o = static_cast<uint8_t*>(o);
    cp.cu_q_lens = cu_q_lens;
    cp.num_seqs = num_seqs;
    cp.T = (int)c.num_q_tokens;
    cp.Hq = (int)c.num_q_heads;
    cp.G = G;
    cp.D = D;
    cp.rows_max = dec_rows;
    cp.v_scale = ap.v_scale;
    cp.sinks = ap.sinks;
    cp.ctrl = ctrl;
    cp.comb = comb;
    cp.part_o = part_o;
    cp.part_ml = part_ml;
    if (launch_combine(cp, Launch{sms * 2, st}) != cudaSuccess) return RPA_ERR_CUDA;
    return RPA_OK;
}
