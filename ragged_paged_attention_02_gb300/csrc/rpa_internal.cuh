// rpa_internal.cuh -- shared definitions of the CUDA side of librpa.
//
// Plan layout, kernel parameters and the small PTX helpers (mbarrier, bulk
// tensor copies, tcgen05, ldmatrix, mma.sync, ex2) used by the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rpa.h"

namespace rpa {

// ---------------------------------------------------------------- plan layout
// Control block (int32 words) at the start of the workspace.
enum Ctrl : int {
    kStatus = 0,
    kNumDecItems = 1,
    kNumPfItems = 2,
    kNumComb = 3,
    kDecChunk = 4,
    kDecCounter = 5,
    kPfCounter = 6,
    kNumPart = 7,
    kNumUnits = 8,
    kSorted = 9,
    kCovLo = 10,   // first token covered by a sequence
    kCovHi = 11,   // end of covered tokens
    kPfCtas = 12,  // prefill CTAs that take work (the rest exit at once)
    kDecCtas = 13, // decode CTAs that take work
    kPlanEpoch = 14,  // the epoch of the call whose plan is complete (the planner writes it last)
    kCtrlWords = 32,
};

// One work item: 8 int32.
struct Item {
    int seq, head, tok0, ntok, kv_begin, kv_end, part, piece;
};
// One work unit (the planner's list): a sequence's query tokens [tok0, tok0 + ntok) against keys
// [kv_begin, kv_end), piece `piece` of `pieces`; `part` is the first partial slot of its split
// sequence (or -1).  Unit u stands for items u H .. u H + H - 1, one per kv head (H the planner's
// kv heads), whose partial slot is part + head * pieces + piece.
struct Unit {
    int seq, tok0, ntok, kv_begin, kv_end, part, piece, pieces;
};
// Item `it` of a unit list of H kv heads
__device__ __forceinline__ Item item_at(const Unit* units, int it, int H) {
    const int u = it / H, h = it - u * H;
    const int4* src = reinterpret_cast<const int4*>(units + u);
    const int4 a = src[0], b = src[1];
    Item r;
    r.seq = a.x;
    r.head = h;
    r.tok0 = a.y;
    r.ntok = a.z;
    r.kv_begin = a.w;
    r.kv_end = b.x;
    r.part = b.y >= 0 ? b.y + h * b.w + b.z : -1;
    r.piece = b.z;
    return r;
}

// One split-KV combine entry: rows [0, rows) of the kv head `head` of the sequence whose first
// query token is q0 merge `pieces` partials starting at slot `part` (32 bytes: two 16-byte loads)
struct __align__(16) Comb {
    int q0, rows, head, part, pieces, pad0, pad1, pad2;
};

// K/V element types inside the kernels (template arguments): 16-bit types feed the MMAs as they
// are; 8-bit types are converted exactly to f16 first.
enum KvType : int { KT_BF16 = 0, KT_F16 = 1, KT_E4M3 = 2, KT_E5M2 = 3, KT_I8 = 4 };
__host__ __device__ constexpr bool kt_8bit(int kt) { return kt >= KT_E4M3; }
__host__ __device__ constexpr bool kt_f16_mma(int kt) { return kt != KT_BF16; }  // MMA operands in f16
// Output element types (o has the q dtype)
enum OutType : int { OT_BF16 = 0, OT_F16 = 1, OT_F32 = 2 };

constexpr int kDecRows = 16;       // rows of a decode tile (one m16 MMA tile)
// latent attention: row width, value width, query rows of a work item
constexpr int kMlaDqk = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaRows = 16;
constexpr int kMaxGroup = 64;      // query heads per kv head (a prefill tile holds 128 / G tokens)
constexpr int kDecWaves = 4;       // target decode items per resident CTA (the most of any kernel)
// ... on the 64-key-tile kernel, whose items pay a Q load into tensor memory and a pipeline ramp
// each, and whose decode rows cost a full tile's tensor work: fewer, longer pieces (fp8_window
// workload: 0.517 ms a step with 2 against 0.527 with 4)
constexpr int kDecWavesTc8 = 2;
constexpr int kMinChunk = 512;     // smallest split-KV piece (keys)
constexpr int kChunkAlign = 64;    // pieces are multiples of this many keys
constexpr int kMaxSort = 8192;     // units sorted by cost on the device
constexpr int kSeqSmem = 4096;     // sequences whose plan scratch fits in shared memory
constexpr int kSeqArrays = 9;      // per-sequence plan scratch arrays of S + 1 ints
constexpr int kPlanThreads = 512;
// rates of the SM-split model (planner): FLOP/ns of one SM on prefill, B/ns one SM can
// stream in the decode kernel, and HBM B/ns.  The first two are the rates measured with
// both kernels running at once (chunked prefill of 512 tokens beside long decodes, D 128):
// lower than either kernel alone, which shares no SMs, L2 or HBM bandwidth.
constexpr int kPfSmGflopsTc = 6500;
constexpr int kPfSmGflopsMma = 800;  // the latent kernel (warp MMAs)
constexpr int kDecSmGBs = 78;
constexpr int kHbmGBs = 6700;

struct PlanParams {
    const int* kv_lens;
    const int* cu_q_lens;
    int num_seqs;
    int T;           // num_q_tokens
    int Hkv;
    int G;           // q heads per kv head
    int P, ps;       // pages_per_seq, page_size
    int causal, has_window, window;
    int dec_rows;    // rows of a decode tile
    int pf_tokens;   // query tokens of a prefill tile
    int dec_slots;   // resident decode CTAs (all SMs)
    // SM split between the decode and prefill kernels when they run concurrently
    int concurrent;      // 1: the two kernels run at the same time on disjoint SMs
    int n_sms, dec_bps, pf_bps;  // SMs, resident CTAs per SM of each kernel
    int pf_mma_rows;     // MMA rows per prefill unit (tile padding included)
    int dec_on_pf;       // 1: decode units become items of the prefill kernel (no decode kernel work)
    int D, kv_elt;
    int pf_sm_gflops;    // prefill FLOP rate of one SM (FLOP/ns)
    int dec_sm_gbs;      // decode bytes one SM can stream (B/ns)
    int hbm_gbs;         // HBM bandwidth (B/ns)
    int force_pf_sms;    // > 0: tuning hook, prefill SMs when both classes have work
    int force_dec_sms;   // > 0: tuning hook, decode SMs
    int dec_waves;       // target decode items per CTA of the kernel that runs them
    int epoch;           // this call's number, published in ctrl[kPlanEpoch] once the plan is out
    int early;           // the inputs are complete at launch: read them before the grid dependency
    int max_units;   // capacity of the unit arrays
    int max_dec_units, max_pf_units;  // capacities of the two unit lists
    int max_part;    // capacity of partial slots
    int max_comb;    // capacity of combine entries
    int* ctrl;
    int* seq_scratch;  // [kSeqArrays * (max_num_seqs + 1)], used when the sequences overflow shared memory
    int* units;        // [max_units * 8]
    unsigned long long* keys;  // [max_units] (only used if > kMaxSort)
    Unit* dec_units;   // the decode kernel's list, in order
    Unit* pf_units;    // the prefill kernel's list, in order
    Comb* comb;
};

struct AttnParams {
    const uint8_t* q;
    const uint8_t* kv;
    uint8_t* o;
    const int* kv_lens;
    const int* page_indices;
    const int* cu_q_lens;
    int T, Hq, Hkv, G, D, ps, P, N;
    int causal, has_window, window, has_cap;
    float qk_log2;      // sm_scale * k_scale * log2(e)  (no cap)
    float cap_exp;      // 2 * sm_scale * k_scale / cap * log2(e)
    float cap_log2;     // cap * log2(e)
    float v_scale;
    int* ctrl;
    const Unit* units;     // the kernel's unit list (item it: item_at(units, it, unit_heads))
    int unit_heads;        // kv heads a unit stands for
    int item_count_word;   // ctrl index of the item count
    int counter_word;      // ctrl index of the work counter
    float* part_o;         // [max_part, kDecRows, D]
    float* part_ml;        // [max_part, kDecRows, 2]
    const float* sinks;    // [Hq] sink logits (natural-log domain), or nullptr
    int odt;               // OutType of o
    int q_f16;             // 8-bit K/V: q holds f16 values (else bf16, rounded to f16 in the kernel)
};

struct DecParams {
    AttnParams a;
    int BR;                 // keys per copied page run: gcd(page_size, 64), >= 4
    int br_shift;           // log2(BR)
    int Tt;                 // query tokens per Q copy: 16 / G
    int debug_stall;        // test hook: the producer issues nothing
    unsigned long long timeout_ns;  // bound of every mbarrier wait
    // >= 0: launched behind the prefill kernel on the same stream (concurrent decode / prefill):
    // the CTAs wait for ctrl[kPlanEpoch] to reach this call's epoch instead of the grid dependency
    // (which is then the prefill kernel), and wait for that dependency only before they exit
    int plan_epoch;
};

struct TcParams {
    AttnParams a;
    int BR;                 // keys per copied page run: gcd(page_size, 64)
    int Tq;                 // query tokens per 128-row tile: 128 / G
    unsigned long long timeout_ns;
};

struct CombParams {
    uint8_t* o;
    const int* cu_q_lens;
    int num_seqs, T, Hq, G, D;
    int rows_max;  // most rows of a combine entry (the decode tile's rows)
    float v_scale;
    const float* sinks;  // [Hq] sink logits (natural-log domain), or nullptr
    int odt;             // OutType of o
    const int* ctrl;
    const Comb* comb;
    const float* part_o;
    const float* part_ml;
};

// ---------------------------------------------------------------- host launchers
struct Launch {
    int grid;
    cudaStream_t stream;
};
// Launch with programmatic stream serialisation (the kernel calls pdl_wait()).
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern k, int grid, int block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}
cudaError_t launch_plan(const PlanParams& p, cudaStream_t st, size_t smem);
constexpr int kCombCtasPerSm = 4;  // combine CTAs resident per SM (its register budget: 64)
cudaError_t launch_combine(const CombParams& p, const Launch& l);
// rows: query rows of a decode tile, 16 (any) or 8 (2-byte K/V, G <= 8: keys on the MMA's M side)
cudaError_t launch_decode_tma(const CUtensorMap& kvm, const CUtensorMap& qm, const DecParams& p, int kt,
                              int rows, const Launch& l);
cudaError_t decode_prepare(int D, int kt, int rows, int* blocks_per_sm);
cudaError_t launch_prefill_tc(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, int kt,
                              const Launch& l);
cudaError_t prefill_tc_prepare(int D, int kt, int* blocks_per_sm);
cudaError_t launch_prefill_tc8(const CUtensorMap& kvm_runs, const CUtensorMap& qm, const TcParams& p, int kt,
                               const Launch& l);
cudaError_t prefill_tc8_prepare(int D, int kt, int* blocks_per_sm);
// latent attention (kt: KT_BF16 or KT_F16); items are tiles of kMlaRows query rows
cudaError_t mla_prepare(int kt, int* blocks_per_sm);
cudaError_t launch_mla(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, int kt, const Launch& l);
// q (n elements of RpaDtype q_dtype: f32, f16 or bf16) rounded to f16 (to_f16) or bf16 into out
cudaError_t launch_q_convert(const void* q, int q_dtype, uint8_t* out, int to_f16, size_t n, const Launch& l);
constexpr int kTcRows = 128;  // rows of a tensor-memory prefill tile
// tensor maps for the gathers (host; no allocation); byte_elems: 1-byte K/V elements, else 2-byte
int encode_kv_map(CUtensorMap* m, const void* kv, int byte_elems, long long N, int ps, int Hkv, int D, int BR);
int encode_q_map(CUtensorMap* m, const void* q, long long T, int Hq, int D, int G, int Tt);
int encode_kv_map_runs(CUtensorMap* m, const void* kv, int byte_elems, long long N, int ps, int Hkv, int D, int BR);
// cache [N, ps, H, D] (2-byte elements; the split cache as H = 2 Hkv): one box = BR slots of one
// row, all its column blocks
int encode_kv_map_heads(CUtensorMap* m, const void* kv, long long N, int ps, int H, int D, int BR);
// occupancy / attributes (call once per device)
size_t plan_smem_bytes();
cudaError_t plan_prepare();

// ---------------------------------------------------------------- one call, host side (rpa_launch.cu)
// The kernels and tiles a configuration uses, with their occupancy and the workspace capacities.
struct KernelSet {
    int G, D, kt, odt;
    int Dv;              // width of V and o (D except for the latent layout)
    int mla;             // latent layout: every item runs on the latent-attention kernel
    int Gp, Hp;          // the planner's heads per kv head and kv heads (latent: blocks of <= 16 q heads)
    int q_conv;          // 1: q is first rounded into the workspace (its type is not the MMA operand type)
    int q_conv_f16;      // ... to f16 (else bf16)
    int q_f16;           // 8-bit K/V: the q the kernels read holds f16 values
    int tc, tc8;         // prefill on the tensor-memory kernel for 2-byte / 8-bit K/V
    int dec_rows, pf_tokens, Tt, BR, br_shift, window;
    float qk_log2, cap_exp, cap_log2, v_scale;
    int sms, dec_bps, pf_bps;
    int max_dec_units, max_pf_units, max_units, max_part, max_comb;
};
// The 64-key-tile kernel in direct mode (2-byte K/V) copies a page run's whole K (or V) tile in
// one box when a run is a whole tile (BR = 64, the map from encode_kv_map_heads); with smaller
// page runs, one box per (run, column block) (the map from encode_kv_map)
constexpr int kTc8Keys = 64;
inline bool tc8_whole_tiles(const KernelSet& ks) { return ks.tc8 && !kt_8bit(ks.kt) && ks.BR == kTc8Keys; }
struct Workspace {
    int* ctrl;
    int* seq_scratch;
    int* units;
    Unit* dec_units;
    Unit* pf_units;
    Comb* comb;
    float* part_o;
    float* part_ml;
    uint8_t* qbuf;  // q in the MMA operand type (when KernelSet::q_conv)
};
// Tensor maps of the last call, re-encoded when the pointers change
struct MapCache {
    CUtensorMap kv, kv_pf, q, q_pf;
    const void* kv_ptr;
    const void* q_ptr;
};
// Profile events of one call: each kernel is timed from an event recorded on its own stream just
// before its launch (after any cross-stream wait) to one recorded just after it.
enum ProfEvent : int {
    kEvStart = 0, kEvPlanEnd, kEvDecStart, kEvDecEnd, kEvPfStart, kEvPfEnd, kEvCombStart, kEvCombEnd,
    kProfEvents
};
struct EnqueueOpts {
    cudaStream_t st;                 // the caller's stream
    int conc;                        // decode on `side` concurrently with prefill on st
    cudaStream_t side;
    cudaEvent_t ev_plan, ev_dec;     // fork / join events (conc)
    cudaEvent_t ev[kProfEvents];     // profile events, or nullptr
    int debug_stall;
    unsigned long long timeout_ns;
    int force_pf_sms, force_dec_sms;
    int epoch;  // this call's number (concurrent decode / prefill on one stream)
    int plan_early;  // RPA_OPT_PLAN_EARLY
};
// Host only: fill ks from a validated configuration (sms = the device's SM count).
void kernels_choose(const RpaCfg& c, int sms, KernelSet* ks);
// Kernel attributes and occupancy on the current device (dec_bps, pf_bps); an error if a kernel
// cannot be resident.
cudaError_t kernels_occupancy(KernelSet* ks);
// The workspace capacities of cfg (host only, after kernels_occupancy).
void kernels_capacity(const RpaCfg& c, KernelSet* ks);
// Both of the above.
cudaError_t kernels_prepare(const RpaCfg& c, KernelSet* ks);
size_t workspace_bytes(const RpaCfg& c, const KernelSet& ks);
Workspace workspace_carve(const RpaCfg& c, const KernelSet& ks, void* base);
// Enqueue one call; returns an RpaStatus.  Allocates nothing.
int enqueue_forward(const RpaCfg& c, const KernelSet& ks, const Workspace& ws, MapCache* maps, const void* q,
                    const void* kv_pages, const int32_t* kv_lens, const int32_t* page_indices,
                    const int32_t* cu_q_lens, int32_t num_seqs, void* o, const EnqueueOpts& eo);

// ---------------------------------------------------------------- device helpers
#ifdef __CUDACC__
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A*B + D, m16n8k16, fp32 accumulate; F16 selects f16 operands, else bf16.
template <bool F16>
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    if constexpr (F16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// 2^x on the special-function unit (hardware instruction).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// 1/x on the special-function unit (hardware instruction, flush-to-zero).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// The softmax denominator of a row whose logits (log2 domain) are relative to `base`, with the
// row's attention sink added: l + 2^(sink log2(e) - base).  The sink starts the row's maximum in
// the definition; any other common base gives the same quotient, and a sink far above the base
// makes the denominator infinite and the row zero, its limit.  A row with no allowed key
// (base -inf) stays zero: its O is zero whatever the denominator.
__device__ __forceinline__ float add_sink(float l, const float* sinks, int qh, float base) {
    if (sinks == nullptr || base == -INFINITY) return l;
    return l + ex2(__ldg(sinks + qh) * 1.4426950408889634f - base);
}

// tanh(x) on the special-function unit (hardware approximation, relative error about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// Paired fp32 arithmetic (one instruction for two lanes of a 64-bit register pair).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;\n" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// max / min of three floats (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Pack two floats into a bf16x2 / f16x2 register (round to nearest even).
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (F16)
        asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e4m3fn bytes -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(v));
    return r;
}
// Two e5m2 bytes -> f16x2 (exact: e5m2 is the upper byte of an IEEE binary16).
__device__ __forceinline__ uint32_t e5m2x2_to_f16x2(uint16_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;\n" : "=r"(r) : "h"(v));
    return r;
}
// f16x2 subtraction
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// Four int8 values -> two f16x2 (exact).  Each byte x is placed, sign bit flipped, as the low
// mantissa byte of the f16 0x6400 (1024): that is 1024 + (x + 128) exactly, and subtracting 1152
// (0x6480) leaves x.  Every step is exact in f16 (11 significant bits).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    lo = hsub2_u32(__byte_perm(u, 0x64646464u, 0x4140), 0x64806480u);
    hi = hsub2_u32(__byte_perm(u, 0x64646464u, 0x4342), 0x64806480u);
}
// Eight 8-bit K/V values (two words, in memory order) -> eight f16 (exact), for KT_E4M3,
// KT_E5M2 or KT_I8.
template <int KT>
__device__ __forceinline__ uint4 cvt8x8_to_f16x8(uint32_t w0, uint32_t w1) {
    uint4 r;
    if constexpr (KT == KT_I8) {
        i8x4_to_f16x4(w0, r.x, r.y);
        i8x4_to_f16x4(w1, r.z, r.w);
    } else if constexpr (KT == KT_E5M2) {
        r = make_uint4(e5m2x2_to_f16x2((uint16_t)(w0 & 0xffff)), e5m2x2_to_f16x2((uint16_t)(w0 >> 16)),
                       e5m2x2_to_f16x2((uint16_t)(w1 & 0xffff)), e5m2x2_to_f16x2((uint16_t)(w1 >> 16)));
    } else {
        r = make_uint4(e4m3x2_to_f16x2((uint16_t)(w0 & 0xffff)), e4m3x2_to_f16x2((uint16_t)(w0 >> 16)),
                       e4m3x2_to_f16x2((uint16_t)(w1 & 0xffff)), e4m3x2_to_f16x2((uint16_t)(w1 >> 16)));
    }
    return r;
}
// f16x2 -> two floats (exact)
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t v) {
    float lo, hi;
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
        : "=f"(lo), "=f"(hi)
        : "r"(v));
    return make_float2(lo, hi);
}
// Two bf16 (one word) -> f16x2, round to nearest even
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack2<true>(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// Output stores in the OutType of o; `e` is the element offset of the first element.
// Two adjacent elements (e even).
__device__ __forceinline__ void store_o2(uint8_t* o, size_t e, float a, float b, int odt) {
    if (odt == OT_F32) *reinterpret_cast<float2*>(o + e * 4) = make_float2(a, b);
    else if (odt == OT_F16) *reinterpret_cast<uint32_t*>(o + e * 2) = pack2<true>(a, b);
    else *reinterpret_cast<uint32_t*>(o + e * 2) = pack2<false>(a, b);
}
// Four consecutive elements (e a multiple of 4).
__device__ __forceinline__ void store_o4(uint8_t* o, size_t e, float a, float b, float c, float d, int odt) {
    if (odt == OT_F32) {
        *reinterpret_cast<float4*>(o + e * 4) = make_float4(a, b, c, d);
    } else if (odt == OT_F16) {
        *reinterpret_cast<uint2*>(o + e * 2) = make_uint2(pack2<true>(a, b), pack2<true>(c, d));
    } else {
        *reinterpret_cast<uint2*>(o + e * 2) = make_uint2(pack2<false>(a, b), pack2<false>(c, d));
    }
}
// Eight consecutive elements v[0..7] * s (e a multiple of 8).
__device__ __forceinline__ void store_o8(uint8_t* o, size_t e, const uint32_t* v, float s, int odt) {
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(v[i]) * s;
    if (odt == OT_F32) {
        *reinterpret_cast<float4*>(o + e * 4) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(o + e * 4 + 16) = make_float4(f[4], f[5], f[6], f[7]);
    } else if (odt == OT_F16) {
        *reinterpret_cast<uint4*>(o + e * 2) =
            make_uint4(pack2<true>(f[0], f[1]), pack2<true>(f[2], f[3]), pack2<true>(f[4], f[5]), pack2<true>(f[6], f[7]));
    } else {
        *reinterpret_cast<uint4*>(o + e * 2) = make_uint4(pack2<false>(f[0], f[1]), pack2<false>(f[2], f[3]),
                                                          pack2<false>(f[4], f[5]), pack2<false>(f[6], f[7]));
    }
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialisation attribute may start before its predecessor in the
// stream ends; it must call pdl_wait() before touching anything the
// predecessor writes.  pdl_trigger() lets the next kernel start early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ void set_status(int* ctrl, int code) {
    atomicCAS(ctrl + kStatus, 0, code);
}

// ---- mbarrier, bulk tensor copies, timer
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Potentially blocking test that suspends the thread for at most about `ns` nanoseconds.
__device__ __forceinline__ bool mbar_try_wait_for(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
// Non-blocking test: has the phase of `parity` completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}
// Wait for the phase of `parity` to complete, giving up after timeout_ns:
// then the status word gets RPA_ERR_TIMEOUT and false is returned.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* ctrl,
                                          uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > timeout_ns) {
            set_status(ctrl, RPA_ERR_TIMEOUT);
            return false;
        }
    }
}
// Wait for *flag (written by another kernel, released with a fence) to equal v, giving up after
// timeout_ns: then the status word gets RPA_ERR_TIMEOUT and false is returned.
__device__ __forceinline__ bool flag_wait(const int* flag, int v, int* ctrl, uint64_t timeout_ns) {
    const uint64_t t0 = global_ns();
    for (;;) {
        int x;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(x) : "l"(flag) : "memory");
        if (x == v) return true;
        if (global_ns() - t0 > timeout_ns) {
            set_status(ctrl, RPA_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(200);
    }
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// 2-D / 3-D tiled tensor copy global -> shared, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n" ::"r"(dst),
        "l"(map), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, uint32_t bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];\n" ::"r"(dst),
        "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// L2 cache policies for bulk copies: evict-first for data read once (streamed K/V), evict-last
// for data several CTAs re-read from L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
// 3-D tiled tensor copy global -> shared with an L2 cache policy.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* map, uint32_t bar, int x, int y, int z,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;\n" ::"r"(dst),
        "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* map, uint32_t bar, int x, int y,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;\n" ::"r"(dst),
        "l"(map), "r"(bar), "r"(x), "r"(y), "l"(pol)
        : "memory");
}

// ---- tcgen05 (5th-generation tensor cores, tensor memory)
// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator,
// A/B major-ness (0 = K-major, 1 = MN-major), N and M of the MMA.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Instruction descriptor, kind::f16 with f16 A and B (fp32 accumulator).
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], the B descriptor as its two 32-bit halves and a compile-time
// accumulate flag:
// an issuing thread that shares its sub-partition with busy warps gets few issue slots, so the
// per-MMA work is kept to an address add or two (the caller offsets the low half, which holds
// the start address, by a constant per MMA).
template <int ACC>
__device__ __forceinline__ void umma_ts_c(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                          uint32_t idesc) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 bd;\n setp.ne.b32 p, %5, 0;\n mov.b64 bd, {%2, %3};\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "n"(ACC)
        : "memory");
}
// D[tmem] (+)= A[smem] * B[smem] in the same lean form (descriptors as 32-bit halves)
template <int ACC>
__device__ __forceinline__ void umma_ss_c(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                          uint32_t idesc) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 ad, bd;\n setp.ne.b32 p, %6, 0;\n mov.b64 ad, {%1, %2};\n"
        " mov.b64 bd, {%3, %4};\n tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p;\n}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "n"(ACC)
        : "memory");
}
// arrive on an mbarrier once every tcgen05.mma issued so far by this thread completes
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
// 32 lanes x 32 columns of 32 bits: thread i gets lane (base + i), 32 consecutive columns
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
          "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
          "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
          "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
#endif

}  // namespace rpa
