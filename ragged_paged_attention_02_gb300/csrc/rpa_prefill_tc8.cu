// rpa_prefill_tc8.cu -- K1 prefill for 8-bit K/V (fp8 e4m3 / e5m2, int8) on the tcgen05 tensor cores.
//
// One persistent CTA per SM takes prefill work items of up to 128 query rows
// of one kv head (Tq = 128 / G tokens x the G query heads of the group, packed
// as the "ragged_paged.zig" page packs its q block into [Tq*G, D]) against a
// key range of one sequence, in tiles of 64 keys.  The page dequantises with
// k.astype(f32) * k_scale -> q dtype; here the 8-bit values (e4m3, e5m2 or
// int8) are converted exactly to f16, both MMAs run in f16 with fp32
// accumulation, k_scale is folded into the logit scale and v_scale into the
// epilogue.  Roles:
//
//   producer warp    Q tile (bf16) into a staging buffer, then per 64-key tile
//                    the raw 8-bit K/V rows of each page run (one bulk tensor
//                    copy per run: K and V of the head) into a ring of raw
//                    stages (2 at D 256, 4 at D 128, 8 at D 64).
//   8 converter      Q (warps on lane quadrants 0-3): bf16 -> f16 (f16 q as it
//   warps            is) into TMEM (the A operand of S = Q K^T).  K and V: each
//                    warp takes 8 key rows of a tile into registers (the
//                    ring slot goes straight back to the producer), then
//                    8-bit -> f16 into
//                    double-buffered, 128-byte swizzled tiles (K-major), keys
//                    outside the item's [kv_begin, kv_end) written as zero
//                    (the page zeroes K/V past kv_len; tail slots may hold any
//                    bits).
//   MMA warp         S = Q K^T (A from TMEM, B from smem) into one of two TMEM
//                    S buffers; O += P V (P from TMEM over S, V MN-major).
//   8 softmax warps  two per TMEM lane quadrant, one per half of the key tile:
//                    scale / softcap / masks in the log2 domain, running max
//                    and sum, P in f16, lazy O rescale (max grows by more than
//                    2^8), epilogue.  Items of at most 64 rows hold each query
//                    row in 2, 4 or 8 TMEM lanes that split the keys.
//
// 2-byte K/V (bf16 or f16) at D = 256 run on the same pipeline in direct mode:
// the producer copies K and V page runs straight into the 128-byte-swizzled
// tiles the MMAs read (one copy per K or V tile when a page run spans the
// 64 keys; K once the QK three tiles back is done, V once that tile's PV is
// done), the MMAs run in the K/V type (P in it too), and the
// converter warps only zero the V rows of keys outside [kv_begin, kv_end) on
// a tile's edges before signalling V ready (K rows there are masked in S).
//
// TMEM: Q (D/2 columns of packed 16-bit pairs, 64 at least), S0, S1 (64 each), O (D) --
// 512 columns at D = 256.  All waits are bounded; on expiry the status word
// gets RPA_ERR_TIMEOUT.
#include <cuda.h>

#include <type_traits>

#include "rpa_internal.cuh"

namespace rpa {

namespace {

constexpr int kM = kTcRows;   // query rows per tile = TMEM lanes
constexpr int kBN = kTc8Keys;  // keys per K/V tile
// warps 0-7 softmax (two per TMEM lane quadrant, one per half of the key tile), 8-15 convert
// (8 key rows of a tile each; 8-11 also convert Q, one TMEM lane quadrant each), 16 producer,
// 17 MMA
constexpr int kThreads = 576;
constexpr int kConv0 = 8, kNConv = 8, kProducer = 16, kMma = 17;
constexpr int kConvRows = kBN / kNConv;  // key rows of a tile per converter warp
// 5 warps share an SM sub-partition's 16384 registers: at most 96 a thread (launch bound 640)
constexpr int kRegBoundThreads = 640;
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kIssueNapNs = 100;  // longest suspension of the MMA thread's idle wait
constexpr int kMaxRaw = 8;             // raw 8-bit stages (the ring at D 64)

enum Meta8 : int { eSeq = 0, eHead, eQStart, eQl, eKl, eKvBegin, eKvEnd, eTok0, eNtok, eNt, eKey0, eStop, ePart };

template <int D, bool DIRECT>
struct G8 {
    static constexpr int CB = D / 64;                  // 128-byte column blocks of a 16-bit row
    static constexpr int ROUNDS = D / 64;              // Q staging rounds (one column block each)
    static constexpr int QSTAGE = kM * 128;            // Q staging: one column block x 128 rows
    static constexpr int RAW = DIRECT ? 0 : kBN * 2 * D;  // one raw 8-bit stage (K and V); none in direct mode
    static constexpr int T16 = CB * kBN * 128;         // one f16 K (or V) tile
    // Ring depths.  Direct mode: 3 K and 3 V tiles (the copies land in them, so a third buffer
    // starts each tile's copies a tile earlier).  8-bit mode: the raw stages hold the copies in
    // flight (2 at D 256; 4 at D 128 and 8 at D 64, the same bytes), then 2 K tiles (K(t)
    // converted once QK(t-2) is done) and 2 V tiles (V(t) once PV(t-2) is done).  A third raw
    // stage at D 256 (in place of a K tile) measured no faster: there the converter and softmax
    // warps, not the copies, set a tile's time
    static constexpr int NRAW = DIRECT ? 0 : 512 / D;
    static constexpr int NBK = DIRECT ? 3 : 2;
    static constexpr int NBV = DIRECT ? 3 : 2;
    static constexpr int DATA = QSTAGE + NRAW * RAW + (NBK + NBV) * T16;
    static constexpr int SMEM = DATA + 1024;
    // TMEM columns: Q (D/2 of packed 16-bit pairs, in a slot of at least 64), S0, S1, O (D)
    static constexpr uint32_t QC = D / 2 < 64 ? 64 : D / 2;
    static constexpr uint32_t TM_Q = 0;
    static constexpr uint32_t TM_S0 = QC, TM_S1 = QC + kBN;
    static constexpr uint32_t TM_O = QC + 2 * kBN;
    static_assert(QC + 2 * kBN + D <= kTmemCols, "TMEM budget");
    static_assert(NRAW <= kMaxRaw, "raw stage barriers");
    static_assert(DATA + 1024 + 4096 <= 227 * 1024, "shared memory budget (dynamic + static)");
};

__device__ __forceinline__ void put_u4(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// One converter warp's key rows (kConvRows cw .. + kConvRows - 1) of one half (K or V) of a raw
// stage ([run][K | V][BR rows][D bytes]; `raw` points at the half's first run): a lane takes 16
// consecutive bytes of a row (D / 16 lanes a row, RPP rows a pass, NP passes).
template <int D>
struct ConvLanes {
    static constexpr int LPR = D / 16, RPP = 32 / LPR, NP = kConvRows / RPP;
};
template <int D>
__device__ __forceinline__ void load_rows(const uint8_t* raw, int cw, int lane, int brs, uint4* v) {
    using C = ConvLanes<D>;
    const int BR = 1 << brs;
    const int e = lane % C::LPR, r0 = lane / C::LPR;
#pragma unroll
    for (int i = 0; i < C::NP; ++i) {
        const int key = kConvRows * cw + r0 + i * C::RPP;
        v[i] = *reinterpret_cast<const uint4*>(raw + (key >> brs) * (2 * BR * D) + (key & (BR - 1)) * D + e * 16);
    }
}
// ... and those rows, converted exactly to f16, into a 128-byte swizzled tile [D / 64][64 rows]
// [128 B]; keys outside [kv_begin, kv_end) become zero.
template <int D, int KT>
__device__ __forceinline__ void store_rows(const uint4* v, uint8_t* dst, int cw, int lane, int k_lo, int kv_begin,
                                           int kv_end) {
    using C = ConvLanes<D>;
    const int e = lane % C::LPR, r0 = lane / C::LPR;
    // the 16 elements are f16 chunks 2e, 2e+1 of column block e / 4; lanes of odd (e / 4) store
    // their second chunk first so that each store of 8 lanes covers all 32 banks
    const bool sw = (e >> 2) & 1;
    const int cb = e >> 2, c0 = (2 * e) & 7;
#pragma unroll
    for (int i = 0; i < C::NP; ++i) {
        const int key = kConvRows * cw + r0 + i * C::RPP;
        const int j = k_lo + key;
        const uint32_t a0 = sw ? v[i].z : v[i].x, a1 = sw ? v[i].w : v[i].y;
        const uint32_t b0 = sw ? v[i].x : v[i].z, b1 = sw ? v[i].y : v[i].w;
        uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
        if (j >= kv_begin && j < kv_end) {
            o0 = cvt8x8_to_f16x8<KT>(a0, a1);
            o1 = cvt8x8_to_f16x8<KT>(b0, b1);
        }
        const int line = cb * kBN + key;
        uint8_t* row = dst + line * 128;
        put_u4(row + ((((c0 + (sw ? 1 : 0)) ^ line) & 7) << 4), o0);
        put_u4(row + ((((c0 + (sw ? 0 : 1)) ^ line) & 7) << 4), o1);
    }
}

// Logits of N keys of a row in the log2 domain, in place: scale (or soft cap), then keys
// outside [lo, hi] (relative to the first) to -inf; returns their max.
template <bool CAP, bool MASK, int N>
__device__ __forceinline__ float tile_logits(uint32_t* sv, float qk, float capl, float capt, int lo, int hi) {
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    const uint64_t qk2 = f32x2(qk, qk), capl2 = f32x2(capl, capl), capt2 = f32x2(capt, capt);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        uint64_t v2 = f32x2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
        float v0, v1;
        if constexpr (CAP) {
            // cap * tanh(x / cap), log2 domain
            f32x2_split(fmul2(v2, capt2), v0, v1);
            f32x2_split(fmul2(f32x2(tanh_approx(v0), tanh_approx(v1)), capl2), v0, v1);
        } else {
            f32x2_split(fmul2(v2, qk2), v0, v1);
        }
        if constexpr (MASK) {
            v0 = (i >= lo && i <= hi) ? v0 : -INFINITY;
            v1 = (i + 1 >= lo && i + 1 <= hi) ? v1 : -INFINITY;
        }
        m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], v0, v1);
        sv[i] = __float_as_uint(v0);
        sv[i + 1] = __float_as_uint(v1);
    }
    return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// Copies of each query row in a 128-row tile (a power of two; see the softmax warps)
__device__ __forceinline__ int row_copies(int rows) { return rows <= 16 ? 8 : rows <= 32 ? 4 : rows <= 64 ? 2 : 1; }

// The N = 32 / F logits of copy c among a lane's 32: kv[i] = sv[c N + i]
template <int F>
__device__ __forceinline__ void pick_keys(const uint32_t* sv, int c, uint32_t* kv) {
    constexpr int N = 32 / F;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        uint32_t x = sv[i];
#pragma unroll
        for (int k = 1; k < F; ++k) x = c == k ? sv[k * N + i] : x;
        kv[i] = x;
    }
}

// Sum of a row's copies (lanes l, l ^ R, l ^ 2R, ...) of 32 O columns, in every lane
__device__ __forceinline__ void add_copies(uint32_t* ov, int R) {
    for (int x = R; x < 32; x <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            ov[i] = __float_as_uint(__uint_as_float(ov[i]) + __uint_as_float(__shfl_xor_sync(0xffffffffu, ov[i], x)));
    }
}

template <int D, int KT>
__global__ void __launch_bounds__(kRegBoundThreads, 1) rpa_prefill_tc8(const __grid_constant__ CUtensorMap kvmap,
                                                               const __grid_constant__ CUtensorMap qmap,
                                                               const TcParams p) {
    // DIRECT: 2-byte K/V copied straight into the MMA tiles (kvmap, 128-byte swizzle: the slot x
    // head-row x column-block map when BR = kBN, else the slot x row map); else 8-bit page runs
    // through the raw ring (kvmap: the page-run map)
    constexpr bool DIRECT = !kt_8bit(KT);
    constexpr bool F16 = kt_f16_mma(KT);  // MMA operands (and P) in f16, else bf16
    using Gm = G8<D, DIRECT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t meta_full[2], meta_free[2];
    __shared__ __align__(8) uint64_t q_full, q_empty, q_ready, qt_free;
    __shared__ __align__(8) uint64_t raw_full[kMaxRaw], raw_empty[kMaxRaw];
    // per S buffer (t mod 2): QK done, P ready (softmax warps; in 8-bit mode also V converted: the
    // converter warps), PV done; per K/V buffer (t mod NB): K ready, and in direct mode V copied, V
    // ready (its edge rows zeroed: converter warps) and the K / V buffer free again (the MMAs that
    // read it are done).  Direct mode keeps V ready apart from P ready: V(t + 2) can be ready before
    // P(t), and each barrier's arrivals must come from one tile at a time.
    __shared__ __align__(8) uint64_t qk_done[2], pv_ready[2], pv_done[2];
    __shared__ __align__(8) uint64_t k_full[3], v_land[3], v_ready[3], k_free[3], v_free[3];
    __shared__ __align__(8) uint64_t o_full, o_free;
    __shared__ __align__(8) uint64_t xchg[4];  // per lane quadrant: the two softmax warps' row maxima / sums
    __shared__ float xm[2][2][kM];             // [tile parity][key half][row] partial row maxima
    __shared__ float xl[2][kM];                // [key half][row] partial row sums
    __shared__ uint32_t tmem_base_sh;
    __shared__ int meta[2][16];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const AttnParams& a = p.a;
    int* ctrl = a.ctrl;
    const uint64_t tmo = p.timeout_ns;
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t q_stage = smem0;                                 // Q staging (bf16)
    const uint32_t raw_base = q_stage + Gm::QSTAGE;                 // NRAW raw 8-bit stages
    const uint32_t k16_base = raw_base + Gm::NRAW * Gm::RAW;        // NBK 16-bit K tiles
    const uint32_t v16_base = k16_base + Gm::NBK * Gm::T16;         // NBV 16-bit V tiles
    // K (V) buffer of global tile g and the parity of its use of that buffer
    auto kbuf = [](uint32_t g) -> int { return (int)(g % (uint32_t)Gm::NBK); };
    auto kpar = [](uint32_t g) -> uint32_t { return (g / (uint32_t)Gm::NBK) & 1u; };
    auto vbuf = [](uint32_t g) -> int { return (int)(g % (uint32_t)Gm::NBV); };
    auto vpar = [](uint32_t g) -> uint32_t { return (g / (uint32_t)Gm::NBV) & 1u; };

    if (tid == 0) {
        for (int i = 0; i < Gm::NRAW; ++i) {
            mbar_init(smem_u32(&raw_full[i]), 1);
            mbar_init(smem_u32(&raw_empty[i]), kNConv);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&meta_full[i]), 1);
            mbar_init(smem_u32(&meta_free[i]), 17);  // 8 softmax + 8 converter warps + MMA thread
            mbar_init(smem_u32(&qk_done[i]), 1);
            mbar_init(smem_u32(&pv_ready[i]), DIRECT ? 8 : 8 + kNConv);
            mbar_init(smem_u32(&pv_done[i]), 1);
        }
        for (int i = 0; i < 3; ++i) {
            // K(t) ready: the converters' arrivals, or in direct mode the copies themselves
            mbar_init(smem_u32(&k_full[i]), DIRECT ? 1 : kNConv);
            mbar_init(smem_u32(&v_land[i]), 1);
            mbar_init(smem_u32(&v_ready[i]), kNConv);
            mbar_init(smem_u32(&k_free[i]), 1);
            mbar_init(smem_u32(&v_free[i]), 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&xchg[i]), 2);  // one arrival per softmax warp
        mbar_init(smem_u32(&q_full), 1);
        mbar_init(smem_u32(&q_empty), 4);
        mbar_init(smem_u32(&q_ready), 4);
        mbar_init(smem_u32(&qt_free), 1);
        mbar_init(smem_u32(&o_full), 1);
        mbar_init(smem_u32(&o_free), 8);
        fence_mbar_init();
    }
    if (warp == kMma) tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    pdl_trigger();
    pdl_wait();  // the planner's items are complete from here on
    const int n_items = a.ctrl[a.item_count_word];
    const bool active = (int)blockIdx.x < a.ctrl[kPfCtas];

    if (!active) {
    } else if (warp == kProducer) {
        // =============================== producer ===============================
        const int BR = p.BR, ps = a.ps, G = a.G, Tq = p.Tq;
        const int runs = kBN / BR;
        const uint32_t run_bytes = (uint32_t)(2 * BR * D);
        const uint32_t q_round_bytes = (uint32_t)(G * Tq * 128);
        int s = 0, ms = 0;
        uint32_t ph = 0, mph = 0, qph = 0;
        uint32_t tgp = 0;  // direct mode: tiles copied so far (all items): tile buffer and phase
        bool ok = true;
        int it = 0;
        if (lane == 0) it = atomicAdd(ctrl + a.counter_word, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        for (;;) {
            if (!mbar_wait(smem_u32(&meta_free[ms]), mph ^ 1u, ctrl, tmo)) break;
            if (it >= n_items) {
                if (lane == 0) {
                    meta[ms][eStop] = 1;
                    mbar_arrive(smem_u32(&meta_full[ms]));
                }
                break;
            }
            const Item item = item_at(a.units, it, a.unit_heads);
            int nxt = 0;
            if (lane == 0) nxt = atomicAdd(ctrl + a.counter_word, 1);
            const int q_start = a.cu_q_lens[item.seq];
            const int ql = a.cu_q_lens[item.seq + 1] - q_start;
            const int kl = a.kv_lens[item.seq];
            const int* ptab = a.page_indices + (size_t)item.seq * a.P;
            const int key0 = item.kv_begin - (item.kv_begin & (BR - 1));
            const int nt = (item.kv_end - key0 + kBN - 1) / kBN;
            if (lane == 0) {
                int* m = meta[ms];
                m[eSeq] = item.seq;
                m[eHead] = item.head;
                m[eQStart] = q_start;
                m[eQl] = ql;
                m[eKl] = kl;
                m[eKvBegin] = item.kv_begin;
                m[eKvEnd] = item.kv_end;
                m[eTok0] = item.tok0;
                m[eNtok] = item.ntok;
                m[eNt] = nt;
                m[eKey0] = key0;
                m[ePart] = item.part;
                m[eStop] = 0;
                mbar_arrive(smem_u32(&meta_full[ms]));
            }
            if (++ms == 2) {
                ms = 0;
                mph ^= 1u;
            }
            // Q: one column block per round through the staging buffer
            for (int rd = 0; rd < Gm::ROUNDS && ok; ++rd) {
                if (!mbar_wait(smem_u32(&q_empty), qph ^ 1u, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                const uint32_t qfb = smem_u32(&q_full);
                if (lane == 0) mbar_arrive_expect_tx(qfb, q_round_bytes);
                __syncwarp();
                if (lane == 0)
                    tma_load_3d(q_stage, &qmap, qfb, rd * 64, item.head * G,
                                q_start + item.tok0);
                qph ^= 1u;
            }
            int win0 = key0 / ps;
            int win = (win0 + lane < a.P) ? __ldg(ptab + win0 + lane) : 0;
            for (int t = 0; t < nt && ok; ++t) {
                const int k_tile = key0 + t * kBN;
                const int lp_last = min(k_tile + kBN - 1, item.kv_end - 1) / ps;
                if (lp_last - win0 >= 32) {
                    win0 = k_tile / ps;
                    win = (win0 + lane < a.P) ? __ldg(ptab + win0 + lane) : 0;
                }
                if constexpr (DIRECT) {
                    // K(t) into K buffer b once QK(t-3) is done, V(t) into V buffer b once PV(t-3) is
                    // done: with runs of a whole tile one copy of all column blocks (kvmap from
                    // encode_kv_map_heads: K of head h is row 2h of a slot, V row 2h + 1), else one
                    // copy per (page run, 128-byte column block), BR rows each
                    static_assert(Gm::NBK == Gm::NBV, "direct mode: K and V rings alike");
                    const int b2 = kbuf(tgp);
                    const uint32_t par = kpar(tgp);
                    ++tgp;
                    const int tasks = runs * Gm::CB;
#pragma unroll 1
                    for (int kv = 0; kv < 2 && ok; ++kv) {
                        if (!mbar_wait(smem_u32(kv ? &v_free[b2] : &k_free[b2]), par ^ 1u, ctrl, tmo)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst0 = (kv ? v16_base : k16_base) + b2 * Gm::T16;
                        if (BR == kBN) {
                            const int lp = k_tile / ps;
                            const int pg = __shfl_sync(0xffffffffu, win, (lp - win0) & 31);
                            const bool want = k_tile < item.kv_end && k_tile + BR > item.kv_begin;
                            const bool good = (unsigned)pg < (unsigned)a.N;
                            const uint32_t fb = smem_u32(kv ? &v_land[b2] : &k_full[b2]);
                            if (lane == 0) {
                                if (want && !good) set_status(ctrl, RPA_ERR_BAD_PAGE_INDEX);
                                mbar_arrive_expect_tx(fb, (want && good) ? (uint32_t)(kBN * D * 2) : 0u);
                                if (want && good)
                                    tma_load_3d(dst0, &kvmap, fb, 0, pg * ps + (k_tile - lp * ps),
                                                (2 * item.head + kv) * Gm::CB);
                            }
                            __syncwarp();
                            continue;
                        }
                        auto task = [&](int tk, int& x, int& y, uint32_t& dst) -> int {
                            const int b = tk / Gm::CB, cb = tk % Gm::CB;
                            const int k0 = k_tile + b * BR;
                            const int lp = k0 / ps;
                            const int pg = __shfl_sync(0xffffffffu, win, (lp - win0) & 31);
                            if (tk >= tasks || k0 >= item.kv_end || k0 + BR <= item.kv_begin) return 0;
                            if ((unsigned)pg >= (unsigned)a.N) return 2;
                            x = (2 * item.head + kv) * D + cb * 64;
                            y = pg * ps + (k0 - lp * ps);
                            dst = dst0 + (uint32_t)(cb * (kBN * 128) + b * BR * 128);
                            return 1;
                        };
                        int n_mine = 0, bad = 0;
                        for (int t0 = 0; t0 < tasks; t0 += 32) {
                            int x, y;
                            uint32_t dst;
                            const int r = task(t0 + lane, x, y, dst);
                            n_mine += r == 1;
                            bad |= r == 2;
                        }
                        const int n_issue = __reduce_add_sync(0xffffffffu, n_mine);
                        if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(ctrl, RPA_ERR_BAD_PAGE_INDEX);
                        const uint32_t fb = smem_u32(kv ? &v_land[b2] : &k_full[b2]);
                        if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)n_issue * (uint32_t)BR * 128u);
                        __syncwarp();
                        for (int t0 = 0; t0 < tasks; t0 += 32) {
                            int x, y;
                            uint32_t dst;
                            if (task(t0 + lane, x, y, dst) == 1) tma_load_2d(dst, &kvmap, fb, x, y);
                        }
                    }
                    continue;
                }
                if (!mbar_wait(smem_u32(&raw_empty[s]), ph ^ 1u, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                const uint32_t stage = raw_base + s * Gm::RAW;
                const int k0 = k_tile + lane * BR;
                const int lp = k0 / ps;
                const int pg = __shfl_sync(0xffffffffu, win, (lp - win0) & 31);
                const bool want = lane < runs && k0 < item.kv_end && k0 + BR > item.kv_begin;
                const bool good = (unsigned)pg < (unsigned)a.N;
                const int n_issue = __popc(__ballot_sync(0xffffffffu, want && good));
                if (__any_sync(0xffffffffu, want && !good) && lane == 0) set_status(ctrl, RPA_ERR_BAD_PAGE_INDEX);
                const uint32_t fb = smem_u32(&raw_full[s]);
                if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)n_issue * run_bytes);
                __syncwarp();
                if (want && good)
                    tma_load_3d(stage + (uint32_t)lane * run_bytes, &kvmap, fb, 0, pg * ps + (k0 - lp * ps),
                                2 * item.head);
                if (++s == Gm::NRAW) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            it = __shfl_sync(0xffffffffu, nxt, 0);
        }
    } else if (warp >= kConv0 && warp < kConv0 + kNConv) {
        // =============================== converters ===============================
        const int cw = warp - kConv0;  // converter warp 0..7; 0..3 also convert Q
        const bool qconv = cw < 4;     // its TMEM lane quadrant is cw (warp % 4)
        const uint32_t lane_addr = tmem + ((uint32_t)((cw & 3) * 32) << 16);
        const int BR = p.BR, brs = __ffs(BR) - 1;
        int s = 0, ms = 0;
        uint32_t ph = 0, mph = 0, qph = 0;
        uint32_t tg = 0, items = 0;  // tiles (all items) and items converted
        for (;;) {
            if (!mbar_wait(smem_u32(&meta_full[ms]), mph, ctrl, tmo)) break;
            const int* mm = meta[ms];
            const int stop = mm[eStop], kv_begin = mm[eKvBegin], kv_end = mm[eKvEnd], nt = mm[eNt],
                      key0 = mm[eKey0], ntok = mm[eNtok];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&meta_free[ms]));
            if (stop) break;
            if (++ms == 2) {
                ms = 0;
                mph ^= 1u;
            }
            // ---- Q: bf16 staging -> f16 TMEM columns; TMEM lane (cw & 3) 32 + lane holds query
            // row (cw & 3) R + lane % R (R = 32 / copies of each row)
            const int R = 32 / row_copies(ntok * a.G);
            const int r = (cw & 3) * R + lane % R;
            if (qconv && items > 0 && !mbar_wait(smem_u32(&qt_free), (items - 1) & 1u, ctrl, tmo)) break;
            bool ok = true;
            for (int rd = 0; rd < (qconv ? Gm::ROUNDS : 0); ++rd) {
                if (!mbar_wait(smem_u32(&q_full), qph, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                qph ^= 1u;
                {
                    uint32_t qv[32];
                    const uint8_t* row = smem + (q_stage - smem0) + r * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 w = *reinterpret_cast<const uint4*>(row + (((c ^ r) & 7) << 4));
                        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            qv[4 * c + k] = (DIRECT || a.q_f16) ? ws[k] : bf16x2_to_f16x2(ws[k]);
                    }
                    tmem_st32(lane_addr + Gm::TM_Q + rd * 32, qv);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&q_empty));
            }
            if (!ok) break;
            if (qconv) {
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&q_ready));
            }
            // ---- K / V tiles: this warp converts keys [kConvRows cw, kConvRows (cw + 1)) of each tile
            for (int t = 0; t < nt; ++t, ++tg) {
                const int b2 = tg & 1;
                const uint32_t par = (tg >> 1) & 1u;
                if constexpr (DIRECT) {
                    // the copies wrote V(t) into its tile: on the tile's edges, zero this warp's rows of
                    // keys outside [kv_begin, kv_end) (page tails may hold any bits; runs outside the
                    // range were not copied), then V is ready
                    const int vb = vbuf(tg);
                    if (!mbar_wait(smem_u32(&v_land[vb]), vpar(tg), ctrl, tmo)) {
                        ok = false;
                        break;
                    }
                    const int k_lo = key0 + t * kBN;
                    if (k_lo < kv_begin || k_lo + kBN > kv_end) {
                        uint8_t* vt = smem + (v16_base - smem0) + vb * Gm::T16;
                        for (int i = lane; i < kConvRows * Gm::CB * 8; i += 32) {
                            const int key = kConvRows * cw + i / (Gm::CB * 8);
                            const int rem = i % (Gm::CB * 8);
                            const int j = k_lo + key;
                            if (j >= kv_begin && j < kv_end) continue;
                            put_u4(vt + ((rem >> 3) * kBN + key) * 128 + (rem & 7) * 16, make_uint4(0, 0, 0, 0));
                        }
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&v_ready[vb]));
                    continue;
                }
                if (!mbar_wait(smem_u32(&raw_full[s]), ph, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                // the warp's K and V rows of the stage into registers, and the stage straight back
                // to the producer: the next copy starts while this tile is being converted
                const uint8_t* raw = smem + (raw_base - smem0) + s * Gm::RAW;
                uint4 kr[ConvLanes<D>::NP], vr[ConvLanes<D>::NP];
                load_rows<D>(raw, cw, lane, brs, kr);
                load_rows<D>(raw + BR * D, cw, lane, brs, vr);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&raw_empty[s]));
                if (++s == Gm::NRAW) {
                    s = 0;
                    ph ^= 1u;
                }
                const int k_lo = key0 + t * kBN;
                // K, then V, both converted exactly by the hardware conversion: K(t) into its buffer
                // once QK(t - NBK), the buffer's last reader, is done
                if (tg >= (uint32_t)Gm::NBK) {
                    const uint32_t gk = tg - Gm::NBK;
                    if (!mbar_wait(smem_u32(&qk_done[gk & 1]), (gk >> 1) & 1u, ctrl, tmo)) {
                        ok = false;
                        break;
                    }
                }
                const int kb = kbuf(tg);
                store_rows<D, KT>(kr, smem + (k16_base - smem0) + kb * Gm::T16, cw, lane, k_lo, kv_begin, kv_end);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&k_full[kb]));
                if (!mbar_wait(smem_u32(&pv_done[b2]), par ^ 1u, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                store_rows<D, KT>(vr, smem + (v16_base - smem0) + b2 * Gm::T16, cw, lane, k_lo, kv_begin, kv_end);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&pv_ready[b2]));
            }
            if (!ok) break;
            ++items;
        }
    } else if (warp == kMma) {
        // =============================== MMA issuer ===============================
        if (lane == 0) {
            constexpr uint32_t idesc_qk = F16 ? umma_idesc_f16(kM, kBN, 0, 0) : umma_idesc_bf16(kM, kBN, 0, 0);
            constexpr uint32_t idesc_pv = F16 ? umma_idesc_f16(kM, D, 0, 1) : umma_idesc_bf16(kM, D, 0, 1);
            int ms = 0;
            uint32_t mph = 0;
            uint32_t tg = 0, items = 0;
            bool ok = true;
            // Per item, QK(t) and PV(t) are issued as soon as their inputs are ready, in either
            // order: QK(t) needs K(t) converted and PV(t-2) issued (it overwrites S(t % 2), which
            // PV(t-2) reads; the tensor pipe runs in issue order); PV(t) needs P(t), V(t) and, for
            // the item's first PV, the previous epilogue done with O.  Readiness is tested without
            // blocking; when nothing is ready the thread naps briefly on a pending barrier, and a
            // thread that sees nothing ready for longer than the wait bound gives up.  Every
            // barrier test and commit costs this thread tens of cycles in series with the tensor
            // pipe, so each MMA group uses one readiness barrier and one commit.
            for (;;) {
                if (!mbar_wait(smem_u32(&meta_full[ms]), mph, ctrl, tmo)) break;
                const int stop = meta[ms][eStop], nt = meta[ms][eNt];
                mbar_arrive(smem_u32(&meta_free[ms]));
                if (stop) break;
                if (++ms == 2) {
                    ms = 0;
                    mph ^= 1u;
                }
                if (!mbar_wait(smem_u32(&q_ready), items & 1u, ctrl, tmo)) break;
                tc_fence_after();
                int tq = 0, tp = 0;  // next QK and next PV of this item
                uint64_t t_idle = 0;
                int idle = 0;
                while (tp < nt) {
                    bool did = false;
                    if (tq < nt && tq <= tp + 1) {
                        const uint32_t g = tg + tq;
                        const int b2 = g & 1, kb = kbuf(g);
                        if (mbar_test(smem_u32(&k_full[kb]), kpar(g))) {
                            tc_fence_after();
                            const uint64_t kd = umma_sdesc(k16_base + kb * Gm::T16, 16, 1024);
                            const uint32_t kd_lo = (uint32_t)kd, kd_hi = (uint32_t)(kd >> 32);
                            const uint32_t sd = tmem + (b2 ? Gm::TM_S1 : Gm::TM_S0), qa = tmem + Gm::TM_Q;
                            umma_ts_c<0>(sd, qa, kd_lo, kd_hi, idesc_qk);
#pragma unroll
                            for (int kk = 1; kk < D / 16; ++kk)
                                umma_ts_c<1>(sd, qa + kk * 8, kd_lo + ((kk >> 2) * (kBN * 128) + (kk & 3) * 32) / 16, kd_hi,
                                             idesc_qk);
                            umma_commit(smem_u32(&qk_done[b2]));
                            if constexpr (DIRECT) umma_commit(smem_u32(&k_free[kb]));
                            if (tq == nt - 1) umma_commit(smem_u32(&qt_free));
                            ++tq;
                            did = true;
                        }
                    }
                    if (tp < tq) {
                        const uint32_t g = tg + tp;
                        const int b2 = g & 1;
                        const uint32_t par = (g >> 1) & 1u;
                        const bool first = tp == 0;
                        if (mbar_test(smem_u32(&pv_ready[b2]), par) &&
                            (!DIRECT || mbar_test(smem_u32(&v_ready[vbuf(g)]), vpar(g))) &&
                            (!first || items == 0 || mbar_test(smem_u32(&o_free), (items - 1) & 1u))) {
                            tc_fence_after();
                            const int vb = vbuf(g);
                            const uint64_t vd = umma_sdesc(v16_base + vb * Gm::T16, kBN * 128, 1024);
                            const uint32_t vd_lo = (uint32_t)vd, vd_hi = (uint32_t)(vd >> 32);
                            const uint32_t od = tmem + Gm::TM_O, pa = tmem + (b2 ? Gm::TM_S1 : Gm::TM_S0);
                            if (first)
                                umma_ts_c<0>(od, pa, vd_lo, vd_hi, idesc_pv);
                            else
                                umma_ts_c<1>(od, pa, vd_lo, vd_hi, idesc_pv);
#pragma unroll
                            for (int kk = 1; kk < kBN / 16; ++kk)
                                umma_ts_c<1>(od, pa + kk * 8, vd_lo + kk * 16 * 128 / 16, vd_hi, idesc_pv);
                            umma_commit(smem_u32(&pv_done[b2]));
                            if constexpr (DIRECT) umma_commit(smem_u32(&v_free[vb]));
                            ++tp;
                            did = true;
                        }
                    }
                    if (did) {
                        idle = 0;
                        t_idle = 0;
                        continue;
                    }
                    // nothing ready: sleep briefly on a barrier the next PV or QK waits for (the two
                    // in turn when both wait), which leaves the sub-partition's issue slots to the
                    // softmax and converter warps
                    {
                        const uint32_t gp = tg + tp, gq = tg + tq;
                        const uint32_t pp = (gp >> 1) & 1u;
                        const bool qk_next = tq < nt && tq <= tp + 1 && (tp >= tq || (idle & 1));
                        if (qk_next)
                            mbar_try_wait_for(smem_u32(&k_full[kbuf(gq)]), kpar(gq), kIssueNapNs);
                        else if (tp < tq)
                            mbar_try_wait_for(smem_u32(&pv_ready[gp & 1]), pp, kIssueNapNs);
                    }
                    if (++idle >= 4) {
                        idle = 0;
                        const uint64_t now = global_ns();
                        if (t_idle == 0) {
                            t_idle = now;
                        } else if (now - t_idle > tmo) {
                            set_status(ctrl, RPA_ERR_TIMEOUT);
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok) break;
                tg += nt;
                umma_commit(smem_u32(&o_full));
                ++items;
            }
        }
        __syncwarp();
    } else {
        // =============================== softmax warps ===============================
        // warp w serves TMEM lanes 32 (w % 4) .. + 31 and key half w / 4 of every tile (32
        // logits a lane); the two warps of a quadrant exchange row maxima every tile and row sums
        // at the item's end through shared memory and the quadrant's xchg barrier.
        // Row copies: an item of at most 64 (32, 16) rows holds each query row in F = 2 (4, 8)
        // lanes of a quadrant (lane l: row q R + l % R, copy c = l / R, R = 32 / F; the Q
        // converters place them so).  Copy c takes keys c n .. c n + n - 1 (n = 32 / F) of the
        // warp's half and leaves P zero in the others, so that each copy's O row sums its own keys;
        // the epilogue adds the copies (lanes l ^ R, l ^ 2R, ...).  The tensor pipe computes 128
        // rows whatever the item's count: copies turn rows that would idle into a split of the
        // exponentials across all four sub-partitions.
        const int q4 = warp & 3, half = warp >> 2;
        const int L = q4 * 32 + lane;  // TMEM lane
        const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t xb = smem_u32(&xchg[q4]);
        constexpr int HC = kBN / 2;  // logits of a lane's row in this warp's half of a tile
        constexpr int HO = D / 2;    // O columns this warp owns
        const int G = a.G, Hq = a.Hq;
        // K and V tiles hold the exact 8-bit values (the scales act on the logits and the output).
        // Soft cap: cap log2(e) tanh(s sm_scale k_scale / cap) with the hardware tanh (relative
        // error about 2^-11, the order of the f16 rounding of P); its argument factor is
        // cap_exp / (2 log2(e)).
        const float qk = a.qk_log2, capl = a.cap_log2, cape = a.cap_exp * (0.5f / 1.4426950408889634f);
        int ms = 0;
        uint32_t mph = 0, tg = 0, items = 0, xph = 0;
        for (;;) {
            if (!mbar_wait(smem_u32(&meta_full[ms]), mph, ctrl, tmo)) break;
            const int* mm = meta[ms];
            const int stop = mm[eStop];
            const int head = mm[eHead], q_start = mm[eQStart], ql = mm[eQl], kl = mm[eKl];
            const int kv_begin = mm[eKvBegin], kv_end = mm[eKvEnd], tok0 = mm[eTok0];
            const int ntok = mm[eNtok], nt = mm[eNt], key0 = mm[eKey0], part = mm[ePart];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&meta_free[ms]));
            if (stop) break;
            if (++ms == 2) {
                ms = 0;
                mph ^= 1u;
            }
            const int rows_used = ntok * G;
            const int R = 32 / row_copies(rows_used);
            const int c = lane / R;           // copy
            const int r = q4 * R + lane % R;  // query row
            const int pos = kl - ql + tok0 + r / G;
            const int pos_lo = kl - ql + tok0, pos_hi = kl - ql + tok0 + ntok - 1;
            // a quadrant whose rows are all past the item's rows computes nothing: its P and O
            // rows are never stored (it still takes part in the barriers, in order)
            const bool idle = q4 * R >= rows_used;
            float m_run = -INFINITY, l_run = 0.f;
            // the item's tiles with F copies of each row (n = 32 / F logits a lane)
            auto run_tiles = [&](auto fc) -> bool {
                constexpr int F = decltype(fc)::value, NK = HC / F;
                for (int t = 0; t < nt; ++t, ++tg) {
                    const int b2 = tg & 1;
                    if (!mbar_wait(smem_u32(&qk_done[b2]), (tg >> 1) & 1u, ctrl, tmo)) return false;
                    tc_fence_after();
                    if (idle) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&pv_ready[b2]));
                        continue;
                    }
                    const int k_lo = key0 + t * kBN;
                    const bool partial = k_lo < kv_begin || k_lo + kBN > kv_end;
                    const bool need_mask = partial || (a.causal && k_lo + kBN - 1 > pos_lo) ||
                                           (a.has_window && k_lo <= pos_hi - a.window);
                    const uint32_t scol = (b2 ? Gm::TM_S1 : Gm::TM_S0) + half * HC;
                    // this half's 32 logits of the lane's row, then the copy's NK of them
                    uint32_t sv[HC];
                    tmem_ld32(lane_addr + scol, sv);
                    tmem_ld_wait();
                    uint32_t kv[NK];
                    pick_keys<F>(sv, c, kv);
                    float mh;
                    if (need_mask) {
                        // keys allowed for this row: [lo, hi] relative to the copy's first key
                        int lo = kv_begin, hi = kv_end - 1;
                        if (a.has_window) lo = max(lo, pos - a.window + 1);
                        if (a.causal) hi = min(hi, pos);
                        const int k_first = k_lo + half * HC + c * NK;
                        lo -= k_first;
                        hi -= k_first;
                        mh = a.has_cap ? tile_logits<true, true, NK>(kv, qk, capl, cape, lo, hi)
                                       : tile_logits<false, true, NK>(kv, qk, capl, cape, lo, hi);
                    } else {
                        mh = a.has_cap ? tile_logits<true, false, NK>(kv, qk, capl, cape, 0, 0)
                                       : tile_logits<false, false, NK>(kv, qk, capl, cape, 0, 0);
                    }
                    // row max over the copies, then over both halves
#pragma unroll
                    for (int x = 32 / F; x < 32; x <<= 1) mh = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, x));
                    xm[tg & 1][half][L] = mh;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xb);
                    if (!mbar_wait(xb, xph, ctrl, tmo)) return false;
                    xph ^= 1u;
                    const float mt = fmaxf(mh, xm[tg & 1][half ^ 1][L]);
                    const bool need = __any_sync(0xffffffffu, mt > m_run + kRescaleLog2);
                    const float m_new = need ? fmaxf(m_run, mt) : m_run;
                    const float alpha = !need ? 1.f : (m_run == -INFINITY ? 0.f : ex2(m_run - m_new));
                    const float base = m_new == -INFINITY ? 0.f : m_new;
                    // P = 2^(x - base) in f16; x - base and the running sums on pairs (f32x2)
                    const uint64_t nbase2 = f32x2(-base, -base);
                    uint64_t ls2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
                    uint32_t own[NK / 2];
#pragma unroll
                    for (int i = 0; i < NK / 2; ++i) {
                        float x0, x1;
                        f32x2_split(fadd2(f32x2(__uint_as_float(kv[2 * i]), __uint_as_float(kv[2 * i + 1])), nbase2),
                                    x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        ls2[i & 1] = fadd2(ls2[i & 1], f32x2(p0, p1));
                        own[i] = pack2<F16>(p0, p1);
                    }
                    // the half's 16 P columns (P[i] at column i / 2): the copy's own, zero elsewhere
                    uint32_t pk[HC / 2];
#pragma unroll
                    for (int k = 0; k < HC / 2; ++k) pk[k] = (F == 1 || k / (NK / 2) == c) ? own[k % (NK / 2)] : 0u;
                    tmem_st16(lane_addr + (b2 ? Gm::TM_S1 : Gm::TM_S0) + half * (HC / 2), pk);
                    float la, lb, lc, ld;
                    f32x2_split(ls2[0], la, lb);
                    f32x2_split(ls2[1], lc, ld);
                    l_run = l_run * alpha + ((la + lb) + (lc + ld));
                    m_run = m_new;
                    if (need && t > 0) {
                        // this warp's half of the O row holds the item's PVs up to tile t-1
                        if (!mbar_wait(smem_u32(&pv_done[(tg - 1) & 1]), ((tg - 1) >> 1) & 1u, ctrl, tmo)) return false;
                        tc_fence_after();
#pragma unroll 1
                        for (int cc = 0; cc < HO / 32; ++cc) {
                            uint32_t ov[32];
                            tmem_ld32(lane_addr + Gm::TM_O + half * HO + cc * 32, ov);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                            tmem_st32(lane_addr + Gm::TM_O + half * HO + cc * 32, ov);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&pv_ready[b2]));
                }
                return true;
            };
            bool ok;
            switch (R) {
                case 32: ok = run_tiles(std::integral_constant<int, 1>{}); break;
                case 16: ok = run_tiles(std::integral_constant<int, 2>{}); break;
                case 8: ok = run_tiles(std::integral_constant<int, 4>{}); break;
                default: ok = run_tiles(std::integral_constant<int, 8>{}); break;
            }
            if (!ok) break;
            if (idle) {
                if (!mbar_wait(smem_u32(&o_full), items & 1u, ctrl, tmo)) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&o_free));
                ++items;
                continue;
            }
            // ---- epilogue: o = O * v_scale / l, this warp's half of the row, the copies added
            for (int x = R; x < 32; x <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, x);
            xl[half][L] = l_run;
            __syncwarp();
            if (lane == 0) mbar_arrive(xb);
            if (!mbar_wait(xb, xph, ctrl, tmo)) break;
            xph ^= 1u;
            const float l_row = l_run + xl[half ^ 1][L];
            if (!mbar_wait(smem_u32(&o_full), items & 1u, ctrl, tmo)) break;
            tc_fence_after();
            // tensor-memory loads and shuffles are warp-collective: every lane takes part, the
            // first copy of each live row stores
            const bool store = c == 0 && r < rows_used;
            if (part >= 0) {
                // a split-KV piece of a decode-class sequence (rows_used <= 16): the unnormalised
                // O, the running max (log2 domain) and the row sum go to partial slot `part`,
                // merged by the combine kernel
                float* prow = a.part_o + ((size_t)part * kDecRows + r) * D + half * HO;
#pragma unroll 1
                for (int cc = 0; cc < HO / 32; ++cc) {
                    uint32_t ov[32];
                    tmem_ld32(lane_addr + Gm::TM_O + half * HO + cc * 32, ov);
                    tmem_ld_wait();
                    add_copies(ov, R);
                    if (store) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            *reinterpret_cast<float4*>(prow + cc * 32 + 4 * i) =
                                make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]),
                                            __uint_as_float(ov[4 * i + 2]), __uint_as_float(ov[4 * i + 3]));
                    }
                }
                if (half == 0 && store)
                    *reinterpret_cast<float2*>(a.part_ml + ((size_t)part * kDecRows + r) * 2) =
                        make_float2(m_run, l_row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&o_free));
                ++items;
                continue;
            }
            const int t_tok = q_start + tok0 + r / G;
            const int qh = head * G + r % G;
            const float l_fin = add_sink(l_row, a.sinks, qh, m_run);  // P was taken relative to m_run
            const float inv = l_fin > 0.f ? a.v_scale / l_fin : 0.f;
            const size_t orow = ((size_t)t_tok * Hq + qh) * D + half * HO;  // element offset of this half row
#pragma unroll 1
            for (int cc = 0; cc < HO / 32; ++cc) {
                uint32_t ov[32];
                tmem_ld32(lane_addr + Gm::TM_O + half * HO + cc * 32, ov);
                tmem_ld_wait();
                add_copies(ov, R);
                if (store) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) store_o8(a.o, orow + cc * 32 + i * 8, ov + 8 * i, inv, a.odt);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&o_free));
            ++items;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int KT>
struct Tc8Kern {
    using Gm = G8<D, !kt_8bit(KT)>;
    static cudaError_t prepare(int* bps) {
        cudaError_t e =
            cudaFuncSetAttribute(rpa_prefill_tc8<D, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bps, rpa_prefill_tc8<D, KT>, kThreads, Gm::SMEM);
    }
    static cudaError_t launch(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, const Launch& l) {
        return launch_pdl(rpa_prefill_tc8<D, KT>, l.grid, kThreads, Gm::SMEM, l.stream, kvm, qm, p);
    }
};

// 8-bit K/V (e4m3, e5m2, int8) at D 64 / 128 / 256; 2-byte K/V (bf16, f16) at D 256 in direct mode
template <int D, typename Op>
cudaError_t tc8_dispatch_kt(int kt, Op op) {
    if (kt == KT_E4M3) return op(Tc8Kern<D, KT_E4M3>{});
    if (kt == KT_E5M2) return op(Tc8Kern<D, KT_E5M2>{});
    if (kt == KT_I8) return op(Tc8Kern<D, KT_I8>{});
    if constexpr (D == 256) {
        if (kt == KT_BF16) return op(Tc8Kern<D, KT_BF16>{});
        if (kt == KT_F16) return op(Tc8Kern<D, KT_F16>{});
    }
    return cudaErrorInvalidValue;
}
template <typename Op>
cudaError_t tc8_dispatch(int D, int kt, Op op) {
    if (D == 64) return tc8_dispatch_kt<64>(kt, op);
    if (D == 128) return tc8_dispatch_kt<128>(kt, op);
    if (D == 256) return tc8_dispatch_kt<256>(kt, op);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t prefill_tc8_prepare(int D, int kt, int* bps) {
    return tc8_dispatch(D, kt, [&](auto k) { return decltype(k)::prepare(bps); });
}

cudaError_t launch_prefill_tc8(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, int kt,
                               const Launch& l) {
    return tc8_dispatch(p.a.D, kt, [&](auto k) { return decltype(k)::launch(kvm, qm, p, l); });
}

}  // namespace rpa
