// rpa_prefill_tc.cu -- K1 prefill on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// One persistent CTA per SM takes prefill work items: up to 256 query rows of
// one kv head, as two 128-row tiles A and B (each Tq = 128 / G tokens x the G
// query heads of the group, packed the way the "ragged_paged.zig" page packs
// its q block into [Tq*G, D]), against a key range of one sequence.  Both
// tiles share every K/V tile, which halves the K/V traffic per FLOP.  Roles:
//
//   producer warp   gathers the two Q tiles and, per 128-key tile, the K and V
//                   rows through the page table with bulk tensor copies (page
//                   runs of the page's createKvAsyncCopyDescriptors) into a
//                   2-stage ring; 128-byte swizzle, rows K-major.
//   MMA warp        one thread issues, per key tile j,
//                     S_A = Q_A K_j^T, S_B = Q_B K_j^T   (both operands in smem)
//                     O_A += P_A V_j, O_B += P_B V_j     (P from TMEM, V MN-major)
//                   in the order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) so that the
//                   tensor cores run one tile's MMAs while the other tile's
//                   softmax works; completion is signalled by tcgen05.commit.
//   2 x 4 softmax   warp group A (warps 0-3) owns S_A/O_A, group B (warps 4-7)
//   warps           S_B/O_B; thread r of a group owns TMEM lane r (one query
//                   row): it loads its S row, applies scale / softcap / masks
//                   (flashAttention's row_ids/col_ids masks) in the log2 domain,
//                   keeps the running max m and sum l, writes P in bf16 over its
//                   S row, and rescales its O row only when the max grows by more
//                   than 2^8 (every P and l use the same stale max, so the result
//                   is unchanged).  At the item's end it normalises O by l and
//                   stores bf16 o.
//
// K/V in f16 run both MMAs in f16 (P in f16); bf16 K/V in bf16.  Q arrives in
// the same type.
//
// Keys of a tile outside the item's [kv_begin, kv_end) are masked in S and
// their V rows are zeroed in shared memory (by group A, before PV_A) since
// tail slots of a page may hold any bits; the page zeroes K/V past kv_len the
// same way.  All waits are bounded; on expiry the status word gets
// RPA_ERR_TIMEOUT.
#include <cuda.h>

#include "rpa_internal.cuh"

namespace rpa {

namespace {

constexpr int kM = kTcRows;      // query rows per tile = TMEM lanes
constexpr int kBN = 128;         // keys per K/V tile
constexpr int kNS = 2;           // K/V stages
constexpr int kThreads = 320;    // warps 0-7 softmax (A: 0-3, B: 4-7), 8 producer, 9 MMA
constexpr int kProducer = 8, kMma = 9;
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;  // rescale O when the row max grows by more than 2^8

enum TcMeta : int { tSeq = 0, tHead, tQStart, tQl, tKl, tKvBegin, tKvEnd, tTok0, tNtok, tNt, tKey0, tStop };

template <int D>
struct TcGeom {
    static constexpr int CB = D / 64;                // 128-byte column blocks of a row
    static constexpr int QTILE = CB * kM * 128;      // one 128-row Q tile
    static constexpr int KBYTES = CB * kBN * 128;    // K (or V) of one stage
    static constexpr int STAGE = 2 * KBYTES;
    static constexpr int DATA = 2 * QTILE + kNS * STAGE;
    // one CTA per SM: it owns all 512 TMEM columns
    static constexpr int SMEM = (DATA + 1024) > 120 * 1024 ? (DATA + 1024) : 120 * 1024;
    // TMEM columns: S_A, S_B, O_A, O_B
    __host__ __device__ static constexpr uint32_t TM_S(int x) { return (uint32_t)(x * kBN); }
    __host__ __device__ static constexpr uint32_t TM_O(int x) { return (uint32_t)(2 * kBN + x * D); }
    static_assert(2 * kBN + 2 * D <= kTmemCols, "TMEM budget");
};

__device__ __forceinline__ void put_u4(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// p = 2^(x * mul - base) for the 32 logits of one S chunk: bf16 (F16: f16) pairs into pk, sums into ls2
template <bool F16>
__device__ __forceinline__ void exp_chunk(const uint32_t* sv, uint64_t mul2, uint64_t nbase2, uint64_t* ls2,
                                          uint32_t* pk) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float x0, x1;
        f32x2_split(ffma2(f32x2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), mul2, nbase2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        ls2[i & 1] = fadd2(ls2[i & 1], f32x2(p0, p1));
        pk[i] = pack2<F16>(p0, p1);
    }
}

template <int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1) rpa_prefill_tc(const __grid_constant__ CUtensorMap kvmap,
                                                              const __grid_constant__ CUtensorMap qmap,
                                                              const TcParams p) {
    using Gm = TcGeom<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full, q_empty, meta_free;
    __shared__ __align__(8) uint64_t kv_full[kNS], kv_empty[kNS];
    __shared__ __align__(8) uint64_t s_full[2], p_full[2];
    __shared__ __align__(8) uint64_t o_full, o_free;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int meta[16];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const AttnParams& a = p.a;
    int* ctrl = a.ctrl;
    const uint64_t tmo = p.timeout_ns;
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t q_base = smem0;                       // Q_A, Q_B
    const uint32_t kv_base = smem0 + 2 * Gm::QTILE;      // kNS stages of [K | V]

    if (tid == 0) {
        mbar_init(smem_u32(&q_full), 1);
        mbar_init(smem_u32(&q_empty), 1);
        mbar_init(smem_u32(&meta_free), 8);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&p_full[i]), 4);
        }
        for (int i = 0; i < kNS; ++i) {
            mbar_init(smem_u32(&kv_full[i]), 1);
            mbar_init(smem_u32(&kv_empty[i]), 1);
        }
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
    const bool active = (int)blockIdx.x < a.ctrl[kPfCtas];  // otherwise SMs left to the decode kernel

    if (!active) {
    } else if (warp == kProducer) {
        // =============================== producer ===============================
        const int BR = p.BR, ps = a.ps, G = a.G, Th = p.Tq / 2;  // tokens per Q tile
        const int tasks = (kBN / BR) * 2 * Gm::CB;
        const uint32_t box_bytes = (uint32_t)BR * 128u;
        const uint64_t pol_keep = l2_policy_evict_last();
        const uint32_t q_bytes = (uint32_t)(2 * Gm::CB * G * Th * 128);
        int s = 0;
        uint32_t qph = 0, ph = 0;
        bool ok = true;
        int it = 0;
        if (lane == 0) it = atomicAdd(ctrl + a.counter_word, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        for (;;) {
            const bool stop = it >= n_items;
            if (!mbar_wait(smem_u32(&q_empty), qph ^ 1u, ctrl, tmo) ||
                !mbar_wait(smem_u32(&meta_free), qph ^ 1u, ctrl, tmo))
                break;
            if (stop) {
                if (lane == 0) {
                    meta[tStop] = 1;
                    mbar_arrive(smem_u32(&q_full));
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
                meta[tSeq] = item.seq;
                meta[tHead] = item.head;
                meta[tQStart] = q_start;
                meta[tQl] = ql;
                meta[tKl] = kl;
                meta[tKvBegin] = item.kv_begin;
                meta[tKvEnd] = item.kv_end;
                meta[tTok0] = item.tok0;
                meta[tNtok] = item.ntok;
                meta[tNt] = nt;
                meta[tKey0] = key0;
                meta[tStop] = 0;
            }
            __syncwarp();
            const uint32_t qfb = smem_u32(&q_full);
            // tile B only when it has tokens: a box wholly past the last query token is not copied
            const int q_tiles = item.ntok > Th ? 2 : 1;
            if (lane == 0) mbar_arrive_expect_tx(qfb, q_bytes / 2 * q_tiles);
            __syncwarp();
            if (lane < q_tiles * Gm::CB) {
                const int tile = lane / Gm::CB, cb = lane % Gm::CB;
                tma_load_3d(q_base + tile * Gm::QTILE + cb * (kM * 128), &qmap, qfb, cb * 64, item.head * G,
                            q_start + item.tok0 + tile * Th);
            }
            qph ^= 1u;
            int win0 = key0 / ps;
            int win = (win0 + lane < a.P) ? __ldg(ptab + win0 + lane) : 0;
            for (int t = 0; t < nt && ok; ++t) {
                const int k_tile = key0 + t * kBN;
                const int lp_last = min(k_tile + kBN - 1, item.kv_end - 1) / ps;
                if (lp_last - win0 >= 32) {
                    win0 = k_tile / ps;
                    win = (win0 + lane < a.P) ? __ldg(ptab + win0 + lane) : 0;
                }
                if (!mbar_wait(smem_u32(&kv_empty[s]), ph ^ 1u, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                const uint32_t stage = kv_base + s * Gm::STAGE;
                // task -> (page run b, K/V, column block cb)
                auto task = [&](int tk, int& x, int& y, uint32_t& dst) -> int {
                    const int per = 2 * Gm::CB;
                    const int b = tk / per, rem = tk % per;
                    const int kv = rem / Gm::CB, cb = rem % Gm::CB;
                    const int k0 = k_tile + b * BR;
                    const int lp = k0 / ps;
                    const int pg = __shfl_sync(0xffffffffu, win, (lp - win0) & 31);
                    if (tk >= tasks || k0 >= item.kv_end || k0 + BR <= item.kv_begin) return 0;
                    if ((unsigned)pg >= (unsigned)a.N) return 2;
                    x = (2 * item.head + kv) * D + cb * 64;
                    y = pg * ps + (k0 - lp * ps);
                    dst = stage + (uint32_t)(kv * Gm::KBYTES + cb * (kBN * 128) + b * BR * 128);
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
                if (__any_sync(0xffffffffu, bad)) {
                    if (lane == 0) set_status(ctrl, RPA_ERR_BAD_PAGE_INDEX);
                    for (int i = lane; i < Gm::STAGE / 16; i += 32)
                        put_u4(smem + (stage - smem0) + i * 16, make_uint4(0, 0, 0, 0));
                    fence_proxy_async_smem();
                }
                __syncwarp();
                const uint32_t fb = smem_u32(&kv_full[s]);
                if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)n_issue * box_bytes);
                __syncwarp();
                // a sequence's K/V is re-read from L2 by the CTAs running its other query tiles
                for (int t0 = 0; t0 < tasks; t0 += 32) {
                    int x, y;
                    uint32_t dst;
                    if (task(t0 + lane, x, y, dst) == 1) tma_load_2d_hint(dst, &kvmap, fb, x, y, pol_keep);
                }
                if (++s == kNS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            it = __shfl_sync(0xffffffffu, nxt, 0);
        }
    } else if (warp == kMma) {
        // =============================== MMA issuer ===============================
        if (lane == 0) {
            constexpr uint32_t idesc_qk = F16 ? umma_idesc_f16(kM, kBN, 0, 0) : umma_idesc_bf16(kM, kBN, 0, 0);
            constexpr uint32_t idesc_pv = F16 ? umma_idesc_f16(kM, D, 0, 1) : umma_idesc_bf16(kM, D, 0, 1);
            int s = 0;
            uint32_t qph = 0, ph = 0;
            uint32_t j_all = 0;   // key tiles issued so far (all items): phase of s_full / p_full
            uint32_t items = 0;   // items finished
            bool ok = true;
            // descriptors are formed once per call and offset per MMA in their low (address) half:
            // the MMA thread shares its sub-partition with two softmax warps, so each MMA costs it
            // only a few issue slots
            auto issue_qk = [&](int x, int ss) {
                const uint64_t qd = umma_sdesc(q_base + x * Gm::QTILE, 16, 1024);
                const uint64_t kd = umma_sdesc(kv_base + ss * Gm::STAGE, 16, 1024);
                const uint32_t qd_lo = (uint32_t)qd, qd_hi = (uint32_t)(qd >> 32);
                const uint32_t kd_lo = (uint32_t)kd, kd_hi = (uint32_t)(kd >> 32);
                const uint32_t sd = tmem + Gm::TM_S(x);
                umma_ss_c<0>(sd, qd_lo, qd_hi, kd_lo, kd_hi, idesc_qk);
#pragma unroll
                for (int kk = 1; kk < D / 16; ++kk)
                    umma_ss_c<1>(sd, qd_lo + ((kk >> 2) * (kM * 128) + (kk & 3) * 32) / 16, qd_hi,
                                 kd_lo + ((kk >> 2) * (kBN * 128) + (kk & 3) * 32) / 16, kd_hi, idesc_qk);
                umma_commit(smem_u32(&s_full[x]));
            };
            auto issue_pv = [&](int x, int ss, uint32_t jj, bool first) -> bool {
                if (!mbar_wait(smem_u32(&p_full[x]), jj & 1u, ctrl, tmo)) return false;
                tc_fence_after();
                const uint64_t vd = umma_sdesc(kv_base + ss * Gm::STAGE + Gm::KBYTES, kBN * 128, 1024);
                const uint32_t vd_lo = (uint32_t)vd, vd_hi = (uint32_t)(vd >> 32);
                const uint32_t od = tmem + Gm::TM_O(x), pa = tmem + Gm::TM_S(x);
                if (first)
                    umma_ts_c<0>(od, pa, vd_lo, vd_hi, idesc_pv);
                else
                    umma_ts_c<1>(od, pa, vd_lo, vd_hi, idesc_pv);
#pragma unroll
                for (int kk = 1; kk < kBN / 16; ++kk)
                    umma_ts_c<1>(od, pa + kk * 8, vd_lo + kk * 16 * 128 / 16, vd_hi, idesc_pv);
                return true;
            };
            for (;;) {
                if (!mbar_wait(smem_u32(&q_full), qph, ctrl, tmo)) break;
                if (meta[tStop]) break;
                const int nt = meta[tNt];
                qph ^= 1u;
                tc_fence_after();
                if (!mbar_wait(smem_u32(&kv_full[s]), ph, ctrl, tmo)) break;
                tc_fence_after();
                issue_qk(0, s);
                issue_qk(1, s);
                if (nt == 1) umma_commit(smem_u32(&q_empty));
                for (int t = 0; t < nt; ++t) {
                    const uint32_t jj = j_all + t;
                    const int cur = s;
                    int nxt_s = s + 1;
                    uint32_t nxt_ph = ph;
                    if (nxt_s == kNS) {
                        nxt_s = 0;
                        nxt_ph ^= 1u;
                    }
                    const bool more = t + 1 < nt;
                    // O_A / O_B are overwritten by this item's first PV: the previous epilogue must be done
                    if (t == 0 && items > 0 && !mbar_wait(smem_u32(&o_free), (items - 1) & 1u, ctrl, tmo)) {
                        ok = false;
                        break;
                    }
                    if (!issue_pv(0, cur, jj, t == 0)) {
                        ok = false;
                        break;
                    }
                    if (more) {
                        if (!mbar_wait(smem_u32(&kv_full[nxt_s]), nxt_ph, ctrl, tmo)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_qk(0, nxt_s);
                    }
                    if (!issue_pv(1, cur, jj, t == 0)) {
                        ok = false;
                        break;
                    }
                    umma_commit(smem_u32(&kv_empty[cur]));
                    if (more) {
                        issue_qk(1, nxt_s);
                        if (t + 2 == nt) umma_commit(smem_u32(&q_empty));
                    }
                    s = nxt_s;
                    ph = nxt_ph;
                }
                if (!ok) break;
                j_all += nt;
                umma_commit(smem_u32(&o_full));
                ++items;
            }
        }
        __syncwarp();
    } else {
        // =============================== softmax warp groups ===============================
        const int x = warp >> 2;           // 0: tile A, 1: tile B
        const int r = tid & 127;           // TMEM lane == row of this tile
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const int G = a.G, Hq = a.Hq, Th = p.Tq / 2;
        int s = 0;
        uint32_t qph = 0, ph = 0;
        uint32_t j_all = 0, items = 0;
        for (;;) {
            if (!mbar_wait(smem_u32(&q_full), qph, ctrl, tmo)) break;
            const int stop = meta[tStop];
            const int head = meta[tHead], q_start = meta[tQStart], ql = meta[tQl], kl = meta[tKl];
            const int kv_begin = meta[tKvBegin], kv_end = meta[tKvEnd], tok0 = meta[tTok0];
            const int ntok = meta[tNtok], nt = meta[tNt], key0 = meta[tKey0];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&meta_free));
            if (stop) break;
            qph ^= 1u;
            // this tile's tokens: [tok0 + x*Th, tok0 + x*Th + ntx)
            const int ttok0 = tok0 + x * Th;
            const int ntx = max(0, min(Th, ntok - x * Th));
            const int pos = kl - ql + ttok0 + r / G;  // key position of this row
            const int pos_lo = kl - ql + ttok0, pos_hi = kl - ql + ttok0 + max(ntx, 1) - 1;
            float m_run = -INFINITY, l_run = 0.f;
            bool ok = true;
            for (int t = 0; t < nt; ++t) {
                const uint32_t jj = j_all + t;
                if (!mbar_wait(smem_u32(&s_full[x]), jj & 1u, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int k_lo = key0 + t * kBN;
                const bool partial = k_lo < kv_begin || k_lo + kBN > kv_end;
                const bool need_mask = partial || (a.causal && k_lo + kBN - 1 > pos_lo) ||
                                       (a.has_window && k_lo <= pos_hi - a.window);
                const uint32_t scol = Gm::TM_S(x);
                // pass 1: row max of the transformed logits; masked or capped values are
                // written back to TMEM so that pass 2 only exponentiates
                const bool rewrite = need_mask || a.has_cap;
                float mt = -INFINITY;
                uint64_t ls2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
                bool need;
                float alpha, m_new;
                if (!rewrite) {
                    // interior tile, no cap.  Pass 1: the extreme raw logit times the scale (the max
                    // for a positive scale, the min for a negative one), chunks 2, 3 then 0, 1, two
                    // loads in flight; chunks 0 and 1 stay in registers for pass 2
                    const bool pos_scale = a.qk_log2 >= 0.f;
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                    float n4[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
                    uint32_t sa[32], sb[32];
#pragma unroll
                    for (int h = 1; h >= 0; --h) {
                        tmem_ld32(lane_addr + scol + (2 * h) * 32, sa);
                        tmem_ld32(lane_addr + scol + (2 * h + 1) * 32, sb);
                        tmem_ld_wait();
                        if (pos_scale) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                m4[i & 3] = fmax3(m4[i & 3], __uint_as_float(sa[2 * i]), __uint_as_float(sa[2 * i + 1]));
                                m4[(i + 2) & 3] = fmax3(m4[(i + 2) & 3], __uint_as_float(sb[2 * i]), __uint_as_float(sb[2 * i + 1]));
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                n4[i & 3] = fmin3(n4[i & 3], __uint_as_float(sa[2 * i]), __uint_as_float(sa[2 * i + 1]));
                                n4[(i + 2) & 3] = fmin3(n4[(i + 2) & 3], __uint_as_float(sb[2 * i]), __uint_as_float(sb[2 * i + 1]));
                            }
                        }
                    }
                    mt = pos_scale ? fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.qk_log2
                                   : fminf(fminf(n4[0], n4[1]), fminf(n4[2], n4[3])) * a.qk_log2;
                    // lazy rescale: move the running max only when it grows by more than 2^8
                    need = __any_sync(0xffffffffu, mt > m_run + kRescaleLog2);  // false if mt == -inf
                    m_new = need ? fmaxf(m_run, mt) : m_run;
                    alpha = !need ? 1.f : (m_run == -INFINITY ? 0.f : ex2(m_run - m_new));
                    const float base = m_new == -INFINITY ? 0.f : m_new;
                    // pass 2: P = 2^(x - base) in bf16 over the consumed S columns (P[i] at column
                    // i/2): chunks 0 and 1 from registers (their P lands in columns 0-31, S chunk 0),
                    // chunks 2 and 3 reloaded while chunk 1 is exponentiated
                    const uint64_t mul2 = f32x2(a.qk_log2, a.qk_log2), nbase2 = f32x2(-base, -base);
                    uint32_t pk[16];
                    exp_chunk<F16>(sa, mul2, nbase2, ls2, pk);
                    tmem_st16(lane_addr + scol, pk);
                    tmem_ld32(lane_addr + scol + 64, sa);
                    exp_chunk<F16>(sb, mul2, nbase2, ls2, pk);
                    tmem_st16(lane_addr + scol + 16, pk);
                    tmem_ld32(lane_addr + scol + 96, sb);
                    tmem_ld_wait();
                    exp_chunk<F16>(sa, mul2, nbase2, ls2, pk);
                    tmem_st16(lane_addr + scol + 32, pk);
                    exp_chunk<F16>(sb, mul2, nbase2, ls2, pk);
                    tmem_st16(lane_addr + scol + 48, pk);
                } else {
                    const bool cap = a.has_cap;
#pragma unroll 1
                    for (int c = 0; c < kBN / 32; ++c) {
                        uint32_t sv[32];
                        tmem_ld32(lane_addr + scol + c * 32, sv);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            float v = __uint_as_float(sv[i]);
                            v = cap ? a.cap_log2 - 2.f * a.cap_log2 * rcp_approx(1.f + ex2(v * a.cap_exp))
                                    : v * a.qk_log2;
                            const int j = k_lo + c * 32 + i;
                            const bool okk = j >= kv_begin && j < kv_end && (!a.causal || j <= pos) &&
                                             (!a.has_window || j > pos - a.window);
                            v = (okk || !need_mask) ? v : -INFINITY;
                            mt = fmaxf(mt, v);
                            sv[i] = __float_as_uint(v);
                        }
                        tmem_st32(lane_addr + scol + c * 32, sv);
                    }
                    tmem_st_wait();
                    need = __any_sync(0xffffffffu, mt > m_run + kRescaleLog2);
                    m_new = need ? fmaxf(m_run, mt) : m_run;
                    alpha = !need ? 1.f : (m_run == -INFINITY ? 0.f : ex2(m_run - m_new));
                    const float base = m_new == -INFINITY ? 0.f : m_new;
                    // pass 2 over the rewritten (already scaled and masked) logits
                    const uint64_t mul2 = f32x2(1.f, 1.f), nbase2 = f32x2(-base, -base);
#pragma unroll 1
                    for (int c = 0; c < kBN / 32; ++c) {
                        uint32_t sv[32], pk[16];
                        tmem_ld32(lane_addr + scol + c * 32, sv);
                        tmem_ld_wait();
                        exp_chunk<F16>(sv, mul2, nbase2, ls2, pk);
                        tmem_st16(lane_addr + scol + c * 16, pk);
                    }
                }
                float la, lb, lc, ld;
                f32x2_split(ls2[0], la, lb);
                f32x2_split(ls2[1], lc, ld);
                const float lsum = (la + lb) + (lc + ld);
                l_run = l_run * alpha + lsum;
                m_run = m_new;
                if (need && t > 0) {
                    // O holds this item's PVs up to tile t-1, all complete: the MMA thread issues
                    // S_x(t) after PV_x(t-1), and a commit (here s_full, waited for above) arrives
                    // once every MMA issued before it is done.  Scale in place.
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(lane_addr + Gm::TM_O(x) + c * 32, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st32(lane_addr + Gm::TM_O(x) + c * 32, ov);
                    }
                }
                tmem_st_wait();
                if (partial && x == 0) {
                    // zero the V rows of keys outside [kv_begin, kv_end) once the stage has landed
                    if (!mbar_wait(smem_u32(&kv_full[s]), ph, ctrl, tmo)) {
                        ok = false;
                        break;
                    }
                    const int j = k_lo + r;  // thread r owns key row r of the tile
                    if (j < kv_begin || j >= kv_end) {
                        uint8_t* vrow = smem + (kv_base - smem0) + s * Gm::STAGE + Gm::KBYTES + r * 128;
#pragma unroll
                        for (int cb = 0; cb < Gm::CB; ++cb)
#pragma unroll
                            for (int c = 0; c < 8; ++c) put_u4(vrow + cb * (kBN * 128) + c * 16, make_uint4(0, 0, 0, 0));
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&p_full[x]));
                if (++s == kNS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            j_all += nt;
            // ---- epilogue: o = O * v_scale / l
            if (!mbar_wait(smem_u32(&o_full), items & 1u, ctrl, tmo)) break;
            tc_fence_after();
            const int rows_used = ntx * G;
            const int t_tok = q_start + ttok0 + r / G;
            const int qh = head * G + r % G;
            const float l_fin = add_sink(l_run, a.sinks, qh, m_run);  // P was taken relative to m_run
            const float inv = l_fin > 0.f ? a.v_scale / l_fin : 0.f;
            const size_t orow = ((size_t)t_tok * Hq + qh) * D;  // element offset of the output row
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(lane_addr + Gm::TM_O(x) + c * 32, ov);
                tmem_ld_wait();
                if (r < rows_used) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) store_o8(a.o, orow + c * 32 + i * 8, ov + 8 * i, inv, a.odt);
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

template <int D, bool F16>
struct TcKern {
    using Gm = TcGeom<D>;
    static cudaError_t prepare(int* bps) {
        cudaError_t e =
            cudaFuncSetAttribute(rpa_prefill_tc<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bps, rpa_prefill_tc<D, F16>, kThreads, Gm::SMEM);
    }
    static cudaError_t launch(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, const Launch& l) {
        return launch_pdl(rpa_prefill_tc<D, F16>, l.grid, kThreads, Gm::SMEM, l.stream, kvm, qm, p);
    }
};

// 2-byte K/V at D 64 / 128: bf16 or f16 MMAs
template <typename Op>
cudaError_t tc_dispatch(int D, int kt, Op op) {
    if (kt != KT_BF16 && kt != KT_F16) return cudaErrorInvalidValue;
    const bool f16 = kt == KT_F16;
    if (D == 64) return f16 ? op(TcKern<64, true>{}) : op(TcKern<64, false>{});
    if (D == 128) return f16 ? op(TcKern<128, true>{}) : op(TcKern<128, false>{});
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t prefill_tc_prepare(int D, int kt, int* bps) {
    return tc_dispatch(D, kt, [&](auto k) { return decltype(k)::prepare(bps); });
}

cudaError_t launch_prefill_tc(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, int kt, const Launch& l) {
    return tc_dispatch(p.a.D, kt, [&](auto k) { return decltype(k)::launch(kvm, qm, p, l); });
}

}  // namespace rpa
