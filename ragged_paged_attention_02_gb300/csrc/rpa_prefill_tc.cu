// rpa_prefill_tc.cu -- K1 prefill on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// One persistent CTA per SM takes prefill work items: 128 query rows of one kv
// head (Tq = 128 / G tokens x the G query heads of the group, packed as the
// "ragged_paged.zig" page packs its q block into [Tq*G, D]) against a key
// range of one sequence.  Roles:
//
//   producer warp   gathers the Q tile and, per 128-key tile, the K and V rows
//                   through the page table with bulk tensor copies (page runs
//                   of the page's createKvAsyncCopyDescriptors), into a
//                   2-stage ring; 128-byte swizzle, K-major rows.
//   MMA warp        one thread issues S = Q K^T (M=128, N=128, K=16 steps,
//                   both operands from shared memory) into one of two TMEM
//                   S buffers, and O += P V with P read from TMEM and V
//                   used MN-major from shared memory; completion is signalled
//                   with tcgen05.commit on mbarriers.
//   4 softmax warps thread r owns TMEM lane r (query row r): it loads its S
//                   row, applies scale / softcap / masks (flashAttention's
//                   row_ids/col_ids masks) in the log2 domain, keeps the
//                   running max m and sum l, writes P in bf16 over its S row,
//                   and rescales its O row only when the max grows by more than
//                   2^8 (the result is the same: every P and l use the same
//                   stale max).  At the item's end it normalises O by l and
//                   stores bf16 o.
//
// Keys of a tile outside the item's [kv_begin, kv_end) are masked in S and
// their V rows are zeroed in shared memory before the PV MMA (tail slots of a
// page may hold any bits; the page zeroes K/V past kv_len the same way).
// All waits are bounded; on expiry the status word gets RPA_ERR_TIMEOUT.
#include <cuda.h>

#include "rpa_internal.cuh"

namespace rpa {

namespace {

constexpr int kM = kTcRows;      // query rows per tile = TMEM lanes
constexpr int kBN = 128;         // keys per K/V tile
constexpr int kNS = 2;           // K/V stages
constexpr int kThreads = 192;    // warps 0-3 softmax, 4 producer, 5 MMA
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;  // rescale O when the row max grows by more than 2^8

enum TcMeta : int { tSeq = 0, tHead, tQStart, tQl, tKl, tKvBegin, tKvEnd, tTok0, tNtok, tNt, tKey0, tStop };

template <int D>
struct TcGeom {
    static constexpr int CB = D / 64;                // 128-byte column blocks of a row
    static constexpr int QBYTES = CB * kM * 128;     // one Q slot
    static constexpr int KBYTES = CB * kBN * 128;    // K (or V) of one stage
    static constexpr int STAGE = 2 * KBYTES;
    static constexpr int DATA = 2 * QBYTES + kNS * STAGE;
    // keep one CTA per SM: it owns all 512 TMEM columns
    static constexpr int SMEM = (DATA + 1024) > 120 * 1024 ? (DATA + 1024) : 120 * 1024;
    static constexpr int TM_S0 = 0, TM_S1 = kBN, TM_O = 2 * kBN;
    static_assert(2 * kBN + D <= kTmemCols, "TMEM budget");
};

__device__ __forceinline__ void put_u4(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

template <int D>
__global__ void __launch_bounds__(kThreads, 1) rpa_prefill_tc(const __grid_constant__ CUtensorMap kvmap,
                                                              const __grid_constant__ CUtensorMap qmap,
                                                              const TcParams p) {
    using Gm = TcGeom<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full[2], q_empty[2], meta_free[2];
    __shared__ __align__(8) uint64_t kv_full[kNS], kv_empty[kNS];
    __shared__ __align__(8) uint64_t s_full[2], p_full[2];
    __shared__ __align__(8) uint64_t pv_done, o_full, o_free;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int meta[2][16];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const AttnParams& a = p.a;
    int* ctrl = a.ctrl;
    const uint64_t tmo = p.timeout_ns;
    const int n_items = a.ctrl[a.item_count_word];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t q_base = smem0;                         // 2 Q slots
    const uint32_t kv_base = smem0 + 2 * Gm::QBYTES;       // kNS stages of [K | V]

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&q_full[i]), 1);
            mbar_init(smem_u32(&q_empty[i]), 1);
            mbar_init(smem_u32(&meta_free[i]), 4);
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&p_full[i]), 4);
        }
        for (int i = 0; i < kNS; ++i) {
            mbar_init(smem_u32(&kv_full[i]), 1);
            mbar_init(smem_u32(&kv_empty[i]), 1);
        }
        mbar_init(smem_u32(&pv_done), 1);
        mbar_init(smem_u32(&o_full), 1);
        mbar_init(smem_u32(&o_free), 4);
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 4) {
        // =============================== producer ===============================
        const int BR = p.BR, ps = a.ps, G = a.G;
        const int tasks = (kBN / BR) * 2 * Gm::CB;
        const uint32_t box_bytes = (uint32_t)BR * 128u;
        const uint32_t q_bytes = (uint32_t)(Gm::CB * G * p.Tq * 128);
        int qs = 0, s = 0;
        uint32_t qph = 0, ph = 0;
        bool ok = true;
        int it = 0;
        if (lane == 0) it = atomicAdd(ctrl + a.counter_word, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        for (;;) {
            const bool stop = it >= n_items;
            // a Q slot (and its meta) for the next item, or for the stop mark
            if (!mbar_wait(smem_u32(&q_empty[qs]), qph ^ 1u, ctrl, tmo) ||
                !mbar_wait(smem_u32(&meta_free[qs]), qph ^ 1u, ctrl, tmo)) {
                ok = false;
                break;
            }
            if (stop) {
                if (lane == 0) {
                    meta[qs][tStop] = 1;
                    mbar_arrive(smem_u32(&q_full[qs]));
                }
                break;
            }
            const Item item = a.items[it];
            int nxt = 0;
            if (lane == 0) nxt = atomicAdd(ctrl + a.counter_word, 1);
            const int q_start = a.cu_q_lens[item.seq];
            const int ql = a.cu_q_lens[item.seq + 1] - q_start;
            const int kl = a.kv_lens[item.seq];
            const int* ptab = a.page_indices + (size_t)item.seq * a.P;
            const int key0 = item.kv_begin - (item.kv_begin & (BR - 1));
            const int nt = (item.kv_end - key0 + kBN - 1) / kBN;
            if (lane == 0) {
                int* m = meta[qs];
                m[tSeq] = item.seq;
                m[tHead] = item.head;
                m[tQStart] = q_start;
                m[tQl] = ql;
                m[tKl] = kl;
                m[tKvBegin] = item.kv_begin;
                m[tKvEnd] = item.kv_end;
                m[tTok0] = item.tok0;
                m[tNtok] = item.ntok;
                m[tNt] = nt;
                m[tKey0] = key0;
                m[tStop] = 0;
            }
            __syncwarp();
            const uint32_t qfb = smem_u32(&q_full[qs]);
            if (lane == 0) mbar_arrive_expect_tx(qfb, q_bytes);
            __syncwarp();
            if (lane < Gm::CB)
                tma_load_3d(q_base + qs * Gm::QBYTES + lane * (kM * 128), &qmap, qfb, lane * 64, item.head * G,
                            q_start + item.tok0);
            if (++qs == 2) {
                qs = 0;
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
                for (int t0 = 0; t0 < tasks; t0 += 32) {
                    int x, y;
                    uint32_t dst;
                    if (task(t0 + lane, x, y, dst) == 1) tma_load_2d(dst, &kvmap, fb, x, y);
                }
                if (++s == kNS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            it = __shfl_sync(0xffffffffu, nxt, 0);
        }
        (void)ok;
    } else if (warp == 5) {
        // =============================== MMA issuer ===============================
        if (lane == 0) {
            constexpr uint32_t idesc_qk = umma_idesc_bf16(kM, kBN, 0, 0);
            constexpr uint32_t idesc_pv = umma_idesc_bf16(kM, D, 0, 1);
            int qs = 0, s = 0;
            uint32_t qph = 0, ph = 0;
            uint32_t g = 0;        // tiles issued so far (all items): S buffer g & 1
            uint32_t items = 0;    // items finished
            bool ok = true;
            // PV of tile gg (stage ss) of the current item; first = first tile of the item
            auto issue_pv = [&](uint32_t gg, int ss, bool first) -> bool {
                const int b = gg & 1;
                if (!mbar_wait(smem_u32(&p_full[b]), (gg >> 1) & 1u, ctrl, tmo)) return false;
                if (first && items > 0 && !mbar_wait(smem_u32(&o_free), (items - 1) & 1u, ctrl, tmo)) return false;
                tc_fence_after();
                const uint32_t vst = kv_base + ss * Gm::STAGE + Gm::KBYTES;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t bdesc = umma_sdesc(vst + kk * 16 * 128, kBN * 128, 1024);
                    umma_ts(tmem + Gm::TM_O, tmem + (b ? Gm::TM_S1 : Gm::TM_S0) + kk * 8, bdesc, idesc_pv,
                            (!first || kk > 0) ? 1 : 0);
                }
                umma_commit(smem_u32(&kv_empty[ss]));
                umma_commit(smem_u32(&pv_done));
                return true;
            };
            for (;;) {
                if (!mbar_wait(smem_u32(&q_full[qs]), qph, ctrl, tmo)) break;
                if (meta[qs][tStop]) break;
                const int nt = meta[qs][tNt];
                tc_fence_after();
                const uint32_t qsl = q_base + qs * Gm::QBYTES;
                int prev_s = 0;
                for (int t = 0; t < nt && ok; ++t) {
                    if (!mbar_wait(smem_u32(&kv_full[s]), ph, ctrl, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int b = g & 1;
                    const uint32_t kst = kv_base + s * Gm::STAGE;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (uint32_t)((kk >> 2) * (kM * 128) + (kk & 3) * 32);
                        const uint32_t koff = (uint32_t)((kk >> 2) * (kBN * 128) + (kk & 3) * 32);
                        umma_ss(tmem + (b ? Gm::TM_S1 : Gm::TM_S0), umma_sdesc(qsl + off, 16, 1024),
                                umma_sdesc(kst + koff, 16, 1024), idesc_qk, kk > 0 ? 1 : 0);
                    }
                    umma_commit(smem_u32(&s_full[b]));
                    if (t == nt - 1) umma_commit(smem_u32(&q_empty[qs]));
                    if (t > 0 && !issue_pv(g - 1, prev_s, t == 1)) {
                        ok = false;
                        break;
                    }
                    prev_s = s;
                    ++g;
                    if (++s == kNS) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok || !issue_pv(g - 1, prev_s, nt == 1)) break;
                umma_commit(smem_u32(&o_full));
                ++items;
                if (++qs == 2) {
                    qs = 0;
                    qph ^= 1u;
                }
            }
        }
        __syncwarp();
    } else {
        // =============================== softmax warps ===============================
        const int r = tid;  // TMEM lane == query row of the tile
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        const int G = a.G, Hq = a.Hq;
        int qs = 0, s = 0;
        uint32_t qph = 0, ph = 0;
        uint32_t g = 0, items = 0;
        for (;;) {
            if (!mbar_wait(smem_u32(&q_full[qs]), qph, ctrl, tmo)) break;
            const int* mm = meta[qs];
            const int stop = mm[tStop];
            const int head = mm[tHead], q_start = mm[tQStart], ql = mm[tQl], kl = mm[tKl];
            const int kv_begin = mm[tKvBegin], kv_end = mm[tKvEnd], tok0 = mm[tTok0], ntok = mm[tNtok];
            const int nt = mm[tNt], key0 = mm[tKey0];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&meta_free[qs]));
            if (stop) break;
            if (++qs == 2) {
                qs = 0;
                qph ^= 1u;
            }
            const int pos = kl - ql + tok0 + r / G;  // key position of this row
            const int pos_lo = kl - ql + tok0, pos_hi = kl - ql + tok0 + ntok - 1;
            float m_run = -INFINITY, l_run = 0.f;
            bool ok = true;
            for (int t = 0; t < nt; ++t) {
                const int b = g & 1;
                if (!mbar_wait(smem_u32(&s_full[b]), (g >> 1) & 1u, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int k_lo = key0 + t * kBN;
                const bool partial = k_lo < kv_begin || k_lo + kBN > kv_end;
                const bool need_mask = partial || (a.causal && k_lo + kBN - 1 > pos_lo) ||
                                       (a.has_window && k_lo <= pos_hi - a.window);
                const uint32_t scol = b ? Gm::TM_S1 : Gm::TM_S0;
                float x[kBN];
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) tmem_ld32(lane_addr + scol + c * 32, reinterpret_cast<uint32_t*>(x) + c * 32);
                tmem_ld_wait();
                float mt = -INFINITY;
#pragma unroll
                for (int i = 0; i < kBN; ++i) {
                    float v = x[i];
                    if (a.has_cap) {
                        const float e = ex2(v * a.cap_exp);
                        v = a.cap_log2 - 2.f * a.cap_log2 * __frcp_rn(1.f + e);
                    } else {
                        v *= a.qk_log2;
                    }
                    if (need_mask) {
                        const int j = k_lo + i;
                        const bool okk = j >= kv_begin && j < kv_end && (!a.causal || j <= pos) &&
                                         (!a.has_window || j > pos - a.window);
                        v = okk ? v : -INFINITY;
                    }
                    x[i] = v;
                    mt = fmaxf(mt, v);
                }
                const bool need = mt > m_run + kRescaleLog2;  // false when mt == -inf
                if (__any_sync(0xffffffffu, need)) {
                    const float m_new = fmaxf(m_run, mt);
                    const float alpha = m_run == -INFINITY ? 0.f : ex2(m_run - m_new);
                    if (t > 0) {
                        // O holds this item's PVs up to tile g-1: wait for it, then scale in place
                        if (!mbar_wait(smem_u32(&pv_done), (g - 1) & 1u, ctrl, tmo)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t ov[32];
                            tmem_ld32(lane_addr + Gm::TM_O + c * 32, ov);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                            tmem_st32(lane_addr + Gm::TM_O + c * 32, ov);
                        }
                        tmem_st_wait();
                    }
                    l_run *= alpha;
                    m_run = m_new;
                }
                const float base = m_run == -INFINITY ? 0.f : m_run;
                uint32_t pk[kBN / 2];
#pragma unroll
                for (int i = 0; i < kBN / 2; ++i) {
                    const float p0 = ex2(x[2 * i] - base);
                    const float p1 = ex2(x[2 * i + 1] - base);
                    l_run += p0 + p1;
                    pk[i] = pack2<false>(p0, p1);
                }
#pragma unroll
                for (int c = 0; c < kBN / 64; ++c) tmem_st32(lane_addr + scol + c * 32, pk + c * 32);
                tmem_st_wait();
                if (partial) {
                    // zero the V rows of keys outside [kv_begin, kv_end) once this stage has landed
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
                if (lane == 0) mbar_arrive(smem_u32(&p_full[b]));
                ++g;
                if (++s == kNS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            // ---- epilogue: o = O * v_scale / l
            if (!mbar_wait(smem_u32(&o_full), items & 1u, ctrl, tmo)) break;
            tc_fence_after();
            const int rows_used = ntok * G;
            const float inv = l_run > 0.f ? a.v_scale / l_run : 0.f;
            const int t_tok = q_start + tok0 + r / G;
            const int qh = head * G + r % G;
            uint8_t* orow = a.o + ((size_t)t_tok * Hq + qh) * (D * 2);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(lane_addr + Gm::TM_O + c * 32, ov);
                tmem_ld_wait();
                if (r < rows_used) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 w;
                        w.x = pack2<false>(__uint_as_float(ov[8 * i + 0]) * inv, __uint_as_float(ov[8 * i + 1]) * inv);
                        w.y = pack2<false>(__uint_as_float(ov[8 * i + 2]) * inv, __uint_as_float(ov[8 * i + 3]) * inv);
                        w.z = pack2<false>(__uint_as_float(ov[8 * i + 4]) * inv, __uint_as_float(ov[8 * i + 5]) * inv);
                        w.w = pack2<false>(__uint_as_float(ov[8 * i + 6]) * inv, __uint_as_float(ov[8 * i + 7]) * inv);
                        put_u4(orow + c * 64 + i * 16, w);
                    }
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
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
struct TcKern {
    using Gm = TcGeom<D>;
    static cudaError_t prepare(int* bps) {
        cudaError_t e = cudaFuncSetAttribute(rpa_prefill_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bps, rpa_prefill_tc<D>, kThreads, Gm::SMEM);
    }
    static cudaError_t launch(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, const Launch& l) {
        rpa_prefill_tc<D><<<l.grid, kThreads, Gm::SMEM, l.stream>>>(kvm, qm, p);
        return cudaGetLastError();
    }
};

}  // namespace

cudaError_t prefill_tc_prepare(int D, int* bps) {
    if (D == 64) return TcKern<64>::prepare(bps);
    if (D == 128) return TcKern<128>::prepare(bps);
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_tc(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, const Launch& l) {
    if (p.a.D == 64) return TcKern<64>::launch(kvm, qm, p, l);
    if (p.a.D == 128) return TcKern<128>::launch(kvm, qm, p, l);
    return cudaErrorInvalidValue;
}

}  // namespace rpa
