// rpa_decode.cu -- K1 decode: paged-KV attention for tiles of <= 16 (or <= 8) query rows.
//
// Decode-class work items (q_len * G <= 16 rows of one kv head, a key range of
// one sequence) are HBM-bound: every key's K and V rows are read once and
// used by at most 16 rows.  The kernel is warp-specialised and persistent:
//
//   producer warp   pulls items from the planner's list, walks each item's
//                   keys in stages of 64, and gathers them through the page
//                   table ("ragged_paged.zig": createKvAsyncCopyDescriptors,
//                   logical page -> page_indices[s, page]) with bulk tensor
//                   copies: one copy per (page run, K/V, 128-byte column
//                   block), K rows of kv head h being combined head 2h and V
//                   rows 2h+1 of each slot.  The Q tile of an item (G
//                   consecutive heads of up to 16/G tokens) comes with the
//                   item's first stage.  A 3-stage mbarrier ring keeps copies
//                   in flight across item boundaries (the page's next-block
//                   prefetch, carried across sequences the same way).
//   4 consumer      each take 16 keys of every stage: S = Q K^T on mma.sync
//   warps           (fp32), scale / softcap / masks in the log2 domain, online
//                   softmax, O += P V; at the item's last stage the four
//                   partial (m, l, O) are merged through shared memory and
//                   written as bf16 o, or as an fp32 split-KV partial for the
//                   combine kernel.
//
// Tiles of at most 8 rows (bf16 K/V, G <= 8; the common decode case) put the
// keys on the MMA's M side instead: S^T = K Q^T and O^T += V^T P^T, half the
// MMAs and accumulator registers of a 16-row tile, three CTAs per SM.
//
// 2-byte K/V only: f16 K/V run the MMAs in f16, bf16 K/V in bf16, and Q
// arrives in that type.  (8-bit K/V take the 64-key-tile tensor-memory kernel,
// decode rows included.)
//
// Every wait is a bounded mbarrier wait (a global-timer deadline): on expiry
// the status word gets RPA_ERR_TIMEOUT and the warp returns.
#include <cuda.h>

#include "rpa_internal.cuh"

namespace rpa {

namespace {

constexpr int kCW = 4;                  // consumer warps
constexpr int kDecThreads = 32 * (kCW + 1);
constexpr int kKS = 64;                 // keys per stage (16 per consumer warp)
// stages in the ring: 3 for 16-row tiles (2 CTAs/SM), 2 for 8-row tiles (3 CTAs/SM)
constexpr int kMetaWords = 16;

// stage meta words
enum Meta : int {
    mItem = 0, mSeq, mHead, mQStart, mQl, mKl, mKvBegin, mKvEnd, mPart, mTok0, mNtok, mSt, mNst,
    mKey0, mStop
};

template <int D, int KT, int ROWS>
struct DecGeom {
    static_assert(!kt_8bit(KT), "2-byte K/V");
    static constexpr int NS = ROWS == 8 ? 2 : 3;   // stages in the ring
    static constexpr int DHQ = D * 2 / 128;        // 128-byte column blocks of a bf16 row
    static constexpr int DH = DHQ;                 // column blocks per K/V box
    static constexpr int QB = DHQ * ROWS * 128;    // Q area: [DHQ][ROWS lines][128 B]
    static constexpr int KVB = kKS * 2 * D * 2;    // K/V area of one stage
    static constexpr int SB = QB + KVB;            // one stage
    static constexpr int SMEM = NS * SB + 1024;    // + alignment slack
    static_assert(QB % 1024 == 0 && KVB % 1024 == 0, "stage alignment");
    static_assert(kCW * ROWS * D * 4 <= KVB, "merge area");
};

__device__ __forceinline__ uint32_t swz128(uint32_t line, uint32_t chunk) {
    return line * 128u + (((chunk ^ line) & 7u) << 4);
}

// resident CTAs per SM the register allocation is sized for (shared memory allows 2 at D <= 128,
// 3 with 8-row tiles; D = 256 fits one)
template <int D, int ROWS>
constexpr int dec_min_blocks() { return D > 128 ? 1 : ROWS == 8 ? 3 : 2; }

// The kernel body; `kvmap` and `qmap` point at the kernel's grid-constant tensor-map parameters.
template <int D, int KT, int ROWS>
__device__ __forceinline__ void decode_body(const CUtensorMap& kvmap, const CUtensorMap& qmap, const DecParams& p) {
    using Gm = DecGeom<D, KT, ROWS>;
    constexpr int kNS = Gm::NS;
    constexpr bool F16 = kt_f16_mma(KT);  // MMA operands in f16 (else bf16)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kNS];
    __shared__ __align__(8) uint64_t empty_bar[kNS];
    __shared__ __align__(8) uint64_t merge_bar;
    __shared__ int meta[kNS][kMetaWords];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const AttnParams& a = p.a;
    int* ctrl = a.ctrl;
    const uint64_t tmo = p.timeout_ns;
    // 1 KiB-aligned base: the 128-byte swizzle pattern follows address bits 7..9
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t smem0 = smem_u32(smem);

    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), kCW);
        }
        mbar_init(smem_u32(&merge_bar), kCW);
        fence_mbar_init();
    }
    __shared__ int s_plan_ok;
    __syncthreads();
    pdl_trigger();
    if (p.plan_epoch >= 0) {
        // behind the prefill kernel on one stream: the planner's items are complete once it has
        // published this call's epoch
        if (tid == 0) s_plan_ok = flag_wait(ctrl + kPlanEpoch, p.plan_epoch, ctrl, tmo) ? 1 : 0;
        __syncthreads();
        if (!s_plan_ok) return;
    } else {
        pdl_wait();  // the planner's items are complete from here on
    }
    if ((int)blockIdx.x >= a.ctrl[kDecCtas]) return;  // SMs left to the prefill kernel
    const int n_items = a.ctrl[a.item_count_word];

    if (warp == kCW) {
        // =============================== producer ===============================
        if (p.debug_stall) return;  // test hook: consumers must time out
        const int BR = p.BR, ps = a.ps;
        const int runs = kKS / BR;  // page runs per stage, one bulk copy each (K and V of the head)
        const uint32_t run_bytes = (uint32_t)(2 * Gm::DH * BR * 128);
        const uint64_t pol_stream = l2_policy_evict_first();
        int s = 0;
        uint32_t ph = 0;
        int it = 0;
        if (lane == 0) it = atomicAdd(ctrl + a.counter_word, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        bool ok = true;
        while (ok && it < n_items) {
            const Item item = item_at(a.units, it, a.unit_heads);
            int nxt = 0;
            if (lane == 0) nxt = atomicAdd(ctrl + a.counter_word, 1);
            const int q_start = a.cu_q_lens[item.seq];
            const int ql = a.cu_q_lens[item.seq + 1] - q_start;
            const int kl = a.kv_lens[item.seq];
            const int* ptab = a.page_indices + (size_t)item.seq * a.P;
            const int key0 = item.kv_begin - (item.kv_begin & (BR - 1));
            const int nst = (item.kv_end - key0 + kKS - 1) / kKS;
            // page ids of 32 consecutive logical pages, one per lane
            int win0 = key0 / ps;
            int win = (win0 + lane < a.P) ? __ldg(ptab + win0 + lane) : 0;
            for (int st = 0; st < nst && ok; ++st) {
                const int k_stage = key0 + st * kKS;
                // make sure the page-id window covers this stage
                const int lp_last = min(k_stage + kKS - 1, item.kv_end - 1) / ps;
                if (lp_last - win0 >= 32) {
                    win0 = k_stage / ps;
                    win = (win0 + lane < a.P) ? __ldg(ptab + win0 + lane) : 0;
                }
                if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1u, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                const uint32_t st_base = smem0 + s * Gm::SB;
                const uint32_t kv_base = st_base + Gm::QB;
                // lane r < runs copies page run r of this stage (BR keys of one page)
                const int k0 = k_stage + lane * BR;
                const int lp = k0 / ps;
                const int pg = __shfl_sync(0xffffffffu, win, (lp - win0) & 31);
                const bool want = lane < runs && k0 < item.kv_end && k0 + BR > item.kv_begin;
                const bool good = (unsigned)pg < (unsigned)a.N;
                const int n_issue = __popc(__ballot_sync(0xffffffffu, want && good));
                if (__any_sync(0xffffffffu, want && !good)) {
                    // a page id outside [0, N): never dereferenced; its keys read as zero
                    if (lane == 0) set_status(ctrl, RPA_ERR_BAD_PAGE_INDEX);
                    for (int i = lane; i < Gm::KVB / 16; i += 32)
                        *reinterpret_cast<uint4*>(smem + (kv_base - smem0) + i * 16) = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                }
                if (lane == 0) {
                    int* m = meta[s];
                    m[mItem] = it;
                    m[mSeq] = item.seq;
                    m[mHead] = item.head;
                    m[mQStart] = q_start;
                    m[mQl] = ql;
                    m[mKl] = kl;
                    m[mKvBegin] = item.kv_begin;
                    m[mKvEnd] = item.kv_end;
                    m[mPart] = item.part;
                    m[mTok0] = item.tok0;
                    m[mNtok] = item.ntok;
                    m[mSt] = st;
                    m[mNst] = nst;
                    m[mKey0] = k_stage;
                    m[mStop] = 0;
                }
                __syncwarp();
                const uint32_t fb = smem_u32(&full_bar[s]);
                if (lane == 0)
                    mbar_arrive_expect_tx(fb, (uint32_t)n_issue * run_bytes +
                                                  (st == 0 ? (uint32_t)(Gm::DHQ * p.Tt * a.G * 128) : 0u));
                __syncwarp();
                if (st == 0 && lane < Gm::DHQ)
                    tma_load_3d(st_base + lane * (ROWS * 128), &qmap, fb, lane * 64, item.head * a.G,
                                q_start + item.tok0);
                // decode K/V is read once: evict it first, so that it does not push out of L2 the
                // K/V a concurrent prefill re-reads
                if (want && good)
                    tma_load_3d_hint(kv_base + (uint32_t)lane * run_bytes, &kvmap, fb, 0, pg * ps + (k0 - lp * ps),
                                     2 * item.head * Gm::DH, pol_stream);
                if (++s == kNS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            it = __shfl_sync(0xffffffffu, nxt, 0);
        }
        if (ok && mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1u, ctrl, tmo)) {
            if (lane == 0) {
                meta[s][mStop] = 1;
                mbar_arrive(smem_u32(&full_bar[s]));
            }
        } else {
            // gave up: let the copies already issued land before leaving
            for (int i = 0; i < kNS; ++i) mbar_wait(smem_u32(&full_bar[i]), 0, ctrl, tmo);
        }
        return;
    }

    if constexpr (ROWS == 16) {
    // =============================== consumers ===============================
    const int w = warp;
    const int G = a.G, Hq = a.Hq;
    const int BR = p.BR, br_shift = p.br_shift;
    const uint32_t PBB = (uint32_t)(2 * Gm::DH * BR * 128);
    int s = 0;
    uint32_t ph = 0, mph = 0;
    uint32_t qf[D / 16][4];
    float o_acc[D / 8][4];
    float m_r[2], l_r[2];
    int pos[2];
    for (;;) {
        if (!mbar_wait(smem_u32(&full_bar[s]), ph, ctrl, tmo)) return;
        const int* m = meta[s];
        if (m[mStop]) return;
        const int st = m[mSt], nst = m[mNst];
        const int kv_begin = m[mKvBegin], kv_end = m[mKvEnd];
        const int kl = m[mKl], ql = m[mQl];
        const int tok0 = m[mTok0], ntok = m[mNtok];
        const uint32_t st_base = smem0 + s * Gm::SB;
        const uint32_t kv_base = st_base + Gm::QB;
        if (st == 0) {
            // Q fragments (A operand) for the whole item, from the stage's Q area
#pragma unroll
            for (int kd = 0; kd < D / 16; ++kd) {
                const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = 2 * kd + (lane >> 4);
                const uint32_t line = (uint32_t)((c >> 3) * 16 + r);
                ldsm_x4(st_base + swz128(line, c & 7), qf[kd][0], qf[kd][1], qf[kd][2], qf[kd][3]);
            }
#pragma unroll
            for (int i = 0; i < D / 8; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
            m_r[0] = m_r[1] = -INFINITY;
            l_r[0] = l_r[1] = 0.f;
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) pos[ri] = kl - ql + tok0 + ((lane >> 2) + ri * 8) / G;
        }

        // ---- this warp's 16 keys: [kw, kw + 16)
        const int kw = m[mKey0] + 16 * w;
        const bool any_in = kw < kv_end && kw + 16 > kv_begin;
        if (any_in) {
            const bool partial = kw < kv_begin || kw + 16 > kv_end;
            if (partial) {
                // keys of this slice outside [kv_begin, kv_end): V rows to zero
                for (int i = lane; i < 16 * Gm::DH * 8; i += 32) {
                    const int row = i / (Gm::DH * 8);
                    const int c = i % (Gm::DH * 8);
                    const int j = kw + row;
                    if (j >= kv_begin && j < kv_end) continue;
                    const int kk = 16 * w + row;
                    const int b = kk >> br_shift, r = kk & (BR - 1);
                    const uint32_t line = (uint32_t)((Gm::DH + (c >> 3)) * BR + r);
                    *reinterpret_cast<uint4*>(smem + (kv_base - smem0) + b * PBB + swz128(line, c & 7)) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // bases of row 0 for the ldmatrix addresses below (K and V blocks of the stage's page runs)
            const uint32_t kb = kv_base, vb = kv_base;

            // ---- S = Q K^T  (16 rows x 16 keys); even and odd k-steps accumulate separately
            // (two independent MMA chains per n-block), summed at the end -- at D 64: at D 128 and 256
            // the registers are spent on Q and O, and one chain per n-block keeps them unspilled
            constexpr bool kTwo = D <= 64;
            float sacc[2][4], sodd[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
                sodd[i][0] = sodd[i][1] = sodd[i][2] = sodd[i][3] = 0.f;
            }
            {
                const int row = (lane & 7) + (lane >> 4) * 8;  // key row of this lane's ldmatrix
#pragma unroll
                for (int kd = 0; kd < D / 16; ++kd) {
                    const int c = 2 * kd + ((lane >> 3) & 1);
                    const int kk = 16 * w + row;
                    const int b = kk >> br_shift, r = kk & (BR - 1);
                    const uint32_t line = (uint32_t)((c >> 3) * BR + r);
                    const uint32_t addr = kb + b * PBB + swz128(line, c & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(addr, b0, b1, b2, b3);
                    mma16816<F16>((kTwo && (kd & 1)) ? sodd[0] : sacc[0], qf[kd], b0, b1);
                    mma16816<F16>((kTwo && (kd & 1)) ? sodd[1] : sacc[1], qf[kd], b2, b3);
                }
                if constexpr (kTwo) {
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sacc[i][e] += sodd[i][e];
                }
            }
            // ---- scale, softcap, masks (log2 domain)
            const bool need_mask = partial || (a.causal && kw + 15 > kl - ql + tok0) ||
                                   (a.has_window && kw <= kl - ql + tok0 + ntok - 1 - a.window);
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int ri = e >> 1;
                    float x = sacc[nb][e];
                    if (a.has_cap) {
                        const float t = ex2(x * a.cap_exp);
                        x = a.cap_log2 - 2.f * a.cap_log2 * rcp_approx(1.f + t);
                    } else {
                        x *= a.qk_log2;
                    }
                    if (need_mask) {
                        const int j = kw + nb * 8 + (lane & 3) * 2 + (e & 1);
                        const bool okk = j >= kv_begin && j < kv_end && (!a.causal || j <= pos[ri]) &&
                                         (!a.has_window || j > pos[ri] - a.window);
                        x = okk ? x : -INFINITY;
                    }
                    sacc[nb][e] = x;
                    mx[ri] = fmaxf(mx[ri], x);
                }
            }
            // lazy rescale: the running max moves only when some row's max grows by more than
            // 2^8 (P and l use the same stale max, so the result is unchanged; P stays <= 2^8)
            float base[2];
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 1));
                mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 2));
            }
            const bool need = __any_sync(0xffffffffu, mx[0] > m_r[0] + 8.f || mx[1] > m_r[1] + 8.f);
            if (need) {
#pragma unroll
                for (int ri = 0; ri < 2; ++ri) {
                    const float m_new = fmaxf(m_r[ri], mx[ri]);
                    const float b = m_new == -INFINITY ? 0.f : m_new;
                    const float alpha = m_r[ri] == -INFINITY ? 0.f : ex2(m_r[ri] - b);
                    m_r[ri] = m_new;
                    l_r[ri] *= alpha;
#pragma unroll
                    for (int nd = 0; nd < D / 8; ++nd) {
                        o_acc[nd][2 * ri] *= alpha;
                        o_acc[nd][2 * ri + 1] *= alpha;
                    }
                }
            }
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) base[ri] = m_r[ri] == -INFINITY ? 0.f : m_r[ri];
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pe = ex2(sacc[nb][e] - base[e >> 1]);
                    sacc[nb][e] = pe;
                    l_r[e >> 1] += pe;
                }
            }
            // ---- O += P V
            {
                uint32_t pa[4];
                pa[0] = pack2<F16>(sacc[0][0], sacc[0][1]);
                pa[1] = pack2<F16>(sacc[0][2], sacc[0][3]);
                pa[2] = pack2<F16>(sacc[1][0], sacc[1][1]);
                pa[3] = pack2<F16>(sacc[1][2], sacc[1][3]);
                const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int nd2 = 0; nd2 < D / 16; ++nd2) {
                    const int c = 2 * nd2 + (lane >> 4);
                    const int kk = 16 * w + row;
                    const int b = kk >> br_shift, r = kk & (BR - 1);
                    const uint32_t line = (uint32_t)((Gm::DH + (c >> 3)) * BR + r);
                    const uint32_t addr = vb + b * PBB + swz128(line, c & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(addr, b0, b1, b2, b3);
                    mma16816<F16>(o_acc[2 * nd2], pa, b0, b1);
                    mma16816<F16>(o_acc[2 * nd2 + 1], pa, b2, b3);
                }
            }
        }

        const uint32_t eb = smem_u32(&empty_bar[s]);
        if (st == nst - 1) {
            // ---- merge the four warps' partials; the stage's own buffers hold them
            float* red_o = reinterpret_cast<float*>(smem + (kv_base - smem0));  // [kCW][16][D]
            float* red_ml = reinterpret_cast<float*>(smem + (st_base - smem0));        // [kCW][16][2]
            float lsum[2];
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                lsum[ri] = l_r[ri] + __shfl_xor_sync(0xffffffffu, l_r[ri], 1);
                lsum[ri] += __shfl_xor_sync(0xffffffffu, lsum[ri], 2);
            }
            const uint32_t mb = smem_u32(&merge_bar);
            __syncwarp();
            if (lane == 0) mbar_arrive(mb);  // A: every warp is done reading the stage
            if (!mbar_wait(mb, mph, ctrl, tmo)) return;
            mph ^= 1u;
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                const int r = (lane >> 2) + ri * 8;
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd)
                    *reinterpret_cast<float2*>(red_o + (w * 16 + r) * D + nd * 8 + (lane & 3) * 2) =
                        make_float2(o_acc[nd][2 * ri], o_acc[nd][2 * ri + 1]);
                if ((lane & 3) == 0) {
                    red_ml[(w * 16 + r) * 2] = m_r[ri];
                    red_ml[(w * 16 + r) * 2 + 1] = lsum[ri];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(mb);  // B: every partial is in shared memory
            if (!mbar_wait(mb, mph, ctrl, tmo)) return;
            mph ^= 1u;
            const int rows_used = ntok * G;
            const int part = m[mPart];
            const int q_start = m[mQStart];
            const int head = m[mHead];
            for (int e = w * 32 + lane; e < 16 * (D / 2); e += kCW * 32) {
                const int r = e / (D / 2);
                const int c = (e % (D / 2)) * 2;
                if (r >= rows_used) break;
                float M = -INFINITY;
#pragma unroll
                for (int ww = 0; ww < kCW; ++ww) M = fmaxf(M, red_ml[(ww * 16 + r) * 2]);
                float L = 0.f, o0 = 0.f, o1 = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int ww = 0; ww < kCW; ++ww) {
                        const float sc = ex2(red_ml[(ww * 16 + r) * 2] - M);
                        L += sc * red_ml[(ww * 16 + r) * 2 + 1];
                        const float2 v = *reinterpret_cast<const float2*>(red_o + (ww * 16 + r) * D + c);
                        o0 += sc * v.x;
                        o1 += sc * v.y;
                    }
                }
                if (part < 0) {
                    const int t = q_start + tok0 + r / G;
                    const int qh = head * G + r % G;
                    L = add_sink(L, a.sinks, qh, M);
                    const float inv = L > 0.f ? a.v_scale / L : 0.f;
                    store_o2(a.o, ((size_t)t * Hq + qh) * D + c, o0 * inv, o1 * inv, a.odt);
                } else {
                    *reinterpret_cast<float2*>(a.part_o + ((size_t)part * kDecRows + r) * D + c) =
                        make_float2(o0, o1);
                    if (c == 0)
                        *reinterpret_cast<float2*>(a.part_ml + ((size_t)part * kDecRows + r) * 2) =
                            make_float2(M, L);
                }
            }
            fence_proxy_async_smem();  // the stage will be refilled by bulk copies
            __syncwarp();
            if (lane == 0) mbar_arrive(eb);
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(eb);
        }
        if (++s == kNS) {
            s = 0;
            ph ^= 1u;
        }
    }
    } else {
    // ====================== consumers, tiles of <= 8 rows: keys on the MMA's M side ======================
    // S^T = K Q^T with A = 16 keys x 16 d of the stage (ldmatrix) and B = Q^T (16 d x 8 rows, registers,
    // loaded once per item); O^T += V^T P^T with A = 16 d x 16 keys (ldmatrix.trans) and B = P^T (16 keys
    // x 8 rows, built from S^T's accumulators with four shuffles).  Half the MMAs of a 16-row tile and
    // half its accumulator registers.  Thread (g = lane / 4, q = lane % 4) holds rows 2q and 2q + 1 of
    // keys g and g + 8 (S^T), and of d = 16 mt + g and + 8 (O^T, m-tile mt).
    const int w = warp;
    const int G = a.G, Hq = a.Hq;
    const int BR = p.BR, br_shift = p.br_shift;
    const uint32_t PBB = (uint32_t)(2 * Gm::DH * BR * 128);
    const int g = lane >> 2, q = lane & 3;
    int s = 0;
    uint32_t ph = 0, mph = 0;
    uint32_t qt[D / 16][2];
    float o_acc[D / 16][4];
    float m_r[2], l_r[2];
    int pos[2];  // kv positions of rows 2q, 2q + 1
    for (;;) {
        if (!mbar_wait(smem_u32(&full_bar[s]), ph, ctrl, tmo)) return;
        const int* m = meta[s];
        if (m[mStop]) return;
        const int st = m[mSt], nst = m[mNst];
        const int kv_begin = m[mKvBegin], kv_end = m[mKvEnd];
        const int kl = m[mKl], ql = m[mQl];
        const int tok0 = m[mTok0], ntok = m[mNtok];
        const uint32_t st_base = smem0 + s * Gm::SB;
        const uint32_t kv_base = st_base + Gm::QB;
        if (st == 0) {
            // Q^T fragments (B operand) for the whole item: rows 0-7 of the stage's Q area, two
            // k-steps per ldmatrix.x4 (matrix i: d chunk 2 kd + i)
#pragma unroll
            for (int kd = 0; kd < D / 16; kd += 2) {
                const int c = 2 * kd + (lane >> 3);
                const uint32_t line = (uint32_t)((c >> 3) * ROWS + (lane & 7));
                ldsm_x4(st_base + swz128(line, c & 7), qt[kd][0], qt[kd][1], qt[kd + 1][0], qt[kd + 1][1]);
            }
#pragma unroll
            for (int i = 0; i < D / 16; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
            m_r[0] = m_r[1] = -INFINITY;
            l_r[0] = l_r[1] = 0.f;
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) pos[ri] = kl - ql + tok0 + (2 * q + ri) / G;
        }

        // ---- this warp's 16 keys: [kw, kw + 16)
        const int kw = m[mKey0] + 16 * w;
        const bool any_in = kw < kv_end && kw + 16 > kv_begin;
        if (any_in) {
            const bool partial = kw < kv_begin || kw + 16 > kv_end;
            if (partial) {
                // keys of this slice outside [kv_begin, kv_end): V rows to zero
                for (int i = lane; i < 16 * Gm::DH * 8; i += 32) {
                    const int row = i / (Gm::DH * 8);
                    const int c = i % (Gm::DH * 8);
                    const int j = kw + row;
                    if (j >= kv_begin && j < kv_end) continue;
                    const int kk = 16 * w + row;
                    const int b = kk >> br_shift, r = kk & (BR - 1);
                    const uint32_t line = (uint32_t)((Gm::DH + (c >> 3)) * BR + r);
                    *reinterpret_cast<uint4*>(smem + (kv_base - smem0) + b * PBB + swz128(line, c & 7)) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }

            // ---- S^T = K Q^T  (16 keys x 8 rows); even and odd k-steps in two MMA chains
            float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sodd[4] = {0.f, 0.f, 0.f, 0.f};
            {
                // A matrices: keys 0-7 / 8-15 (lane bit 3) of d chunk 2 kd / 2 kd + 1 (lane bit 4)
                const int kk = 16 * w + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int b = kk >> br_shift, r = kk & (BR - 1);
#pragma unroll
                for (int kd = 0; kd < D / 16; ++kd) {
                    const int c = 2 * kd + (lane >> 4);
                    const uint32_t line = (uint32_t)((c >> 3) * BR + r);
                    uint32_t af[4];
                    ldsm_x4(kv_base + b * PBB + swz128(line, c & 7), af[0], af[1], af[2], af[3]);
                    mma16816<F16>((kd & 1) ? sodd : sacc, af, qt[kd][0], qt[kd][1]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[e] += sodd[e];
            }
            // ---- scale, softcap, masks (log2 domain); sacc[e]: key g + 8 (e >> 1), row 2q + (e & 1)
            const bool need_mask = partial || (a.causal && kw + 15 > kl - ql + tok0) ||
                                   (a.has_window && kw <= kl - ql + tok0 + ntok - 1 - a.window);
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int ri = e & 1;
                float x = sacc[e];
                if (a.has_cap) {
                    const float t = ex2(x * a.cap_exp);
                    x = a.cap_log2 - 2.f * a.cap_log2 * rcp_approx(1.f + t);
                } else {
                    x *= a.qk_log2;
                }
                if (need_mask) {
                    const int j = kw + g + 8 * (e >> 1);
                    const bool okk = j >= kv_begin && j < kv_end && (!a.causal || j <= pos[ri]) &&
                                     (!a.has_window || j > pos[ri] - a.window);
                    x = okk ? x : -INFINITY;
                }
                sacc[e] = x;
                mx[ri] = fmaxf(mx[ri], x);
            }
            // row max over the warp's 16 keys: the eight lanes of a row differ in lane bits 2-4
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 4));
                mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 8));
                mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 16));
            }
            // lazy rescale: the running max moves only when some row's max grows by more than 2^8
            const bool need = __any_sync(0xffffffffu, mx[0] > m_r[0] + 8.f || mx[1] > m_r[1] + 8.f);
            if (need) {
#pragma unroll
                for (int ri = 0; ri < 2; ++ri) {
                    const float m_new = fmaxf(m_r[ri], mx[ri]);
                    const float bse = m_new == -INFINITY ? 0.f : m_new;
                    const float alpha = m_r[ri] == -INFINITY ? 0.f : ex2(m_r[ri] - bse);
                    m_r[ri] = m_new;
                    l_r[ri] *= alpha;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        o_acc[mt][ri] *= alpha;
                        o_acc[mt][ri + 2] *= alpha;
                    }
                }
            }
            float base[2];
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) base[ri] = m_r[ri] == -INFINITY ? 0.f : m_r[ri];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float pe = ex2(sacc[e] - base[e & 1]);
                sacc[e] = pe;
                l_r[e & 1] += pe;
            }
            // ---- P^T as the B operand: b0 = P[key 2q, 2q + 1][row g], b1 = P[key 2q + 8, 2q + 9][row g].
            // P[key k][row n] (k < 8) sits in lane 4k + n/2, element n % 2 (keys 8-15: elements 2, 3).
            uint32_t pb0, pb1;
            {
                const uint32_t w01 = pack2<F16>(sacc[0], sacc[1]);  // key g:     rows 2q, 2q + 1
                const uint32_t w23 = pack2<F16>(sacc[2], sacc[3]);  // key g + 8: rows 2q, 2q + 1
                const int src0 = 8 * q + (g >> 1), src1 = src0 + 4;   // lanes of keys 2q, 2q + 1
                const uint32_t x0 = __shfl_sync(0xffffffffu, w01, src0);
                const uint32_t x1 = __shfl_sync(0xffffffffu, w01, src1);
                const uint32_t y0 = __shfl_sync(0xffffffffu, w23, src0);
                const uint32_t y1 = __shfl_sync(0xffffffffu, w23, src1);
                const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;  // row g's half of each word
                pb0 = __byte_perm(x0, x1, sel);
                pb1 = __byte_perm(y0, y1, sel);
            }
            // ---- O^T += V^T P^T: A matrices: d chunk 2 mt / 2 mt + 1 (lane bit 3) of keys 0-7 / 8-15
            // (lane bit 4), transposed
            {
                const int kk = 16 * w + (lane & 7) + (lane >> 4) * 8;
                const int b = kk >> br_shift, r = kk & (BR - 1);
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const int c = 2 * mt + ((lane >> 3) & 1);
                    const uint32_t line = (uint32_t)((Gm::DH + (c >> 3)) * BR + r);
                    uint32_t af[4];
                    ldsm_x4_t(kv_base + b * PBB + swz128(line, c & 7), af[0], af[1], af[2], af[3]);
                    mma16816<F16>(o_acc[mt], af, pb0, pb1);
                }
            }
        }

        const uint32_t eb = smem_u32(&empty_bar[s]);
        if (st == nst - 1) {
            // ---- merge the four warps' partials; the stage's own buffers hold them
            float* red_o = reinterpret_cast<float*>(smem + (kv_base - smem0));  // [kCW][ROWS][D]
            float* red_ml = reinterpret_cast<float*>(smem + (st_base - smem0)); // [kCW][ROWS][2]
            float lsum[2];
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                lsum[ri] = l_r[ri] + __shfl_xor_sync(0xffffffffu, l_r[ri], 4);
                lsum[ri] += __shfl_xor_sync(0xffffffffu, lsum[ri], 8);
                lsum[ri] += __shfl_xor_sync(0xffffffffu, lsum[ri], 16);
            }
            const uint32_t mb = smem_u32(&merge_bar);
            __syncwarp();
            if (lane == 0) mbar_arrive(mb);  // A: every warp is done reading the stage
            if (!mbar_wait(mb, mph, ctrl, tmo)) return;
            mph ^= 1u;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    red_o[(w * ROWS + 2 * q + (e & 1)) * D + 16 * mt + g + 8 * (e >> 1)] = o_acc[mt][e];
            if (g == 0) {
#pragma unroll
                for (int ri = 0; ri < 2; ++ri) {
                    red_ml[(w * ROWS + 2 * q + ri) * 2] = m_r[ri];
                    red_ml[(w * ROWS + 2 * q + ri) * 2 + 1] = lsum[ri];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(mb);  // B: every partial is in shared memory
            if (!mbar_wait(mb, mph, ctrl, tmo)) return;
            mph ^= 1u;
            const int rows_used = ntok * G;
            const int part = m[mPart];
            const int q_start = m[mQStart];
            const int head = m[mHead];
            for (int e = w * 32 + lane; e < ROWS * (D / 2); e += kCW * 32) {
                const int r = e / (D / 2);
                const int c = (e % (D / 2)) * 2;
                if (r >= rows_used) break;
                float M = -INFINITY;
#pragma unroll
                for (int ww = 0; ww < kCW; ++ww) M = fmaxf(M, red_ml[(ww * ROWS + r) * 2]);
                float L = 0.f, o0 = 0.f, o1 = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int ww = 0; ww < kCW; ++ww) {
                        const float sc = ex2(red_ml[(ww * ROWS + r) * 2] - M);
                        L += sc * red_ml[(ww * ROWS + r) * 2 + 1];
                        const float2 v = *reinterpret_cast<const float2*>(red_o + (ww * ROWS + r) * D + c);
                        o0 += sc * v.x;
                        o1 += sc * v.y;
                    }
                }
                if (part < 0) {
                    const int t = q_start + tok0 + r / G;
                    const int qh = head * G + r % G;
                    L = add_sink(L, a.sinks, qh, M);
                    const float inv = L > 0.f ? a.v_scale / L : 0.f;
                    store_o2(a.o, ((size_t)t * Hq + qh) * D + c, o0 * inv, o1 * inv, a.odt);
                } else {
                    *reinterpret_cast<float2*>(a.part_o + ((size_t)part * kDecRows + r) * D + c) =
                        make_float2(o0, o1);
                    if (c == 0)
                        *reinterpret_cast<float2*>(a.part_ml + ((size_t)part * kDecRows + r) * 2) =
                            make_float2(M, L);
                }
            }
            fence_proxy_async_smem();  // the stage will be refilled by bulk copies
            __syncwarp();
            if (lane == 0) mbar_arrive(eb);
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(eb);
        }
        if (++s == kNS) {
            s = 0;
            ph ^= 1u;
        }
    }
    }
}

template <int D, int KT, int ROWS>
__global__ void __launch_bounds__(kDecThreads, dec_min_blocks<D, ROWS>()) rpa_decode_attn(
    const __grid_constant__ CUtensorMap kvmap, const __grid_constant__ CUtensorMap qmap, const DecParams p) {
    decode_body<D, KT, ROWS>(kvmap, qmap, p);
    // behind the prefill kernel: this grid completes only after it (the combine kernel and the
    // next call depend on this grid alone)
    if (p.plan_epoch >= 0) pdl_wait();
}

template <int D, int KT, int ROWS>
struct DecKern {
    using Gm = DecGeom<D, KT, ROWS>;
    static constexpr auto fn() { return rpa_decode_attn<D, KT, ROWS>; }
    static cudaError_t prepare(int* bps) {
        cudaError_t e = cudaFuncSetAttribute(fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::SMEM);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bps, fn(), kDecThreads, Gm::SMEM);
    }
    static cudaError_t launch(const CUtensorMap& kvm, const CUtensorMap& qm, const DecParams& p,
                              const Launch& l) {
        return launch_pdl(fn(), l.grid, kDecThreads, Gm::SMEM, l.stream, kvm, qm, p);
    }
};

// The instantiations: 2-byte K/V at D 64 / 128 / 256 with 8- or 16-row tiles (8-bit K/V take the
// 64-key-tile tensor-memory kernel).  `op` is called with the kernel type, or the result is
// cudaErrorInvalidValue.
template <typename Op>
cudaError_t dec_dispatch(int D, int kt, int rows, Op op) {
    if (kt_8bit(kt)) return cudaErrorInvalidValue;
    const bool f16 = kt == KT_F16;
    if (rows == 8) {
        if (D == 64) return f16 ? op(DecKern<64, KT_F16, 8>{}) : op(DecKern<64, KT_BF16, 8>{});
        if (D == 128) return f16 ? op(DecKern<128, KT_F16, 8>{}) : op(DecKern<128, KT_BF16, 8>{});
        if (D == 256) return f16 ? op(DecKern<256, KT_F16, 8>{}) : op(DecKern<256, KT_BF16, 8>{});
    } else if (rows == 16) {
        if (D == 64) return f16 ? op(DecKern<64, KT_F16, 16>{}) : op(DecKern<64, KT_BF16, 16>{});
        if (D == 128) return f16 ? op(DecKern<128, KT_F16, 16>{}) : op(DecKern<128, KT_BF16, 16>{});
        if (D == 256) return f16 ? op(DecKern<256, KT_F16, 16>{}) : op(DecKern<256, KT_BF16, 16>{});
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_prepare(int D, int kt, int rows, int* bps) {
    return dec_dispatch(D, kt, rows, [&](auto k) { return decltype(k)::prepare(bps); });
}

cudaError_t launch_decode_tma(const CUtensorMap& kvm, const CUtensorMap& qm, const DecParams& p, int kt,
                              int rows, const Launch& l) {
    return dec_dispatch(p.a.D, kt, rows, [&](auto k) { return decltype(k)::launch(kvm, qm, p, l); });
}

}  // namespace rpa
