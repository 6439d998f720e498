// rpa_mla.cu -- latent attention over a paged latent cache.
//
// The latent form of the "from_qwen_ops.rs" page ("The latent-attention family at whole-tile
// widths": a 512-wide latent and a 64-wide rope part, sixteen or more heads of 576): every slot of
// a page holds one row of DQ = 576 elements per kv head; a key is that whole row and its value is
// the row's first DV = 512 elements.  q is [T, Hq, 576], o is [T, Hq, 512].  Masks, soft cap,
// scales and sinks are those of the rest of the library.
//
// Work items are tiles of 16 query rows (the tokens x heads of a block of G' <= 16 query heads that
// share one kv head) against a key range; long key ranges are split into pieces that the combine
// kernel merges.  One persistent CTA per SM:
//
//   producer warp   per item its Q tile (nine 128-byte column blocks, into one of two Q buffers),
//                   then per 64-key stage one bulk tensor copy per page run of the latent rows
//                   ("ragged_paged.zig": createKvAsyncCopyDescriptors, logical page ->
//                   page_indices[s, page]) into a 2-stage mbarrier ring, crossing item boundaries.
//   8 consumer      S = Q K^T: warp w takes k-steps [9 (w % 4), 9 (w % 4) + 9) of the 576-wide
//   warps           contraction for keys 32 (w / 4) .. + 31 of the stage (mma.sync, fp32; four
//                   independent accumulator chains; its Q fragments from the item's Q buffer),
//                   the partial sums meet in shared memory and warp w adds up keys 8w .. 8w+7; scale / soft cap
//                   / masks in the log2 domain; the row maxima meet in shared memory, every warp
//                   forms the same running max, writes its P (bf16 / f16) to shared memory and
//                   keeps its own partial row sum; then
//                   O += P V: warp w owns value columns 64w .. 64w+63 of all 16 rows (V is the first
//                   512 columns of the very rows of the stage).  Lazy rescale (the max grows by more
//                   than 2^8).  At the item's end the row sums meet in shared memory and each warp
//                   writes its 64 columns of o, or of an fp32 split-KV partial.
//
// Why not the tensor-memory MMAs here: with the query rows on the M side an fp32 accumulator of
// 512 value columns fills all 512 columns of a tensor-memory lane, which leaves no room for S; with
// the keys on the M side (S^T = K Q^T at M = 64, N = 16; O^T += V^T P^T at M = 128, N = 16) each
// MMA of these shapes measured ~60-80 cycles whatever its size, ~3.5k cycles of tensor pipe a 64-key
// stage for 52 of them, longer than this kernel's whole stage.  The rows of a decode tile are few
// (the heads that share a latent row), so the warp MMAs keep O in registers (32 floats a thread).
//
// Every wait is a bounded mbarrier wait (a global-timer deadline): on expiry the status word gets
// RPA_ERR_TIMEOUT and the warp returns.
#include <cuda.h>

#include "rpa_internal.cuh"

namespace rpa {

namespace {

constexpr int kMlaCW = 8;                      // consumer warps
constexpr int kMlaThreads = 32 * (kMlaCW + 1);
constexpr int kQK = kMlaDqk;                   // 576
constexpr int kV = kMlaDv;                     // 512
constexpr int kCBQ = kQK / 64;                 // 128-byte column blocks of a latent row (9)
constexpr int kRows = kMlaRows;                // query rows of an item (16)
constexpr int kKS = 64;                        // keys per stage
constexpr int kNS = 2;                         // stages
constexpr int kStage = kKS * kQK * 2;          // 73728 bytes
constexpr int kQBuf = kCBQ * kRows * 128;      // 18432 bytes: [9 column blocks][16 rows][128 B]
constexpr int kPBuf = kRows * kKS * 2;         // P: [16 rows][64 keys] 16-bit, 2048 bytes
constexpr int kMlaSmem = kNS * kStage + 2 * kQBuf + kPBuf + 1024;
constexpr float kRescaleLog2 = 8.f;
constexpr int kSPad = 72;                      // row stride (floats) of the partial-S exchange
constexpr int kKSteps = kQK / 16;              // k-steps of the QK contraction (36)
constexpr int kKSlices = 4;                    // the contraction split four ways, the keys two ways
constexpr int kSliceSteps = kKSteps / kKSlices;  // 9
static_assert(kKSlices * 2 == kMlaCW && kKSteps % kKSlices == 0, "warp split of S");

enum MlaMeta : int { mSeq = 0, mHead, mQStart, mQl, mKl, mKvBegin, mKvEnd, mPart, mTok0, mNtok, mSt, mNst, mKey0,
                     mQb, mStop, mWords = 16 };

__device__ __forceinline__ uint32_t swz128(uint32_t line, uint32_t chunk) {
    return line * 128u + (((chunk ^ line) & 7u) << 4);
}

template <bool F16>
__global__ void __launch_bounds__(kMlaThreads, 1) rpa_mla_attn(const __grid_constant__ CUtensorMap kvmap,
                                                               const __grid_constant__ CUtensorMap qmap,
                                                               const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kNS], empty_bar[kNS], q_full[2], q_empty[2];
    // exchanges among the consumer warps (bounded mbarrier waits, so that a warp that gives up
    // cannot leave the others waiting on a hardware barrier): row maxima posted, P complete,
    // row sums posted
    __shared__ __align__(8) uint64_t x_s, x_p, x_p2, x_sum;
    __shared__ int meta[kNS][mWords];
    __shared__ float red_m[kNS][kMlaCW][kRows];  // [ring slot][warp]: its keys' row maxima (that stage)
    __shared__ int red_f[kNS][kMlaCW];           // [ring slot][warp]: some row outgrew the running max
    __shared__ float red_l[kMlaCW][kRows];  // per warp: its row sums (item end)
    // per k-slice: the partial S over its k-steps (both key halves), [row][key] with rows padded to
    // 72 floats (the fragment stores and loads of a half warp then touch 32 distinct banks)
    __shared__ __align__(16) float red_s[kKSlices][kRows][kSPad];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const AttnParams& a = p.a;
    int* ctrl = a.ctrl;
    const uint64_t tmo = p.timeout_ns;
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t ring0 = smem0;                    // kNS stages
    const uint32_t qbuf0 = smem0 + kNS * kStage;     // 2 Q buffers
    const uint32_t pbuf = qbuf0 + 2 * kQBuf;         // P

    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), kMlaCW);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&q_full[i]), 1);
            mbar_init(smem_u32(&q_empty[i]), kMlaCW);
        }
        mbar_init(smem_u32(&x_s), kMlaCW);
        mbar_init(smem_u32(&x_p2), kMlaCW);
        mbar_init(smem_u32(&x_p), kMlaCW);
        mbar_init(smem_u32(&x_sum), kMlaCW);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();
    pdl_wait();  // the planner's items are complete from here on
    if ((int)blockIdx.x >= a.ctrl[kPfCtas]) return;
    const int n_items = a.ctrl[a.item_count_word];
    const int Gv = a.G;  // query heads of an item's block (G')

    if (warp == kMlaCW) {
        // =============================== producer ===============================
        const int BR = p.BR, ps = a.ps;
        const int runs = kKS / BR;
        const uint32_t run_bytes = (uint32_t)(kCBQ * BR * 128);
        const uint64_t pol_stream = l2_policy_evict_first();
        const int Tt = kRows / Gv;  // tokens of a Q box
        int s = 0, qb = 0;
        uint32_t ph = 0, qph = 0;
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
            // kv head of this block of query heads (the latent row it reads)
            const int kvh = (item.head * Gv) / (a.Hq / a.Hkv);
            // Q of the item into Q buffer qb, once the item that used it last is done
            if (!mbar_wait(smem_u32(&q_empty[qb]), qph ^ 1u, ctrl, tmo)) {
                ok = false;
                break;
            }
            {
                const uint32_t qfb = smem_u32(&q_full[qb]);
                if (lane == 0) mbar_arrive_expect_tx(qfb, (uint32_t)(kCBQ * Tt * Gv * 128));
                __syncwarp();
                if (lane < kCBQ)
                    tma_load_3d(qbuf0 + qb * kQBuf + lane * (kRows * 128), &qmap, qfb, lane * 64, item.head * Gv,
                                q_start + item.tok0);
            }
            int win0 = key0 / ps;
            int win = (win0 + lane < a.P) ? __ldg(ptab + win0 + lane) : 0;
            for (int st = 0; st < nst && ok; ++st) {
                const int k_stage = key0 + st * kKS;
                const int lp_last = min(k_stage + kKS - 1, item.kv_end - 1) / ps;
                if (lp_last - win0 >= 32) {
                    win0 = k_stage / ps;
                    win = (win0 + lane < a.P) ? __ldg(ptab + win0 + lane) : 0;
                }
                if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1u, ctrl, tmo)) {
                    ok = false;
                    break;
                }
                const uint32_t stage = ring0 + s * kStage;
                const int k0 = k_stage + lane * BR;
                const int lp = k0 / ps;
                const int pg = __shfl_sync(0xffffffffu, win, (lp - win0) & 31);
                const bool want = lane < runs && k0 < item.kv_end && k0 + BR > item.kv_begin;
                const bool good = (unsigned)pg < (unsigned)a.N;
                const int n_issue = __popc(__ballot_sync(0xffffffffu, want && good));
                if (__any_sync(0xffffffffu, want && !good)) {
                    // a page id outside [0, N): never dereferenced; its keys read as zero
                    if (lane == 0) set_status(ctrl, RPA_ERR_BAD_PAGE_INDEX);
                    for (int i = lane; i < kStage / 16; i += 32)
                        *reinterpret_cast<uint4*>(smem + (stage - smem0) + i * 16) = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                }
                if (lane == 0) {
                    int* m = meta[s];
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
                    m[mQb] = qb;
                    m[mStop] = 0;
                }
                __syncwarp();
                const uint32_t fb = smem_u32(&full_bar[s]);
                if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)n_issue * run_bytes);
                __syncwarp();
                if (want && good)
                    tma_load_3d_hint(stage + (uint32_t)lane * run_bytes, &kvmap, fb, 0, pg * ps + (k0 - lp * ps),
                                     kvh * kCBQ, pol_stream);
                if (++s == kNS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (++qb == 2) {
                qb = 0;
                qph ^= 1u;
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
            for (int i = 0; i < 2; ++i) mbar_wait(smem_u32(&q_full[i]), 0, ctrl, tmo);
        }
        return;
    }

    // =============================== consumers ===============================
    const int w = warp;
    const int Hq = a.Hq;
    const int BR = p.BR, br_shift = __ffs(BR) - 1;
    const uint32_t run_bytes = (uint32_t)(kCBQ * BR * 128);
    int s = 0;
    uint32_t ph = 0, xph_s = 0, xph_p = 0, xph_p2 = 0, xph_sum = 0;
    // this warp's k-slice of the QK contraction and key half of the stage
    const int kslice = w & (kKSlices - 1), khalf = w / kKSlices;
    const int kd0 = kslice * kSliceSteps;
    uint32_t qph[2] = {0u, 0u};
    // every consumer warp arrives, then waits (bounded) for the others
    auto exchange = [&](uint64_t& bar, uint32_t& xph) -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar));
        const bool ok = mbar_wait(smem_u32(&bar), xph, ctrl, tmo);
        xph ^= 1u;
        return ok;
    };
    float o_acc[8][4];  // rows (lane / 4, + 8) x value columns 64w + 8 nd + 2 (lane % 4) (+1)
    float m_r[2], l_r[2];
    int pos[2];
    // this warp's keys: 8w .. 8w + 7 of every stage (the n-tile of S it computes)
    for (;;) {
        if (!mbar_wait(smem_u32(&full_bar[s]), ph, ctrl, tmo)) return;
        const int* m = meta[s];
        if (m[mStop]) return;
        const int st = m[mSt], nst = m[mNst];
        const int kv_begin = m[mKvBegin], kv_end = m[mKvEnd];
        const int kl = m[mKl], ql = m[mQl];
        const int tok0 = m[mTok0], ntok = m[mNtok];
        const int qb = m[mQb];
        const int part = m[mPart], q_start = m[mQStart], head = m[mHead];
        const int k_stage = m[mKey0];  // (the stage's meta words are rewritten once every warp releases it)
        const uint32_t stage = ring0 + s * kStage;
        const uint32_t qbase = qbuf0 + qb * kQBuf;
        if (st == 0) {
            if (!mbar_wait(smem_u32(&q_full[qb]), qph[qb], ctrl, tmo)) return;
            qph[qb] ^= 1u;

#pragma unroll
            for (int nd = 0; nd < 8; ++nd) o_acc[nd][0] = o_acc[nd][1] = o_acc[nd][2] = o_acc[nd][3] = 0.f;
            m_r[0] = m_r[1] = -INFINITY;
            l_r[0] = l_r[1] = 0.f;
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) pos[ri] = kl - ql + tok0 + ((lane >> 2) + ri * 8) / Gv;
        }
        if (k_stage < kv_begin || k_stage + kKS > kv_end) {
            // keys of the stage outside [kv_begin, kv_end): their P is zero, but their V rows may
            // hold any bits (page tails, runs not copied); this warp zeroes its value columns
            // (column block w) of those rows before its PV
            for (int i = lane; i < kKS * 8; i += 32) {
                const int kk = i >> 3, c = i & 7;
                const int j = k_stage + kk;
                if (j >= kv_begin && j < kv_end) continue;
                const int b = kk >> br_shift, r = kk & (BR - 1);
                *reinterpret_cast<uint4*>(smem + (stage - smem0) + b * run_bytes + swz128((uint32_t)(w * BR + r), c)) =
                    make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();  // the stage will be refilled by bulk copies
            __syncwarp();
        }

        // ---- S = Q K^T: this warp's k-slice for its 32 keys (four n-tiles, independent chains),
        // then the partial sums meet in shared memory and the warp adds up its keys 8w .. 8w+7
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            float sp[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) sp[nt][0] = sp[nt][1] = sp[nt][2] = sp[nt][3] = 0.f;
#pragma unroll
            for (int i = 0; i < kSliceSteps; ++i) {
                // the Q fragment of k-step kd0 + i (A, 16 rows x 16): read from the item's Q buffer
                uint32_t qa[4];
                {
                    const int qr = (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int qc = 2 * (kd0 + i) + (lane >> 4);
                    ldsm_x4(qbase + swz128((uint32_t)((qc >> 3) * kRows + qr), qc & 7), qa[0], qa[1], qa[2], qa[3]);
                }
                const int c = 2 * (kd0 + i) + ((lane >> 3) & 1);  // chunk of this lane's matrix
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    // keys 32 khalf + 16 np + (lane & 7) (+ 8 for lanes 16-31): b0, b1 the first
                    // n-tile, b2, b3 the second
                    const int kk = 32 * khalf + 16 * np + (lane & 7) + (lane >> 4) * 8;
                    const int b = kk >> br_shift, r = kk & (BR - 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(stage + b * run_bytes + swz128((uint32_t)((c >> 3) * BR + r), c & 7), b0, b1, b2, b3);
                    mma16816<F16>(sp[2 * np], qa, b0, b1);
                    mma16816<F16>(sp[2 * np + 1], qa, b2, b3);
                }
            }
            const int r0 = lane >> 2, qq = 2 * (lane & 3);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int key = 32 * khalf + 8 * nt + qq;
                *reinterpret_cast<float2*>(&red_s[kslice][r0][key]) = make_float2(sp[nt][0], sp[nt][1]);
                *reinterpret_cast<float2*>(&red_s[kslice][r0 + 8][key]) = make_float2(sp[nt][2], sp[nt][3]);
            }
            if (!exchange(x_s, xph_s)) return;
#pragma unroll
            for (int ks = 0; ks < kKSlices; ++ks) {
                const float2 u = *reinterpret_cast<const float2*>(&red_s[ks][r0][8 * w + qq]);
                const float2 v = *reinterpret_cast<const float2*>(&red_s[ks][r0 + 8][8 * w + qq]);
                sacc[0] += u.x;
                sacc[1] += u.y;
                sacc[2] += v.x;
                sacc[3] += v.y;
            }
        }
        // ---- scale, soft cap, masks (log2 domain); sacc[e]: row (lane / 4) + 8 (e >> 1), key
        // 8w + 2 (lane % 4) + (e & 1)
        const int kw = k_stage + 8 * w;
        const bool need_mask = kw < kv_begin || kw + 8 > kv_end || (a.causal && kw + 7 > kl - ql + tok0) ||
                               (a.has_window && kw <= kl - ql + tok0 + ntok - 1 - a.window);
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int ri = e >> 1;
            float x = sacc[e];
            if (a.has_cap) {
                const float t = ex2(x * a.cap_exp);
                x = a.cap_log2 - 2.f * a.cap_log2 * rcp_approx(1.f + t);
            } else {
                x *= a.qk_log2;
            }
            if (need_mask) {
                const int j = kw + 2 * (lane & 3) + (e & 1);
                const bool okk = j >= kv_begin && j < kv_end && (!a.causal || j <= pos[ri]) &&
                                 (!a.has_window || j > pos[ri] - a.window);
                x = okk ? x : -INFINITY;
            }
            sacc[e] = x;
            mx[ri] = fmaxf(mx[ri], x);
        }
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 1));
            mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 2));
        }
        // Lazy maximum.  A row's exponent base is its running max, which moves only when some key
        // outgrows it by more than 2^8 (always so on an item's first stage with a live key).  Each
        // warp posts its keys' row maxima and whether any row of its keys grew, and writes P against
        // the running max (all warps hold the same one); after the P exchange all read the flags.  If
        // some row grew, the stage's row maxima form the new running max, O and the sums are rescaled
        // and P is written again, behind one more exchange.
        const bool grow = __any_sync(0xffffffffu, mx[0] > m_r[0] + kRescaleLog2 || mx[1] > m_r[1] + kRescaleLog2);
        if ((lane & 3) == 0) {
            red_m[s][w][lane >> 2] = mx[0];
            red_m[s][w][(lane >> 2) + 8] = mx[1];
        }
        if (lane == 0) red_f[s][w] = grow ? 1 : 0;
        float lsum[2] = {0.f, 0.f};
        // P of this warp's 8 keys into the shared P tile [16 rows][64 keys] (128-byte rows,
        // swizzled): keys 8w + 2 (lane % 4), + 1 are word lane % 4 of chunk w of the row
        auto write_p = [&]() {
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                const float bse = m_r[ri] == -INFINITY ? 0.f : m_r[ri];
                const float p0 = ex2(sacc[2 * ri] - bse), p1 = ex2(sacc[2 * ri + 1] - bse);
                lsum[ri] = p0 + p1;
                const int row = (lane >> 2) + 8 * ri;
                *reinterpret_cast<uint32_t*>(smem + (pbuf - smem0) + swz128((uint32_t)row, (uint32_t)w) + 4 * (lane & 3)) =
                    pack2<F16>(p0, p1);
            }
        };
        if (!grow) write_p();
        // P complete.  The next stage's partial S, maxima and P are written only after this
        // warp's PV of this stage; every warp has read this stage's partial S before it arrives here.
        if (!exchange(x_p, xph_p)) return;
        bool need = false;
#pragma unroll
        for (int ww = 0; ww < kMlaCW; ++ww) need |= red_f[s][ww] != 0;
        if (need) {
            // (the same flags and maxima in every warp: the same new running max)
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                float mt = -INFINITY;
#pragma unroll
                for (int ww = 0; ww < kMlaCW; ++ww) mt = fmaxf(mt, red_m[s][ww][(lane >> 2) + 8 * ri]);
                const float m_new = fmaxf(m_r[ri], mt);
                const float bse = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = m_r[ri] == -INFINITY ? 0.f : ex2(m_r[ri] - bse);
                m_r[ri] = m_new;
                l_r[ri] *= alpha;
#pragma unroll
                for (int nd = 0; nd < 8; ++nd) {
                    o_acc[nd][2 * ri] *= alpha;
                    o_acc[nd][2 * ri + 1] *= alpha;
                }
            }
            write_p();
            if (!exchange(x_p2, xph_p2)) return;
        }
        l_r[0] += lsum[0];
        l_r[1] += lsum[1];

        // ---- O += P V: this warp's value columns 64w .. 64w+63 (column block w of the rows)
#pragma unroll
        for (int ks = 0; ks < kKS / 16; ++ks) {
            uint32_t pa[4];
            {
                const int pr = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int pc = 2 * ks + (lane >> 4);
                ldsm_x4(pbuf + swz128((uint32_t)pr, (uint32_t)pc), pa[0], pa[1], pa[2], pa[3]);
            }
            // V rows (keys) 16 ks + (lane & 7) + 8 ((lane >> 3) & 1), chunks 2 nd2 + (lane >> 4)
            const int kk = 16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int b = kk >> br_shift, r = kk & (BR - 1);
            const uint32_t vbase = stage + b * run_bytes + (uint32_t)((w * BR + r) * 128);
#pragma unroll
            for (int nd2 = 0; nd2 < 4; ++nd2) {
                const int c = 2 * nd2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + (((c ^ (w * BR + r)) & 7) << 4), b0, b1, b2, b3);
                mma16816<F16>(o_acc[2 * nd2], pa, b0, b1);
                mma16816<F16>(o_acc[2 * nd2 + 1], pa, b2, b3);
            }
        }
        // this warp is done with the stage's K/V
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
        if (st == nst - 1) {
            // ---- epilogue: the Q buffer back to the producer, the row sums over the warps, then
            // this warp's 64 columns
            if (lane == 0) mbar_arrive(smem_u32(&q_empty[qb]));
            float lsum[2];
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                lsum[ri] = l_r[ri] + __shfl_xor_sync(0xffffffffu, l_r[ri], 1);
                lsum[ri] += __shfl_xor_sync(0xffffffffu, lsum[ri], 2);
            }
            if ((lane & 3) == 0) {
                red_l[w][lane >> 2] = lsum[0];
                red_l[w][(lane >> 2) + 8] = lsum[1];
            }
            // red_l is rewritten only at the next item's end, after its x_s and x_p exchanges
            if (!exchange(x_sum, xph_sum)) return;
            const int rows_used = ntok * Gv;
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                const int rr = (lane >> 2) + 8 * ri;
                float L = 0.f;
#pragma unroll
                for (int ww = 0; ww < kMlaCW; ++ww) L += red_l[ww][rr];
                if (rr >= rows_used) continue;
                const int qh = head * Gv + rr % Gv;
                const int col0 = 64 * w + 2 * (lane & 3);
                if (part < 0) {
                    L = add_sink(L, a.sinks, qh, m_r[ri]);
                    const float inv = L > 0.f ? a.v_scale / L : 0.f;
                    const int t = q_start + tok0 + rr / Gv;
                    const size_t orow = ((size_t)t * Hq + qh) * kV;
#pragma unroll
                    for (int nd = 0; nd < 8; ++nd)
                        store_o2(a.o, orow + col0 + 8 * nd, o_acc[nd][2 * ri] * inv, o_acc[nd][2 * ri + 1] * inv, a.odt);
                } else {
                    float* prow = a.part_o + ((size_t)part * kDecRows + rr) * kV;
#pragma unroll
                    for (int nd = 0; nd < 8; ++nd)
                        *reinterpret_cast<float2*>(prow + col0 + 8 * nd) = make_float2(o_acc[nd][2 * ri], o_acc[nd][2 * ri + 1]);
                    if (w == 0 && (lane & 3) == 0)
                        *reinterpret_cast<float2*>(a.part_ml + ((size_t)part * kDecRows + rr) * 2) = make_float2(m_r[ri], L);
                }
            }
        }
        if (++s == kNS) {
            s = 0;
            ph ^= 1u;
        }
    }
}

template <bool F16>
struct MlaKern {
    static cudaError_t prepare(int* bps) {
        cudaError_t e = cudaFuncSetAttribute(rpa_mla_attn<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(bps, rpa_mla_attn<F16>, kMlaThreads, kMlaSmem);
    }
    static cudaError_t launch(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, const Launch& l) {
        return launch_pdl(rpa_mla_attn<F16>, l.grid, kMlaThreads, kMlaSmem, l.stream, kvm, qm, p);
    }
};

}  // namespace

cudaError_t mla_prepare(int kt, int* bps) {
    if (kt == KT_BF16) return MlaKern<false>::prepare(bps);
    if (kt == KT_F16) return MlaKern<true>::prepare(bps);
    return cudaErrorInvalidValue;
}

cudaError_t launch_mla(const CUtensorMap& kvm, const CUtensorMap& qm, const TcParams& p, int kt, const Launch& l) {
    if (kt == KT_BF16) return MlaKern<false>::launch(kvm, qm, p, l);
    if (kt == KT_F16) return MlaKern<true>::launch(kvm, qm, p, l);
    return cudaErrorInvalidValue;
}

}  // namespace rpa
