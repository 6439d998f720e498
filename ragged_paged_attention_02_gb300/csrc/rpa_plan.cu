// rpa_plan.cu -- K0: the device-side work planner.
//
// One CTA reads cu_q_lens / kv_lens, validates them, and turns the ragged
// batch into work items for the attention kernels.  It replaces the
// sequential grid walk of the "ragged_paged.zig" page (run: the q-block loop
// over sequences and the kv-block loop bounded by kv_len), which a GPU does
// not need: every (sequence, kv head, query tile, key range) is independent.
//
//  * decode-class sequences (q_len * G <= decode tile rows) become units
//    (sequence, key piece); their keys are split into pieces of `chunk` keys
//    so that the kernel that runs them has about dec_waves items per resident CTA
//    (split-KV; partial results are merged by the combine kernel);
//  * prefill-class sequences become units (sequence, query tile);
//  * each unit expands to one item per kv head;
//  * decode units are sorted by cost (keys to visit), longest first, so that
//    the persistent kernel finishes together; prefill sequences are ordered by
//    their heaviest unit, longest first, and a sequence's units stay together
//    (by cost) so that the CTAs running at any moment share one sequence's K/V
//    in L2; ties keep unit order.
//
// The key range of a unit is the band its rows can see (page: flashAttention
// row_ids / col_ids masks): causal rows end at position p, windowed rows start
// after p - sliding_window.  Everything here is integer and deterministic.
#include "rpa_internal.cuh"

namespace rpa {

namespace {

constexpr int kUnitSmem = 1024;    // unit descriptors kept in shared memory (else global)
// with at most kUnitSmem units the sort touches keys [0, 3 kUnitSmem) (its range starts below
// kUnitSmem and spans at most twice the keys), below the descriptors
static_assert(3 * kUnitSmem <= kMaxSort / 2 && kUnitSmem * 8 * 4 <= kMaxSort / 2 * 8,
              "unit descriptors share the key array's upper half");

// The plan of call `epoch` is complete (control words included): a decode kernel launched behind
// the prefill kernel waits for this word instead of the planner grid.
__device__ __forceinline__ void publish_epoch(int* ctrl, int epoch) {
    __threadfence();
    asm volatile("st.release.gpu.global.b32 [%0], %1;\n" ::"l"(ctrl + kPlanEpoch), "r"(epoch) : "memory");
}

__device__ __forceinline__ void key_band(int kl, int ql, int i0, int i1, const PlanParams& p,
                                         int& lo, int& hi) {
    const int p_lo = kl - ql + i0;
    const int p_hi = kl - ql + i1 - 1;
    hi = p.causal ? min(kl, p_hi + 1) : kl;
    lo = p.has_window ? max(0, p_lo - p.window + 1) : 0;
    if (hi < lo) hi = lo;
}

// Exclusive scan of N ints per thread over the whole block (one pass for all N): r gets the
// thread's offsets, tot the block's sums.  s_scan holds 33 N ints.
template <int N>
__device__ void block_scan(const int (&v)[N], int (&r)[N], int (&tot)[N], int* s_scan) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int x[N];
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = v[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const int y = __shfl_up_sync(0xffffffffu, x[i], o);
            if (lane >= o) x[i] += y;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int i = 0; i < N; ++i) s_scan[warp * N + i] = x[i];
    }
    __syncthreads();
    if (warp == 0) {
        int w[N], ww[N];
#pragma unroll
        for (int i = 0; i < N; ++i) ww[i] = w[i] = lane < nwarps ? s_scan[lane * N + i] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int y = __shfl_up_sync(0xffffffffu, ww[i], o);
                if (lane >= o) ww[i] += y;
            }
        }
#pragma unroll
        for (int i = 0; i < N; ++i) {
            s_scan[lane * N + i] = ww[i] - w[i];
            if (lane == 31) s_scan[32 * N + i] = ww[i];
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < N; ++i) {
        r[i] = x[i] - v[i] + s_scan[warp * N + i];
        tot[i] = s_scan[32 * N + i];
    }
    __syncthreads();
}

// Sums of two 64-bit values per thread over the block (all threads get them).  s_red holds 64.
__device__ void block_sum64x2(unsigned long long& a, unsigned long long& b, unsigned long long* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if (lane == 0) {
        s_red[warp] = a;
        s_red[32 + warp] = b;
    }
    __syncthreads();
    unsigned long long x = lane < nwarps ? s_red[lane] : 0ull, y = lane < nwarps ? s_red[32 + lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        x += __shfl_xor_sync(0xffffffffu, x, o);
        y += __shfl_xor_sync(0xffffffffu, y, o);
    }
    __syncthreads();
    a = x;
    b = y;
}
// Minimum of one 64-bit value per thread over the block (all threads get it).  s_red holds 32.
__device__ unsigned long long block_min64(unsigned long long v, unsigned long long* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w < v ? w : v;
    }
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    unsigned long long t = lane < nwarps ? s_red[lane] : ~0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, t, o);
        t = w < t ? w : t;
    }
    __syncthreads();
    return t;
}

// first s in [0, n) with ends[s] > u (ends non-decreasing, ends[n-1] > u)
__device__ __forceinline__ int upper_seq(const int* ends, int n, int u) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (ends[mid] > u) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kPlanThreads, 1) rpa_plan_kernel(PlanParams p) {
    extern __shared__ __align__(16) unsigned long long s_keys[];  // kMaxSort keys, then sequence scratch
    __shared__ int s_scan[33 * 5];
    __shared__ unsigned long long s_red[64];
    __shared__ int s_bad;
    __shared__ int s_split[2];                // prefill CTAs, decode CTAs
    const int tid = threadIdx.x;
    const int S = p.num_seqs;
    int* ctrl = p.ctrl;
    pdl_trigger();  // the attention kernels may start their prologue now
    // Launched as a programmatic dependent of the kernel before it on the stream, the planner may
    // run while that kernel does.  Unless the caller has said that the inputs are complete at
    // launch (RPA_OPT_PLAN_EARLY), it waits for that kernel before reading them; either way it
    // waits before rewriting what earlier kernels read (below)
    if (!p.early) pdl_wait();
    // per-sequence scratch (shared memory when it fits): class, count, decode / prefill
    // unit ends, partial offset, combine offset, decode sequences with a partial last piece before
    // this one, first query token (S + 1 entries: cu_q_lens), kv_len
    int* seq_base = S <= kSeqSmem ? reinterpret_cast<int*>(s_keys + kMaxSort) : p.seq_scratch;
    int* s_cls = seq_base;
    int* s_cnt = s_cls + S + 1;
    int* s_dend = s_cnt + S + 1;
    int* s_pend = s_dend + S + 1;
    int* s_part = s_pend + S + 1;
    int* s_comb = s_part + S + 1;
    int* s_ppre = s_comb + S + 1;
    int* s_q0 = s_ppre + S + 1;
    int* s_kl = s_q0 + S + 1;
    const int Tq = max(1, p.pf_tokens);  // query tokens per prefill tile

    if (tid == 0) s_bad = 0;
    __syncthreads();

    // ---- 1. validate and classify each sequence; per-thread sums of decode (key, kv head)
    // pairs and of the keys prefill units visit, reduced over the block below
    unsigned long long my_total = 0ull, my_pf_keys = 0ull;
    for (int s = tid; s < S; s += blockDim.x) {
        const int q0 = p.cu_q_lens[s], q1 = p.cu_q_lens[s + 1], kl = p.kv_lens[s];
        const int ql = q1 - q0;
        s_q0[s] = q0;
        if (s == S - 1) s_q0[S] = q1;
        s_kl[s] = kl;
        const bool bad = q0 < 0 || ql < 0 || kl < 0 || kl > p.P * p.ps || ql > kl || q1 > p.T;
        int cls = 0, cnt = 0;
        if (bad) {
            s_bad = 1;
        } else if (ql > 0) {
            if ((long long)ql * p.G <= p.dec_rows) {
                int lo, hi;
                key_band(kl, ql, 0, ql, p, lo, hi);
                cls = 1;
                cnt = hi - lo;
                my_total += (unsigned long long)cnt * (unsigned long long)p.Hkv;
            } else {
                cls = 2;
                cnt = (ql + Tq - 1) / Tq;
                unsigned long long keys = 0;
                int wmax = 0;
                for (int k = 0; k < cnt; ++k) {
                    int lo, hi;
                    key_band(kl, ql, k * Tq, min(ql, (k + 1) * Tq), p, lo, hi);
                    keys += (unsigned long long)(hi - lo);
                    wmax = max(wmax, hi - lo);
                }
                my_pf_keys += keys;
                s_comb[s] = wmax;  // the sequence's heaviest unit (sort weight); combine offsets are decode-only
            }
        }
        s_cls[s] = cls;
        s_cnt[s] = cnt;
    }
    __syncthreads();
    if (s_bad) {
        pdl_wait();  // the previous call's kernels read the control words until they finish
        if (tid == 0) {
            for (int w = 1; w < kCtrlWords; ++w) ctrl[w] = 0;
            ctrl[kStatus] = RPA_ERR_BAD_LENGTHS;
            publish_epoch(ctrl, p.epoch);
        }
        return;
    }

    block_sum64x2(my_total, my_pf_keys, s_red);
    const unsigned long long s_total = my_total, s_pf_keys = my_pf_keys;

    // ---- 2. SMs for each kernel, then the split-KV chunk for decode units
    {
        const unsigned long long dec_bytes = s_total * (unsigned long long)(2 * p.D * p.kv_elt);
        const unsigned long long pf_flops =
            s_pf_keys * (unsigned long long)p.Hkv * (unsigned long long)p.pf_mma_rows * (unsigned long long)(4 * p.D);
        const bool both = p.concurrent && dec_bytes > 0 && pf_flops > 0;
        // minimise max(prefill time, decode time) over the prefill SM count x (times in ns; one
        // x per thread, the first minimum wins: (time << 16 | x) is unique and orders that way)
        unsigned long long mine = ~0ull;
        if (both) {
            for (int x = 1 + tid; x < p.n_sms; x += blockDim.x) {
                const unsigned long long tp = pf_flops / ((unsigned long long)x * p.pf_sm_gflops);
                const unsigned long long bw =
                    min((unsigned long long)p.hbm_gbs, (unsigned long long)(p.n_sms - x) * p.dec_sm_gbs);
                const unsigned long long td = dec_bytes / bw;
                const unsigned long long c = tp > td ? tp : td;
                const unsigned long long k = (min(c, (1ull << 47) - 1) << 16) | (unsigned long long)x;
                mine = k < mine ? k : mine;
            }
        }
        const unsigned long long best = block_min64(mine, s_red);
        if (tid == 0) {
            int pf_sms = p.n_sms, dec_sms = p.n_sms;
            if (both) {
                int best_x = (int)(best & 0xFFFFull);
                if (p.force_pf_sms > 0) best_x = min(p.force_pf_sms, p.n_sms - 1);
                pf_sms = best_x;
                dec_sms = p.n_sms - best_x;
            }
            if (p.force_dec_sms > 0) dec_sms = min(p.force_dec_sms, p.n_sms);
            s_split[0] = pf_sms * p.pf_bps;
            s_split[1] = dec_sms * p.dec_bps;
        }
    }
    __syncthreads();
    int chunk;
    {
        // pieces for about dec_waves items per CTA of the kernel that runs them
        const int dec_ctas = p.dec_on_pf ? s_split[0] : s_split[1];
        const unsigned long long target = (unsigned long long)p.dec_waves * (unsigned long long)max(1, dec_ctas);
        unsigned long long c = (s_total + target - 1) / target;
        if (c < (unsigned long long)kMinChunk) c = kMinChunk;
        c = (c + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
        if (c > (1ull << 30)) c = 1ull << 30;
        chunk = (int)c;
    }

    // ---- 3. prefix sums: unit ends per class, partial slots, combine entries
    int carry_d = 0, carry_p = 0, carry_part = 0, carry_comb = 0, carry_pp = 0;
    for (int base = 0; base < S; base += blockDim.x) {
        const int s = base + tid;
        int du = 0, pu = 0, pa = 0, cb = 0, pp = 0;
        if (s < S) {
            const int cls = s_cls[s], cnt = s_cnt[s];
            if (cls == 1) {
                du = (cnt + chunk - 1) / chunk;
                pp = cnt % chunk != 0 ? 1 : 0;  // a last piece shorter than the chunk
                if (du > 1) {
                    pa = du * p.Hkv;
                    cb = p.Hkv;
                }
            } else if (cls == 2) {
                pu = cnt;
            }
        }
        const int v[5] = {du, pu, pa, cb, pp};
        int off[5], tot[5];
        block_scan<5>(v, off, tot, s_scan);
        if (s < S) {
            s_ppre[s] = carry_pp + off[4];
            s_dend[s] = carry_d + off[0] + du;
            s_pend[s] = carry_p + off[1] + pu;
            if (s_cls[s] != 2) {  // partial and combine offsets are read for decode sequences only
                s_part[s] = carry_part + off[2];
                s_comb[s] = carry_comb + off[3];
            }
        }
        carry_d += tot[0];
        carry_p += tot[1];
        carry_part += tot[2];
        carry_comb += tot[3];
        carry_pp += tot[4];
    }
    const int n_dec = carry_d, n_pf = carry_p, n_units = n_dec + n_pf;
    // decode pieces of a whole chunk (all of a sequence's but a shorter last one) share the highest
    // decode cost, so their sorted order is unit order: they go straight to their ranks, and only
    // the shorter pieces and the prefill units are sorted, after them
    const int n_full = n_dec - carry_pp;
    if (n_units > p.max_units || n_dec > p.max_dec_units || (p.dec_on_pf ? n_units : n_pf) > p.max_pf_units ||
        carry_part > p.max_part || carry_comb > p.max_comb) {
        // cannot happen with the create-time sizing; refuse rather than overflow
        pdl_wait();
        if (tid == 0) {
            for (int w = 1; w < kCtrlWords; ++w) ctrl[w] = 0;
            ctrl[kStatus] = RPA_ERR_INVALID_ARG;
            publish_epoch(ctrl, p.epoch);
        }
        return;
    }
    __syncthreads();

    // ---- 4. unit descriptors and sort keys.  Descriptors of up to kUnitSmem units sit in the
    // upper half of the key array (the sort then touches only keys below 3 kUnitSmem)
    const bool do_sort = n_units <= kMaxSort && S < 65536;  // key fields: unit < 2^16, seq < 2^16
    int* units = n_units <= kUnitSmem ? reinterpret_cast<int*>(s_keys + kMaxSort / 2) : p.units;
    for (int u = tid; u < n_units; u += blockDim.x) {
        int d[8];
        int cost, wseq = 0;
        int cls_bit;
        int pos;  // the key's slot: a whole-chunk piece at its rank, the others in the range sorted below
        if (u < n_dec) {
            const int s = upper_seq(s_dend, S, u);
            const int k = u - (s_dend[s] - (s_cnt[s] + chunk - 1) / chunk);  // piece index
            const int ql = s_q0[s + 1] - s_q0[s], kl = s_kl[s];
            int lo, hi;
            key_band(kl, ql, 0, ql, p, lo, hi);
            const int pieces = (s_cnt[s] + chunk - 1) / chunk;
            const int kb = lo + k * chunk;
            const int ke = min(hi, kb + chunk);
            d[0] = s; d[1] = 0; d[2] = ql; d[3] = kb; d[4] = ke;
            d[5] = pieces > 1 ? s_part[s] : -1;
            d[6] = k; d[7] = pieces;
            cost = ke - kb;
            cls_bit = 0;
            pos = cost == chunk ? (s_dend[s] - pieces - s_ppre[s]) + k : n_full + s_ppre[s];
        } else {
            const int v = u - n_dec;
            const int s = upper_seq(s_pend, S, v);
            const int k = v - (s_pend[s] - s_cnt[s]);  // tile index
            const int ql = s_q0[s + 1] - s_q0[s], kl = s_kl[s];
            const int t0 = k * Tq;
            const int nt = min(Tq, ql - t0);
            int lo, hi;
            key_band(kl, ql, t0, t0 + nt, p, lo, hi);
            d[0] = s; d[1] = t0; d[2] = nt; d[3] = lo; d[4] = hi;
            d[5] = -1; d[6] = 0; d[7] = 1;
            cost = hi - lo;
            wseq = s_comb[s];
            cls_bit = 1;
            pos = u;
        }
        int4* dst = reinterpret_cast<int4*>(units + (size_t)u * 8);
        dst[0] = make_int4(d[0], d[1], d[2], d[3]);
        dst[1] = make_int4(d[4], d[5], d[6], d[7]);
        // decode: cost descending.  Prefill: sequences by their heaviest unit descending (the
        // longest work starts first), a sequence's units together (its K/V stays in L2), then
        // cost descending; weights and costs in 16-key buckets.  Fields: class 1 | weight 16 |
        // sequence 18 | cost 16 | unit 13 (units < 8192, sequences < 65536 when sorting).
        if (do_sort)
            s_keys[pos] = cls_bit == 0
                            ? ((unsigned long long)(0x7FFFFFFF - cost) << 32) | (unsigned long long)u
                            : (1ull << 63) | ((unsigned long long)(0xFFFF - min(wseq >> 4, 0xFFFF)) << 47) |
                                  ((unsigned long long)d[0] << 29) |
                                  ((unsigned long long)(0xFFFF - min(cost >> 4, 0xFFFF)) << 13) |
                                  (unsigned long long)u;
    }

    // ---- 5. bitonic sort of the keys (ascending: decode first, then cost descending) in
    // [n_full, n_units), or in all of [0, n_units) when that range's power-of-two span would not
    // fit the key array (the same order either way)
    int base = n_full, n_sort = n_units - n_full;
    int n2 = 32;
    while (n2 < n_sort) n2 <<= 1;
    if (base + n2 > kMaxSort) {
        base = 0;
        n_sort = n_units;
        n2 = 32;
        while (n2 < n_units) n2 <<= 1;
    }
    unsigned long long* keys = s_keys + base;
    if (do_sort && n_sort > 1) {
        for (int i = n_sort + tid; i < n2; i += blockDim.x) keys[i] = ~0ull;
        __syncthreads();
        // merge widths up to 32: every warp sorts its 32 keys in registers, by shuffles
        for (int i = tid; i < n2; i += blockDim.x) {
            unsigned long long v = keys[i];
#pragma unroll
            for (int k = 2; k <= 32; k <<= 1) {
                const bool up = (i & k) == 0;
#pragma unroll
                for (int j = k >> 1; j > 0; j >>= 1) {
                    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, j);
                    const bool lower = (i & j) == 0;
                    const unsigned long long lo = v < o ? v : o, hi = v < o ? o : v;
                    v = (lower == up) ? lo : hi;
                }
            }
            keys[i] = v;
        }
        __syncthreads();
        for (int k = 64; k <= n2; k <<= 1) {
            // strides >= 32: pairs in different warps, through shared memory
            for (int j = k >> 1; j >= 32; j >>= 1) {
                for (int i = tid; i < n2; i += blockDim.x) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const unsigned long long a = keys[i], b = keys[ixj];
                        const bool up = (i & k) == 0;
                        if ((a > b) == up) {
                            keys[i] = b;
                            keys[ixj] = a;
                        }
                    }
                }
                __syncthreads();
            }
            // strides < 32: both keys of a pair sit in one warp, exchanged by shuffles
            for (int i = tid; i < n2; i += blockDim.x) {
                unsigned long long v = keys[i];
                const bool up = (i & k) == 0;
#pragma unroll
                for (int j = 16; j > 0; j >>= 1) {
                    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, j);
                    const bool lower = (i & j) == 0;
                    const unsigned long long lo = v < o ? v : o, hi = v < o ? o : v;
                    v = (lower == up) ? lo : hi;
                }
                keys[i] = v;
            }
            __syncthreads();
        }
    }
    __syncthreads();

    // With RPA_OPT_PLAN_EARLY the planner may get here while the previous call is still merging:
    // the phases above touch only the inputs, shared memory and scratch no earlier kernel reads;
    // what follows rewrites what they read
    pdl_wait();

    // ---- 6. the unit lists in sorted order (each unit stands for one item per kv head); a
    // thread writes one 16-byte half of a unit, consecutive threads consecutive halves
    for (int c = tid; c < 2 * n_units; c += blockDim.x) {
        const int r = c >> 1, hf = c & 1;
        // unit index: low 32 bits of a decode key, low 13 bits of a prefill key
        const unsigned long long key = do_sort ? s_keys[r] : 0ull;
        const int u = !do_sort ? r : (int)((key >> 63) ? (key & 0x1FFFull) : (key & 0xFFFFFFFFull));
        // decode units come first; with dec_on_pf they lead the prefill kernel's list instead
        const bool is_dec = r < n_dec && !p.dec_on_pf;
        Unit* dst = is_dec ? p.dec_units + r : p.pf_units + (p.dec_on_pf ? r : r - n_dec);
        reinterpret_cast<int4*>(dst)[hf] = reinterpret_cast<const int4*>(units + (size_t)u * 8)[hf];
    }
    // ---- 7. combine entries of split decode sequences, a 16-byte half of one a thread: thread
    // index c -> sequence c / 2H, half (c mod 2H) of its H entries, stepped without divisions
    {
        const int W = 2 * p.Hkv;
        const int ds = (int)blockDim.x / W, dr = (int)blockDim.x - ds * W;
        int s = tid / W, rem = tid - s * W;
        for (; s < S; s += ds, rem += dr) {
            if (rem >= W) {
                rem -= W;
                if (++s >= S) break;
            }
            if (s_cls[s] != 1) continue;
            const int pieces = s_dend[s] - (s > 0 ? s_dend[s - 1] : 0);  // the sequence's decode units
            if (pieces <= 1) continue;
            const int h = rem >> 1;
            // Comb: q0, rows, head, part | pieces, 0, 0, 0
            int4* d4 = reinterpret_cast<int4*>(p.comb + s_comb[s] + h);
            if ((rem & 1) == 0)
                d4[0] = make_int4(s_q0[s], (s_q0[s + 1] - s_q0[s]) * p.G, h, s_part[s] + h * pieces);
            else
                d4[1] = make_int4(pieces, 0, 0, 0);
        }
    }
    // every thread's unit-list and combine-entry stores, before the plan is published
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        ctrl[kNumDecItems] = p.dec_on_pf ? 0 : n_dec * p.Hkv;
        ctrl[kNumPfItems] = (p.dec_on_pf ? n_units : n_pf) * p.Hkv;
        ctrl[kNumComb] = carry_comb;
        ctrl[kDecChunk] = chunk;
        ctrl[kDecCounter] = 0;
        ctrl[kPfCounter] = 0;
        ctrl[kNumPart] = carry_part;
        ctrl[kNumUnits] = n_units;
        ctrl[kSorted] = do_sort ? 1 : 0;
        ctrl[kCovLo] = S > 0 ? s_q0[0] : 0;
        ctrl[kCovHi] = S > 0 ? s_q0[S] : 0;
        ctrl[kPfCtas] = s_split[0];
        ctrl[kDecCtas] = s_split[1];
        ctrl[kStatus] = 0;
        publish_epoch(ctrl, p.epoch);
    }
}

}  // namespace

size_t plan_smem_bytes() { return sizeof(unsigned long long) * kMaxSort + sizeof(int) * kSeqArrays * (kSeqSmem + 1); }

cudaError_t launch_plan(const PlanParams& p, cudaStream_t st, size_t smem) {
    return launch_pdl(rpa_plan_kernel, 1, kPlanThreads, smem, st, p);
}

cudaError_t plan_prepare() {
    return cudaFuncSetAttribute(rpa_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)plan_smem_bytes());
}

}  // namespace rpa
