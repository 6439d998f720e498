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
//    so that the decode kernel has about kDecWaves items per resident CTA
//    (split-KV; partial results are merged by the combine kernel);
//  * prefill-class sequences become units (sequence, query tile);
//  * each unit expands to one item per kv head;
//  * decode units are sorted by cost (keys to visit), longest first, so that
//    the persistent kernel finishes together; prefill units are sorted by
//    sequence, then cost, so that the CTAs running at any moment share one
//    sequence's K/V in L2; ties keep unit order.
//
// The key range of a unit is the band its rows can see (page: flashAttention
// row_ids / col_ids masks): causal rows end at position p, windowed rows start
// after p - sliding_window.  Everything here is integer and deterministic.
#include "rpa_internal.cuh"

namespace rpa {

namespace {

__device__ __forceinline__ void key_band(int kl, int ql, int i0, int i1, const PlanParams& p,
                                         int& lo, int& hi) {
    const int p_lo = kl - ql + i0;
    const int p_hi = kl - ql + i1 - 1;
    hi = p.causal ? min(kl, p_hi + 1) : kl;
    lo = p.has_window ? max(0, p_lo - p.window + 1) : 0;
    if (hi < lo) hi = lo;
}

// Exclusive scan of one int per thread over the whole block; *total gets the sum.
__device__ int block_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? s_warp[lane] : 0;
        int ww = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, ww, o);
            if (lane >= o) ww += y;
        }
        s_warp[lane] = ww - w;
        if (lane == 31) s_warp[32] = ww;
    }
    __syncthreads();
    const int r = x - v + s_warp[warp];
    *total = s_warp[32];
    __syncthreads();
    return r;
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
    extern __shared__ unsigned long long s_keys[];  // kMaxSort
    __shared__ int s_warp[33];
    __shared__ int s_bad;
    __shared__ unsigned long long s_total;
    const int tid = threadIdx.x;
    const int S = p.num_seqs;
    int* ctrl = p.ctrl;
    // per-sequence scratch: class, count, decode/prefill unit end, partial offset, combine offset
    int* s_cls = p.seq_scratch;
    int* s_cnt = s_cls + p.num_seqs + 1;
    int* s_dend = s_cnt + p.num_seqs + 1;
    int* s_pend = s_dend + p.num_seqs + 1;
    int* s_part = s_pend + p.num_seqs + 1;
    int* s_comb = s_part + p.num_seqs + 1;
    const int Tq = max(1, p.pf_tokens);  // query tokens per prefill tile

    if (tid == 0) {
        s_bad = 0;
        s_total = 0ull;
    }
    __syncthreads();

    // ---- 1. validate and classify each sequence
    for (int s = tid; s < S; s += blockDim.x) {
        const int q0 = p.cu_q_lens[s], q1 = p.cu_q_lens[s + 1], kl = p.kv_lens[s];
        const int ql = q1 - q0;
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
                atomicAdd(&s_total, (unsigned long long)cnt * (unsigned long long)p.Hkv);
            } else {
                cls = 2;
                cnt = (ql + Tq - 1) / Tq;
            }
        }
        s_cls[s] = cls;
        s_cnt[s] = cnt;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            for (int w = 1; w < kCtrlWords; ++w) ctrl[w] = 0;
            ctrl[kStatus] = RPA_ERR_BAD_LENGTHS;
        }
        return;
    }

    // ---- 2. split-KV chunk for decode units
    int chunk;
    {
        const unsigned long long target = (unsigned long long)kDecWaves * (unsigned long long)max(1, p.dec_slots);
        unsigned long long c = (s_total + target - 1) / target;
        if (c < (unsigned long long)kMinChunk) c = kMinChunk;
        c = (c + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
        if (c > (1ull << 30)) c = 1ull << 30;
        chunk = (int)c;
    }

    // ---- 3. prefix sums: unit ends per class, partial slots, combine entries
    int carry_d = 0, carry_p = 0, carry_part = 0, carry_comb = 0;
    for (int base = 0; base < S; base += blockDim.x) {
        const int s = base + tid;
        int du = 0, pu = 0, pa = 0, cb = 0;
        if (s < S) {
            const int cls = s_cls[s], cnt = s_cnt[s];
            if (cls == 1) {
                du = (cnt + chunk - 1) / chunk;
                if (du > 1) {
                    pa = du * p.Hkv;
                    cb = p.Hkv;
                }
            } else if (cls == 2) {
                pu = cnt;
            }
        }
        int tot;
        const int od = block_scan(du, s_warp, &tot);
        const int td = tot;
        const int op = block_scan(pu, s_warp, &tot);
        const int tp = tot;
        const int oa = block_scan(pa, s_warp, &tot);
        const int ta = tot;
        const int oc = block_scan(cb, s_warp, &tot);
        const int tc = tot;
        if (s < S) {
            s_dend[s] = carry_d + od + du;
            s_pend[s] = carry_p + op + pu;
            s_part[s] = carry_part + oa;
            s_comb[s] = carry_comb + oc;
        }
        carry_d += td;
        carry_p += tp;
        carry_part += ta;
        carry_comb += tc;
    }
    const int n_dec = carry_d, n_pf = carry_p, n_units = n_dec + n_pf;
    if (n_units > p.max_units || n_dec > p.max_dec_units || n_pf > p.max_pf_units ||
        carry_part > p.max_part || carry_comb > p.max_comb) {
        // cannot happen with the create-time sizing; refuse rather than overflow
        if (tid == 0) {
            for (int w = 1; w < kCtrlWords; ++w) ctrl[w] = 0;
            ctrl[kStatus] = RPA_ERR_INVALID_ARG;
        }
        return;
    }
    __syncthreads();

    // ---- 4. unit descriptors and sort keys
    const bool do_sort = n_units <= kMaxSort && S < 65536;  // key fields: unit < 2^16, seq < 2^16
    for (int u = tid; u < n_units; u += blockDim.x) {
        int d[8];
        int cost;
        int cls_bit;
        if (u < n_dec) {
            const int s = upper_seq(s_dend, S, u);
            const int k = u - (s_dend[s] - (s_cnt[s] + chunk - 1) / chunk);  // piece index
            const int q0 = p.cu_q_lens[s], ql = p.cu_q_lens[s + 1] - q0, kl = p.kv_lens[s];
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
        } else {
            const int v = u - n_dec;
            const int s = upper_seq(s_pend, S, v);
            const int k = v - (s_pend[s] - s_cnt[s]);  // tile index
            const int q0 = p.cu_q_lens[s], ql = p.cu_q_lens[s + 1] - q0, kl = p.kv_lens[s];
            const int t0 = k * Tq;
            const int nt = min(Tq, ql - t0);
            int lo, hi;
            key_band(kl, ql, t0, t0 + nt, p, lo, hi);
            d[0] = s; d[1] = t0; d[2] = nt; d[3] = lo; d[4] = hi;
            d[5] = -1; d[6] = 0; d[7] = 1;
            cost = hi - lo;
            cls_bit = 1;
        }
        int4* dst = reinterpret_cast<int4*>(p.units + (size_t)u * 8);
        dst[0] = make_int4(d[0], d[1], d[2], d[3]);
        dst[1] = make_int4(d[4], d[5], d[6], d[7]);
        if (do_sort)
            s_keys[u] = cls_bit == 0
                            ? ((unsigned long long)(0x7FFFFFFF - cost) << 32) | (unsigned long long)u
                            : (1ull << 63) | ((unsigned long long)d[0] << 47) |
                                  ((unsigned long long)(0x7FFFFFFF - cost) << 16) | (unsigned long long)u;
    }

    // ---- 5. bitonic sort of the keys (ascending: decode first, then cost descending)
    int n2 = 1;
    while (n2 < n_units) n2 <<= 1;
    if (do_sort) {
        for (int i = n_units + tid; i < n2; i += blockDim.x) s_keys[i] = ~0ull;
        __syncthreads();
        for (int k = 2; k <= n2; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = tid; i < n2; i += blockDim.x) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const unsigned long long a = s_keys[i], b = s_keys[ixj];
                        const bool up = (i & k) == 0;
                        if ((a > b) == up) {
                            s_keys[i] = b;
                            s_keys[ixj] = a;
                        }
                    }
                }
                __syncthreads();
            }
        }
    }
    __syncthreads();

    // ---- 6. items (one per kv head) in sorted unit order
    for (int r = tid; r < n_units; r += blockDim.x) {
        // unit index: low 32 bits of a decode key, low 16 bits of a prefill key
        const unsigned long long key = do_sort ? s_keys[r] : 0ull;
        const int u = !do_sort ? r : (int)((key >> 63) ? (key & 0xFFFFull) : (key & 0xFFFFFFFFull));
        const int4* src = reinterpret_cast<const int4*>(p.units + (size_t)u * 8);
        const int4 a = src[0], b = src[1];
        const bool is_dec = r < n_dec;
        Item* dst = is_dec ? p.dec_items + (size_t)r * p.Hkv : p.pf_items + (size_t)(r - n_dec) * p.Hkv;
        for (int h = 0; h < p.Hkv; ++h) {
            Item it;
            it.seq = a.x;
            it.head = h;
            it.tok0 = a.y;
            it.ntok = a.z;
            it.kv_begin = a.w;
            it.kv_end = b.x;
            it.part = b.y >= 0 ? b.y + h * b.w + b.z : -1;
            it.piece = b.z;
            dst[h] = it;
        }
    }
    // ---- 7. combine entries of split decode sequences
    for (int s = tid; s < S; s += blockDim.x) {
        if (s_cls[s] != 1) continue;
        const int pieces = (s_cnt[s] + chunk - 1) / chunk;
        if (pieces <= 1) continue;
        for (int h = 0; h < p.Hkv; ++h) {
            Comb c;
            c.seq = s;
            c.head = h;
            c.part = s_part[s] + h * pieces;
            c.pieces = pieces;
            p.comb[s_comb[s] + h] = c;
        }
    }
    if (tid == 0) {
        ctrl[kNumDecItems] = n_dec * p.Hkv;
        ctrl[kNumPfItems] = n_pf * p.Hkv;
        ctrl[kNumComb] = carry_comb;
        ctrl[kDecChunk] = chunk;
        ctrl[kDecCounter] = 0;
        ctrl[kPfCounter] = 0;
        ctrl[kNumPart] = carry_part;
        ctrl[kNumUnits] = n_units;
        ctrl[kSorted] = do_sort ? 1 : 0;
        ctrl[kCovLo] = S > 0 ? p.cu_q_lens[0] : 0;
        ctrl[kCovHi] = S > 0 ? p.cu_q_lens[S] : 0;
        ctrl[kStatus] = 0;
    }
}

}  // namespace

size_t plan_smem_bytes() { return sizeof(unsigned long long) * kMaxSort; }

cudaError_t launch_plan(const PlanParams& p, cudaStream_t st, size_t smem) {
    rpa_plan_kernel<<<1, kPlanThreads, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t plan_prepare() {
    return cudaFuncSetAttribute(rpa_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)plan_smem_bytes());
}

}  // namespace rpa
