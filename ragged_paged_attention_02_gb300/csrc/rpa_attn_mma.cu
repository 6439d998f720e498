// rpa_attn_mma.cu -- K1 prefill (warp-MMA): paged-KV flash attention for query tiles.
//
// One persistent CTA pulls work items (sequence, kv head, query tile, key
// range) from the planner's list and runs the blockwise online softmax of the
// "ragged_paged.zig" page (flashAttention) over the item's keys:
//
//   * page-table gather: key j of sequence s lives in physical page
//     page_indices[s, j / page_size], slot j % page_size; the K row (combined
//     head 2h) and the V row (2h+1) are adjacent, so one key is 2*D*elt
//     contiguous bytes, fetched with 16-byte cp.async into a multi-stage
//     shared-memory ring (page: createKvAsyncCopyDescriptors / waitKvDma);
//     keys past the item's range are zero-filled, never read (page: K/V tail
//     zeroing);
//   * GQA packing: tile row r is query token tok0 + r / G, query head
//     h*G + r % G (page: q block reshaped to [Tq*G, D]);
//   * S = Q K^T on mma.sync m16n8k16 (fp32 accumulate), scaled by
//     sm_scale*k_scale in the log2 domain, soft-capped as
//     cap*tanh(x/cap) = cap - 2cap/(1 + e^{2x/cap}), then masked (tail, causal
//     p < j, window p - sw >= j) to -inf;
//   * online softmax with running max / sum per row (row max by warp shuffle),
//     P in bf16 (f16 for f16 and 8-bit K/V), O += P V on mma.sync;
//   * epilogue: O * v_scale / l in o's type, or the unnormalised fp32 partial
//     and (max, sum) of a split-KV piece for the combine kernel.
//
// 8-bit K/V (e4m3, e5m2, int8): the bytes are converted to f16 in shared
// memory (exact), Q is taken to f16 (bf16 q rounded, f16 q as it is), and the
// MMAs run in f16; k_scale is folded into the logit scale and v_scale into the
// epilogue.  f16 K/V run the MMAs in f16 with f16 Q.
//
// The body is written for WM row-warps x WN key-warps; the prefill kernel
// uses WM=4, WN=1: 64 rows, all warps share each stage of keys.  (WN > 1
// splits the keys of a stage across warps and merges them at the end.)
#include "rpa_internal.cuh"

namespace rpa {

namespace {

template <int D, int KT, int WM, int WN, int BK, int STAGES>
struct KCfg {
    static constexpr bool FP8 = kt_8bit(KT);
    static constexpr int kThreads = 32 * WM * WN;
    static constexpr int kRows = 16 * WM;
    static constexpr int kKeys = WN * BK;          // keys per stage
    static constexpr int kCh = D / 8;              // 16-byte chunks per 16-bit row
    static constexpr int kRowB = D * 2;            // bytes of a 16-bit row
    static constexpr int kQBytes = kRows * kRowB;
    static constexpr int kTileBytes = 2 * kKeys * kRowB;                 // K and V, 16-bit
    static constexpr int kRawBytes = FP8 ? kKeys * 2 * D : kTileBytes;  // one stage as loaded
    static constexpr int kStageRegion = STAGES * kRawBytes + (FP8 ? kTileBytes : 0);
    static constexpr int kMergeBytes = WN > 1 ? WN * 16 * (D + 2) * 4 : 0;
    static constexpr int kSmem =
        kQBytes + (kStageRegion > kMergeBytes ? kStageRegion : kMergeBytes);
    static_assert(WN == 1 || WM == 1, "either rows or keys are split across warps");
    static_assert(BK % 16 == 0 && D % 64 == 0, "tile shape");
};

__device__ __forceinline__ uint32_t swz(int row, int ch) { return (uint32_t)((ch ^ (row & 7)) << 4); }

template <int D, int KT, int WM, int WN, int BK, int STAGES>
__device__ __forceinline__ void attn_body(const AttnParams& p) {
    using C = KCfg<D, KT, WM, WN, BK, STAGES>;
    constexpr bool FP8 = C::FP8;
    constexpr bool F16 = kt_f16_mma(KT);
    constexpr int kThreads = C::kThreads;
    constexpr int kKeys = C::kKeys;
    constexpr int kCh = C::kCh;
    constexpr int kRowB = C::kRowB;
    constexpr int kKvElt = FP8 ? 1 : 2;

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* q_s = smem;
    uint8_t* stage_s = smem + C::kQBytes;
    __shared__ int s_item;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp % WM, wn = warp / WM;
    pdl_trigger();
    pdl_wait();  // the planner's items are complete from here on
    if ((int)blockIdx.x >= p.ctrl[kPfCtas]) return;  // SMs left to the decode kernel
    const int n_items = p.ctrl[p.item_count_word];
    const int G = p.G, Hq = p.Hq, ps = p.ps;
    const size_t kv_slot_stride = (size_t)2 * p.Hkv * D * kKvElt;

    for (;;) {
        if (tid == 0) s_item = atomicAdd(p.ctrl + p.counter_word, 1);
        __syncthreads();
        const int it_idx = s_item;
        if (it_idx >= n_items) break;
        const Item item = item_at(p.units, it_idx, p.unit_heads);
        const int s = item.seq, h = item.head;
        const int q_start = p.cu_q_lens[s];
        const int ql = p.cu_q_lens[s + 1] - q_start;
        const int kl = p.kv_lens[s];
        const int rows_used = item.ntok * G;
        const int kv_begin = item.kv_begin, kv_end = item.kv_end;
        const int* ptab = p.page_indices + (size_t)s * p.P;

        // ---- Q tile -> shared (swizzled 16-bit rows); rows past the item are zero
        for (int c = tid; c < C::kRows * kCh; c += kThreads) {
            const int r = c / kCh, ch = c % kCh;
            uint8_t* dst = q_s + r * kRowB + swz(r, ch);
            const bool valid = r < rows_used;
            const int t = q_start + item.tok0 + r / G;
            const int qh = h * G + r % G;
            const uint8_t* src = p.q + ((size_t)t * Hq + qh) * (D * 2) + ch * 16;
            if constexpr (FP8) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (valid) v = __ldg(reinterpret_cast<const uint4*>(src));
                // bf16 -> f16 for the f16 MMAs (f16 q as it is)
                uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t o4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) o4[k] = p.q_f16 ? w[k] : bf16x2_to_f16x2(w[k]);
                *reinterpret_cast<uint4*>(dst) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            } else {
                cp_async16(smem_u32(dst), valid ? (const void*)src : (const void*)p.q, valid);
            }
        }

        // ---- one stage of keys: K/V rows gathered through the page table
        auto load_stage = [&](int tile, int buf) {
            const int key0 = kv_begin + tile * kKeys;
            uint8_t* raw = stage_s + buf * C::kRawBytes;
            constexpr int CPK = FP8 ? kCh : 2 * kCh;  // 16-byte chunks per key (K then V)
#pragma unroll 4
            for (int c = tid; c < kKeys * CPK; c += kThreads) {
                const int kk = c / CPK, w = c % CPK;
                const int j = key0 + kk;
                bool valid = j < kv_end;
                const uint8_t* src = p.kv;
                if (valid) {
                    const int pg = __ldg(ptab + j / ps);
                    if ((unsigned)pg >= (unsigned)p.N) {
                        set_status(p.ctrl, RPA_ERR_BAD_PAGE_INDEX);
                        valid = false;
                    } else {
                        src = p.kv + ((size_t)pg * ps + (j % ps)) * kv_slot_stride +
                              (size_t)(2 * h) * (D * kKvElt) + w * 16;
                    }
                }
                uint32_t dst;
                if constexpr (FP8) {
                    dst = smem_u32(raw + kk * (2 * D) + w * 16);
                } else {
                    const int isv = w >= kCh;
                    const int ch = w - isv * kCh;
                    dst = smem_u32(raw + isv * (kKeys * kRowB) + kk * kRowB + swz(kk, ch));
                }
                cp_async16(dst, src, valid);
            }
        };

        // per-thread rows: lane/4 and lane/4 + 8 of this warp's 16
        int pos[2];
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            const int r = wm * 16 + (lane >> 2) + ri * 8;
            pos[ri] = kl - ql + item.tok0 + r / G;
        }
        float m_r[2] = {-INFINITY, -INFINITY};
        float l_r[2] = {0.f, 0.f};
        float o_acc[D / 8][4];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;

        const int n_tiles = (kv_end - kv_begin + kKeys - 1) / kKeys;
#pragma unroll
        for (int st = 0; st < STAGES - 1; ++st) {
            if (st < n_tiles) load_stage(st, st);
            cp_async_commit();
        }

        for (int tile = 0; tile < n_tiles; ++tile) {
            cp_async_wait<STAGES - 2>();
            __syncthreads();
            {
                const int nt = tile + STAGES - 1;
                if (nt < n_tiles) load_stage(nt, nt % STAGES);
                cp_async_commit();
            }
            const uint8_t* kt;
            if constexpr (FP8) {
                // 8-bit -> f16 (exact) into the single converted tile
                const uint8_t* raw = stage_s + (tile % STAGES) * C::kRawBytes;
                uint8_t* conv = stage_s + STAGES * C::kRawBytes;
                constexpr int U = 2 * D / 8;  // 8-element units per key (K then V)
                for (int c = tid; c < kKeys * U; c += kThreads) {
                    const int kk = c / U, w = c % U;
                    const int isv = w >= D / 8;
                    const int ch = w - isv * (D / 8);
                    const uint2 b = *reinterpret_cast<const uint2*>(raw + kk * (2 * D) + w * 8);
                    const uint4 o4 = cvt8x8_to_f16x8<KT>(b.x, b.y);
                    *reinterpret_cast<uint4*>(conv + isv * (kKeys * kRowB) + kk * kRowB + swz(kk, ch)) = o4;
                }
                __syncthreads();
                kt = conv;
            } else {
                kt = stage_s + (tile % STAGES) * C::kRawBytes;
            }
            const uint32_t qb = smem_u32(q_s);
            const uint32_t kb = smem_u32(kt);
            const uint32_t vb = kb + kKeys * kRowB;

            // ---- S = Q K^T  (16 rows x BK keys per warp)
            float sacc[BK / 8][4];
#pragma unroll
            for (int i = 0; i < BK / 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
            for (int kd = 0; kd < D / 16; ++kd) {
                uint32_t a[4];
                {
                    const int r = wm * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = 2 * kd + (lane >> 4);
                    ldsm_x4(qb + r * kRowB + swz(r, ch), a[0], a[1], a[2], a[3]);
                }
#pragma unroll
                for (int nb2 = 0; nb2 < BK / 16; ++nb2) {
                    const int key = wn * BK + nb2 * 16 + (lane & 7) + (lane >> 4) * 8;
                    const int ch = 2 * kd + ((lane >> 3) & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + key * kRowB + swz(key, ch), b0, b1, b2, b3);
                    mma16816<F16>(sacc[2 * nb2], a, b0, b1);
                    mma16816<F16>(sacc[2 * nb2 + 1], a, b2, b3);
                }
            }

            // ---- scale, softcap, mask (log2 domain)
            const int kbase = kv_begin + tile * kKeys + wn * BK;
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nb = 0; nb < BK / 8; ++nb) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = kbase + nb * 8 + (lane & 3) * 2 + (e & 1);
                    const int ri = e >> 1;
                    float x = sacc[nb][e];
                    if (p.has_cap) {
                        const float t = ex2(x * p.cap_exp);
                        x = p.cap_log2 - 2.f * p.cap_log2 * rcp_approx(1.f + t);
                    } else {
                        x *= p.qk_log2;
                    }
                    const bool ok = j < kv_end && (!p.causal || j <= pos[ri]) &&
                                    (!p.has_window || j > pos[ri] - p.window);
                    x = ok ? x : -INFINITY;
                    sacc[nb][e] = x;
                    mx[ri] = fmaxf(mx[ri], x);
                }
            }
            float base[2];
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 1));
                mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 2));
                const float m_new = fmaxf(m_r[ri], mx[ri]);
                base[ri] = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = ex2(m_r[ri] - base[ri]);
                m_r[ri] = m_new;
                l_r[ri] *= alpha;
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd) {
                    o_acc[nd][2 * ri] *= alpha;
                    o_acc[nd][2 * ri + 1] *= alpha;
                }
            }
#pragma unroll
            for (int nb = 0; nb < BK / 8; ++nb) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pe = ex2(sacc[nb][e] - base[e >> 1]);
                    sacc[nb][e] = pe;
                    l_r[e >> 1] += pe;
                }
            }

            // ---- O += P V
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                uint32_t a[4];
                a[0] = pack2<F16>(sacc[2 * kk][0], sacc[2 * kk][1]);
                a[1] = pack2<F16>(sacc[2 * kk][2], sacc[2 * kk][3]);
                a[2] = pack2<F16>(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
                a[3] = pack2<F16>(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
                for (int nd2 = 0; nd2 < D / 16; ++nd2) {
                    const int key = wn * BK + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = 2 * nd2 + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + key * kRowB + swz(key, ch), b0, b1, b2, b3);
                    mma16816<F16>(o_acc[2 * nd2], a, b0, b1);
                    mma16816<F16>(o_acc[2 * nd2 + 1], a, b2, b3);
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();

        // ---- epilogue
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            l_r[ri] += __shfl_xor_sync(0xffffffffu, l_r[ri], 1);
            l_r[ri] += __shfl_xor_sync(0xffffffffu, l_r[ri], 2);
        }
        if constexpr (WN == 1) {
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                const int r = wm * 16 + (lane >> 2) + ri * 8;
                if (r >= rows_used) continue;
                const int t = q_start + item.tok0 + r / G;
                const int qh = h * G + r % G;
                if (item.part < 0) {
                    const float l = add_sink(l_r[ri], p.sinks, qh, m_r[ri]);
                    const float inv = l > 0.f ? p.v_scale / l : 0.f;
                    const size_t orow = ((size_t)t * Hq + qh) * D;  // element offset of the output row
#pragma unroll
                    for (int nd = 0; nd < D / 8; ++nd)
                        store_o2(p.o, orow + nd * 8 + (lane & 3) * 2, o_acc[nd][2 * ri] * inv,
                                 o_acc[nd][2 * ri + 1] * inv, p.odt);
                } else {
                    float* prow = p.part_o + ((size_t)item.part * kDecRows + r) * D;
#pragma unroll
                    for (int nd = 0; nd < D / 8; ++nd)
                        *reinterpret_cast<float2*>(prow + nd * 8 + (lane & 3) * 2) =
                            make_float2(o_acc[nd][2 * ri], o_acc[nd][2 * ri + 1]);
                    if ((lane & 3) == 0)
                        *reinterpret_cast<float2*>(p.part_ml + ((size_t)item.part * kDecRows + r) * 2) =
                            make_float2(m_r[ri], l_r[ri]);
                }
            }
        } else {
            // merge the WN key-split warps through shared memory
            float* red_o = reinterpret_cast<float*>(stage_s);  // [WN][16][D]
            float* red_ml = red_o + WN * 16 * D;               // [WN][16][2]
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                const int r = (lane >> 2) + ri * 8;
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd)
                    *reinterpret_cast<float2*>(red_o + (wn * 16 + r) * D + nd * 8 + (lane & 3) * 2) =
                        make_float2(o_acc[nd][2 * ri], o_acc[nd][2 * ri + 1]);
                if ((lane & 3) == 0) {
                    red_ml[(wn * 16 + r) * 2] = m_r[ri];
                    red_ml[(wn * 16 + r) * 2 + 1] = l_r[ri];
                }
            }
            __syncthreads();
            for (int e = tid; e < 16 * (D / 2); e += kThreads) {
                const int r = e / (D / 2);
                const int c = (e % (D / 2)) * 2;
                if (r >= rows_used) continue;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < WN; ++w) M = fmaxf(M, red_ml[(w * 16 + r) * 2]);
                float L = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
                for (int w = 0; w < WN; ++w) {
                    const float sc = M == -INFINITY ? 0.f : ex2(red_ml[(w * 16 + r) * 2] - M);
                    L += sc * red_ml[(w * 16 + r) * 2 + 1];
                    const float2 v = *reinterpret_cast<const float2*>(red_o + (w * 16 + r) * D + c);
                    o0 += sc * v.x;
                    o1 += sc * v.y;
                }
                const int t = q_start + item.tok0 + r / G;
                const int qh = h * G + r % G;
                if (item.part < 0) {
                    const float Ls = add_sink(L, p.sinks, qh, M);
                    const float inv = Ls > 0.f ? p.v_scale / Ls : 0.f;
                    store_o2(p.o, ((size_t)t * Hq + qh) * D + c, o0 * inv, o1 * inv, p.odt);
                } else {
                    *reinterpret_cast<float2*>(p.part_o + ((size_t)item.part * kDecRows + r) * D + c) =
                        make_float2(o0, o1);
                    if (c == 0)
                        *reinterpret_cast<float2*>(p.part_ml + ((size_t)item.part * kDecRows + r) * 2) =
                            make_float2(M, L);
                }
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- instantiations
// prefill: 64 rows (4 warps), all warps share each stage
template <int D>
struct PfShape {
    static constexpr int WM = 4, WN = 1, BK = (D >= 256 ? 32 : 64), STAGES = (D >= 256 ? 2 : 3);
};

template <int D, int KT>
__global__ void __launch_bounds__(128) rpa_prefill_attn(const AttnParams p) {
    using S = PfShape<D>;
    attn_body<D, KT, S::WM, S::WN, S::BK, S::STAGES>(p);
}

template <int D, int KT>
struct Kern {
    using S = PfShape<D>;
    using C = KCfg<D, KT, S::WM, S::WN, S::BK, S::STAGES>;
    static_assert(C::kThreads == 128, "launch bounds");
    static cudaError_t prepare(int* blocks_per_sm) {
        cudaError_t e = cudaFuncSetAttribute(rpa_prefill_attn<D, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, rpa_prefill_attn<D, KT>, C::kThreads,
                                                             C::kSmem);
    }
    static cudaError_t launch(const AttnParams& p, const Launch& l) {
        return launch_pdl(rpa_prefill_attn<D, KT>, l.grid, C::kThreads, C::kSmem, l.stream, p);
    }
};

// The configurations routed here: 8-bit K/V at D 64 (the tensor-memory kernels cover 2-byte K/V
// at every head size and 8-bit K/V at D 128 / 256).
template <typename Op>
cudaError_t mma_dispatch(int D, int kt, Op op) {
    if (D == 64) {
        if (kt == KT_E4M3) return op(Kern<64, KT_E4M3>{});
        if (kt == KT_E5M2) return op(Kern<64, KT_E5M2>{});
        if (kt == KT_I8) return op(Kern<64, KT_I8>{});
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const AttnParams& p, int kt, const Launch& l) {
    return mma_dispatch(p.D, kt, [&](auto k) { return decltype(k)::launch(p, l); });
}
cudaError_t attn_prepare(int D, int kt, int* pf_bps) {
    return mma_dispatch(D, kt, [&](auto k) { return decltype(k)::prepare(pf_bps); });
}

}  // namespace rpa
