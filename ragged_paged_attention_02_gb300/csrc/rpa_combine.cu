// rpa_combine.cu -- K2: split-KV merge and output completion.
//
// A decode item whose keys were split into pieces leaves, per piece i and row
// r, the unnormalised partial O_i = sum_j 2^{x_j - m_i} v_j together with m_i
// (log2-domain max) and l_i = sum_j 2^{x_j - m_i}.  The merge is the same
// algebra as the page's online-softmax step (flashAttention: m_next, alpha,
// beta, l_next) applied across pieces instead of across key blocks:
//
//   M = max_i m_i,   L = sum_i 2^{m_i - M} l_i,   o = v_scale * sum_i 2^{m_i - M} O_i / L
//
// With attention sinks the row's sink term 2^{s log2(e) - M} joins L here, once: the pieces
// leave it out.
//
// Each warp merges 128 columns of one row of one entry at a time (the tasks of an entry on
// consecutive warps).  Its partial O loads (up to eight pieces, all in flight at once) go out as soon
// as the entry is read; beside them, lanes over the pieces reduce the row's m and l to M, the scale
// factors 2^(m_i - M) and 1 / L (shuffles).  No block barrier: a task costs two dependent rounds of
// loads.  Entries hold at most `rows_max` rows (the decode tile's rows: the planner classifies a
// sequence as decode only when q_len * G fits).
//
// The same kernel writes zeros into the rows of tokens that no sequence
// covers (outside [cu_q_lens[0], cu_q_lens[num_seqs])), so that o is always
// fully defined; after a length error the planner marks every row uncovered.
#include "rpa_internal.cuh"

namespace rpa {

namespace {

constexpr int kCombThreads = 256;
constexpr int kBatch = 6;  // pieces whose partial O loads a lane has in flight at once

__global__ void __launch_bounds__(kCombThreads, kCombCtasPerSm) rpa_combine_kernel(const CombParams p) {
    pdl_trigger();  // the next call's planner may start its first phases now
    pdl_wait();     // the attention kernels' partials are complete from here on
    const int n_comb = p.ctrl[kNumComb];
    const int D = p.D, G = p.G, Hq = p.Hq;
    const int lane = threadIdx.x & 31;
    const int rmax = max(1, min(p.rows_max, kDecRows));
    const int quads = D / 4;
    const int nchunk = (quads + 31) / 32;  // 128-column chunks of a row
    const int per_entry = rmax * nchunk;
    const int warps = gridDim.x * (kCombThreads / 32);
    for (int task = blockIdx.x * (kCombThreads / 32) + (threadIdx.x >> 5); task < n_comb * per_entry;
         task += warps) {
        const int e = task / per_entry, rem = task - e * per_entry;
        const int r = rem / nchunk, c4 = (rem - r * nchunk) * 32 + lane;
        const int4* cp = reinterpret_cast<const int4*>(p.comb + e);
        const int4 c0 = cp[0], c1 = cp[1];
        const int q0 = c0.x, rows = c0.y, head = c0.z, part = c0.w, pieces = c1.x;
        if (r >= rows) continue;  // the same for every lane of the warp
        const bool act = c4 < quads;
        const float* ml = p.part_ml + ((size_t)part * kDecRows + r) * 2;  // piece k at + k kDecRows 2
        // piece k's four columns at pv[k * kstride] (float4 units)
        const float4* pv = reinterpret_cast<const float4*>(p.part_o + ((size_t)part * kDecRows + r) * D) + c4;
        const int kstride = kDecRows * D / 4;
        // few pieces: every partial O load in flight before the m / l reduction
        const bool held = pieces <= kBatch;
        float4 v[kBatch];
        if (held) {
#pragma unroll
            for (int k = 0; k < kBatch; ++k)
                if (act && k < pieces) v[k] = pv[k * kstride];
        }
        // the row's M, and L over all pieces (lanes over the pieces, 32 at a time)
        float M = -INFINITY;
        for (int k = lane; k < pieces; k += 32) M = fmaxf(M, ml[(size_t)k * kDecRows * 2]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f, sc_mine = 0.f;  // sc_mine: 2^(m_lane - M) for piece `lane` (the first 32)
        if (M != -INFINITY) {
            for (int k = lane; k < pieces; k += 32) {
                const float2 w = *reinterpret_cast<const float2*>(ml + (size_t)k * kDecRows * 2);
                const float sc = ex2(w.x - M);
                if (k < 32) sc_mine = sc;
                L += sc * w.y;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        const int qh = head * G + r % G;
        L = add_sink(L, p.sinks, qh, M);  // the sink joins once, over all pieces
        const float inv = L > 0.f ? p.v_scale / L : 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            if (held) {
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    if (k < pieces) {
                        const float sc = __shfl_sync(0xffffffffu, sc_mine, k);
                        if (act) {
                            acc.x += sc * v[k].x;
                            acc.y += sc * v[k].y;
                            acc.z += sc * v[k].z;
                            acc.w += sc * v[k].w;
                        }
                    }
                }
            } else {
                // many pieces: batches of kBatch loads; every lane runs every step (shuffles)
                for (int k0 = 0; k0 < pieces; k0 += kBatch) {
#pragma unroll
                    for (int k = 0; k < kBatch; ++k)
                        if (act && k0 + k < pieces) v[k] = pv[(k0 + k) * kstride];
#pragma unroll
                    for (int k = 0; k < kBatch; ++k) {
                        if (k0 + k < pieces) {
                            const int kk = k0 + k;
                            const float sc = kk < 32 ? __shfl_sync(0xffffffffu, sc_mine, kk)
                                                     : ex2(ml[(size_t)kk * kDecRows * 2] - M);
                            if (act) {
                                acc.x += sc * v[k].x;
                                acc.y += sc * v[k].y;
                                acc.z += sc * v[k].z;
                                acc.w += sc * v[k].w;
                            }
                        }
                    }
                }
            }
        }
        if (act)
            store_o4(p.o, ((size_t)(q0 + r / G) * Hq + qh) * D + 4 * c4, acc.x * inv, acc.y * inv, acc.z * inv,
                     acc.w * inv, p.odt);
    }
    // zero rows of uncovered tokens: [0, lo) and [hi, T)
    const int lo = min(max(p.ctrl[kCovLo], 0), p.T);
    const int hi = min(max(p.ctrl[kCovHi], lo), p.T);
    const size_t row16 = (size_t)Hq * D * (p.odt == OT_F32 ? 4 : 2) / 16;  // 16-byte words per token row
    const size_t n_lo = (size_t)lo * row16;
    const size_t n_hi = (size_t)(p.T - hi) * row16;
    uint4* o16 = reinterpret_cast<uint4*>(p.o);
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_lo + n_hi;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t w = i < n_lo ? i : (size_t)hi * row16 + (i - n_lo);
        o16[w] = z;
    }
}

}  // namespace

cudaError_t launch_combine(const CombParams& p, const Launch& l) {
    return launch_pdl(rpa_combine_kernel, l.grid, kCombThreads, 0, l.stream, p);
}

}  // namespace rpa
