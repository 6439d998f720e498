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
// Work goes out in units of a few rows of one entry (one group of four columns per thread).  An
// entry of at most eight pieces merges in registers; longer ones first reduce each row's m and l
// (a warp per row) into shared-memory scale factors.  Entries hold at most `rows_max` rows (the
// decode tile's rows: the planner classifies a sequence as decode only when q_len * G fits).
//
// The same kernel writes zeros into the rows of tokens that no sequence
// covers (outside [cu_q_lens[0], cu_q_lens[num_seqs])), so that o is always
// fully defined; after a length error the planner marks every row uncovered.
#include "rpa_internal.cuh"

namespace rpa {

namespace {

constexpr int kCombThreads = 256;
constexpr int kCombCache = 64;  // pieces whose per-row scale factors are kept in shared memory
constexpr int kDirect = 8;      // entries of at most this many pieces merge without shared memory

__global__ void __launch_bounds__(kCombThreads, 2) rpa_combine_kernel(const CombParams p) {
    __shared__ float s_sc[kCombCache][kDecRows];  // 2^(m_i - M) of piece i and row r
    __shared__ float s_M[kDecRows], s_inv[kDecRows];
    pdl_wait();  // the attention kernels' partials are complete from here on
    const int n_comb = p.ctrl[kNumComb];
    const int D = p.D, G = p.G, Hq = p.Hq;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // a unit of work: rpu rows of one entry, so that each thread merges one group of four
    // columns (more units than entries keep more SMs busy)
    const int quads = D / 4;
    const int rmax = max(1, min(p.rows_max, kDecRows));
    const int rpu = max(1, min(rmax, kCombThreads / quads));
    const int upe = (rmax + rpu - 1) / rpu;
    for (int u = blockIdx.x; u < n_comb * upe; u += gridDim.x) {
        const int e = u / upe, r0 = (u % upe) * rpu;
        const Comb c = p.comb[e];
        const int q0 = p.cu_q_lens[c.seq];
        const int rows = (p.cu_q_lens[c.seq + 1] - q0) * G;
        const int r1 = min(rows, r0 + rpu);
        if (r0 >= rows) continue;  // the same for every thread of the block
        const float* ml = p.part_ml + (size_t)c.part * kDecRows * 2;  // [pieces][kDecRows][2]
        if (c.pieces <= kDirect) {
            // few pieces: each thread merges its four columns of a row on its own (the row's m and
            // l are re-read by the row's threads; all loads are issued before the sums)
            for (int x = tid; x < (r1 - r0) * quads; x += kCombThreads) {
                const int r = r0 + x / quads, col = (x % quads) * 4;
                float2 mlk[kDirect];
                float4 v[kDirect];
                float M = -INFINITY;
#pragma unroll
                for (int k = 0; k < kDirect; ++k) {
                    if (k < c.pieces) {
                        const size_t pr = (size_t)(c.part + k) * kDecRows + r;
                        mlk[k] = *reinterpret_cast<const float2*>(p.part_ml + pr * 2);
                        v[k] = *reinterpret_cast<const float4*>(p.part_o + pr * D + col);
                        M = fmaxf(M, mlk[k].x);
                    }
                }
                float L = 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M != -INFINITY) {
#pragma unroll
                    for (int k = 0; k < kDirect; ++k) {
                        if (k < c.pieces) {
                            const float sc = ex2(mlk[k].x - M);
                            L += sc * mlk[k].y;
                            acc.x += sc * v[k].x;
                            acc.y += sc * v[k].y;
                            acc.z += sc * v[k].z;
                            acc.w += sc * v[k].w;
                        }
                    }
                }
                const int t = q0 + r / G;
                const int qh = c.head * G + r % G;
                L = add_sink(L, p.sinks, qh, M);  // the sink joins once, over all pieces
                const float inv = L > 0.f ? p.v_scale / L : 0.f;
                store_o4(p.o, ((size_t)t * Hq + qh) * D + col, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv,
                         p.odt);
            }
            continue;  // the same for every thread of the block
        }
        // 1. per row (a warp per row, lanes over the pieces): M, the scale factors and 1 / L
        for (int r = r0 + warp; r < r1; r += kCombThreads / 32) {
            float M = -INFINITY;
            for (int k = lane; k < c.pieces; k += 32) M = fmaxf(M, ml[((size_t)k * kDecRows + r) * 2]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            float L = 0.f;
            if (M != -INFINITY) {
                for (int k = lane; k < c.pieces; k += 32) {
                    const float2 v = *reinterpret_cast<const float2*>(ml + ((size_t)k * kDecRows + r) * 2);
                    const float sc = ex2(v.x - M);
                    if (k < kCombCache) s_sc[k][r] = sc;
                    L += sc * v.y;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
            if (lane == 0) {
                L = add_sink(L, p.sinks, c.head * G + r % G, M);  // the sink joins once, over all pieces
                s_M[r] = M;
                s_inv[r] = L > 0.f ? p.v_scale / L : 0.f;
            }
        }
        __syncthreads();
        // 2. each thread: four columns of a row, summed over the pieces (loads of several pieces
        // in flight at once)
        for (int x = tid; x < (r1 - r0) * quads; x += kCombThreads) {
            const int r = r0 + x / quads, col = (x % quads) * 4;
            const float M = s_M[r];
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (M != -INFINITY) {
                const float* po = p.part_o + ((size_t)c.part * kDecRows + r) * D + col;
#pragma unroll 4
                for (int k = 0; k < c.pieces; ++k) {
                    const float sc = k < kCombCache ? s_sc[k][r] : ex2(ml[((size_t)k * kDecRows + r) * 2] - M);
                    const float4 v = *reinterpret_cast<const float4*>(po + (size_t)k * kDecRows * D);
                    acc.x += sc * v.x;
                    acc.y += sc * v.y;
                    acc.z += sc * v.z;
                    acc.w += sc * v.w;
                }
            }
            const float inv = s_inv[r];
            const int t = q0 + r / G;
            const int qh = c.head * G + r % G;
            store_o4(p.o, ((size_t)t * Hq + qh) * D + col, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv, p.odt);
        }
        __syncthreads();
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
