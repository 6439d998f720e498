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
// The same kernel writes zeros into the rows of tokens that no sequence
// covers (outside [cu_q_lens[0], cu_q_lens[num_seqs])), so that o is always
// fully defined; after a length error the planner marks every row uncovered.
#include "rpa_internal.cuh"

namespace rpa {

namespace {

__global__ void __launch_bounds__(256) rpa_combine_kernel(const CombParams p) {
    pdl_wait();  // the attention kernels' partials are complete from here on
    const int n_comb = p.ctrl[kNumComb];
    const int D = p.D, G = p.G, Hq = p.Hq;
    for (int e = blockIdx.x; e < n_comb; e += gridDim.x) {
        const Comb c = p.comb[e];
        const int q0 = p.cu_q_lens[c.seq];
        const int rows = (p.cu_q_lens[c.seq + 1] - q0) * G;
        for (int x = threadIdx.x; x < rows * (D / 2); x += blockDim.x) {
            const int r = x / (D / 2);
            const int col = (x % (D / 2)) * 2;
            float M = -INFINITY;
            for (int k = 0; k < c.pieces; ++k)
                M = fmaxf(M, p.part_ml[((size_t)(c.part + k) * kDecRows + r) * 2]);
            float L = 0.f, o0 = 0.f, o1 = 0.f;
            if (M != -INFINITY) {
                for (int k = 0; k < c.pieces; ++k) {
                    const size_t pr = (size_t)(c.part + k) * kDecRows + r;
                    const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + pr * 2);
                    const float sc = ex2(ml.x - M);
                    L += sc * ml.y;
                    const float2 v = *reinterpret_cast<const float2*>(p.part_o + pr * D + col);
                    o0 += sc * v.x;
                    o1 += sc * v.y;
                }
            }
            const float inv = L > 0.f ? p.v_scale / L : 0.f;
            const int t = q0 + r / G;
            const int qh = c.head * G + r % G;
            *reinterpret_cast<uint32_t*>(p.o + (((size_t)t * Hq + qh) * D + col) * 2) =
                pack2<false>(o0 * inv, o1 * inv);
        }
    }
    // zero rows of uncovered tokens: [0, lo) and [hi, T)
    const int lo = min(max(p.ctrl[kCovLo], 0), p.T);
    const int hi = min(max(p.ctrl[kCovHi], lo), p.T);
    const size_t row16 = (size_t)Hq * D * 2 / 16;  // 16-byte words per token row
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
    return launch_pdl(rpa_combine_kernel, l.grid, 256, 0, l.stream, p);
}

}  // namespace rpa
