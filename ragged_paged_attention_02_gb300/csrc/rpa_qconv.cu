// rpa_qconv.cu -- q in the tensor cores' operand type.
//
// The MMAs take both operands in one type (bf16 with bf16 K/V, f16 with f16
// and 8-bit K/V).  A q of another type (f32 q, or a 16-bit q of the other
// 16-bit type) is rounded to that type, to nearest even, into the workspace
// before the attention kernels read it.  An HBM-bound pass: each thread moves
// eight elements at a time (16 or 32 bytes in, 16 out).
#include "rpa_internal.cuh"

namespace rpa {

namespace {

constexpr int kQcThreads = 256;

__device__ __forceinline__ void load8(const uint8_t* q, size_t i, int q_dtype, float* f) {
    if (q_dtype == RPA_DT_F32) {
        const float4 a = *reinterpret_cast<const float4*>(q + i * 4);
        const float4 b = *reinterpret_cast<const float4*>(q + i * 4 + 16);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else {
        const uint4 v = *reinterpret_cast<const uint4*>(q + i * 2);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (q_dtype == RPA_DT_F16) {
                const float2 h = f16x2_to_f32x2(w[k]);
                f[2 * k] = h.x;
                f[2 * k + 1] = h.y;
            } else {
                f[2 * k] = __uint_as_float(w[k] << 16);
                f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
            }
        }
    }
}

__global__ void __launch_bounds__(kQcThreads) rpa_q_convert_kernel(const uint8_t* __restrict__ q, int q_dtype,
                                                                    uint8_t* __restrict__ out, int to_f16, size_t n8) {
    for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < n8; g += (size_t)gridDim.x * blockDim.x) {
        float f[8];
        load8(q, g * 8, q_dtype, f);
        uint4 o;
        if (to_f16)
            o = make_uint4(pack2<true>(f[0], f[1]), pack2<true>(f[2], f[3]), pack2<true>(f[4], f[5]),
                           pack2<true>(f[6], f[7]));
        else
            o = make_uint4(pack2<false>(f[0], f[1]), pack2<false>(f[2], f[3]), pack2<false>(f[4], f[5]),
                           pack2<false>(f[6], f[7]));
        *reinterpret_cast<uint4*>(out + g * 16) = o;
    }
}

}  // namespace

cudaError_t launch_q_convert(const void* q, int q_dtype, uint8_t* out, int to_f16, size_t n, const Launch& l) {
    // n = T * Hq * D, a multiple of 64 (head_dim in {64, 128, 256})
    const size_t n8 = n / 8;
    const size_t want = (n8 + kQcThreads - 1) / kQcThreads;
    const int grid = (int)(want < (size_t)l.grid ? (want > 0 ? want : 1) : (size_t)l.grid);
    rpa_q_convert_kernel<<<grid, kQcThreads, 0, l.stream>>>(static_cast<const uint8_t*>(q), q_dtype, out, to_f16, n8);
    return cudaGetLastError();
}

}  // namespace rpa
