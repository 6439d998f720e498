// rpa_tmap.cu -- tensor maps (bulk-copy descriptors) for the decode gather.
//
// Host code only.  The encoder is the driver's cuTensorMapEncodeTiled,
// fetched through the runtime's driver entry point so that the library does
// not link libcuda directly.  Encoding fills a 128-byte descriptor on the
// host; it allocates nothing.
#include <cuda.h>
#include <cuda_runtime.h>

#include "rpa_internal.cuh"

namespace rpa {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

}  // namespace

// K/V pages viewed as a 2-D tensor: rows = N * page_size slots, each row the
// 2 * Hkv * D elements of one slot (combined heads: K of head h at 2h, V at
// 2h+1).  One box = BR slots x one 128-byte column block (2-byte elements,
// 128-byte swizzle) or BR slots x one whole D-byte row (1-byte elements, no
// swizzle).  The copies move bits: a 2-byte map serves bf16 and f16 alike.
int encode_kv_map(CUtensorMap* m, const void* kv, int fp8, long long N, int ps, int Hkv, int D, int BR) {
    EncodeTiledFn fn = encoder();
    if (!fn) return -1;
    const cuuint64_t dims[2] = {(cuuint64_t)(2 * Hkv * D), (cuuint64_t)(N * ps)};
    const cuuint64_t strides[1] = {(cuuint64_t)(2 * Hkv * D) * (fp8 ? 1u : 2u)};
    const cuuint32_t box[2] = {(cuuint32_t)(fp8 ? D : 64), (cuuint32_t)BR};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(kv), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

// K/V pages viewed as a 3-D tensor for the decode gather: (row elements of one
// 128-byte column block, slots, column blocks of a slot row).  One box = BR
// slots of kv head h: its K column blocks then its V column blocks, landing in
// shared memory as [2*D/64][BR][128 B] (2-byte elements, 128-byte swizzle);
// for 1-byte elements the box is (D bytes, BR slots, K and V) landing as
// [2][BR][D] (no swizzle).
// The slot dimension comes before the column-block dimension so that the BR
// rows of one column block are consecutive 128-byte lines.
int encode_kv_map_runs(CUtensorMap* m, const void* kv, int fp8, long long N, int ps, int Hkv, int D, int BR) {
    EncodeTiledFn fn = encoder();
    if (!fn) return -1;
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r;
    if (fp8) {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)(N * ps), (cuuint64_t)(2 * Hkv)};
        const cuuint64_t strides[2] = {(cuuint64_t)(2 * Hkv * D), (cuuint64_t)D};
        const cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)BR, 2u};
        r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(kv), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[3] = {64u, (cuuint64_t)(N * ps), (cuuint64_t)(2 * Hkv * D / 64)};
        const cuuint64_t strides[2] = {(cuuint64_t)(2 * Hkv * D * 2), 128u};
        const cuuint32_t box[3] = {64u, (cuuint32_t)BR, (cuuint32_t)(2 * D / 64)};
        r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kv), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

// A cache whose slots hold H rows of D 2-byte elements ([N, ps, H, D]) viewed as (64 elements of
// a column block, slots, column blocks of a slot: H * D / 64).  One box = BR slots of one row,
// landing as [D/64][BR][128 B] (128-byte swizzle): the MMA tile layout of BR keys.  Serves the
// latent cache (H = Hkv) and the split K/V cache seen as 2 Hkv rows (K of head h at 2h, V at
// 2h + 1), one box then being a page run's whole K (or V) tile.
int encode_kv_map_heads(CUtensorMap* m, const void* kv, long long N, int ps, int H, int D, int BR) {
    EncodeTiledFn fn = encoder();
    if (!fn) return -1;
    const cuuint64_t dims[3] = {64u, (cuuint64_t)(N * ps), (cuuint64_t)(H * D / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)(H * D * 2), 128u};
    const cuuint32_t box[3] = {64u, (cuuint32_t)BR, (cuuint32_t)(D / 64)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kv), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

// q viewed as (D, Hq, T): one box = 64 elements x the G heads of a kv group x
// Tt tokens, 128-byte swizzle; tokens past T read as zero.  q holds 2-byte
// elements (bf16 or f16: the copy moves bits).
int encode_q_map(CUtensorMap* m, const void* q, long long T, int Hq, int D, int G, int Tt) {
    EncodeTiledFn fn = encoder();
    if (!fn) return -1;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2u, (cuuint64_t)Hq * D * 2u};
    const cuuint32_t box[3] = {64u, (cuuint32_t)G, (cuuint32_t)Tt};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

}  // namespace rpa
