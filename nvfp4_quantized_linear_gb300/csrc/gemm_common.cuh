// Pieces shared by the tensor-core kernels (the two GEMMs and the transform
// quantizer): tile order, tensor-map builders.
#pragma once

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace nvfp4 {
namespace gemm_detail {

struct Tile {
    int mb, nb;
};

// 512-byte scale tiles (128 rows x 4 scale columns) per 128-row band in one
// 256-element K stage: NVFP4 has a scale per 16 elements (4 tiles), MXFP4 one
// per 32 (2 tiles).
template <bool kMx>
constexpr int kSfTilesPerStage = kMx ? 2 : 4;

// Tiles are walked column by column (row band fastest) inside groups of
// `group` row bands (at most): the CTAs resident at one time work on a few
// weight column bands, so each weight tile is streamed from DRAM about once
// and shared by the row bands through L2, while the group's activation rows
// stay resident in L2 across columns.  Both GEMM kernels use groups of 8192
// activation rows (64 bands of 128 rows, or 32 pair tiles of 256 rows): on the
// Qwen gate_up shape (M = 16384, K = 5120) the CTA-pair kernel measured
// 1278 us with 32-tile groups against 1327 us with 64 and 1311 / 1385 us with
// 16 / 8.
__device__ __forceinline__ Tile tile_coord(int tile, int num_m, int num_n, int group = 64)
{
    const int G = num_m < group ? num_m : group;
    const int per_group = G * num_n;
    const int grp = tile / per_group;
    const int first_m = grp * G;
    const int gm = min(G, num_m - first_m);
    const int within = tile - grp * per_group;
    return {first_m + within % gm, within / gm};
}

__device__ __forceinline__ uint32_t bf16_bits_rn(float f)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}


inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2-D map over a packed FP4 operand [rows, row_bytes] with boxes of
// `box_bytes` (64 or 128) x `box_rows`, swizzled with the same width, zero
// fill outside the tensor.
inline bool make_operand_map(CUtensorMap *map, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows,
                             uint32_t box_bytes = 128)
{
    auto encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_bytes, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle swz = box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map of the bf16 output [m, n_out] (row stride ldo elements) for TMA stores
// of 16-column x 32-row boxes, no swizzle.  The TMA skips elements outside
// [0, n_out) x [0, m).  Requires a 16-B aligned base and ldo % 8 == 0.
inline bool make_output_map(CUtensorMap *map, void *base, uint64_t n_out, uint64_t m, uint64_t ldo)
{
    auto encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    cuuint64_t dims[2] = {n_out, m};
    cuuint64_t strides[1] = {ldo * 2};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map of the bf16 output [m, n_out] (row stride ldo elements) for TMA stores
// of 64-column x 32-row boxes (128-byte rows) with the 128-byte swizzle; the
// TMA skips elements outside [0, n_out) x [0, m).  Requires a 16-B aligned base
// and ldo % 8 == 0.
inline bool make_output_map_sw128(CUtensorMap *map, void *base, uint64_t n_out, uint64_t m, uint64_t ldo)
{
    auto encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    cuuint64_t dims[2] = {n_out, m};
    cuuint64_t strides[1] = {ldo * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map of a tiled scale tensor viewed as [bands, band_bytes / 8] 8-byte
// elements (one row per 128-row band), for copies of `box_elems` elements of
// two consecutive bands at once (the scale tiles of one K stage of a 256-row
// operand tile); zero fill past the last band or the band's end.  band_bytes
// is a multiple of 512 and the base 16-B aligned.
inline bool make_scale_bands_map(CUtensorMap *map, const void *base, uint64_t band_bytes, uint64_t bands,
                                 uint32_t box_elems)
{
    auto encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    cuuint64_t dims[2] = {band_bytes / 8, bands};
    cuuint64_t strides[1] = {band_bytes};
    cuuint32_t box[2] = {box_elems, 2};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map of a bf16 activation [m, k] (row stride ld elements) for copies of 256
// columns x 16 rows (the fused small-m linear's per-stage slice), no swizzle,
// zero fill past m and k.  Requires a 16-B aligned base and ld % 8 == 0.
inline bool make_x_slice_map(CUtensorMap *map, const void *base, uint64_t k, uint64_t m, uint64_t ld)
{
    auto encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    cuuint64_t dims[2] = {k, m};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {256, 16};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over bf16 rows [rows, cols] (row stride ld elements) with boxes of
// 64 columns x 128 rows, 128-byte swizzle (the K-major operand layout of a
// kind::f16 MMA), zero fill outside the tensor.  Requires a 16-B aligned base
// and ld % 8 == 0.
inline bool make_bf16_rows_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t ld)
{
    auto encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gemm_detail
}  // namespace nvfp4
