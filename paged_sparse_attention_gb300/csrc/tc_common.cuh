// Shared pieces of the tcgen05 attention kernels (bf16, head_dim 128, page 128):
// tile geometry, the 128B-swizzled shared-memory operand descriptors and the host
// side tensor-map construction for TMA.
#pragma once
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "sm103_ptx.cuh"

namespace oomb {
namespace tc {

constexpr int kTile = 128;                         // rows of a query tile == tokens per page
constexpr int kD = 128;                            // head dim
constexpr uint32_t kTileBytes = kTile * kD * 2;    // one bf16 128x128 operand tile: 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;    // one 128 x 64 TMA box (128B rows)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// A 128x128 bf16 tile is held as two [128 rows][64 cols] boxes with the 128-byte
// swizzle; rows are 128 B apart and 8-row groups 1024 B apart.
//
// K-major operand (rows = M or N, 128-wide K split over the two boxes): the
// 16-wide K step kk starts in box kk/4 at byte (kk%4)*32 of the row.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_saddr, int kk, uint32_t box_bytes = kHalfBytes) {
  return smem_desc(tile_saddr + (uint32_t)(kk >> 2) * box_bytes + (uint32_t)(kk & 3) * 32u, 16, 1024,
                   kSwizzle128B);
}
// MN-major operand (rows = K, 128-wide M/N split over the two boxes, LBO = box
// stride): the 16-row K step kk starts at row 16*kk.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile_saddr, int kk, uint32_t box_bytes = kHalfBytes) {
  return smem_desc(tile_saddr + (uint32_t)kk * 2048u, box_bytes, 1024, kSwizzle128B);
}

// Byte offset of element (row, col) of a 128x128 bf16 tile stored in the layout above
// (for threads that write operands to shared memory themselves).
__device__ __forceinline__ uint32_t swz_offset(int row, int col) {
  const int box = col >> 6, c = col & 63;
  const int chunk = (c >> 3) ^ (row & 7);
  return (uint32_t)box * kHalfBytes + (uint32_t)row * 128u + (uint32_t)chunk * 16u + (uint32_t)(c & 7) * 2u;
}

__device__ __forceinline__ uint32_t tmem_lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }

// ------------------------------------------------------------------ host side
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map over a [rows, 128] bf16 matrix with [128 rows x 64 cols] boxes, 128B swizzle.
inline bool make_tmap_rows(CUtensorMap* m, const void* base, uint64_t rows) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, kTile};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a token-major [n, H, 128] bf16 tensor: box = `rows` tokens of one
// head, 64 columns; tokens beyond n read as zero.
inline bool make_tmap_heads(CUtensorMap* m, const void* base, int n, int H, int rows = kTile) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)n};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of the K/V source a tensor map must cover.
inline uint64_t kv_rows(const AttnArgs& a) {
  if (a.kv.staged) return (uint64_t)2 * a.g.Hkv * a.kv.stage_stride * kTile;
  return (uint64_t)a.g.num_phys * a.g.Hkv * kTile;
}

}  // namespace tc
}  // namespace oomb
