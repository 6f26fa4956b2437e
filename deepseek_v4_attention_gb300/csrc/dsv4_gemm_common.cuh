// dsv4_gemm_common.cuh -- what the block-scaled GEMM kernels share
// (dsv4_gemm.cu: one CTA per tile; dsv4_gemm_pair.cu: CTA pairs): tile sizes,
// kernel parameters, the tile order, the weight-scale words and the
// tensor-map encoding.
#pragma once

#include <string.h>

#include "dsv4_device.cuh"
#include "dsv4_internal.h"

namespace dsv4 {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 128;
constexpr int kTmemCols = 512;
constexpr int kRasterM = 16;   // m-blocks per raster group (G = 1); 8 measured worse

constexpr uint32_t kSfaBytes = kBM * 4;    // 512 B

struct Params {
  int64_t T;
  int G, N, K;
  int m_tiles, n_tiles, num_tiles, k_blocks, packs;
  int64_t t_al;
  const int32_t* a_scale;  // int32 [G][packs][t_al]
  const uint8_t* b_scale;
  int b_scale_ld;          // K / 128
  __nv_bfloat16* out;      // [T][G*N] or null
  uint8_t* q_out;          // [T][G*N]
  int32_t* q_scale;        // [ceil(G*N/512)][t_al]
  int* status;             // device status word
  // fused A only
  const uint16_t* o;       // bf16 [T][H][512]
  const int64_t* positions;
  const float* cache;      // fp32 [max_pos][64]
  int64_t max_pos;
  int H, hpg;
  int raster_m;            // > 0: tiles in groups of raster_m m-blocks (G = 1), see tile_coords
  int prefetch_l2;         // launched to overlap the previous kernel: before waiting for it,
                           // prefetch the first tile's remaining weight k-blocks into L2
};

// Tile order.  Default: m-blocks fastest, then column tiles, then groups (the
// column tiles of one group's m-block run in the same wave and share its A tile
// in L2).  raster_m > 0 (a single group with many m-blocks, the dense wo_b):
// groups of raster_m m-blocks, column tiles within a group, so that a wave
// re-reads only its group's share of A (measured at T = 4096: DRAM reads of
// wo_b 536 -> 411 MB).
__device__ __forceinline__ void tile_coords(const Params& p, int tile, int& g, int& n_blk,
                                            int& m_blk) {
  if (p.raster_m > 0) {
    const int per_group = p.raster_m * p.n_tiles;
    const int grp = tile / per_group;
    const int idx = tile - grp * per_group;
    const int rest_m = p.m_tiles - grp * p.raster_m;
    const int m_in = rest_m < p.raster_m ? rest_m : p.raster_m;   // the last group may be short
    n_blk = idx / m_in;
    m_blk = grp * p.raster_m + (idx - n_blk * m_in);
    g = 0;
    return;
  }
  m_blk = tile % p.m_tiles;
  const int rest = tile / p.m_tiles;
  n_blk = rest % p.n_tiles;
  g = rest / p.n_tiles;
}

// Packed scale word of weight row block `rb` for k-blocks 4j..4j+3 (bytes
// beyond the last k-block are 0).
__device__ __forceinline__ uint32_t b_scale_word(const Params& p, int rb, int j) {
  const uint8_t* row = p.b_scale + static_cast<int64_t>(rb) * p.b_scale_ld;
  uint32_t w = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int kb = 4 * j + b;
    if (kb < p.k_blocks) w |= static_cast<uint32_t>(__ldg(row + kb)) << (8 * b);
  }
  return w;
}

// ----------------------------------------------------------- host side --
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
            const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
            CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t elem_strides[3] = {1, 1, 1};
  return fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides_bytes,
            box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

}  // namespace dsv4
