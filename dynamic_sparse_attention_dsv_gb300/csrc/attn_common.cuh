// Pieces shared by the sparse attention forward and backward kernels: tensor
// maps over Q/K/V, the per-launch parameter block and tile addressing.
#pragma once
#include "common.cuh"

namespace dsv {

// Tensor maps used by one attention launch (all over bf16 [P*S][d] tensors).
struct AttnMaps {
  CUtensorMap q_cube;   // 4D [P*T][Y][X][d], box (64, gx, gy, gt): one query group
  CUtensorMap k_rows;   // 2D [P*S][d], box (64, 1): row gather of selected keys
  CUtensorMap v_rows;
  CUtensorMap k_tile;   // 2D [P*S][d], box (64, 128): contiguous key tiles (dense)
  CUtensorMap v_tile;
};

struct AttnParams {
  Geometry geo;
  int32_t d;
  float scale_log2;          // scale * log2(e)
  float scale;
  const int32_t* idx;
  const __nv_bfloat16* Q;
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const __nv_bfloat16* O;    // bwd: forward output
  const __nv_bfloat16* dO;   // bwd
  const float* LSE;          // bwd
  __nv_bfloat16* out;        // fwd: O; bwd: dQ
  float* lse_out;            // fwd
  int32_t* status;
};

// 4D map over a [P*T][Y][X][d] view of a [P][S][d] tensor.
inline bool make_cube_map(CUtensorMap* m, const void* base, const Geometry& geo, int d, int P) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  memset(m, 0, sizeof(*m));
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)geo.X, (cuuint64_t)geo.Y, (cuuint64_t)P * geo.T};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)geo.X * d * 2, (cuuint64_t)geo.Y * geo.X * d * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)geo.gx, (cuuint32_t)geo.gy, (cuuint32_t)geo.gt};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool make_attn_maps(AttnMaps* m, const void* Q, const void* K, const void* V, const Geometry& geo, int d,
                           int P) {
  const uint64_t rows = (uint64_t)P * geo.S;
  return make_cube_map(&m->q_cube, Q, geo, d, P) &&
         make_map_2d(&m->k_rows, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, rows, 64, 1) &&
         make_map_2d(&m->v_rows, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, rows, 64, 1) &&
         make_map_2d(&m->k_tile, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, rows, 64, 128) &&
         make_map_2d(&m->v_tile, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, rows, 64, 128);
}

// Issues the loads of one 128-row key (or value) tile into `dst` (K-major,
// 128-byte swizzle, d/64 atoms of 16 KB). Called by all 32 lanes of a warp;
// lane 0 has already posted the expected byte count on `bar`.
// Sparse: rows idx_row[t*128 + i] (padded with the row's last key past k).
// Dense: rows t*128 .. t*128+127.
template <int D>
__device__ __forceinline__ void load_kv_tile(uint8_t* dst, const CUtensorMap* rows_map, const CUtensorMap* tile_map,
                                             uint64_t* bar, const int32_t* idx_row, int k, int t, int prow0,
                                             int lane) {
  constexpr int kAtoms = D / 64;
  if (idx_row) {
    int r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = t * 128 + lane * 4 + i;
      r[i] = prow0 + __ldg(idx_row + (j < k ? j : k - 1));
    }
#pragma unroll
    for (int a = 0; a < kAtoms; ++a)
      tma_gather4(dst + a * 16384 + lane * 512, rows_map, bar, a * 64, r[0], r[1], r[2], r[3]);
  } else if (lane == 0) {
#pragma unroll
    for (int a = 0; a < kAtoms; ++a) tma_load_2d(dst + a * 16384, tile_map, bar, a * 64, prow0 + t * 128);
  }
}

}  // namespace dsv
