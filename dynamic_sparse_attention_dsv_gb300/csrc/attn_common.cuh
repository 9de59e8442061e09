// Pieces shared by the sparse attention forward and backward kernels: tensor
// maps over Q/K/V, the per-launch parameter block and tile addressing.
#pragma once
#include "common.cuh"

namespace dsv {

// Tensor maps used by one attention launch (all over bf16 [P*S][d] tensors).
struct AttnMaps {
  CUtensorMap q_cube;   // 4D [P*T][Y][X][d], box (64, gx, gy, gt): one query group
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
  uint64_t wait_ns;          // limit of each pipeline wait
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
         make_map_2d(&m->k_tile, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, rows, 64, 128) &&
         make_map_2d(&m->v_tile, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, rows, 64, 128);
}

// ---------------------------------------------------------------------------
// Row gather of selected K/V rows with cp.async by W producer warps. A warp
// instruction copies whole rows (d*2 bytes = d/8 16-byte chunks, consecutive
// lanes on consecutive chunks) into the K-major 128-byte swizzled tile layout
// the tensor cores read. The tile's instructions are dealt round-robin to the
// W warps (instruction pw + i*W for warp pw), so W need not divide the tile.
// The rate at which an SM issues these copies grows with the number of
// issuing warps (up to ~33 B/clk per SM on random 256-byte rows from L2), so a
// kernel that is bound by its gathers uses more of them.
constexpr int kGatherWarps = 2;

template <int D, int W = kGatherWarps>
struct Gather {
  static constexpr int kChunksPerRow = D / 8;                      // 16-byte chunks per row
  static constexpr int kRowsPerInstr = 32 / kChunksPerRow;         // rows per warp instruction
  static constexpr int kInstr = 128 / kRowsPerInstr;               // warp instructions per tile and tensor
  static constexpr int kIters = (kInstr + W - 1) / W;              // instructions per lane per tensor
  __device__ static bool valid(int pw, int i) { return kInstr % W == 0 || pw + i * W < kInstr; }
  __device__ static int row(int pw, int i, int lane) { return (pw + i * W) * kRowsPerInstr + lane / kChunksPerRow; }
};

// Key rows (absolute row in the [P*S][d] tensor) this lane copies for tile t.
// Slots past k repeat the row's last key, so every copied row is a real key.
template <int D, int W = kGatherWarps>
__device__ __forceinline__ void gather_rows(int (&rows)[Gather<D, W>::kIters], const int32_t* idx_row, int k, int t,
                                            int prow0, int pw, int lane) {
  using Gt = Gather<D, W>;
#pragma unroll
  for (int i = 0; i < Gt::kIters; ++i) {
    if (!Gt::valid(pw, i)) break;
    const int slot = t * 128 + Gt::row(pw, i, lane);
    rows[i] = prow0 + __ldg(idx_row + (slot < k ? slot : k - 1));
  }
}

template <int D, int W = kGatherWarps>
__device__ __forceinline__ void gather_tile(uint8_t* dst, const __nv_bfloat16* src,
                                            const int (&rows)[Gather<D, W>::kIters], int pw, int lane) {
  using Gt = Gather<D, W>;
  const int chunk = lane % Gt::kChunksPerRow;
  const uint32_t base = smem_u32(dst) + (chunk >> 3) * 16384;
#pragma unroll
  for (int i = 0; i < Gt::kIters; ++i) {
    if (!Gt::valid(pw, i)) break;
    const int row = Gt::row(pw, i, lane);
    cp_async_16(base + row * 128 + (((chunk & 7) ^ (row & 7)) << 4), src + (int64_t)rows[i] * D + chunk * 8);
  }
}

// Dense tiles (rows t*128 .. t*128+127 of the problem) by one TMA box per
// 64-column atom, issued by one thread that has posted the byte count.
template <int D>
__device__ __forceinline__ void load_dense_tile(uint8_t* dst, const CUtensorMap* tile_map, uint64_t* bar, int t,
                                                int prow0) {
#pragma unroll
  for (int a = 0; a < D / 64; ++a) tma_load_2d(dst + a * 16384, tile_map, bar, a * 64, prow0 + t * 128);
}

}  // namespace dsv
