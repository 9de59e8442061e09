// Host-side pieces shared by every libdsv entry point: status strings,
// validation, the tensor-map encoder and the head dispatcher.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace dsv {

dsv_status validate_common(const dsv_shape& s, const dsv_group& g, bool need_d_supported) {
  if (s.B < 1 || s.H < 1 || s.T < 1 || s.Y < 1 || s.X < 1) return DSV_ERR_INVALID_ARG;
  if (g.gt < 1 || g.gy < 1 || g.gx < 1) return DSV_ERR_INVALID_ARG;
  if (s.T % g.gt || s.Y % g.gy || s.X % g.gx) return DSV_ERR_INVALID_ARG;
  const int64_t S = s.T * s.Y * s.X;
  if (S >= (int64_t(1) << 31) || s.T > (1 << 20) || s.Y > (1 << 20) || s.X > (1 << 20)) return DSV_ERR_UNSUPPORTED;
  if (S % 128) return DSV_ERR_UNSUPPORTED;
  if (s.B * s.H > kMaxProblems) return DSV_ERR_UNSUPPORTED;
  const int64_t G = int64_t(g.gt) * g.gy * g.gx;
  if (G != 64 && G != 128) return DSV_ERR_UNSUPPORTED;
  if (need_d_supported && s.d != 64 && s.d != 128) return DSV_ERR_UNSUPPORTED;
  return DSV_OK;
}

static std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t cols,
                 uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  memset(m, 0, sizeof(*m));
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dsv

using namespace dsv;

extern "C" const char* dsv_status_string(dsv_status s) {
  switch (s) {
    case DSV_OK: return "DSV_OK";
    case DSV_ERR_INVALID_ARG: return "DSV_ERR_INVALID_ARG: bad pointer, size, alignment or shape";
    case DSV_ERR_UNSUPPORTED: return "DSV_ERR_UNSUPPORTED: request outside the supported sizes";
    case DSV_ERR_WORKSPACE: return "DSV_ERR_WORKSPACE: workspace missing or too small";
    case DSV_ERR_CUDA: return "DSV_ERR_CUDA: a CUDA launch or API call failed";
    case DSV_ERR_TIMEOUT: return "DSV_ERR_TIMEOUT: a bounded device wait ran out";
    case DSV_ERR_OVERFLOW: return "DSV_ERR_OVERFLOW: reserved";
    case DSV_ERR_CANDIDATES: return "DSV_ERR_CANDIDATES: a top-k row failed its consistency check";
  }
  return "DSV_ERR_UNKNOWN";
}

extern "C" uint64_t dsv_set_wait_limit_ns(uint64_t ns) { return g_wait_limit_ns.exchange(ns); }

extern "C" dsv_status dsv_read_status(const int32_t* dev_status, int32_t* host_out, void* stream) {
  if (!dev_status || !host_out) return DSV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_out, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return DSV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DSV_ERR_CUDA;
  return DSV_OK;
}

static int64_t round_half_up(double x) { return static_cast<int64_t>(std::floor(x + 0.5)); }

extern "C" dsv_status dsv_plan_heads(const int32_t* k_cov, int32_t n, int64_t S, int64_t n_groups, double lo_frac,
                                     double hi_frac, double dense_frac, int32_t* k_h, uint8_t* dense,
                                     int64_t* idx_offset, int64_t* idx_total) {
  if (!k_cov || !k_h || !dense || !idx_offset || !idx_total || n < 0 || S < 1 || n_groups < 1)
    return DSV_ERR_INVALID_ARG;
  if (!(lo_frac >= 0.0) || !(hi_frac >= lo_frac) || !(dense_frac >= 0.0)) return DSV_ERR_INVALID_ARG;
  const int64_t lo = std::max<int64_t>(1, round_half_up(lo_frac * (double)S));
  const int64_t hi = std::min<int64_t>(S, round_half_up(hi_frac * (double)S));
  int64_t total = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (k_cov[i] < 1 || k_cov[i] > S) return DSV_ERR_INVALID_ARG;
    if ((double)k_cov[i] > dense_frac * (double)S) {
      dense[i] = 1;
      k_h[i] = static_cast<int32_t>(S);
      idx_offset[i] = -1;
    } else {
      dense[i] = 0;
      const int64_t k = std::min(std::max<int64_t>(k_cov[i], lo), hi);
      k_h[i] = static_cast<int32_t>(k);
      idx_offset[i] = total;
      total += n_groups * k;
    }
  }
  *idx_total = total;
  return DSV_OK;
}

// Head-wise context-parallel re-balancing: longest processing time first.
extern "C" dsv_status dsv_plan_gpus(const int64_t* cost, int32_t n, int32_t n_gpus, int32_t equal_counts,
                                    int32_t* gpu_of, int64_t* load) {
  if (!cost || !gpu_of || n < 1 || n_gpus < 1) return DSV_ERR_INVALID_ARG;
  for (int32_t p = 0; p < n; ++p)
    if (cost[p] < 0) return DSV_ERR_INVALID_ARG;
  const int32_t cap = equal_counts ? (n + n_gpus - 1) / n_gpus : n;
  std::vector<int32_t> order(n);
  for (int32_t p = 0; p < n; ++p) order[p] = p;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return cost[a] > cost[b]; });
  std::vector<int64_t> ld(n_gpus, 0);
  std::vector<int32_t> cnt(n_gpus, 0);
  for (const int32_t p : order) {
    int32_t best = -1;
    for (int32_t g = 0; g < n_gpus; ++g)
      if (cnt[g] < cap && (best < 0 || ld[g] < ld[best])) best = g;
    gpu_of[p] = best;
    ld[best] += cost[p];
    ++cnt[best];
  }
  if (load)
    for (int32_t g = 0; g < n_gpus; ++g) load[g] = ld[g];
  return DSV_OK;
}
