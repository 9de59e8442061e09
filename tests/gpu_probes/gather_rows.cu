// Row-gather probe (test infrastructure): random 256-byte rows (d = 128
// bf16) from an L2-resident tensor into shared memory, by cp.async issued
// from W warps or by TMA tile::gather4 (box 64 columns x 1 row, four rows
// per instruction) issued from I lanes. Every CTA moves `tiles` tiles of 128
// rows (32 KB) through a two-stage buffer; both methods write the same
// layout (two 64-column halves of 128 rows x 128 B), and each block copies
// its last tile out, so the methods' results can be compared byte for byte.
// Prints GB/s and B/clk/SM per method and exits non-zero on any difference
// or error. Every wait is bounded.
#include <cstdio>
#include <cstdlib>
#include <vector>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t par) {
  for (long long it = 0; it < (1ll << 26); ++it) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0,1,0,p;\n}"
                 : "=r"(ok) : "r"(sa(b)), "r"(par) : "memory");
    if (ok) return true;
  }
  return false;
}

__device__ void copy_out(const uint8_t* tile, uint8_t* out) {
  for (int i = threadIdx.x; i < 32768 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(out + (size_t)blockIdx.x * 32768)[i] = reinterpret_cast<const uint4*>(tile)[i];
}

__global__ void __launch_bounds__(256) k_cpasync(const uint16_t* K, const int* rows, int tiles, int W, int* err,
                                                 uint8_t* out) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* r = rows + (size_t)blockIdx.x * tiles * 128;
  if (warp < W) {
    for (int t = 0; t < tiles; ++t) {
      uint8_t* dst = smem + (t & 1) * 32768;
      // 64 warp instructions per tile (2 rows of 16 chunks each), dealt to W warps
      for (int i = warp; i < 64; i += W) {
        const int row = i * 2 + lane / 16, chunk = lane % 16;
        const uint16_t* src = K + (size_t)r[t * 128 + row] * 128 + chunk * 8;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                         sa(dst + (chunk >> 3) * 16384 + row * 128 + (chunk & 7) * 16)),
                     "l"(src)
                     : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  __syncthreads();
  copy_out(smem + ((tiles - 1) & 1) * 32768, out);
}

__global__ void __launch_bounds__(256) k_gather4(const __grid_constant__ CUtensorMap map, const int* rows, int tiles,
                                                 int I, int* err, uint8_t* out) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t full[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* r = rows + (size_t)blockIdx.x * tiles * 128;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(full + s)), "r"(I));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // issuing lanes: lane 0 of warps 0..I-1; each takes 1/I of the tile's 64 gather4 instructions
  if (lane == 0 && warp < I) {
    for (int t = 0; t < tiles; ++t) {
      const int s = t & 1;
      if (t >= 2 && !bar_wait(full + s, ((t >> 1) - 1) & 1)) { atomicAdd(err, 1); break; }
      uint8_t* dst = smem + s * 32768;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(full + s)), "r"(32768 / I)
                   : "memory");
      for (int i = warp; i < 64; i += I) {
        const int a = i & 1, r4 = (i >> 1) * 4;   // atom (64 columns) and first of four rows
        const int* rr = r + t * 128 + r4;
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
            "%3, %4, %5, %6}], [%7];" ::"r"(sa(dst + a * 16384 + r4 * 128)),
            "l"((uint64_t)&map), "r"(a * 64), "r"(rr[0]), "r"(rr[1]), "r"(rr[2]), "r"(rr[3]), "r"(sa(full + s))
            : "memory");
      }
    }
    // drain: the last two stages' copies land before the block exits
    for (int t = tiles - 2; t < tiles; ++t)
      if (t >= 0 && !bar_wait(full + (t & 1), (t >> 1) & 1)) atomicAdd(err, 1);
  }
  __syncthreads();
  copy_out(smem + ((tiles - 1) & 1) * 32768, out);
}

int main() {
  const int nrows = 131072;   // 32 MB of K rows (d = 128 bf16): L2-resident
  const int blocks = 152 * 2, tiles = 96;
  uint16_t* K;
  int *rows, *err;
  cudaMalloc(&K, (size_t)nrows * 256);
  {
    std::vector<uint16_t> hk((size_t)nrows * 128);
    for (size_t i = 0; i < hk.size(); ++i) hk[i] = (uint16_t)(i * 2654435761u >> 16);
    cudaMemcpy(K, hk.data(), hk.size() * 2, cudaMemcpyHostToDevice);
  }
  uint8_t *out_ref, *out;
  cudaMalloc(&out_ref, (size_t)blocks * 32768);
  cudaMalloc(&out, (size_t)blocks * 32768);
  std::vector<int> h((size_t)blocks * tiles * 128);
  srand(1);
  for (auto& x : h) x = rand() % nrows;
  cudaMalloc(&rows, h.size() * 4);
  cudaMemcpy(rows, h.data(), h.size() * 4, cudaMemcpyHostToDevice);
  cudaMalloc(&err, 4);
  cudaMemset(err, 0, 4);
  cudaFuncSetAttribute(k_cpasync, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536 + 1024);
  cudaFuncSetAttribute(k_gather4, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536 + 1024);
  cudaDeviceProp pr;
  cudaGetDeviceProperties(&pr, 0);
  int clk_khz = 0;
  cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, 0);
  const double bytes = (double)blocks * tiles * 128 * 256;
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  auto report = [&](const char* name, float ms) {
    const double gbs = bytes / (ms * 1e-3) / 1e9;
    printf("%-28s %8.3f ms  %8.1f GB/s  %6.1f B/clk/SM (at %d MHz, %d SMs)\n", name, ms, gbs,
           gbs * 1e9 / (pr.multiProcessorCount * (double)clk_khz * 1e3), clk_khz / 1000, pr.multiProcessorCount);
  };
  for (int W : {7, 4, 2}) {
    float ms = 1e30f;
    for (int rep = 0; rep < 5; ++rep) {
      cudaEventRecord(a);
      k_cpasync<<<blocks, 256, 65536 + 1024>>>(K, rows, tiles, W, err, out_ref);
      cudaEventRecord(b);
      cudaEventSynchronize(b);
      float m;
      cudaEventElapsedTime(&m, a, b);
      if (rep) ms = m < ms ? m : ms;
    }
    char name[64];
    snprintf(name, sizeof name, "cp.async, %d warps", W);
    report(name, ms);
  }
  // tensor map: [nrows][128] bf16, box 64 x 1, no swizzle (layout is not checked here)
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&enc, 12000, cudaEnableDefault, &q);
  CUtensorMap map;
  cuuint64_t dims[2] = {128, (cuuint64_t)nrows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t es[2] = {1, 1};
  if (!enc || enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    printf("tensor map failed\n");
    return 1;
  }
  for (int I : {1, 4}) {
    float ms = 1e30f;
    for (int rep = 0; rep < 5; ++rep) {
      cudaEventRecord(a);
      k_gather4<<<blocks, 256, 65536 + 1024>>>(map, rows, tiles, I, err, out);
      cudaEventRecord(b);
      cudaEventSynchronize(b);
      float m;
      cudaEventElapsedTime(&m, a, b);
      if (rep) ms = m < ms ? m : ms;
    }
    char name[64];
    snprintf(name, sizeof name, "TMA gather4, %d issuing lane%s", I, I > 1 ? "s" : "");
    report(name, ms);
    std::vector<uint8_t> a_h((size_t)blocks * 32768), b_h((size_t)blocks * 32768);
    cudaMemcpy(a_h.data(), out_ref, a_h.size(), cudaMemcpyDeviceToHost);
    cudaMemcpy(b_h.data(), out, b_h.size(), cudaMemcpyDeviceToHost);
    if (a_h != b_h) {
      printf("gather4 (%d lanes) and cp.async tiles differ\n", I);
      return 2;
    }
  }
  int herr = 0;
  cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  cudaError_t e = cudaGetLastError();
  printf("errors %d, cuda %s\n", herr, cudaGetErrorString(e));
  return (herr || e != cudaSuccess) ? 1 : 0;
}
