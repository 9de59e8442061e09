// Rate of one tcgen05.mma kind::f16 instruction, M = 128, N = 128 or 256,
// K = 16 (bf16 operands, fp32 accumulation in TMEM), with both operands in
// shared memory (ss) or A in TMEM (ts): one thread issues 8160 accumulations
// and times them with clock64, on one CTA and on one CTA per SM. The
// accumulations go into one TMEM accumulator (a dependent chain) or, at
// N = 128, round-robin into two or three independent accumulators (columns
// 0, 128, 256), which shows whether the N = 128 rate is set by the chain's
// dependency or by the instruction's throughput. The operands are zero, so
// the accumulator must read back as zero (checked on the first 32 lanes x 32
// columns).
#include <cstdio>
#include <cstdlib>
#include <cuda_runtime.h>

#include "../../dynamic_sparse_attention_dsv_gb300/csrc/ptx.cuh"
using namespace dsv;

constexpr uint32_t kColA = 384;   // the ts form's A operand: zero bf16 pairs in columns 384..415

// kChains is a template argument so that the issuing loop stays a few
// instructions per MMA: a runtime modulo in it costs more than the MMA itself
template <int kChains>
__global__ void __launch_bounds__(128, 1) k_rate(int variant, int iters, long long* out, int* bad) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = sm;           // 128 rows x 128 B, 128-byte swizzle
  uint8_t* sB = sm + 16384;   // 256 rows x 128 B
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 49152);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  for (int i = threadIdx.x; i < 49152 / 16; i += blockDim.x) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x < 32) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  if (threadIdx.x < 32) {
    uint32_t z[32];
    for (int i = 0; i < 32; ++i) z[i] = 0u;
    tmem_st32(tbase + kColA, z);
    tmem_st_wait();
  }
  if (threadIdx.x >= 32 && threadIdx.x < 128) {
    uint32_t z[32];
    for (int i = 0; i < 32; ++i) z[i] = 0u;
    tmem_st32(tbase + ((uint32_t)((threadIdx.x >> 5) * 32) << 16) + kColA, z);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  bool ok = true;
  if (threadIdx.x == 0) {
    const bool n256 = variant & 1, ts = variant & 2;
    const uint32_t id = n256 ? instr_desc(128, 256, 1, 0, 0) : instr_desc(128, 128, 1, 0, 0);
    const uint64_t da = smem_desc(smem_u32(sA), 16, 1024), db = smem_desc(smem_u32(sB), 16, 1024);
    const long long t0 = clock64();
    for (int i0 = 0; i0 < iters; i0 += 4 * kChains) {
#pragma unroll
      for (int j = 0; j < 4 * kChains; ++j) {
        const int i = i0 + j;
        const uint32_t off = ((j / kChains) & 3) * 32;   // the four K steps of one 64-element atom
        const uint32_t acc = tbase + 128u * (j % kChains);
        if (ts) mma_f16_ts(acc, tbase + kColA + ((j / kChains) & 3) * 8, desc_at(db, off), id, i >= kChains ? 1u : 0u);
        else mma_f16_ss(acc, desc_at(da, off), desc_at(db, off), id, i >= kChains ? 1u : 0u);
      }
    }
    mma_commit(bar);
    ok = mbar_wait(bar, 0, 2000000000ull);
    const long long t1 = clock64();
    out[blockIdx.x] = ok ? t1 - t0 : -1;
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (threadIdx.x < 32 && ok) {
    tc_fence_after();
    uint32_t v[32];
    tmem_ld32(tbase, v);
    tmem_ld_wait(v);
    for (int i = 0; i < 32; ++i)
      if (v[i] != 0u) atomicAdd(bad, 1);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tbase, 512);
}

int main() {
  const int iters = 8160, smem = 120 * 1024;
  if (cudaFuncSetAttribute(k_rate<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k_rate<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k_rate<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 2;
  int nsm = 0;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  long long* d;
  int* bad;
  cudaMalloc(&d, 1024 * sizeof(long long));
  cudaMalloc(&bad, sizeof(int));
  long long h[1024];
  const char* names[4] = {"ss N=128", "ss N=256", "ts N=128", "ts N=256"};
  // (variant, accumulators): N = 256 fills 256 columns, so it runs one chain
  const int runs[][2] = {{0, 1}, {1, 1}, {2, 1}, {3, 1}, {0, 2}, {0, 3}, {2, 2}, {2, 3}};
  int fails = 0;
  for (int grid : {1, nsm}) {
    for (const auto& r : runs) {
      const int v = r[0], chains = r[1];
      cudaMemset(bad, 0, sizeof(int));
      for (int rep = 0; rep < 2; ++rep) {   // warm-up, then the timed launch
        if (chains == 1) k_rate<1><<<grid, 128, smem>>>(v, iters, d, bad);
        else if (chains == 2) k_rate<2><<<grid, 128, smem>>>(v, iters, d, bad);
        else k_rate<3><<<grid, 128, smem>>>(v, iters, d, bad);
      }
      const cudaError_t e = cudaDeviceSynchronize();
      int hb = 0;
      cudaMemcpy(h, d, grid * sizeof(long long), cudaMemcpyDeviceToHost);
      cudaMemcpy(&hb, bad, sizeof(int), cudaMemcpyDeviceToHost);
      double s = 0;
      bool timeout = false;
      for (int i = 0; i < grid; ++i) {
        s += (double)h[i];
        timeout = timeout || h[i] < 0;
      }
      const int N = (v & 1) ? 256 : 128;
      const double cyc = s / grid / iters;
      printf("grid %3d %s x%d: %.1f cycles per MMA, %.0f MAC/clk per SM, nonzero accumulators %d, %s\n", grid,
             names[v], chains, cyc, 128.0 * N * 16 / cyc, hb, cudaGetErrorString(e));
      fails += (e != cudaSuccess) || timeout || hb != 0;
    }
  }
  return fails ? 1 : 0;
}
