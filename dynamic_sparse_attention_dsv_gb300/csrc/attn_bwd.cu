// Query-grouped sparse attention, backward pass.
//
// "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT
// Training" (gist.science technical summary, section 2.1): stage 2 trains
// with attention restricted to the critical KV pairs, so gradients flow
// through the selected (query, key) pairs only; the index sets are constants
// of the step. Recomputation from the saved LSE follows the usual
// memory-efficient attention practice.
//
// Group-major kernel (every problem): one CTA per (query group, problem),
// looping over the group's 128-key tiles:
//   S = Q K^T, dP = dO V^T                        tcgen05 (smem x smem) -> TMEM
//   P = exp2(S*scale*log2e - LSE*log2e), dS = P (dP - Delta)   registers
//   dQ += dS K                                    accumulated in TMEM, written once
//   sparse problems only: dV_tile = P^T dO, dK_tile = dS^T Q -> TMEM, then
//   converted to int64 fixed point (2^-32 units) and added into per-key
//   accumulators. Integer addition is associative, so dK/dV do not depend on
//   the order in which groups arrive.
// Key-major kernel (dense problems): one CTA per (128-key tile, problem),
// looping over all 128-token query tiles with dV, dK accumulated in TMEM;
// no cross-CTA reduction at all.
#include <algorithm>
#include <vector>

#include "attn_common.cuh"

namespace dsv {

constexpr int kBwdThreads = 192;
constexpr int kBwdChunkProblems = 4;   // sparse problems per accumulator chunk

template <int D>
struct BwdCfg {
  static constexpr int kTile = 128 * D * 2;      // one [128][D] bf16 tile
  static constexpr int kStages = D == 128 ? 1 : 2;
  static constexpr int kOffDO = kTile;           // Q at 0
  static constexpr int kOffK = 2 * kTile;
  static constexpr int kOffV = kOffK + kStages * kTile;
  static constexpr int kOffP = kOffV + kStages * kTile;   // [128 q][128 keys] bf16 = 32 KB
  static constexpr int kOffDS = kOffP + 32768;
  static constexpr int kOffBar = kOffDS + 32768;   // barriers at +0, key slots at +128
  static constexpr int kSmemUsed = kOffBar + 1024 + 1024;
  static constexpr int kSmem = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
};

// round(v * 2^32) as int64 for |v| < 2^30, from the float's bits (no FP64).
__device__ __forceinline__ int64_t f2fix(float v) {
  const uint32_t b = __float_as_uint(v);
  const int e = (int)((b >> 23) & 0xFF) - 127;
  if (e < -33) return 0;
  const uint64_t m = (b & 0x7FFFFFu) | 0x800000u;   // v = m * 2^(e-23)
  const int sh = e + 9;                              // v * 2^32 = m * 2^(e+9)
  const uint64_t mag = sh >= 0 ? (m << sh) : ((m + (1ull << (-sh - 1))) >> (-sh));
  return (b >> 31) ? -(int64_t)mag : (int64_t)mag;
}

__device__ __forceinline__ void red_global_u64(int64_t* addr, int64_t v) {
  asm volatile("red.global.add.u64 [%0], %1;" ::"l"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ void compute_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Writes 8 bf16 values (packed in 4 words) at 16-byte chunk `chunk` (0..15)
// of row `row` of a [128][128] bf16 K-major tile with the 128-byte swizzle.
__device__ __forceinline__ void st_sw128_chunk(uint8_t* tile, int row, int chunk, uint4 v) {
  const int atom = chunk >> 3, c = chunk & 7;
  *reinterpret_cast<uint4*>(tile + atom * 16384 + row * 128 + ((c ^ (row & 7)) << 4)) = v;
}

// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_attn_bwd_q(const __grid_constant__ AttnMaps maps, const __grid_constant__ CUtensorMap do_cube,
                 const AttnParams prm, const ProblemTable tab) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;
  uint8_t* sDO = sm + C::kOffDO;
  uint8_t* sK = sm + C::kOffK;
  uint8_t* sV = sm + C::kOffV;
  uint8_t* sP = sm + C::kOffP;
  uint8_t* sDS = sm + C::kOffDS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;       // [2]
  uint64_t* v_full = bars + 3;       // [2]
  uint64_t* kv_empty = bars + 5;     // [2]
  uint64_t* sdp_full = bars + 7;
  uint64_t* ps_full = bars + 8;
  uint64_t* part_full = bars + 9;
  uint64_t* part_empty = bars + 10;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 12);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, lp = blockIdx.y, p = tab.p[lp];
  const Geometry& geo = prm.geo;
  const bool dense = (prm.idx == nullptr) || (tab.off[lp] < 0);
  const bool partials = !dense && prm.dK_acc != nullptr;
  const int k = dense ? geo.S : tab.k[lp];
  const int nt = (k + 127) / 128;
  const int32_t* idx_row = dense ? nullptr : prm.idx + tab.off[lp] + (int64_t)g * k;
  const int G = geo.G;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;

  if (G < 128) {
    for (int i = tid; i < (128 - G) * (D / 64) * 8; i += blockDim.x) {
      const int a = i / ((128 - G) * 8), rem = i % ((128 - G) * 8);
      reinterpret_cast<uint4*>(sQ + a * 16384 + G * 128)[rem] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(sDO + a * 16384 + G * 128)[rem] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 5) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(v_full + i, 1);
      mbar_init(kv_empty + i, 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(ps_full, 4);
    mbar_init(part_full, 1);
    mbar_init(part_empty, 4);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA
    const int ct = g / (geo.ncy * geo.ncx), cy = (g / geo.ncx) % geo.ncy, cx = g % geo.ncx;
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * G * D * 2);
      for (int a = 0; a < D / 64; ++a) {
        tma_load_4d(sQ + a * 16384, &maps.q_cube, q_full, a * 64, cx * geo.gx, cy * geo.gy, p * geo.T + ct * geo.gt);
        tma_load_4d(sDO + a * 16384, &do_cube, q_full, a * 64, cx * geo.gx, cy * geo.gy, p * geo.T + ct * geo.gt);
      }
    }
    const int prow0 = p * geo.S;
    for (int t = 0; t < nt; ++t) {
      const int s = t % C::kStages;
      if (t >= C::kStages && !mbar_wait_warp(kv_empty + s, ((t / C::kStages) - 1) & 1, kWaitLimitNs)) {
        if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(k_full + s, C::kTile);
      __syncwarp();
      load_kv_tile<D>(sK + s * C::kTile, &maps.k_rows, &maps.k_tile, k_full + s, idx_row, k, t, prow0, lane);
      if (lane == 0) mbar_arrive_expect_tx(v_full + s, C::kTile);
      __syncwarp();
      load_kv_tile<D>(sV + s * C::kTile, &maps.v_rows, &maps.v_tile, v_full + s, idx_row, k, t, prow0, lane);
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id_sdp = instr_desc(128, 128, 1, 0, 0);   // Q K^T, dO V^T
      constexpr uint32_t id_dq = instr_desc(128, D, 1, 0, 1);      // dS K (B = K, MN-major)
      constexpr uint32_t id_kv = instr_desc(128, D, 1, 1, 1);      // P^T dO, dS^T Q (A, B MN-major)
      const uint32_t aq = smem_u32(sQ), ado = smem_u32(sDO), ap = smem_u32(sP), ads = smem_u32(sDS);
      bool ok = mbar_wait(q_full, 0, kWaitLimitNs);
      for (int t = 0; ok && t < nt; ++t) {
        const int s = t % C::kStages;
        if (!mbar_wait(k_full + s, (t / C::kStages) & 1, kWaitLimitNs) ||
            !mbar_wait(v_full + s, (t / C::kStages) & 1, kWaitLimitNs) ||
            (t >= 1 && !mbar_wait(part_empty, (t - 1) & 1, kWaitLimitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ak = smem_u32(sK + s * C::kTile), av = smem_u32(sV + s * C::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ss(tbase + kColS, smem_desc(aq + off, 16, 1024), smem_desc(ak + off, 16, 1024), id_sdp, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ss(tbase + kColDP, smem_desc(ado + off, 16, 1024), smem_desc(av + off, 16, 1024), id_sdp,
                     kk > 0);
        }
        mma_commit(sdp_full);
        if (!mbar_wait(ps_full, t & 1, kWaitLimitNs)) { ok = false; break; }
        tc_fence_after();
        // dQ += dS K   (K over the 128 keys of the tile)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offa = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ss(tbase + kColDQ, smem_desc(ads + offa, 16, 1024), smem_desc(ak + kk * 2048, 16384, 1024), id_dq,
                     (t > 0 || kk > 0) ? 1u : 0u);
        }
        if (partials) {
          // dV_tile = P^T dO, dK_tile = dS^T Q   (K over the 128 queries)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            mma_f16_ss(tbase + kColS, smem_desc(ap + kk * 2048, 16384, 1024), smem_desc(ado + kk * 2048, 16384, 1024),
                       id_kv, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            mma_f16_ss(tbase + kColDP, smem_desc(ads + kk * 2048, 16384, 1024), smem_desc(aq + kk * 2048, 16384, 1024),
                       id_kv, kk > 0);
          }
        }
        mma_commit(kv_empty + s);
        mma_commit(part_full);
      }
      if (!ok) raise_status(prm.status, DSV_ERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------ compute (warps 0-3)
    const int row = warp * 32 + lane;
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    const float sc = prm.scale_log2;
    float lse2 = INFINITY, delta = 0.f;
    int tok = 0;
    if (row < G) {
      tok = token_of(geo, g, row);
      const int64_t o = ((int64_t)p * geo.S + tok) * D;
      const uint4* orow = reinterpret_cast<const uint4*>(prm.O + o);
      const uint4* drow = reinterpret_cast<const uint4*>(prm.dO + o);
      float acc = 0.f;
      for (int c = 0; c < D / 8; ++c) {
        const uint4 a = orow[c], b = drow[c];
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(b2[e]);
          acc = fmaf(x.x, y.x, acc);
          acc = fmaf(x.y, y.y, acc);
        }
      }
      delta = acc;
      lse2 = prm.LSE[(int64_t)p * geo.S + tok] * 1.4426950408889634f;
    }
    // A wait that runs out clears `ok`; later waits are skipped but every
    // warp still passes every named barrier, so the CTA always terminates.
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
      ok = ok && mbar_wait_warp(sdp_full, t & 1, kWaitLimitNs);
      tc_fence_after();
      const int nvalid = min(128, k - t * 128);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t sr[32], dr[32];
        tmem_ld32(lane_addr + kColS + c * 32, sr);
        tmem_ld32(lane_addr + kColDP + c * 32, dr);
        tmem_ld_wait(sr);
        reg_fence(dr);
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int j = c * 32 + e;
          const float p0 = j < nvalid ? ex2_fast(__uint_as_float(sr[e]) * sc - lse2) : 0.f;
          const float p1 = j + 1 < nvalid ? ex2_fast(__uint_as_float(sr[e + 1]) * sc - lse2) : 0.f;
          const float d0 = p0 * (__uint_as_float(dr[e]) - delta);
          const float d1 = p1 * (__uint_as_float(dr[e + 1]) - delta);
          pw[e >> 1] = pack_bf16x2(p0, p1);
          dw[e >> 1] = pack_bf16x2(d0, d1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          st_sw128_chunk(sP, row, c * 4 + q, make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]));
          st_sw128_chunk(sDS, row, c * 4 + q, make_uint4(dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ps_full);
      ok = ok && mbar_wait_warp(part_full, t & 1, kWaitLimitNs);
      tc_fence_after();
      if (partials) {
        // Drain dV_tile (cols 0..D) and dK_tile (cols 128..128+D): TMEM lane =
        // key slot. Rows are staged as int64 in the P/dS area (64 rows per
        // round), then added with consecutive threads on consecutive columns.
        int64_t* stage = reinterpret_cast<int64_t*>(sP);
        const int slot_key = t * 128 + row;
        const int krow = slot_key < k ? __ldg(idx_row + slot_key) : -1;
        int* keys = reinterpret_cast<int*>(sm + C::kOffBar + 128);   // [128] key of each slot
        keys[row] = krow;
        for (int tensor = 0; tensor < 2; ++tensor) {
          const uint32_t col = tensor == 0 ? kColS : kColDP;
          const float mul = tensor == 0 ? 1.f : prm.scale;
          int64_t* acc = tensor == 0 ? prm.dV_acc : prm.dK_acc;
          for (int half = 0; half < 2; ++half) {
            compute_barrier();   // staging area free; keys[] visible
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              tmem_ld32(lane_addr + col + c * 32, v);
              tmem_ld_wait(v);
              if ((row >> 6) == half) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  const float x = __uint_as_float(v[e]) * mul;
                  int64_t fx = 0;
                  if (fabsf(x) < prm.overflow_limit) fx = f2fix(x);
                  else raise_status(prm.status, DSV_ERR_OVERFLOW);
                  stage[(row & 63) * D + c * 32 + e] = fx;
                }
              }
            }
            compute_barrier();
            for (int i = tid; i < 64 * D; i += 128) {
              const int r = i / D, cc = i % D;
              const int kr = keys[half * 64 + r];
              const int64_t val = stage[i];
              if (kr >= 0 && val != 0) red_global_u64(acc + ((int64_t)lp * geo.S + kr) * D + cc, val);
            }
          }
        }
        compute_barrier();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(part_empty);
    }
    // ----------------------------------------------------------- dQ out
    if (!ok) {
      if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
    } else {
      tc_fence_after();
      __nv_bfloat16* qrow = prm.out + ((int64_t)p * geo.S + tok) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + kColDQ + c * 32, o);
        tmem_ld_wait(o);
        if (row < G) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * prm.scale, __uint_as_float(o[2 * e + 1]) * prm.scale);
          uint4* dst = reinterpret_cast<uint4*>(qrow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------
// Key-major dK/dV for dense problems. grid = (S/128, problems).
template <int D>
struct KvCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kOffV = kTile;            // K at 0
  static constexpr int kOffQ = 2 * kTile;
  static constexpr int kOffDO = 3 * kTile;
  static constexpr int kOffP = 4 * kTile;        // P^T [128 keys][128 q] bf16
  static constexpr int kOffDS = kOffP + 32768;
  static constexpr int kOffStat = kOffDS + 32768;   // LSE2[128], Delta[128]
  static constexpr int kOffBar = kOffStat + 1024;
  static constexpr int kSmemUsed = kOffBar + 1024 + 1024;
  static constexpr int kSmem = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
};

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_attn_bwd_kv(const __grid_constant__ AttnMaps maps, const __grid_constant__ CUtensorMap q_tile,
                  const __grid_constant__ CUtensorMap do_tile, const AttnParams prm, const float* delta_all,
                  __nv_bfloat16* dK, __nv_bfloat16* dV, const ProblemTable tab) {
  using C = KvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sm;
  uint8_t* sV = sm + C::kOffV;
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sDO = sm + C::kOffDO;
  uint8_t* sP = sm + C::kOffP;
  uint8_t* sDS = sm + C::kOffDS;
  float* sLse = reinterpret_cast<float*>(sm + C::kOffStat);
  float* sDelta = sLse + 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = bars + 2;
  uint64_t* sdp_full = bars + 3;
  uint64_t* ps_full = bars + 4;
  uint64_t* mma_done = bars + 5;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kt = blockIdx.x, lp = blockIdx.y, p = tab.p[lp];
  const Geometry& geo = prm.geo;
  const int nq = geo.S / 128;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;

  if (warp == 5) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(kv_full, 1);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(sdp_full, 1);
    mbar_init(ps_full, 4);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const int prow0 = p * geo.S;

  if (warp == 4) {
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::kTile);
      for (int a = 0; a < D / 64; ++a) {
        tma_load_2d(sK + a * 16384, &maps.k_tile, kv_full, a * 64, prow0 + kt * 128);
        tma_load_2d(sV + a * 16384, &maps.v_tile, kv_full, a * 64, prow0 + kt * 128);
      }
      for (int u = 0; u < nq; ++u) {
        if (u >= 1 && !mbar_wait(q_empty, (u - 1) & 1, kWaitLimitNs)) {
          raise_status(prm.status, DSV_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * C::kTile);
        for (int a = 0; a < D / 64; ++a) {
          tma_load_2d(sQ + a * 16384, &q_tile, q_full, a * 64, prow0 + u * 128);
          tma_load_2d(sDO + a * 16384, &do_tile, q_full, a * 64, prow0 + u * 128);
        }
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t id_sdp = instr_desc(128, 128, 1, 0, 0);   // K Q^T, V dO^T
      constexpr uint32_t id_acc = instr_desc(128, D, 1, 0, 1);     // P^T dO, dS^T Q (B MN-major)
      const uint32_t ak = smem_u32(sK), av = smem_u32(sV), aq = smem_u32(sQ), ado = smem_u32(sDO);
      const uint32_t ap = smem_u32(sP), ads = smem_u32(sDS);
      bool ok = mbar_wait(kv_full, 0, kWaitLimitNs);
      for (int u = 0; ok && u < nq; ++u) {
        if (!mbar_wait(q_full, u & 1, kWaitLimitNs)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ss(tbase + kColS, smem_desc(ak + off, 16, 1024), smem_desc(aq + off, 16, 1024), id_sdp, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ss(tbase + kColDP, smem_desc(av + off, 16, 1024), smem_desc(ado + off, 16, 1024), id_sdp, kk > 0);
        }
        mma_commit(sdp_full);
        if (!mbar_wait(ps_full, u & 1, kWaitLimitNs)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offa = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ss(tbase + kColDV, smem_desc(ap + offa, 16, 1024), smem_desc(ado + kk * 2048, 16384, 1024), id_acc,
                     (u > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offa = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ss(tbase + kColDK, smem_desc(ads + offa, 16, 1024), smem_desc(aq + kk * 2048, 16384, 1024), id_acc,
                     (u > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(q_empty);
        mma_commit(mma_done);
      }
      if (!ok) raise_status(prm.status, DSV_ERR_TIMEOUT);
    }
  } else {
    const int row = warp * 32 + lane;   // key slot of the tile
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    const float sc = prm.scale_log2;
    // as in the group-major kernel: no early exit from a loop with named barriers
    bool ok = true;
    for (int u = 0; u < nq; ++u) {
      // P^T/dS^T smem and the S/dP TMEM columns are free once tile u-1's MMAs are done
      if (u >= 1) ok = ok && mbar_wait_warp(mma_done, (u - 1) & 1, kWaitLimitNs);
      sLse[row] = prm.LSE[(int64_t)prow0 + u * 128 + row] * 1.4426950408889634f;
      sDelta[row] = delta_all[(int64_t)prow0 + u * 128 + row];
      compute_barrier();
      ok = ok && mbar_wait_warp(sdp_full, u & 1, kWaitLimitNs);
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t sr[32], dr[32];
        tmem_ld32(lane_addr + kColS + c * 32, sr);
        tmem_ld32(lane_addr + kColDP + c * 32, dr);
        tmem_ld_wait(sr);
        reg_fence(dr);
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int q = c * 32 + e;
          const float p0 = ex2_fast(__uint_as_float(sr[e]) * sc - sLse[q]);
          const float p1 = ex2_fast(__uint_as_float(sr[e + 1]) * sc - sLse[q + 1]);
          const float d0 = p0 * (__uint_as_float(dr[e]) - sDelta[q]);
          const float d1 = p1 * (__uint_as_float(dr[e + 1]) - sDelta[q + 1]);
          pw[e >> 1] = pack_bf16x2(p0, p1);
          dw[e >> 1] = pack_bf16x2(d0, d1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          st_sw128_chunk(sP, row, c * 4 + q, make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]));
          st_sw128_chunk(sDS, row, c * 4 + q, make_uint4(dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      compute_barrier();   // sLse/sDelta reads done before the next tile overwrites them
      if (lane == 0) mbar_arrive(ps_full);
    }
    if (ok && !mbar_wait_warp(mma_done, (nq - 1) & 1, kWaitLimitNs)) ok = false;
    if (!ok) {
      if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
    } else {
      tc_fence_after();
      const int64_t o = ((int64_t)prow0 + kt * 128 + row) * D;
      for (int tensor = 0; tensor < 2; ++tensor) {
        const uint32_t col = tensor == 0 ? kColDV : kColDK;
        const float mul = tensor == 0 ? 1.f : prm.scale;
        __nv_bfloat16* dst_row = (tensor == 0 ? dV : dK) + o;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_addr + col + c * 32, v);
          tmem_ld_wait(v);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
          uint4* dst = reinterpret_cast<uint4*>(dst_row + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tbase, 512);
}

// Delta_i = sum_c dO_ic O_ic for every row of the listed problems.
__global__ void k_bwd_delta(const __nv_bfloat16* __restrict__ O, const __nv_bfloat16* __restrict__ dO, int S, int d,
                            float* __restrict__ delta, const ProblemTable tab) {
  const int lp = blockIdx.y, p = tab.p[lp];
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= S) return;
  const int64_t o = ((int64_t)p * S + s) * d;
  const uint4* a = reinterpret_cast<const uint4*>(O + o);
  const uint4* b = reinterpret_cast<const uint4*>(dO + o);
  float acc = 0.f;
  for (int c = 0; c < d / 8; ++c) {
    const uint4 x = a[c], y = b[c];
    const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&x);
    const __nv_bfloat162* y2 = reinterpret_cast<const __nv_bfloat162*>(&y);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 u = __bfloat1622float2(x2[e]), v = __bfloat1622float2(y2[e]);
      acc = fmaf(u.x, v.x, acc);
      acc = fmaf(u.y, v.y, acc);
    }
  }
  delta[(int64_t)p * S + s] = acc;
}

// Fixed-point accumulators (local problem lp) -> bf16 dK, dV of problem p.
__global__ void k_fix_to_bf16(const int64_t* __restrict__ acc_k, const int64_t* __restrict__ acc_v, int64_t per,
                              __nv_bfloat16* dK, __nv_bfloat16* dV, const ProblemTable tab) {
  const int lp = blockIdx.y, p = tab.p[lp];
  const int64_t base_l = (int64_t)lp * per, base_p = (int64_t)p * per;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < per; i += (int64_t)gridDim.x * blockDim.x) {
    dK[base_p + i] = __float2bfloat16_rn((float)acc_k[base_l + i] * 2.3283064365386963e-10f);
    dV[base_p + i] = __float2bfloat16_rn((float)acc_v[base_l + i] * 2.3283064365386963e-10f);
  }
}

template <int D>
static cudaError_t configure_bwd() {
  static bool done = false;
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_attn_bwd_q<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_attn_bwd_kv<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::kSmem);
  if (e == cudaSuccess) done = true;
  return e;
}

template <int D>
static cudaError_t launch_bwd_q(const AttnMaps& maps, const CUtensorMap& do_cube, const AttnParams& prm,
                                const ProblemTable& tab, int n_groups, cudaStream_t st) {
  k_attn_bwd_q<D><<<dim3(n_groups, tab.n), kBwdThreads, BwdCfg<D>::kSmem, st>>>(maps, do_cube, prm, tab);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_bwd_kv(const AttnMaps& maps, const CUtensorMap& q_tile, const CUtensorMap& do_tile,
                                 const AttnParams& prm, const float* delta, __nv_bfloat16* dK, __nv_bfloat16* dV,
                                 const ProblemTable& tab, int S, cudaStream_t st) {
  k_attn_bwd_kv<D><<<dim3(S / 128, tab.n), kBwdThreads, KvCfg<D>::kSmem, st>>>(maps, q_tile, do_tile, prm, delta,
                                                                                dK, dV, tab);
  return cudaGetLastError();
}

struct BwdWs {
  int64_t* acc_k;
  int64_t* acc_v;
  float* delta;
};

static size_t carve_bwd(void* base, const dsv_shape& s, BwdWs* w) {
  Carver c(base);
  const size_t S = (size_t)(s.T * s.Y * s.X), P = (size_t)(s.B * s.H);
  const size_t hc = std::min<size_t>(P, kBwdChunkProblems);
  w->acc_k = c.take<int64_t>(hc * S * s.d);
  w->acc_v = c.take<int64_t>(hc * S * s.d);
  w->delta = c.take<float>(P * S);
  return c.used + 256;
}

}  // namespace dsv

using namespace dsv;

extern "C" size_t dsv_sparse_attn_bwd_workspace_size(dsv_shape shape, dsv_group group) {
  if (validate_common(shape, group, true) != DSV_OK) return 0;
  BwdWs w;
  return carve_bwd(nullptr, shape, &w);
}

extern "C" dsv_status dsv_sparse_attn_bwd(const void* Q, const void* K, const void* V, const void* O,
                                          const float* LSE, const void* dO, const int32_t* idx,
                                          const int32_t* k_per_head, const int64_t* idx_offset, dsv_shape shape,
                                          dsv_group group, float scale, void* dQ, void* dK, void* dV,
                                          void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                          void* stream) {
  dsv_status v = validate_common(shape, group, true);
  if (v != DSV_OK) return v;
  if (!Q || !K || !V || !O || !LSE || !dO || !dQ || !dK || !dV || !(scale > 0.f)) return DSV_ERR_INVALID_ARG;
  for (const void* ptr : {Q, K, V, O, dO, (const void*)dQ, (const void*)dK, (const void*)dV})
    if (!aligned(ptr, 16)) return DSV_ERR_INVALID_ARG;
  if (idx && (!k_per_head || !idx_offset || !aligned(idx, 4))) return DSV_ERR_INVALID_ARG;
  BwdWs w;
  const size_t need = carve_bwd(nullptr, shape, &w);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DSV_ERR_WORKSPACE;
  carve_bwd(workspace, shape, &w);
  const Geometry geo = make_geometry(shape, group);
  const int P = (int)(shape.B * shape.H), d = (int)shape.d;
  std::vector<int> sparse, dense;
  for (int i = 0; i < P; ++i) {
    if (!idx || idx_offset[i] < 0) {
      dense.push_back(i);
    } else {
      if (k_per_head[i] < 1 || k_per_head[i] > geo.S) return DSV_ERR_INVALID_ARG;
      sparse.push_back(i);
    }
  }
  AttnMaps maps;
  CUtensorMap do_cube, q_tile, do_tile;
  if (!make_attn_maps(&maps, Q, K, V, geo, d, P) || !make_cube_map(&do_cube, dO, geo, d, P) ||
      !make_map_2d(&q_tile, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, (uint64_t)P * geo.S, 64, 128) ||
      !make_map_2d(&do_tile, dO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, (uint64_t)P * geo.S, 64, 128))
    return DSV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((d == 128 ? configure_bwd<128>() : configure_bwd<64>()) != cudaSuccess) return DSV_ERR_CUDA;

  AttnParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.geo = geo;
  prm.d = d;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.idx = idx;
  prm.O = static_cast<const __nv_bfloat16*>(O);
  prm.dO = static_cast<const __nv_bfloat16*>(dO);
  prm.LSE = LSE;
  prm.out = static_cast<__nv_bfloat16*>(dQ);
  prm.overflow_limit = 1073741824.0f / (float)geo.n_groups;
  prm.status = dev_status;
  auto* dKp = static_cast<__nv_bfloat16*>(dK);
  auto* dVp = static_cast<__nv_bfloat16*>(dV);
  const int64_t per = (int64_t)geo.S * d;

  // sparse problems: dQ + fixed-point dK/dV, in chunks of accumulators
  for (size_t c0 = 0; c0 < sparse.size(); c0 += kBwdChunkProblems) {
    ProblemTable tab;
    memset(&tab, 0, sizeof(tab));
    tab.n = (int)std::min<size_t>(kBwdChunkProblems, sparse.size() - c0);
    for (int i = 0; i < tab.n; ++i) {
      const int p = sparse[c0 + i];
      tab.p[i] = p;
      tab.k[i] = k_per_head[p];
      tab.off[i] = idx_offset[p];
    }
    const size_t bytes = (size_t)tab.n * per * sizeof(int64_t);
    if (cudaMemsetAsync(w.acc_k, 0, bytes, st) != cudaSuccess || cudaMemsetAsync(w.acc_v, 0, bytes, st) != cudaSuccess)
      return DSV_ERR_CUDA;
    AttnParams pc = prm;
    pc.dK_acc = w.acc_k;
    pc.dV_acc = w.acc_v;
    const cudaError_t e = d == 128 ? launch_bwd_q<128>(maps, do_cube, pc, tab, geo.n_groups, st)
                                   : launch_bwd_q<64>(maps, do_cube, pc, tab, geo.n_groups, st);
    if (e != cudaSuccess) return DSV_ERR_CUDA;
    k_fix_to_bf16<<<dim3(592, tab.n), 256, 0, st>>>(w.acc_k, w.acc_v, per, dKp, dVp, tab);
    if (cudaGetLastError() != cudaSuccess) return DSV_ERR_CUDA;
  }
  // dense problems: dQ group-major, dK/dV key-major
  if (!dense.empty()) {
    ProblemTable tab;
    memset(&tab, 0, sizeof(tab));
    tab.n = (int)dense.size();
    for (int i = 0; i < tab.n; ++i) {
      tab.p[i] = dense[i];
      tab.k[i] = geo.S;
      tab.off[i] = -1;
    }
    k_bwd_delta<<<dim3((geo.S + 255) / 256, tab.n), 256, 0, st>>>(prm.O, prm.dO, geo.S, d, w.delta, tab);
    if (cudaGetLastError() != cudaSuccess) return DSV_ERR_CUDA;
    AttnParams pd = prm;
    pd.dK_acc = nullptr;
    pd.dV_acc = nullptr;
    cudaError_t e = d == 128 ? launch_bwd_q<128>(maps, do_cube, pd, tab, geo.n_groups, st)
                             : launch_bwd_q<64>(maps, do_cube, pd, tab, geo.n_groups, st);
    if (e == cudaSuccess)
      e = d == 128 ? launch_bwd_kv<128>(maps, q_tile, do_tile, pd, w.delta, dKp, dVp, tab, geo.S, st)
                   : launch_bwd_kv<64>(maps, q_tile, do_tile, pd, w.delta, dKp, dVp, tab, geo.S, st);
    if (e != cudaSuccess) return DSV_ERR_CUDA;
  }
  return DSV_OK;
}
