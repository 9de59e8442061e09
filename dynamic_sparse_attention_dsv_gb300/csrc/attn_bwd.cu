// Query-grouped sparse attention, backward pass.
//
// "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT
// Training" (gist.science technical summary, section 2.1): stage 2 trains
// with attention restricted to the critical KV pairs, so gradients flow
// through the selected (query, key) pairs only; the index sets are constants
// of the step. Recomputation from the saved LSE follows the usual
// memory-efficient attention practice.
//
// Group-major kernel (sparse problems): one CTA per (query group, problem),
// looping over the group's 128-key tiles:
//   S = Q K^T, dP = dO V^T                        tcgen05 (smem x smem) -> TMEM
//   P = exp2(S*scale*log2e - LSE*log2e), dS' = scale P (dP - Delta)   registers
//   dQ += dS' K                                   accumulated in TMEM, written once
//   dV_tile = P^T dO, dK_tile = dS'^T Q -> TMEM, written as bf16 partial
//   rows, one per (group, selected key) pair.
// Ordered dK/dV reduction (no atomics on the data): a bitmap of which groups
// selected each key gives every (key, group) pair a slot, off[key] + the
// number of lower groups that selected the key (each 32-group bitmap word
// carries the count of the key's lower words), so the partials of one key
// lie contiguously in ascending group order; a reduce kernel sums each key's
// slots in that order in fp32. The result is the same bits on every run.
// Dense problems: dQ by a group-major pass without partials (k_attn_bwd_dq,
// dS kept in TMEM), dK/dV by a key-major kernel: one CTA per (128-key tile,
// problem), looping over all 128-token query tiles with dV, dK accumulated in
// TMEM; no cross-CTA reduction at all.
#include <algorithm>
#include <type_traits>
#include <vector>

#include "attn_common.cuh"

namespace dsv {

constexpr int kBwdThreads = 192;                       // key-major kernel
// Group-major kernel: three warpgroups. Registers per thread at launch are
// 16384 / (3 warps x 32 lanes) per SM sub-partition, rounded down to 8; the
// warpgroups then rebalance them (softmax up, loaders down) so that the three
// shares add up to exactly the launch total.
constexpr int kBwdQThreads = 384;
constexpr int kBwdQLaunchRegs = 168;
constexpr int kRegsSoftmax = 232, kRegsDrain = 136, kRegsLoad = 136;
static_assert(kRegsSoftmax + kRegsDrain + kRegsLoad == 3 * kBwdQLaunchRegs, "register split must equal the launch");
// Warps 8-10 gather the selected K/V rows, warp 11 issues the MMAs.
constexpr int kBwdGatherWarps = 3;
constexpr int kMaxUnits = 48;                       // work units per group-major launch
constexpr size_t kPartialBudget = 48ull << 30;      // bytes of bf16 dK/dV partials in flight
constexpr int kMaxBlocks = 1024;                    // 256-key blocks per problem (S <= 2^18)

// A unit is a range of groups of one problem whose dK/dV partials are
// produced and reduced by one launch.
struct UnitTable {
  int32_t n;
  int32_t p[kMaxUnits];        // problem (b*H + h)
  int32_t k[kMaxUnits];        // keys per group (S for dense problems)
  int32_t g0[kMaxUnits];       // first group of the unit
  int32_t ng[kMaxUnits];       // groups in the unit
  int32_t nwords[kMaxUnits];   // bitmap words per key (ceil(ng / 32))
  int32_t flags[kMaxUnits];    // bit 0: first unit of its problem, bit 1: last unit
  int64_t off[kMaxUnits];      // idx offset of row (p, 0); -1 = dense
  int64_t part_base[kMaxUnits];   // first partial slot of the unit
  int64_t bits_base[kMaxUnits];   // first bitmap word of the unit
};

struct CscParams {
  uint64_t* bits;              // per unit [S][nwords]: low 32 bits: bit (key, group) set if the group selected
                               // the key; high 32 bits: number of set bits in the key's lower words
  int32_t* off;                // per unit [S + 1]: first slot of each key within its 256-key block
  int32_t* bpre;               // per unit [S/256 + 1]: first slot of each 256-key block; last = total
  __nv_bfloat16* part_v;       // [slots][d]
  __nv_bfloat16* part_k;       // [slots][d]
  float* acc_v;                // [S][d] fp32 running sums of a problem split over several units
  float* acc_k;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
};

template <int D>
struct BwdCfg {
  static constexpr int kTile = 128 * D * 2;      // one [128][D] bf16 tile
  static constexpr int kKStages = 2;
  static constexpr int kVStages = D == 128 ? 1 : 2;
  static constexpr int kOffDO = kTile;           // Q at 0
  static constexpr int kOffK = 2 * kTile;
  static constexpr int kOffV = kOffK + kKStages * kTile;
  static constexpr int kOffP = kOffV + kVStages * kTile;  // [128 q][128 keys] bf16 = 32 KB
  static constexpr int kOffDS = kOffP + 32768;
  static constexpr int kOffBar = kOffDS + 32768;
  static constexpr int kSmemUsed = kOffBar + 1024 + 1024;
  static constexpr int kSmem = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
  // TMEM columns: S and dP of a tile share one 128-column region (dP(t) is
  // computed once S(t) is in registers, S(t+1) once dP(t) is), which leaves
  // room for the dQ accumulator and separate dV and dK regions: each job
  // drains while the tensor cores compute the other.
  static constexpr uint32_t kColSDP = 0, kColDQ = 128, kColDV = 128 + D, kColDK = 128 + 2 * D;
};
static_assert(BwdCfg<128>::kSmemUsed <= 232448, "group-major backward exceeds shared memory");
static_assert(BwdCfg<128>::kColDK + 128 <= 512 && BwdCfg<64>::kColDK + 64 <= 512, "TMEM budget");

// Writes 8 bf16 values (packed in 4 words) at 16-byte chunk `chunk` (0..15)
// of row `row` of a [128][128] bf16 K-major tile with the 128-byte swizzle.
__device__ __forceinline__ void st_sw128_chunk(uint8_t* tile, int row, int chunk, uint4 v) {
  const int atom = chunk >> 3, c = chunk & 7;
  *reinterpret_cast<uint4*>(tile + atom * 16384 + row * 128 + ((c ^ (row & 7)) << 4)) = v;
}

// Columns 32c..32c+31 of one dS row: dS = P (scale dP - scale Delta) from
// the row's fp32 P and dP, packed to bf16 and written to the K-major tile.
__device__ __forceinline__ void ds_chunk(uint8_t* sDS, int row, int c, const uint32_t (&p)[32],
                                         const uint32_t (&dp)[32], float dsc, float ndd) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = q * 8 + e * 2;
      w[e] = pack_bf16x2(__uint_as_float(p[i]) * fmaf(__uint_as_float(dp[i]), dsc, ndd),
                         __uint_as_float(p[i + 1]) * fmaf(__uint_as_float(dp[i + 1]), dsc, ndd));
    }
    st_sw128_chunk(sDS, row, c * 4 + q, make_uint4(w[0], w[1], w[2], w[3]));
  }
}

// ---------------------------------------------------------------------------
// Group-major backward. Warps 0-3 turn S, dP into P, dS (shared memory);
// warps 4-7 drain the dV/dK partial rows to their slots and write dQ at the
// end; warps 8-10 gather the selected K/V rows (cp.async); warp 11 issues
// the MMAs. Per 128-key tile t, in the order the MMAs are issued:
//   dP(t) = dO V^T     once S(t) is in registers (same TMEM columns)
//   dV(t) = P(t)^T dO  once P(t) is in shared memory and dV(t-1) drained
//   S(t+1) = Q K^T     once dP(t) is in registers
//   dQ += dS(t) K; dK(t) = dS(t)^T Q  once dS(t) is in shared memory
// so the softmax warps compute P(t) while dP(t) runs and dS(t) while S(t+1)
// runs, and the drain of one job overlaps the other job's MMAs.
template <int D>
__global__ void __launch_bounds__(kBwdQThreads, 1)
    k_attn_bwd_q(const __grid_constant__ AttnMaps maps, const __grid_constant__ CUtensorMap do_cube,
                 const AttnParams prm, const CscParams csc, const UnitTable tab) {
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
  uint64_t* k_empty = bars + 3;      // [2]
  uint64_t* v_full = bars + 5;       // [2]
  uint64_t* v_empty = bars + 7;      // [2]
  uint64_t* s_full = bars + 9;       // S(t) in TMEM
  uint64_t* s_free = bars + 10;      // S(t) in registers: dP(t) may overwrite its columns
  uint64_t* dp_full = bars + 11;     // dP(t) in TMEM
  uint64_t* dp_free = bars + 12;     // dP(t) in registers: S(t+1) may overwrite its columns
  uint64_t* p_full = bars + 13;      // P(t) in shared memory
  uint64_t* p_free = bars + 14;      // P(t) read by the dV MMAs
  uint64_t* ds_full = bars + 15;     // dS(t) in shared memory
  uint64_t* ds_free = bars + 16;     // dS(t) read by the dQ and dK MMAs
  uint64_t* dv_full = bars + 17;     // dV partials of tile t in TMEM
  uint64_t* dv_free = bars + 18;     // ... drained to their slots
  uint64_t* dk_full = bars + 19;
  uint64_t* dk_free = bars + 20;
  uint64_t* dq_done = bars + 21;
  uint64_t* mma_drain = bars + 22;   // every MMA issued has completed (unwind)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 23);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.y;
  if ((int)blockIdx.x >= tab.ng[u]) return;   // units of a launch may hold fewer groups than the grid
  const int g = tab.g0[u] + blockIdx.x, p = tab.p[u];
  const Geometry& geo = prm.geo;
  // every unit here is a sparse problem (dense ones take k_attn_bwd_dq and k_attn_bwd_kv)
  const int k = tab.k[u];
  const int nt = (k + 127) / 128;
  const int32_t* idx_row = prm.idx + tab.off[u] + (int64_t)g * k;
  const int G = geo.G;
  constexpr int kProdWarp = 8, kMmaWarp = 8 + kBwdGatherWarps;

  if (G < 128) {
    for (int i = tid; i < (128 - G) * (D / 64) * 8; i += blockDim.x) {
      const int a = i / ((128 - G) * 8), rem = i % ((128 - G) * 8);
      reinterpret_cast<uint4*>(sQ + a * 16384 + G * 128)[rem] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(sDO + a * 16384 + G * 128)[rem] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {   // one arrival per gathering lane
      mbar_init(k_full + i, 32u * kBwdGatherWarps);
      mbar_init(v_full + i, 32u * kBwdGatherWarps);
      mbar_init(k_empty + i, 1);
      mbar_init(v_empty + i, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 4);
    mbar_init(p_full, 4);
    mbar_init(p_free, 1);
    mbar_init(ds_full, 4);
    mbar_init(ds_free, 1);
    mbar_init(dv_full, 1);
    mbar_init(dv_free, 4);
    mbar_init(dk_full, 1);
    mbar_init(dk_free, 4);
    mbar_init(dq_done, 1);
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp >= kProdWarp) {
   setmaxnreg_dec<kRegsLoad>();   // the whole warpgroup (warps 8-11) executes this one instruction
   if (warp < kMmaWarp) {
    // ----------------------------------------------------------- producers
    const int pw = warp - kProdWarp;
    const int ct = g / (geo.ncy * geo.ncx), cy = (g / geo.ncx) % geo.ncy, cx = g % geo.ncx;
    if (pw == 0 && lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * G * D * 2);
      for (int a = 0; a < D / 64; ++a) {
        tma_load_4d(sQ + a * 16384, &maps.q_cube, q_full, a * 64, cx * geo.gx, cy * geo.gy, p * geo.T + ct * geo.gt);
        tma_load_4d(sDO + a * 16384, &do_cube, q_full, a * 64, cx * geo.gx, cy * geo.gy, p * geo.T + ct * geo.gt);
      }
    }
    const int prow0 = p * geo.S;
    int rows[Gather<D, kBwdGatherWarps>::kIters], nxt[Gather<D, kBwdGatherWarps>::kIters];
    gather_rows<D, kBwdGatherWarps>(nxt, idx_row, k, 0, prow0, pw, lane);
    for (int t = 0; t < nt; ++t) {
      const int ks = t % C::kKStages, vs = t % C::kVStages;
#pragma unroll
      for (int i = 0; i < Gather<D, kBwdGatherWarps>::kIters; ++i) rows[i] = nxt[i];
      if (t + 1 < nt) gather_rows<D, kBwdGatherWarps>(nxt, idx_row, k, t + 1, prow0, pw, lane);
      if (t >= C::kKStages && !mbar_wait_warp(k_empty + ks, ((t / C::kKStages) - 1) & 1, prm.wait_ns)) {
        if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
        break;
      }
      gather_tile<D, kBwdGatherWarps>(sK + ks * C::kTile, prm.K, rows, pw, lane);
      cp_async_arrive_noinc(k_full + ks);
      if (t >= C::kVStages && !mbar_wait_warp(v_empty + vs, ((t / C::kVStages) - 1) & 1, prm.wait_ns)) {
        if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
        break;
      }
      gather_tile<D, kBwdGatherWarps>(sV + vs * C::kTile, prm.V, rows, pw, lane);
      cp_async_arrive_noinc(v_full + vs);
    }
    // the warp leaves only once the copies it started have landed (a
    // timed-out pipeline may not have consumed them)
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (pw == 0 && lane == 0) mbar_wait(q_full, 0, kDrainLimitNs);
   } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id_sdp = instr_desc(128, 128, 1, 0, 0);   // Q K^T, dO V^T
      constexpr uint32_t id_dq = instr_desc(128, D, 1, 0, 1);      // dS K (B = K, MN-major)
      constexpr uint32_t id_kv = instr_desc(128, D, 1, 1, 1);      // P^T dO, dS^T Q (MN-major)
      // base descriptors (K-major), built once; an operand is a fixed offset from one of
      // them, and the MN-major form differs only by a constant in the stride field
      constexpr uint64_t kMn = (uint64_t)((16384 >> 4) - (16 >> 4)) << 16;
      const uint64_t dq_k = smem_desc(smem_u32(sQ), 16, 1024), ddo_k = smem_desc(smem_u32(sDO), 16, 1024);
      const uint64_t dp_k = smem_desc(smem_u32(sP), 16, 1024), dds_k = smem_desc(smem_u32(sDS), 16, 1024);
      bool ok = mbar_wait(q_full, 0, prm.wait_ns);
      auto issue_s = [&](int t) -> bool {   // S(t) = Q K(t)^T
        const int ks = t % C::kKStages;
        if (!mbar_wait(k_full + ks, (t / C::kKStages) & 1, prm.wait_ns)) return false;
        fence_proxy_async_smem();   // rows written by cp.async (generic proxy) -> tensor core reads
        tc_fence_after();
        const uint64_t dk = smem_desc(smem_u32(sK + ks * C::kTile), 16, 1024);
        const uint64_t dq = opaque(dq_k);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ss(tbase + C::kColSDP, desc_at(dq, off), desc_at(dk, off), id_sdp, kk > 0);
        }
        mma_commit(s_full);
        return true;
      };
      if (ok && nt > 0) ok = issue_s(0);
      for (int t = 0; ok && t < nt; ++t) {
        const int ks = t % C::kKStages, vs = t % C::kVStages;
        // dP(t) = dO V(t)^T into the columns S(t) has left
        if (!mbar_wait(s_free, t & 1, prm.wait_ns) ||
            !mbar_wait(v_full + vs, (t / C::kVStages) & 1, prm.wait_ns)) { ok = false; break; }
        fence_proxy_async_smem();
        tc_fence_after();
        {
          const uint64_t dv = smem_desc(smem_u32(sV + vs * C::kTile), 16, 1024);
          const uint64_t ddo = opaque(ddo_k);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_f16_ss(tbase + C::kColSDP, desc_at(ddo, off), desc_at(dv, off), id_sdp, kk > 0);
          }
        }
        mma_commit(dp_full);
        mma_commit(v_empty + vs);
        // dV(t) = P(t)^T dO
        if (!mbar_wait(p_full, t & 1, prm.wait_ns) ||
            (t >= 1 && !mbar_wait(dv_free, (t - 1) & 1, prm.wait_ns))) { ok = false; break; }
        tc_fence_after();
        {
          const uint64_t a = opaque(dp_k + kMn), b = opaque(ddo_k + kMn);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f16_ss(tbase + C::kColDV, desc_at(a, kk * 2048), desc_at(b, kk * 2048), id_kv, kk > 0);
        }
        mma_commit(dv_full);
        mma_commit(p_free);
        // S(t+1) into the columns dP(t) has left
        if (t + 1 < nt && (!mbar_wait(dp_free, t & 1, prm.wait_ns) || !issue_s(t + 1))) { ok = false; break; }
        // dQ += dS(t) K(t), then dK(t) = dS(t)^T Q
        if (!mbar_wait(ds_full, t & 1, prm.wait_ns)) { ok = false; break; }
        tc_fence_after();
        {
          const uint64_t dk_m = smem_desc(smem_u32(sK + ks * C::kTile), 16, 1024) + kMn;
          const uint64_t dds = opaque(dds_k);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t offa = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_f16_ss(tbase + C::kColDQ, desc_at(dds, offa), desc_at(dk_m, kk * 2048), id_dq,
                       (t > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(k_empty + ks);
        if (t >= 1 && !mbar_wait(dk_free, (t - 1) & 1, prm.wait_ns)) { ok = false; break; }
        tc_fence_after();
        {
          const uint64_t a = opaque(dds_k + kMn), b = opaque(dq_k + kMn);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f16_ss(tbase + C::kColDK, desc_at(a, kk * 2048), desc_at(b, kk * 2048), id_kv, kk > 0);
        }
        mma_commit(dk_full);
        mma_commit(ds_free);
      }
      if (ok) mma_commit(dq_done);
      else raise_status(prm.status, DSV_ERR_TIMEOUT);
      // every MMA issued completes before TMEM is released
      mma_commit(mma_drain);
      mbar_wait(mma_drain, 0, kDrainLimitNs);
    }
   }
  } else if (warp < 4) {
    // ------------------------------------------- S, dP -> P, dS (warps 0-3)
    setmaxnreg_inc<kRegsSoftmax>();
    const int row = warp * 32 + lane;
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    const float sc = prm.scale_log2;
    float lse2 = INFINITY, delta = 0.f;
    if (row < G) {
      const int tok = token_of(geo, g, row);
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
    // dS is produced pre-multiplied by the attention scale (scale dS = P (scale dP - scale Delta)),
    // so dQ = (scale dS) K and dK = (scale dS)^T Q need no scaling afterwards
    const float dsc = prm.scale, ndd = -delta * prm.scale;
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
      const int nvalid = min(128, k - t * 128);
      ok = ok && mbar_wait_warp(s_full, t & 1, prm.wait_ns);
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_addr + C::kColSDP + c * 32, sr[c]);
      tmem_ld_wait(sr[0]);
      reg_fence(sr[1]);
      reg_fence(sr[2]);
      reg_fence(sr[3]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);   // S(t) in registers: dP(t) may take its columns
      // P (fp32, in place of S), while dP(t) is computed. The exponential is
      // taken for every column (the padding columns hold finite scores of a
      // repeated key) and the padding zeroed afterwards: a choice around the
      // exponential itself costs far more than the exponential.
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) sr[c][e] = __float_as_uint(ex2_fast(fmaf(__uint_as_float(sr[c][e]), sc, -lse2)));
      if (nvalid < 128) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e >= nvalid) sr[c][e] = 0u;
      }
      // P(t-1) is free once its dV MMAs completed
      if (t >= 1) ok = ok && mbar_wait_warp(p_free, (t - 1) & 1, prm.wait_ns);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const uint32_t* x = &sr[q >> 2][(q & 3) * 8];
        st_sw128_chunk(sP, row, q,
                       make_uint4(pack_bf16x2(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                  pack_bf16x2(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                  pack_bf16x2(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                  pack_bf16x2(__uint_as_float(x[6]), __uint_as_float(x[7]))));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      // dS = P (scale dP - scale Delta), 32 columns at a time with the next
      // chunk's TMEM load in flight
      ok = ok && mbar_wait_warp(dp_full, t & 1, prm.wait_ns);
      tc_fence_after();
      uint32_t da[2][32];
      tmem_ld32(lane_addr + C::kColSDP, da[0]);
      tmem_ld32(lane_addr + C::kColSDP + 32, da[1]);
      tmem_ld_wait(da[0]);
      reg_fence(da[1]);
      // dS(t-1) is free once its dQ and dK MMAs completed
      if (t >= 1) ok = ok && mbar_wait_warp(ds_free, (t - 1) & 1, prm.wait_ns);
      ds_chunk(sDS, row, 0, sr[0], da[0], dsc, ndd);
      tmem_ld32(lane_addr + C::kColSDP + 64, da[0]);
      ds_chunk(sDS, row, 1, sr[1], da[1], dsc, ndd);
      tmem_ld_wait(da[0]);
      tmem_ld32(lane_addr + C::kColSDP + 96, da[1]);
      ds_chunk(sDS, row, 2, sr[2], da[0], dsc, ndd);
      tmem_ld_wait(da[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dp_free);   // dP(t) in registers: S(t+1) may take its columns
      ds_chunk(sDS, row, 3, sr[3], da[1], dsc, ndd);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    if (!ok && lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
  } else if (warp >= 4 && warp < 8) {
    // -------------------------------- dV/dK partial drain, then dQ (warps 4-7)
    setmaxnreg_dec<kRegsDrain>();
    const int q = warp - 4;
    const int row = q * 32 + lane;   // key slot of the tile for the partials; query row for dQ
    const uint32_t lane_addr = tbase + ((uint32_t)(q * 32) << 16);
    bool ok = true;
    // Slot of this key row for tile t: off[key] + groups below ours that chose it.
    const int gl = g - tab.g0[u];
    const uint64_t* bits_u = csc.bits + tab.bits_base[u];
    const int32_t* off_u = csc.off + (int64_t)u * (geo.S + 1);
    const int32_t* bpre_u = csc.bpre + (int64_t)u * (kMaxBlocks + 1);
    auto slot_of = [&](int j) -> int64_t {
      const uint64_t x = __ldg(bits_u + (int64_t)j * tab.nwords[u] + (gl >> 5));
      const int r = (int)(x >> 32) + __popc((uint32_t)x & ((1u << (gl & 31)) - 1u));
      return tab.part_base[u] + __ldg(bpre_u + (j >> 8)) + __ldg(off_u + j) + r;
    };
    int j_next = row < k ? __ldg(idx_row + row) : -1;
    int64_t pos_next = j_next >= 0 ? slot_of(j_next) : 0;
    for (int t = 0; t < nt; ++t) {
      // The drain reads 16 rows per TMEM load, each row's 64 columns split
      // over two threads (lane l and l + 16), so one store instruction covers
      // 16 rows x 64 bytes instead of 32 rows x 32: half the cache lines per
      // instruction. Thread `lane` stores row 16h + (lane & 15) of the warp's 32.
      const int64_t pos = pos_next;
      const int64_t hpos0 = __shfl_sync(0xffffffffu, pos, lane & 15);
      const int64_t hpos1 = __shfl_sync(0xffffffffu, pos, 16 + (lane & 15));
      const int hrow0 = t * 128 + q * 32 + (lane & 15);   // row of the first half within the problem's keys
      const int nslot = (t + 1) * 128 + row;
      j_next = (t + 1 < nt && nslot < k) ? __ldg(idx_row + nslot) : -1;   // next tile's key, loaded early
      for (int jb = 0; jb < 2; ++jb) {   // dV, then dK
        ok = ok && mbar_wait_warp(jb == 0 ? dv_full : dk_full, t & 1, prm.wait_ns);
        tc_fence_after();
        const uint32_t col = jb == 0 ? C::kColDV : C::kColDK;
        __nv_bfloat16* part = jb == 0 ? csc.part_v : csc.part_k;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb) {
            const int dcol = cb * 64 + (lane >= 16 ? 32 : 0);
            uint32_t v[32];
            tmem_ld16x2<32>(lane_addr + ((uint32_t)(16 * h) << 16) + col + cb * 64, v);
            tmem_ld_wait(v);
            if (hrow0 + 16 * h < k) {
              __nv_bfloat16* dst = part + (h ? hpos1 : hpos0) * D + dcol;
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)
                pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
              st_global_v8(dst, pk);
              st_global_v8(dst + 16, pk + 8);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(jb == 0 ? dv_free : dk_free);
        if (jb == 0) pos_next = j_next >= 0 ? slot_of(j_next) : 0;   // overlaps the next job's MMAs
      }
    }
    // ----------------------------------------------------------- dQ out
    ok = ok && mbar_wait_warp(dq_done, 0, prm.wait_ns);
    if (!ok) {
      if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
    } else {
      tc_fence_after();
      const int tok = row < G ? token_of(geo, g, row) : 0;
      __nv_bfloat16* qrow = prm.out + ((int64_t)p * geo.S + tok) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + C::kColDQ + c * 32, o);
        tmem_ld_wait(o);
        if (row < G) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1]));
          uint4* dst = reinterpret_cast<uint4*>(qrow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------
// Key-major dK/dV for dense problems. grid = (S/128, problems). One CTA owns
// a 128-key tile and loops over every 128-query tile u:
//   S^T = K Q^T, dP^T = V dO^T       tcgen05 (smem x smem) -> TMEM
//   P^T, dS^T (registers, key per thread), written back to TMEM as bf16 in
//   place of S^T and dP^T
//   dV += P^T dO, dK += dS^T Q       tcgen05 with A in TMEM (no shared-memory
//                                    copy of P or dS) -> TMEM accumulators
// Q, dO and the tile's LSE*log2(e) and Delta rows are double-buffered, so the
// next tile's copies overlap this tile's work. Warps 0-3 compute P and dS,
// warp 4 loads, warp 5 issues the MMAs.
template <int D>
struct KvCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kOffV = kTile;            // K at 0
  static constexpr int kOffQ = 2 * kTile;        // [2 stages]
  static constexpr int kOffDO = 4 * kTile;       // [2 stages]
  static constexpr int kOffStat = 6 * kTile;     // [2 stages][LSE2[128], Delta[128]]
  static constexpr int kOffBar = kOffStat + 2 * 1024;
  static constexpr int kSmemUsed = kOffBar + 256 + 1024;
  static constexpr int kSmem = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
};
static_assert(KvCfg<128>::kSmemUsed <= 232448, "key-major backward exceeds shared memory");

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_attn_bwd_kv(const __grid_constant__ AttnMaps maps, const __grid_constant__ CUtensorMap q_tile,
                  const __grid_constant__ CUtensorMap do_tile, const AttnParams prm, const float* delta_all,
                  const float* lse2_all, __nv_bfloat16* dK, __nv_bfloat16* dV, const ProblemTable tab) {
  using C = KvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sm;
  uint8_t* sV = sm + C::kOffV;
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sDO = sm + C::kOffDO;
  float* sStat = reinterpret_cast<float*>(sm + C::kOffStat);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;      // [2] Q, dO, LSE2 and Delta of the stage's query tile
  uint64_t* q_empty = bars + 3;     // [2] the stage's MMAs (and so its P/dS pass) are done
  uint64_t* sdp_full = bars + 5;    // S^T, dP^T of tile u in TMEM
  uint64_t* ps_half = bars + 6;     // [2] P^T, dS^T of queries 0-63 / 64-127 of tile u in TMEM
  uint64_t* mma_drain = bars + 8;   // every MMA issued has completed (end, or unwind)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 9);

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
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + i, 1);
      mbar_init(q_empty + i, 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(ps_half, 4);
    mbar_init(ps_half + 1, 4);
    mbar_init(mma_drain, 1);
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
      int issued = 0;
      for (int u = 0; u < nq; ++u) {
        const int st = u & 1;
        if (u >= 2 && !mbar_wait(q_empty + st, ((u >> 1) - 1) & 1, prm.wait_ns)) {
          raise_status(prm.status, DSV_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(q_full + st, 2 * C::kTile + 1024);
        for (int a = 0; a < D / 64; ++a) {
          tma_load_2d(sQ + st * C::kTile + a * 16384, &q_tile, q_full + st, a * 64, prow0 + u * 128);
          tma_load_2d(sDO + st * C::kTile + a * 16384, &do_tile, q_full + st, a * 64, prow0 + u * 128);
        }
        bulk_load(sStat + st * 256, lse2_all + (int64_t)prow0 + u * 128, 512, q_full + st);
        bulk_load(sStat + st * 256 + 128, delta_all + (int64_t)prow0 + u * 128, 512, q_full + st);
        issued = u + 1;
      }
      // the block leaves only once every copy it started has landed
      mbar_wait(kv_full, 0, kDrainLimitNs);
      for (int u = max(0, issued - 2); u < issued; ++u) mbar_wait(q_full + (u & 1), (u >> 1) & 1, kDrainLimitNs);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t id_sdp = instr_desc(128, 128, 1, 0, 0);   // K Q^T, V dO^T
      constexpr uint32_t id_acc = instr_desc(128, D, 1, 0, 1);     // P^T dO, dS^T Q (A in TMEM, B MN-major)
      const uint32_t ak = smem_u32(sK), av = smem_u32(sV);
      bool ok = mbar_wait(kv_full, 0, prm.wait_ns);
      for (int u = 0; ok && u < nq; ++u) {
        const int st = u & 1;
        const uint32_t aq = smem_u32(sQ + st * C::kTile), ado = smem_u32(sDO + st * C::kTile);
        if (!mbar_wait(q_full + st, (u >> 1) & 1, prm.wait_ns)) { ok = false; break; }
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
        // P^T and dS^T: bf16 pairs in the first 64 columns of the S^T and dP^T regions; the
        // MMAs of the first 64 queries run while the second 64 are computed
        for (int h = 0; h < 2; ++h) {
          if (!mbar_wait(ps_half + h, u & 1, prm.wait_ns)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
            mma_f16_ts(tbase + kColDV, tbase + kColS + kk * 8, smem_desc(ado + kk * 2048, 16384, 1024), id_acc,
                       (u > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
            mma_f16_ts(tbase + kColDK, tbase + kColDP + kk * 8, smem_desc(aq + kk * 2048, 16384, 1024), id_acc,
                       (u > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(q_empty + st);
      }
      if (!ok) raise_status(prm.status, DSV_ERR_TIMEOUT);
      // every MMA issued completes before the results are read and TMEM is released
      mma_commit(mma_drain);
      mbar_wait(mma_drain, 0, kDrainLimitNs);
    }
  } else {
    const int row = warp * 32 + lane;   // key slot of the tile
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    const float sc = prm.scale_log2;
    bool ok = true;
    for (int u = 0; ok && u < nq; ++u) {
      const int st = u & 1;
      // the stage's LSE2 and Delta rows arrived with its Q and dO
      ok = ok && mbar_wait_warp(q_full + st, (u >> 1) & 1, prm.wait_ns);
      ok = ok && mbar_wait_warp(sdp_full, u & 1, prm.wait_ns);
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = sStat + st * 256;
      const float* dl = lse2 + 128;
      // 32 queries at a time; P^T and dS^T of chunk c go to columns 16c .. 16c+15,
      // which hold S^T / dP^T values already read (chunks <= c)
      uint32_t sr[2][32], dr[2][32];
      tmem_ld32(lane_addr + kColS, sr[0]);
      tmem_ld32(lane_addr + kColDP, dr[0]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int b = c & 1;
        tmem_ld_wait(sr[b]);
        reg_fence(dr[b]);
        if (c + 1 < 4) {
          tmem_ld32(lane_addr + kColS + (c + 1) * 32, sr[b ^ 1]);
          tmem_ld32(lane_addr + kColDP + (c + 1) * 32, dr[b ^ 1]);
        }
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int q = c * 32 + e;
          const float p0 = ex2_fast(fmaf(__uint_as_float(sr[b][e]), sc, -lse2[q]));
          const float p1 = ex2_fast(fmaf(__uint_as_float(sr[b][e + 1]), sc, -lse2[q + 1]));
          pw[e >> 1] = pack_bf16x2(p0, p1);
          dw[e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dr[b][e]) - dl[q]),
                                   p1 * (__uint_as_float(dr[b][e + 1]) - dl[q + 1]));
        }
        tmem_st16(lane_addr + kColS + c * 16, pw);
        tmem_st16(lane_addr + kColDP + c * 16, dw);
        if (c & 1) {   // queries 0-63 (c = 1) or 64-127 (c = 3) complete
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(ps_half + (c >> 1));
        }
      }
    }
    ok = ok && mbar_wait_warp(mma_drain, 0, prm.wait_ns);
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

// ---------------------------------------------------------------------------
// dQ of a dense problem, group-major: one CTA per (query group, problem)
// over all S keys in 128-key tiles. With no dK/dV partials to produce, the
// group-major kernel's shared-memory copies of P and dS are not needed: dS
// goes back to TMEM as bf16 in place of dP, and dQ += dS K takes its A
// operand from there. Two TMEM regions alternate between tiles (S, then dP,
// then dS of tile t in region t % 2), so tile t+1's S is computed while tile
// t's P and dS are. Warps 0-3: P, dS and the final dQ rows (one query per
// thread); warp 4 loads (TMA); warp 5 issues the MMAs.
template <int D>
struct DqCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kKStages = 3, kVStages = 2;
  static constexpr int kOffDO = kTile;       // Q at 0
  static constexpr int kOffK = 2 * kTile;
  static constexpr int kOffV = kOffK + kKStages * kTile;
  static constexpr int kOffBar = kOffV + kVStages * kTile;
  static constexpr int kSmemUsed = kOffBar + 256 + 1024;
  static constexpr int kSmem = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
  static constexpr uint32_t kColR0 = 0, kColDQ = 128, kColR1 = 256;
};
static_assert(DqCfg<128>::kSmemUsed <= 232448, "dense dQ kernel exceeds shared memory");

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_attn_bwd_dq(const __grid_constant__ AttnMaps maps, const __grid_constant__ CUtensorMap do_cube,
                  const AttnParams prm, const float* delta_all, const UnitTable tab) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;
  uint8_t* sDO = sm + C::kOffDO;
  uint8_t* sK = sm + C::kOffK;
  uint8_t* sV = sm + C::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;       // [3]
  uint64_t* k_empty = bars + 4;      // [3]
  uint64_t* v_full = bars + 7;       // [2]
  uint64_t* v_empty = bars + 9;      // [2]
  uint64_t* s_full = bars + 11;      // [2] S of the region's tile in TMEM
  uint64_t* s_free = bars + 13;      // S(t) in registers: dP(t) may overwrite it
  uint64_t* dp_full = bars + 14;     // dP(t) in TMEM
  uint64_t* ds_full = bars + 15;     // dS(t) in TMEM
  uint64_t* dq_done = bars + 16;
  uint64_t* mma_drain = bars + 17;   // every MMA issued has completed (unwind)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 18);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.y;
  if ((int)blockIdx.x >= tab.ng[u]) return;
  const int g = tab.g0[u] + blockIdx.x, p = tab.p[u];
  const Geometry& geo = prm.geo;
  const int G = geo.G, nt = geo.S / 128, prow0 = p * geo.S;

  if (G < 128) {   // padding query rows stay zero: the Q/dO boxes write only the group's G rows
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
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_full + 1, 1);
    mbar_init(s_free, 4);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 4);
    mbar_init(dq_done, 1);
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 4) {
    if (lane == 0) {
      const int ct = g / (geo.ncy * geo.ncx), cy = (g / geo.ncx) % geo.ncy, cx = g % geo.ncx;
      mbar_arrive_expect_tx(q_full, 2 * G * D * 2);
      for (int a = 0; a < D / 64; ++a) {
        tma_load_4d(sQ + a * 16384, &maps.q_cube, q_full, a * 64, cx * geo.gx, cy * geo.gy, p * geo.T + ct * geo.gt);
        tma_load_4d(sDO + a * 16384, &do_cube, q_full, a * 64, cx * geo.gx, cy * geo.gy, p * geo.T + ct * geo.gt);
      }
      int k_issued = 0, v_issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int ks = t % C::kKStages, vs = t % C::kVStages;
        if (t >= C::kKStages && !mbar_wait(k_empty + ks, ((t / C::kKStages) - 1) & 1, prm.wait_ns)) {
          raise_status(prm.status, DSV_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(k_full + ks, C::kTile);
        load_dense_tile<D>(sK + ks * C::kTile, &maps.k_tile, k_full + ks, t, prow0);
        k_issued = t + 1;
        if (t >= C::kVStages && !mbar_wait(v_empty + vs, ((t / C::kVStages) - 1) & 1, prm.wait_ns)) {
          raise_status(prm.status, DSV_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(v_full + vs, C::kTile);
        load_dense_tile<D>(sV + vs * C::kTile, &maps.v_tile, v_full + vs, t, prow0);
        v_issued = t + 1;
      }
      // the block leaves only once every copy it started has landed
      for (int t = max(0, k_issued - C::kKStages); t < k_issued; ++t)
        mbar_wait(k_full + t % C::kKStages, (t / C::kKStages) & 1, kDrainLimitNs);
      for (int t = max(0, v_issued - C::kVStages); t < v_issued; ++t)
        mbar_wait(v_full + t % C::kVStages, (t / C::kVStages) & 1, kDrainLimitNs);
      mbar_wait(q_full, 0, kDrainLimitNs);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t id_sdp = instr_desc(128, 128, 1, 0, 0);   // Q K^T, dO V^T
      constexpr uint32_t id_dq = instr_desc(128, D, 1, 0, 1);      // dS K (A in TMEM, B = K MN-major)
      constexpr uint64_t kMn = (uint64_t)((16384 >> 4) - (16 >> 4)) << 16;
      const uint64_t dq_k = smem_desc(smem_u32(sQ), 16, 1024), ddo_k = smem_desc(smem_u32(sDO), 16, 1024);
      auto region = [&](int t) -> uint32_t { return tbase + ((t & 1) ? C::kColR1 : C::kColR0); };
      auto issue_s = [&](int t) -> bool {   // S(t) = Q K(t)^T into the tile's region
        const int ks = t % C::kKStages;
        if (!mbar_wait(k_full + ks, (t / C::kKStages) & 1, prm.wait_ns)) return false;
        tc_fence_after();
        const uint64_t dk = smem_desc(smem_u32(sK + ks * C::kTile), 16, 1024);
        const uint64_t dq = opaque(dq_k);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ss(region(t), desc_at(dq, off), desc_at(dk, off), id_sdp, kk > 0);
        }
        mma_commit(s_full + (t & 1));
        return true;
      };
      bool ok = mbar_wait(q_full, 0, prm.wait_ns);
      if (ok && nt > 0) ok = issue_s(0);
      if (ok && nt > 1) ok = issue_s(1);
      for (int t = 0; ok && t < nt; ++t) {
        const int ks = t % C::kKStages, vs = t % C::kVStages;
        // dP(t) = dO V(t)^T into the columns S(t) has left
        if (!mbar_wait(s_free, t & 1, prm.wait_ns) ||
            !mbar_wait(v_full + vs, (t / C::kVStages) & 1, prm.wait_ns)) { ok = false; break; }
        tc_fence_after();
        {
          const uint64_t dv = smem_desc(smem_u32(sV + vs * C::kTile), 16, 1024);
          const uint64_t ddo = opaque(ddo_k);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_f16_ss(region(t), desc_at(ddo, off), desc_at(dv, off), id_sdp, kk > 0);
          }
        }
        mma_commit(dp_full);
        mma_commit(v_empty + vs);
        // dQ += dS(t) K(t), dS as bf16 pairs in the region's first 64 columns
        if (!mbar_wait(ds_full, t & 1, prm.wait_ns)) { ok = false; break; }
        tc_fence_after();
        {
          const uint64_t dk_m = smem_desc(smem_u32(sK + ks * C::kTile), 16, 1024) + kMn;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f16_ts(tbase + C::kColDQ, region(t) + kk * 8, desc_at(dk_m, kk * 2048), id_dq,
                       (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(k_empty + ks);
        // S(t+2) into this region, after dQ(t) has read its dS (the MMAs run in issue order)
        if (t + 2 < nt && !issue_s(t + 2)) { ok = false; break; }
      }
      if (ok) mma_commit(dq_done);
      else raise_status(prm.status, DSV_ERR_TIMEOUT);
      mma_commit(mma_drain);
      mbar_wait(mma_drain, 0, kDrainLimitNs);
    }
  } else {
    // ---------------------------------------------- P, dS, dQ rows (warps 0-3)
    const int row = warp * 32 + lane;
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    const float sc = prm.scale_log2;
    float lse2 = INFINITY, delta = 0.f;
    int tok = 0;
    if (row < G) {
      tok = token_of(geo, g, row);
      lse2 = prm.LSE[(int64_t)prow0 + tok] * 1.4426950408889634f;
      delta = delta_all[(int64_t)prow0 + tok];
    }
    // dS pre-multiplied by the attention scale, so dQ = (scale dS) K needs no scaling afterwards
    const float dsc = prm.scale, ndd = -delta * prm.scale;
    bool ok = true;
    for (int t = 0; ok && t < nt; ++t) {
      const uint32_t rb = lane_addr + ((t & 1) ? C::kColR1 : C::kColR0);
      ok = ok && mbar_wait_warp(s_full + (t & 1), (t >> 1) & 1, prm.wait_ns);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(rb + c * 32, sr[c]);
      tmem_ld_wait(sr[0]);
      reg_fence(sr[1]);
      reg_fence(sr[2]);
      reg_fence(sr[3]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);   // S(t) in registers: dP(t) may take its columns
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) sr[c][e] = __float_as_uint(ex2_fast(fmaf(__uint_as_float(sr[c][e]), sc, -lse2)));
      ok = ok && mbar_wait_warp(dp_full, t & 1, prm.wait_ns);
      if (!ok) break;
      tc_fence_after();
      // dS of 32 columns at a time, written as 16 bf16-pair columns at 16c over dP values
      // already read (chunks <= c), the next chunk's load in flight
      uint32_t da[2][32];
      tmem_ld32(rb, da[0]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int b = c & 1;
        tmem_ld_wait(da[b]);
        if (c + 1 < 4) tmem_ld32(rb + (c + 1) * 32, da[b ^ 1]);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          w[e >> 1] = pack_bf16x2(__uint_as_float(sr[c][e]) * fmaf(__uint_as_float(da[b][e]), dsc, ndd),
                                  __uint_as_float(sr[c][e + 1]) * fmaf(__uint_as_float(da[b][e + 1]), dsc, ndd));
        tmem_st16(rb + c * 16, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    ok = ok && mbar_wait_warp(dq_done, 0, prm.wait_ns);
    if (!ok) {
      if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
    } else {
      tc_fence_after();
      __nv_bfloat16* qrow = prm.out + ((int64_t)prow0 + tok) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + C::kColDQ + c * 32, o);
        tmem_ld_wait(o);
        if (row < G) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1]));
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

// Delta_i = sum_c dO_ic O_ic for every row of the listed problems. Each
// thread takes one 16-byte chunk of a row (d / 8 threads per row, a divisor
// of the warp), so the loads are coalesced; the row's threads then reduce in
// a fixed order by shuffles.
// With `lse2` non-null it also writes LSE_i * log2(e) (the exponent offset of
// the key-major kernel, which stages it per query tile).
__global__ void __launch_bounds__(256) k_bwd_delta(const __nv_bfloat16* __restrict__ O,
                                                   const __nv_bfloat16* __restrict__ dO, int S, int d,
                                                   float* __restrict__ delta, const float* __restrict__ LSE,
                                                   float* __restrict__ lse2, const ProblemTable tab) {
  const int lp = blockIdx.y, p = tab.p[lp];
  const int cpr = d / 8;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t s = gid / cpr;
  const int c = (int)(gid % cpr);
  float acc = 0.f;
  if (s < S) {
    const int64_t o = ((int64_t)p * S + s) * d + c * 8;
    const uint4 x = *reinterpret_cast<const uint4*>(O + o), y = *reinterpret_cast<const uint4*>(dO + o);
    const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&x);
    const __nv_bfloat162* y2 = reinterpret_cast<const __nv_bfloat162*>(&y);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 u = __bfloat1622float2(x2[e]), v = __bfloat1622float2(y2[e]);
      acc = fmaf(u.x, v.x, acc);
      acc = fmaf(u.y, v.y, acc);
    }
  }
  for (int m = cpr / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (s < S && c == 0) {
    delta[(int64_t)p * S + s] = acc;
    if (lse2) lse2[(int64_t)p * S + s] = LSE[(int64_t)p * S + s] * 1.4426950408889634f;
  }
}

// ---------------------------------------------------------------------------
// Ordered dK/dV reduction: slot map.
constexpr int kCscKeys = 256;
constexpr int kCscStride = kCscKeys + 1;   // words per bitmap column in shared memory (bank spread)

// One CTA per (256-key block, unit) builds the block's part of the selection
// bitmap in shared memory. Index rows are ascending, so each thread binary-
// searches a group's row for the block's first key and walks the row while
// the keys stay inside the block. The words then go out with, in each word's
// high half, the count of the key's set bits in its lower words, and every
// key's slot offset within the block plus the block's total are written.
// Keys outside the block (including values outside [0, S)) are ignored.

__global__ void __launch_bounds__(256) k_csc_build(const int32_t* __restrict__ idx, uint64_t* bits, int S,
                                                   int32_t* off, int32_t* bsum, const UnitTable tab) {
  extern __shared__ uint32_t sb[];                 // [nw][kCscStride]: word w of each key of the block
  __shared__ int cnt[kCscKeys];
  __shared__ int wsum[8];
  const int u = blockIdx.y, kb = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int j0 = kb * kCscKeys;
  if (j0 >= S) return;
  const int j1 = min(j0 + kCscKeys, S);
  const int nw = tab.nwords[u], ng = tab.ng[u], k = tab.k[u];
  for (int i = tid; i < kCscStride * nw; i += 256) sb[i] = 0u;
  __syncthreads();
  // Each thread takes kPair groups (gl and gl + 256) at once, so the steps of
  // their binary searches (and of their scans) have two loads in flight.
  constexpr int kPair = 2;
  for (int gb = tid; gb < ng; gb += 256 * kPair) {
    const int32_t* row[kPair];
    int lo[kPair], hi[kPair];                      // first position whose key is >= j0
#pragma unroll
    for (int e = 0; e < kPair; ++e) {
      const int gl = gb + e * 256;
      row[e] = idx + tab.off[u] + (int64_t)(tab.g0[u] + min(gl, ng - 1)) * k;
      lo[e] = 0;
      hi[e] = gl < ng ? k : 0;
    }
    while (lo[0] < hi[0] || lo[1] < hi[1]) {
      int mid[kPair], v[kPair];
#pragma unroll
      for (int e = 0; e < kPair; ++e) {
        mid[e] = (lo[e] + hi[e]) >> 1;
        v[e] = lo[e] < hi[e] ? __ldg(row[e] + mid[e]) : 0;
      }
#pragma unroll
      for (int e = 0; e < kPair; ++e)
        if (lo[e] < hi[e]) {
          if (v[e] < j0) lo[e] = mid[e] + 1;
          else hi[e] = mid[e];
        }
    }
    // scan from there to the first key >= j1, eight keys of each row per step
    int s[kPair];
    bool live[kPair];
#pragma unroll
    for (int e = 0; e < kPair; ++e) {
      s[e] = lo[e];
      live[e] = gb + e * 256 < ng;
    }
    while (live[0] || live[1]) {
      int key[kPair][8];
#pragma unroll
      for (int e = 0; e < kPair; ++e)
#pragma unroll
        for (int i = 0; i < 8; ++i) key[e][i] = live[e] && s[e] + i < k ? __ldg(row[e] + s[e] + i) : j1;
#pragma unroll
      for (int e = 0; e < kPair; ++e) {
        if (!live[e]) continue;
        const int gl = gb + e * 256;
        const uint32_t bit = 1u << (gl & 31);
        uint32_t* col = sb + (gl >> 5) * kCscStride;
        bool done = s[e] + 8 >= k;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (key[e][i] >= j0 && key[e][i] < j1) atomicOr(col + (key[e][i] - j0), bit);
          done = done || key[e][i] >= j1;
        }
        s[e] += 8;
        live[e] = !done;
      }
    }
  }
  __syncthreads();
  // one warp per key: words with their lower-word counts, coalesced
  uint64_t* out = bits + tab.bits_base[u];
  for (int jj = w; jj < kCscKeys; jj += 8) {
    const int j = j0 + jj;
    uint32_t carry = 0;
    for (int i0 = 0; i0 < nw; i0 += 32) {
      const int i = i0 + lane;
      const uint32_t word = i < nw ? sb[i * kCscStride + jj] : 0u;
      const uint32_t x = __popc(word);
      uint32_t incl = x;
#pragma unroll
      for (int dd = 1; dd < 32; dd <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, dd);
        if (lane >= dd) incl += y;
      }
      if (i < nw && j < j1) out[(int64_t)j * nw + i] = ((uint64_t)(carry + incl - x) << 32) | word;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) cnt[jj] = j < j1 ? (int)carry : 0;
  }
  __syncthreads();
  // slot offsets of the block's keys and the block total
  const int c = cnt[tid];
  int x = c;
#pragma unroll
  for (int dd = 1; dd < 32; dd <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, dd);
    if (lane >= dd) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  int before = 0;
  for (int i = 0; i < w; ++i) before += wsum[i];
  if (j0 + tid < S) off[(int64_t)u * (S + 1) + j0 + tid] = before + x - c;
  if (tid == 255) bsum[(int64_t)u * (kMaxBlocks + 1) + kb] = before + x;
}

// In place: block totals -> exclusive block offsets; entry nblk = total.
__global__ void __launch_bounds__(1024) k_csc_bscan(int nblk, int32_t* bsum) {
  __shared__ int wsum[32];
  const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int32_t* b = bsum + (int64_t)u * (kMaxBlocks + 1);
  const int v = tid < nblk ? b[tid] : 0;
  int x = v;
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  int before = 0;
  for (int i = 0; i < w; ++i) before += wsum[i];
  if (tid < nblk) b[tid] = before + x - v;
  if (tid == nblk - 1) b[nblk] = before + x;
}

// Per key: dV = sum of its partial rows in slot (= group) order, same for dK;
// fp32 sums. A problem split over several units carries fp32 running sums.
template <int D>
__global__ void __launch_bounds__(256) k_csc_reduce(const CscParams csc, int S, const UnitTable tab) {
  constexpr int E = D / 32;                          // elements per lane
  const int u = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + warp;
  if (j >= S) return;
  const int32_t* o = csc.off + (int64_t)u * (S + 1);
  const int32_t* bp = csc.bpre + (int64_t)u * (kMaxBlocks + 1);
  const int nblk = (S + 255) / 256;
  const int64_t a = tab.part_base[u] + bp[j >> 8] + o[j];
  const int64_t b = tab.part_base[u] + (j + 1 == S ? bp[nblk] : bp[(j + 1) >> 8] + o[j + 1]);
  const bool first = tab.flags[u] & 1, last = tab.flags[u] & 2;
  float sv[E], sk[E];
  const int64_t arow = (int64_t)j * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    sv[e] = first ? 0.f : csc.acc_v[arow + e];
    sk[e] = first ? 0.f : csc.acc_k[arow + e];
  }
  // slots are summed one after the other in ascending order; the rows of the
  // next kBatch slots are loaded first so that more of them are in flight
  constexpr int kBatch = 8;
  auto add_row = [&](const uint32_t (&xv)[E / 2], const uint32_t (&xk)[E / 2]) {
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv[e]));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xk[e]));
      sv[2 * e] += x.x;
      sv[2 * e + 1] += x.y;
      sk[2 * e] += y.x;
      sk[2 * e + 1] += y.y;
    }
  };
  // one 8-byte (d = 128) or 4-byte (d = 64) load per lane and tensor
  auto load_row = [&](int64_t slot, uint32_t (&xv)[E / 2], uint32_t (&xk)[E / 2]) {
    const __nv_bfloat16* pv = csc.part_v + slot * D + lane * E;
    const __nv_bfloat16* pk = csc.part_k + slot * D + lane * E;
    if constexpr (E == 4) {
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(pv)), c = __ldg(reinterpret_cast<const uint2*>(pk));
      xv[0] = a.x;
      xv[1] = a.y;
      xk[0] = c.x;
      xk[1] = c.y;
    } else {
      xv[0] = __ldg(reinterpret_cast<const uint32_t*>(pv));
      xk[0] = __ldg(reinterpret_cast<const uint32_t*>(pk));
    }
  };
  auto batch = [&](auto n, int64_t s) {   // n slots from s: all loads, then the adds in order
    constexpr int N = decltype(n)::value;
    uint32_t xv[N][E / 2], xk[N][E / 2];
#pragma unroll
    for (int i = 0; i < N; ++i) load_row(s + i, xv[i], xk[i]);
#pragma unroll
    for (int i = 0; i < N; ++i) add_row(xv[i], xk[i]);
  };
  int64_t s = a;
  for (; s + kBatch <= b; s += kBatch) batch(std::integral_constant<int, kBatch>{}, s);
  if (s + 4 <= b) {   // the ragged end: at most one batch of four, one of two and one slot
    batch(std::integral_constant<int, 4>{}, s);
    s += 4;
  }
  if (s + 2 <= b) {
    batch(std::integral_constant<int, 2>{}, s);
    s += 2;
  }
  if (s < b) batch(std::integral_constant<int, 1>{}, s);
  if (last) {
    const int64_t orow = ((int64_t)tab.p[u] * S + j) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      *reinterpret_cast<__nv_bfloat162*>(csc.dV + orow + e) = __floats2bfloat162_rn(sv[e], sv[e + 1]);
      *reinterpret_cast<__nv_bfloat162*>(csc.dK + orow + e) = __floats2bfloat162_rn(sk[e], sk[e + 1]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      csc.acc_v[arow + e] = sv[e];
      csc.acc_k[arow + e] = sk[e];
    }
  }
}

template <int D>
static cudaError_t launch_bwd_q(const AttnMaps& maps, const CUtensorMap& do_cube, const AttnParams& prm,
                                const CscParams& csc, const UnitTable& tab, int max_ng, cudaStream_t st) {
  k_attn_bwd_q<D><<<dim3(max_ng, tab.n), kBwdQThreads, BwdCfg<D>::kSmem, st>>>(maps, do_cube, prm, csc, tab);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_bwd_dq(const AttnMaps& maps, const CUtensorMap& do_cube, const AttnParams& prm,
                                const float* delta, const UnitTable& tab, int max_ng, cudaStream_t st) {
  k_attn_bwd_dq<D><<<dim3(max_ng, tab.n), kBwdThreads, DqCfg<D>::kSmem, st>>>(maps, do_cube, prm, delta, tab);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_bwd_kv(const AttnMaps& maps, const CUtensorMap& q_tile, const CUtensorMap& do_tile,
                                 const AttnParams& prm, const float* delta, const float* lse2, __nv_bfloat16* dK,
                                 __nv_bfloat16* dV, const ProblemTable& tab, int S, cudaStream_t st) {
  k_attn_bwd_kv<D><<<dim3(S / 128, tab.n), kBwdThreads, KvCfg<D>::kSmem, st>>>(maps, q_tile, do_tile, prm, delta,
                                                                                lse2, dK, dV, tab);
  return cudaGetLastError();
}

template <int D>
static cudaError_t configure_bwd() {
  static bool done = false;
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_attn_bwd_q<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_attn_bwd_kv<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_attn_bwd_dq<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmem);
  // The warpgroups' register shares add up to kBwdQLaunchRegs per thread; a
  // build that launched with any other count would never satisfy the softmax
  // warpgroup's increase, so it is refused here instead of launched.
  // the slot-map bitmap of a 256-key block: up to S / 64 groups, 32 per word
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_csc_build, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kCscStride * (256 * kMaxBlocks / 64 / 32) * (int)sizeof(uint32_t));
  cudaFuncAttributes a;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, k_attn_bwd_q<D>);
  if (e == cudaSuccess && a.numRegs != kBwdQLaunchRegs) e = cudaErrorInvalidConfiguration;
  if (e == cudaSuccess) done = true;
  return e;
}

// ---------------------------------------------------------------------------
// Host planning: units, launches and workspace.
struct BwdPlan {
  std::vector<UnitTable> launches;   // sparse problems (partials)
  UnitTable dense;                   // dense problems (dQ only)
  int max_ng = 1;                    // largest unit (grid x of the group-major launches)
  size_t slots = 0;                  // partial slots needed by the largest launch
  size_t bits_words = 0;             // bitmap words needed by the largest launch
  bool split = false;                // some problem spans several units
};

// Units and launches for a budget of bf16 partial bytes in flight per launch.
static BwdPlan plan_bwd(const dsv_shape& shape, const Geometry& geo, bool any_sparse, const int32_t* k_per_head,
                        const int64_t* idx_offset, size_t budget = kPartialBudget) {
  BwdPlan pl;
  memset(&pl.dense, 0, sizeof(pl.dense));
  const int P = (int)(shape.B * shape.H);
  const size_t slot_bytes = (size_t)shape.d * 2 * sizeof(__nv_bfloat16);
  const size_t cap = std::max<size_t>(1, budget / slot_bytes);
  UnitTable cur;
  memset(&cur, 0, sizeof(cur));
  size_t cur_slots = 0, cur_words = 0;
  auto flush = [&]() {
    if (cur.n == 0) return;
    pl.launches.push_back(cur);
    pl.slots = std::max(pl.slots, cur_slots);
    pl.bits_words = std::max(pl.bits_words, cur_words);
    memset(&cur, 0, sizeof(cur));
    cur_slots = cur_words = 0;
  };
  auto add = [&](int p, int k, int64_t off, int g0, int ng, int flags) {
    const size_t slots = (size_t)ng * k;
    const int nw = (ng + 31) / 32;
    const size_t words = (size_t)geo.S * nw;
    if (cur.n == kMaxUnits || cur_slots + slots > cap || (flags != 3 && cur.n > 0)) flush();
    const int i = cur.n++;
    cur.p[i] = p;
    cur.k[i] = k;
    cur.g0[i] = g0;
    cur.ng[i] = ng;
    cur.nwords[i] = nw;
    cur.flags[i] = flags;
    cur.off[i] = off;
    cur.part_base[i] = (int64_t)cur_slots;
    cur.bits_base[i] = (int64_t)cur_words;
    cur_slots += slots;
    cur_words += words;
    pl.max_ng = std::max(pl.max_ng, ng);
    if (flags != 3) flush();   // a unit of a split problem runs alone
  };
  for (int p = 0; p < P; ++p) {
    const bool dense = !any_sparse || idx_offset[p] < 0;
    if (dense) {
      const int i = pl.dense.n++;
      pl.dense.p[i] = p;
      pl.dense.k[i] = geo.S;
      pl.dense.g0[i] = 0;
      pl.dense.ng[i] = geo.n_groups;
      pl.dense.off[i] = -1;
      pl.dense.flags[i] = 3;
      continue;
    }
    const int k = k_per_head[p];
    const size_t pairs = (size_t)geo.n_groups * k;
    if (pairs <= cap) {
      add(p, k, idx_offset[p], 0, geo.n_groups, 3);
    } else {
      pl.split = true;
      const int per = (int)std::max<size_t>(1, cap / (size_t)k);
      for (int g0 = 0; g0 < geo.n_groups; g0 += per) {
        const int ng = std::min(per, geo.n_groups - g0);
        add(p, k, idx_offset[p], g0, ng, (g0 == 0 ? 1 : 0) | (g0 + ng == geo.n_groups ? 2 : 0));
      }
    }
  }
  flush();
  return pl;
}

struct BwdWs {
  __nv_bfloat16* part_v;
  __nv_bfloat16* part_k;
  uint64_t* bits;
  int32_t* off;
  int32_t* bpre;
  float* acc_v;
  float* acc_k;
  float* delta;
  float* lse2;
};

static size_t carve_bwd(void* base, const dsv_shape& s, const BwdPlan& pl, BwdWs* w) {
  Carver c(base);
  const size_t S = (size_t)(s.T * s.Y * s.X), P = (size_t)(s.B * s.H);
  w->part_v = c.take<__nv_bfloat16>(pl.slots * s.d);
  w->part_k = c.take<__nv_bfloat16>(pl.slots * s.d);
  w->bits = c.take<uint64_t>(pl.bits_words);
  w->off = c.take<int32_t>((size_t)kMaxUnits * (S + 1));
  w->bpre = c.take<int32_t>((size_t)kMaxUnits * (kMaxBlocks + 1));
  w->acc_v = c.take<float>(pl.split ? S * s.d : 0);
  w->acc_k = c.take<float>(pl.split ? S * s.d : 0);
  w->delta = c.take<float>(pl.dense.n ? P * S : 0);
  w->lse2 = c.take<float>(pl.dense.n ? P * S : 0);
  return c.used + 256;
}

}  // namespace dsv

using namespace dsv;

extern "C" size_t dsv_sparse_attn_bwd_workspace_size(dsv_shape shape, dsv_group group, const int32_t* k_per_head,
                                                     const int64_t* idx_offset) {
  if (validate_common(shape, group, true) != DSV_OK) return 0;
  const Geometry geo = make_geometry(shape, group);
  const int P = (int)(shape.B * shape.H);
  const bool any_sparse = k_per_head != nullptr;
  if (any_sparse && !idx_offset) return 0;
  if (any_sparse)
    for (int i = 0; i < P; ++i)
      if (idx_offset[i] >= 0 && (k_per_head[i] < 1 || k_per_head[i] > geo.S)) return 0;
  const BwdPlan pl = plan_bwd(shape, geo, any_sparse, k_per_head, idx_offset);
  BwdWs w;
  return carve_bwd(nullptr, shape, pl, &w);
}

extern "C" size_t dsv_sparse_attn_bwd_min_workspace_size(dsv_shape shape, dsv_group group,
                                                         const int32_t* k_per_head, const int64_t* idx_offset) {
  if (validate_common(shape, group, true) != DSV_OK) return 0;
  const Geometry geo = make_geometry(shape, group);
  const int P = (int)(shape.B * shape.H);
  const bool any_sparse = k_per_head != nullptr;
  if (any_sparse && !idx_offset) return 0;
  if (any_sparse)
    for (int i = 0; i < P; ++i)
      if (idx_offset[i] >= 0 && (k_per_head[i] < 1 || k_per_head[i] > geo.S)) return 0;
  // the smallest of the plans dsv_sparse_attn_bwd tries (budgets halving from
  // kPartialBudget to one query group per launch): any workspace at least this
  // large fits one of them
  const size_t slot_bytes = (size_t)shape.d * 2 * sizeof(__nv_bfloat16);
  size_t least = SIZE_MAX;
  for (size_t budget = kPartialBudget;; budget /= 2) {
    const BwdPlan pl = plan_bwd(shape, geo, any_sparse, k_per_head, idx_offset, budget);
    BwdWs w;
    least = std::min(least, carve_bwd(nullptr, shape, pl, &w));
    if (budget < slot_bytes) break;
  }
  return least;
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
  const Geometry geo = make_geometry(shape, group);
  const int P = (int)(shape.B * shape.H), d = (int)shape.d;
  if (idx)
    for (int i = 0; i < P; ++i) {
      if (idx_offset[i] < 0) continue;
      if (k_per_head[i] < 1 || k_per_head[i] > geo.S) return DSV_ERR_INVALID_ARG;
      if (geo.S > 256 * kMaxBlocks) return DSV_ERR_UNSUPPORTED;   // slot map covers S <= 2^18
    }
  if (!workspace || !aligned(workspace, 256)) return DSV_ERR_WORKSPACE;
  // The largest budget of partials in flight whose plan fits the workspace: a
  // smaller workspace only means more, smaller launches (a problem's groups
  // split over several, with fp32 running sums; the summation order, and so
  // every result bit, stays the same).
  BwdPlan pl;
  BwdWs w;
  bool fits = false;
  const size_t slot_bytes = (size_t)d * 2 * sizeof(__nv_bfloat16);
  for (size_t budget = kPartialBudget;; budget /= 2) {
    pl = plan_bwd(shape, geo, idx != nullptr, k_per_head, idx_offset, budget);
    if (carve_bwd(nullptr, shape, pl, &w) <= workspace_bytes) {
      fits = true;
      break;
    }
    if (budget < slot_bytes) break;   // one group per launch already
  }
  if (!fits) return DSV_ERR_WORKSPACE;
  carve_bwd(workspace, shape, pl, &w);
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
  prm.K = static_cast<const __nv_bfloat16*>(K);
  prm.V = static_cast<const __nv_bfloat16*>(V);
  prm.O = static_cast<const __nv_bfloat16*>(O);
  prm.dO = static_cast<const __nv_bfloat16*>(dO);
  prm.LSE = LSE;
  prm.out = static_cast<__nv_bfloat16*>(dQ);
  prm.status = dev_status;
  prm.wait_ns = wait_limit_ns();
  CscParams csc;
  memset(&csc, 0, sizeof(csc));
  csc.bits = w.bits;
  csc.off = w.off;
  csc.bpre = w.bpre;
  csc.part_v = w.part_v;
  csc.part_k = w.part_k;
  csc.acc_v = w.acc_v;
  csc.acc_k = w.acc_k;
  csc.dK = static_cast<__nv_bfloat16*>(dK);
  csc.dV = static_cast<__nv_bfloat16*>(dV);

  // sparse problems: dQ + ordered dK/dV
  for (const UnitTable& tab : pl.launches) {
    int max_ng = 1, max_nw = 1;
    for (int i = 0; i < tab.n; ++i) {
      max_ng = std::max(max_ng, tab.ng[i]);
      max_nw = std::max(max_nw, tab.nwords[i]);
    }
    k_csc_build<<<dim3((geo.S + kCscKeys - 1) / kCscKeys, tab.n), 256, (size_t)kCscStride * max_nw * sizeof(uint32_t),
                  st>>>(idx, w.bits, geo.S, w.off, w.bpre, tab);
    k_csc_bscan<<<tab.n, 1024, 0, st>>>((geo.S + 255) / 256, w.bpre);
    cudaError_t e = d == 128 ? launch_bwd_q<128>(maps, do_cube, prm, csc, tab, max_ng, st)
                             : launch_bwd_q<64>(maps, do_cube, prm, csc, tab, max_ng, st);
    if (e != cudaSuccess) return DSV_ERR_CUDA;
    if (d == 128) k_csc_reduce<128><<<dim3((geo.S + 7) / 8, tab.n), 256, 0, st>>>(csc, geo.S, tab);
    else k_csc_reduce<64><<<dim3((geo.S + 7) / 8, tab.n), 256, 0, st>>>(csc, geo.S, tab);
    if (cudaGetLastError() != cudaSuccess) return DSV_ERR_CUDA;
  }
  // dense problems: dQ group-major, dK/dV key-major
  if (pl.dense.n) {
    ProblemTable ptab;
    memset(&ptab, 0, sizeof(ptab));
    ptab.n = pl.dense.n;
    for (int i = 0; i < ptab.n; ++i) {
      ptab.p[i] = pl.dense.p[i];
      ptab.k[i] = geo.S;
      ptab.off[i] = -1;
    }
    k_bwd_delta<<<dim3((unsigned)(((int64_t)geo.S * (d / 8) + 255) / 256), ptab.n), 256, 0, st>>>(
        prm.O, prm.dO, geo.S, d, w.delta, prm.LSE, w.lse2, ptab);
    if (cudaGetLastError() != cudaSuccess) return DSV_ERR_CUDA;
    for (int c0 = 0; c0 < pl.dense.n; c0 += kMaxUnits) {
      UnitTable dt = pl.dense;
      dt.n = std::min(kMaxUnits, pl.dense.n - c0);
      for (int i = 0; i < dt.n; ++i) {
        dt.p[i] = pl.dense.p[c0 + i];
        dt.k[i] = geo.S;
        dt.g0[i] = 0;
        dt.ng[i] = geo.n_groups;
        dt.off[i] = -1;
      }
      cudaError_t e = d == 128 ? launch_bwd_dq<128>(maps, do_cube, prm, w.delta, dt, geo.n_groups, st)
                               : launch_bwd_dq<64>(maps, do_cube, prm, w.delta, dt, geo.n_groups, st);
      if (e != cudaSuccess) return DSV_ERR_CUDA;
    }
    const cudaError_t e =
        d == 128 ? launch_bwd_kv<128>(maps, q_tile, do_tile, prm, w.delta, w.lse2, csc.dK, csc.dV, ptab, geo.S, st)
                 : launch_bwd_kv<64>(maps, q_tile, do_tile, prm, w.delta, w.lse2, csc.dK, csc.dV, ptab, geo.S, st);
    if (e != cudaSuccess) return DSV_ERR_CUDA;
  }
  return DSV_OK;
}
