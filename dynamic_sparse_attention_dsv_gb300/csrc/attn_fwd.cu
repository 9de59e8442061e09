// Query-grouped sparse attention, forward pass.
//
// "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video DiT
// Training" (gist.science technical summary): section 2.1 computes full
// attention on the critical KV pairs only; section 2.2 groups adjacent
// queries so a group shares one key index set. The dense case (FlashAttention
// in stage 1, or a head the dispatcher keeps dense) is the same kernel over
// all S keys.
//
// One CTA per (query group, problem). The group's G (64 or 128) queries form
// the M = 128 rows of every MMA (G = 64 leaves rows 64..127 zero). Per
// 128-key tile:
//   cp.async row gather of the selected K and V rows into swizzled shared memory
//   S  = Q K^T        tcgen05.mma kind::f16, A = Q in TMEM (copied there once
//                     per CTA), B = K (smem) -> TMEM
//   P  = exp2(S*scale*log2e - m) in registers, written back to TMEM as bf16
//   O += P V          tcgen05.mma with A = P in TMEM, B = V (MN-major) -> TMEM
// The running max m is raised lazily (only when it grows by more than 8 in
// log2 units, which bounds P by 2^8), so O is rescaled rarely.
//
// Warps 0-7: softmax and epilogue, two warps per query row (TMEM lane): warp
// w takes key columns 64*(w/4) .. +63 of the rows in lane quarter w%4 and
// half of O's columns; the pair exchanges its partial row maxima (and row
// sums at the end) through shared memory. Warps 8-11 and 13-15: producers
// (cp.async row gather of the selected K/V rows, which bounds the kernel, so
// seven warps issue them; TMA boxes for dense tiles and the query cube).
// Warp 12: MMA issuer. The four warpgroups rebalance their registers after
// launch (softmax up, the rest down).
#include "attn_common.cuh"

namespace dsv {

template <int D>
struct FwdCfg {
  static constexpr int kStages = D == 128 ? 3 : 4;
  static constexpr int kTile = 128 * D * 2;            // bytes of one 128-row bf16 tile
  static constexpr int kOffK = kTile;                  // Q first
  static constexpr int kOffV = kOffK + kStages * kTile;
  static constexpr int kOffBar = kOffV + kStages * kTile;   // barriers; pair status flags at +192
  static constexpr int kOffX = kOffBar + 256;                // [2 halves][128 rows] fp32 exchange
  static constexpr int kSmemUsed = kOffX + 1024 + 1024;
  // at least half the SM's shared memory, so one CTA owns the SM's TMEM
  static constexpr int kSmem = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
  static constexpr int kGatherW = 7;                   // producer warps: 8-11 and 13-15
  static constexpr int kThreads = 512;
  static constexpr int kLaunchRegs = 128;              // 16384 / (4 warps x 32 lanes) per SM sub-partition
  static constexpr int kRegsSoftmax = 168, kRegsLoad = 96, kRegsMma = 80;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;               // S buffers at 0 and 128
  static constexpr uint32_t kColQ = 384;               // Q as bf16 pairs, D/2 columns
};

static_assert(FwdCfg<128>::kSmemUsed <= 232448 && FwdCfg<64>::kSmemUsed <= 232448, "forward exceeds shared memory");
static_assert(FwdCfg<128>::kOffX == FwdCfg<128>::kOffBar + 256, "status flags live in the barrier block");
static_assert(2 * FwdCfg<128>::kRegsSoftmax + FwdCfg<128>::kRegsLoad + FwdCfg<128>::kRegsMma ==
                  4 * FwdCfg<128>::kLaunchRegs,
              "register split must equal the launch");

template <int D>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1)
    k_attn_fwd(const __grid_constant__ AttnMaps maps, const AttnParams prm, const ProblemTable tab) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;
  uint8_t* sK = sm + C::kOffK;
  uint8_t* sV = sm + C::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;                  // [kStages <= 4]
  uint64_t* v_full = bars + 5;                  // [kStages]
  uint64_t* kv_empty = bars + 9;                // [kStages]
  uint64_t* s_full = bars + 13;                 // [2]
  uint64_t* p_full = bars + 15;                 // [2]
  uint64_t* o_ready = bars + 17;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 18);
  uint64_t* q_tm = bars + 19;                   // Q copied into TMEM by the eight softmax warps
  uint64_t* mma_done = bars + 20;               // every MMA issued has completed (unwind)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, lp = blockIdx.y;
  const int p = tab.p[lp];
  const Geometry& geo = prm.geo;
  const bool dense = (prm.idx == nullptr) || (tab.off[lp] < 0);
  const int k = dense ? geo.S : tab.k[lp];
  const int nt = (k + 127) / 128;
  const int32_t* idx_row = dense ? nullptr : prm.idx + tab.off[lp] + (int64_t)g * k;
  const int G = geo.G;

  // rows G..127 of Q stay zero (G = 64)
  if (G < 128) {
    for (int i = tid; i < (128 - G) * (D / 64) * 8; i += blockDim.x) {
      const int a = i / ((128 - G) * 8), rem = i % ((128 - G) * 8);
      reinterpret_cast<uint4*>(sQ + a * 16384 + G * 128)[rem] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  constexpr int kProdWarp = 8, kMmaWarp = 12;
  constexpr int W = C::kGatherW;
  if (warp == kMmaWarp) {
    tmem_alloc(tslot, C::kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(q_full, 1);
    const uint32_t fills = dense ? 1u : 32u * W;   // TMA tx arrival, or one per gathering lane
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(k_full + i, fills);
      mbar_init(v_full + i, fills);
      mbar_init(kv_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 8);
    }
    mbar_init(o_ready, 1);
    mbar_init(q_tm, 8);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  // ------------------------------------------------------------- producers
  // Producers leave only once their own copies have landed (a timed-out
  // pipeline may not have consumed them): cp.async by waiting for all of this
  // thread's copies, TMA by waiting for the last phase of each barrier armed.
  auto produce = [&](const int pw) {
    const int ct = g / (geo.ncy * geo.ncx), cy = (g / geo.ncx) % geo.ncy, cx = g % geo.ncx;
    if (pw == 0 && lane == 0) {
      prefetch_tmap(&maps.q_cube);
      mbar_arrive_expect_tx(q_full, G * D * 2);
      for (int a = 0; a < D / 64; ++a)
        tma_load_4d(sQ + a * 16384, &maps.q_cube, q_full, a * 64, cx * geo.gx, cy * geo.gy, p * geo.T + ct * geo.gt);
    }
    const int prow0 = p * geo.S;
    if (idx_row) {
      int rows[Gather<D, W>::kIters], nxt[Gather<D, W>::kIters];
      gather_rows<D, W>(nxt, idx_row, k, 0, prow0, pw, lane);
      for (int t = 0; t < nt; ++t) {
        const int s = t % C::kStages;
#pragma unroll
        for (int i = 0; i < Gather<D, W>::kIters; ++i) rows[i] = nxt[i];
        if (t + 1 < nt) gather_rows<D, W>(nxt, idx_row, k, t + 1, prow0, pw, lane);
        if (t >= C::kStages && !mbar_wait_warp(kv_empty + s, ((t / C::kStages) - 1) & 1, prm.wait_ns)) {
          if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
          break;
        }
        gather_tile<D, W>(sK + s * C::kTile, prm.K, rows, pw, lane);
        cp_async_arrive_noinc(k_full + s);
        gather_tile<D, W>(sV + s * C::kTile, prm.V, rows, pw, lane);
        cp_async_arrive_noinc(v_full + s);
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (pw == 0) {
      int issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int s = t % C::kStages;
        if (t >= C::kStages && !mbar_wait_warp(kv_empty + s, ((t / C::kStages) - 1) & 1, prm.wait_ns)) {
          if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(k_full + s, C::kTile);
          load_dense_tile<D>(sK + s * C::kTile, &maps.k_tile, k_full + s, t, prow0);
          mbar_arrive_expect_tx(v_full + s, C::kTile);
          load_dense_tile<D>(sV + s * C::kTile, &maps.v_tile, v_full + s, t, prow0);
        }
        issued = t + 1;
      }
      if (lane == 0)
        for (int t = max(0, issued - C::kStages); t < issued; ++t) {
          mbar_wait(k_full + t % C::kStages, (t / C::kStages) & 1, kDrainLimitNs);
          mbar_wait(v_full + t % C::kStages, (t / C::kStages) & 1, kDrainLimitNs);
        }
    }
    if (pw == 0 && lane == 0) mbar_wait(q_full, 0, kDrainLimitNs);
  };
  if (warp >= kProdWarp && warp < kMmaWarp) {
    setmaxnreg_dec<C::kRegsLoad>();
    produce(warp - kProdWarp);
  } else if (warp > kMmaWarp) {
    setmaxnreg_dec<C::kRegsMma>();   // the same instruction as warp 12 (one warpgroup)
    produce(warp - kMmaWarp - 1 + (kMmaWarp - kProdWarp));
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA (warp 12)
    setmaxnreg_dec<C::kRegsMma>();
    if (lane == 0) {
      constexpr uint32_t idesc_qk = instr_desc(128, 128, 1, 0, 0);
      constexpr uint32_t idesc_pv = instr_desc(128, D, 1, 0, 1);
      // Q is read from TMEM: the shared-memory operand traffic of S = Q K^T halves
      bool ok = mbar_wait(q_tm, 0, prm.wait_ns);
      tc_fence_after();
      auto issue_pv = [&](int t) -> bool {
        const int s = t % C::kStages, b = t & 1;
        if (!mbar_wait(p_full + b, (t >> 1) & 1, prm.wait_ns)) return false;
        if (!mbar_wait(v_full + s, (t / C::kStages) & 1, prm.wait_ns)) return false;
        fence_proxy_async_smem();   // rows written by cp.async (generic proxy) -> tensor core reads
        tc_fence_after();
        const uint64_t dv0 = smem_desc(smem_u32(sV + s * C::kTile), 16384, 1024);
        const uint32_t ta = tbase + b * 128, to = tbase + C::kColO;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f16_ts(to, ta + kk * 8, desc_at(dv0, kk * 2048), idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(kv_empty + s);
        mma_commit(o_ready);
        return true;
      };
      for (int t = 0; ok && t < nt; ++t) {
        const int s = t % C::kStages, b = t & 1;
        if (!mbar_wait(k_full + s, (t / C::kStages) & 1, prm.wait_ns)) { ok = false; break; }
        fence_proxy_async_smem();
        tc_fence_after();
        const uint64_t dk0 = smem_desc(smem_u32(sK + s * C::kTile), 16, 1024);
        const uint32_t ts = tbase + b * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_f16_ts(ts, tbase + C::kColQ + kk * 8, desc_at(dk0, off), idesc_qk, kk > 0);
        }
        mma_commit(s_full + b);
        if (t >= 1 && !issue_pv(t - 1)) { ok = false; break; }
      }
      if (ok && nt > 0) ok = issue_pv(nt - 1);
      if (!ok) raise_status(prm.status, DSV_ERR_TIMEOUT);
      // every MMA issued completes before TMEM is released
      mma_commit(mma_done);
      mbar_wait(mma_done, 0, kDrainLimitNs);
    }
  } else {
    // ----------------------------------------------------- softmax (warps 0-7)
    setmaxnreg_inc<C::kRegsSoftmax>();
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tbase + ((uint32_t)(quarter * 32) << 16);
    const uint32_t pair_bar = 1 + quarter;   // named barrier of warps quarter and quarter + 4
    float* xch = reinterpret_cast<float*>(sm + C::kOffX);
    volatile int* xok = reinterpret_cast<volatile int*>(sm + C::kOffBar + 192);
    // Publishes v (and this warp's status), returns the partner's v; both warps
    // leave with the same status. The second barrier keeps the next exchange
    // from overwriting a value the partner has not read yet.
    auto exchange = [&](float v, bool& ok_io) -> float {
      xch[half * 128 + row] = v;
      if (lane == 0) xok[half * 4 + quarter] = ok_io ? 1 : 0;
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
      const float other = xch[(half ^ 1) * 128 + row];
      ok_io = ok_io && xok[(half ^ 1) * 4 + quarter] != 0;
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
      return other;
    };
    constexpr int kOChunks = D / 64;   // 32-column chunks of O per warp
    const float sc = prm.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = mbar_wait_warp(q_full, 0, prm.wait_ns);
    {
      // this warp's 32 rows of Q, half of the columns, from the swizzled tile into TMEM
      constexpr int kQc = D / 16;   // 16-byte chunks
      uint32_t qv[kQc * 4];
#pragma unroll
      for (int c = 0; c < kQc; ++c) {
        const int cg = half * kQc + c, atom = cg >> 3, c8 = cg & 7;
        const uint4 v = *reinterpret_cast<const uint4*>(sQ + atom * 16384 + row * 128 + ((c8 ^ (row & 7)) << 4));
        qv[4 * c] = v.x;
        qv[4 * c + 1] = v.y;
        qv[4 * c + 2] = v.z;
        qv[4 * c + 3] = v.w;
      }
      if (ok) {
        if constexpr (D == 128) tmem_st32(lane_addr + C::kColQ + half * (D / 4), qv);
        else tmem_st16(lane_addr + C::kColQ + half * (D / 4), qv);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_tm);
    }
    for (int t = 0; t < nt; ++t) {
      const int b = t & 1;
      ok = ok && mbar_wait_warp(s_full + b, (t >> 1) & 1, prm.wait_ns);
      tc_fence_after();
      uint32_t r[2][32];
      tmem_ld32(lane_addr + b * 128 + half * 64, r[0]);
      tmem_ld32(lane_addr + b * 128 + half * 64 + 32, r[1]);
      tmem_ld_wait(r[0]);
      reg_fence(r[1]);
      const int nvalid = min(128, k - t * 128) - half * 64;   // valid columns of this warp's half
      const bool full = nvalid >= 64;   // every tile but a group's last
      float mx = -INFINITY;
      if (full) {
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // independent chains
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            m4[e >> 3 & 3] = max3f(m4[e >> 3 & 3], __uint_as_float(r[c][e]), __uint_as_float(r[c][e + 1]));
        mx = fmaxf(max3f(m4[0], m4[1], m4[2]), m4[3]);
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e < nvalid) mx = fmaxf(mx, __uint_as_float(r[c][e]));
      }
      float mt = mx * sc;   // sc > 0
      mt = fmaxf(mt, exchange(mt, ok));
      if (!ok) break;   // both warps of the pair leave at the same tile
      bool waited = false;
      const bool want = t > 0 && mt > m + 8.f;
      if (t == 0) {
        m = mt;
      } else if (__any_sync(0xffffffffu, want)) {
        // O must be quiescent: wait for PV(t-1), then rescale the rows whose
        // max grew (warp-collective TMEM access; other rows use factor 1)
        ok = ok && mbar_wait_warp(o_ready, (t - 1) & 1, prm.wait_ns);
        waited = true;
        const float f = want ? ex2_fast(m - mt) : 1.f;
        if (ok) {
          tc_fence_after();
#pragma unroll 1
          for (int c = half * kOChunks; c < (half + 1) * kOChunks; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_addr + C::kColO + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(lane_addr + C::kColO + c * 32, o);
          }
          tmem_st_wait();
        }
        l *= f;
        if (want) m = mt;
      }
      uint32_t pk[32];
      float lsum = 0.f;
      if (full) {
        // two-wide fp32 for the exponent argument and the running sum
        const uint64_t sc2 = f32x2(sc, sc), nm2 = f32x2(-m, -m);
        uint64_t ls2 = f32x2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[c][e]), __uint_as_float(r[c][e + 1])), sc2, nm2), x0, x1);
            const float p0 = ex2_fast(x0), p1 = ex2_fast(x1);
            ls2 = add_f32x2(ls2, f32x2(p0, p1));
            pk[(c * 32 + e) >> 1] = pack_bf16x2(p0, p1);
          }
        float l0, l1;
        f32x2_split(ls2, l0, l1);
        lsum = l0 + l1;
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int j = c * 32 + e;
            const float p0 = j < nvalid ? ex2_fast(__uint_as_float(r[c][e]) * sc - m) : 0.f;
            const float p1 = j + 1 < nvalid ? ex2_fast(__uint_as_float(r[c][e + 1]) * sc - m) : 0.f;
            lsum += p0 + p1;
            pk[j >> 1] = pack_bf16x2(p0, p1);
          }
      }
      l += lsum;
      // P of keys 64*half .. +63, packed two per column, in place of S
      tmem_st32(lane_addr + b * 128 + half * 32, pk);
      tmem_st_wait();
      if (t >= 1 && !waited) ok = ok && mbar_wait_warp(o_ready, (t - 1) & 1, prm.wait_ns);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + b);
    }
    // ---------------------------------------------------------- epilogue
    if (nt > 0) ok = ok && mbar_wait_warp(o_ready, (nt - 1) & 1, prm.wait_ns);
    l += exchange(l, ok);
    if (!ok) {
      if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
    } else if (row < G) {
      tc_fence_after();
      const int tok = token_of(geo, g, row);
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = prm.out + ((int64_t)p * geo.S + tok) * D;
#pragma unroll 1
      for (int c = half * kOChunks; c < (half + 1) * kOChunks; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + C::kColO + c * 32, o);
        tmem_ld_wait(o);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
      if (half == 0) prm.lse_out[(int64_t)p * geo.S + tok] = (m + __log2f(l)) * 0.69314718055994531f;
    } else {
      // padded rows still take part in the TMEM loads (warp-collective)
      tc_fence_after();
#pragma unroll 1
      for (int c = half * kOChunks; c < (half + 1) * kOChunks; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + C::kColO + c * 32, o);
        tmem_ld_wait(o);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tbase, C::kTmemCols);
}

template <int D>
static cudaError_t launch_fwd(const AttnMaps& maps, const AttnParams& prm, const ProblemTable& tab, int n_groups,
                              cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(k_attn_fwd<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<D>::kSmem);
    if (e != cudaSuccess) return e;
    // The warpgroups' register shares add up to kLaunchRegs per thread; a build
    // that launched with another count would stall the softmax increase, so
    // it is refused instead of launched.
    cudaFuncAttributes a;
    e = cudaFuncGetAttributes(&a, k_attn_fwd<D>);
    if (e != cudaSuccess) return e;
    if (a.numRegs != FwdCfg<D>::kLaunchRegs) return cudaErrorInvalidConfiguration;
    configured = true;
  }
  k_attn_fwd<D><<<dim3(n_groups, tab.n), FwdCfg<D>::kThreads, FwdCfg<D>::kSmem, st>>>(maps, prm, tab);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// True attention mass of the selected keys. For query i the selected keys'
// share of its softmax over all keys is exp(LSE_sel,i - LSE_all,i), with both
// LSEs from the forward (on the index sets, and dense). One block per problem;
// the mean runs in fp64 in a fixed order (strided per-thread sums, then a
// fixed tree), so every run gives the same bits.
constexpr int kMassThreads = 256;

__global__ void __launch_bounds__(kMassThreads) k_attn_mass(const float* __restrict__ lse_sel,
                                                            const float* __restrict__ lse_all, int64_t S,
                                                            float* mass, float* per_query) {
  __shared__ double part[kMassThreads];
  const int p = blockIdx.x, tid = threadIdx.x;
  const float* a = lse_sel + (int64_t)p * S;
  const float* b = lse_all + (int64_t)p * S;
  double acc = 0.0;
  for (int64_t i = tid; i < S; i += kMassThreads) {
    const float m = expf(a[i] - b[i]);
    if (per_query) per_query[(int64_t)p * S + i] = m;
    acc += (double)m;
  }
  part[tid] = acc;
  __syncthreads();
  for (int w = kMassThreads / 2; w > 0; w >>= 1) {
    if (tid < w) part[tid] += part[tid + w];
    __syncthreads();
  }
  if (tid == 0) mass[p] = (float)(part[0] / (double)S);
}

}  // namespace dsv

using namespace dsv;

extern "C" size_t dsv_sparse_attn_fwd_workspace_size(dsv_shape shape, dsv_group group) {
  (void)shape;
  (void)group;
  return 0;
}

extern "C" dsv_status dsv_sparse_attn_fwd(const void* Q, const void* K, const void* V, const int32_t* idx,
                                          const int32_t* k_per_head, const int64_t* idx_offset, dsv_shape shape,
                                          dsv_group group, float scale, void* O, float* LSE, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_status, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  dsv_status v = validate_common(shape, group, true);
  if (v != DSV_OK) return v;
  if (!Q || !K || !V || !O || !LSE || !(scale > 0.f)) return DSV_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(LSE, 4))
    return DSV_ERR_INVALID_ARG;
  if (idx && (!k_per_head || !idx_offset || !aligned(idx, 4))) return DSV_ERR_INVALID_ARG;
  const Geometry geo = make_geometry(shape, group);
  const int P = (int)(shape.B * shape.H);
  const int d = (int)shape.d;
  ProblemTable tab;
  memset(&tab, 0, sizeof(tab));
  tab.n = P;
  for (int i = 0; i < P; ++i) {
    tab.p[i] = i;
    const bool dense = !idx || idx_offset[i] < 0;
    tab.k[i] = dense ? geo.S : k_per_head[i];
    tab.off[i] = dense ? -1 : idx_offset[i];
    if (!dense && (tab.k[i] < 1 || tab.k[i] > geo.S)) return DSV_ERR_INVALID_ARG;
  }
  AttnMaps maps;
  if (!make_attn_maps(&maps, Q, K, V, geo, d, P)) return DSV_ERR_CUDA;
  AttnParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.geo = geo;
  prm.d = d;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.idx = idx;
  prm.K = static_cast<const __nv_bfloat16*>(K);
  prm.V = static_cast<const __nv_bfloat16*>(V);
  prm.out = static_cast<__nv_bfloat16*>(O);
  prm.lse_out = LSE;
  prm.status = dev_status;
  prm.wait_ns = wait_limit_ns();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d == 128 ? launch_fwd<128>(maps, prm, tab, geo.n_groups, st)
                                 : launch_fwd<64>(maps, prm, tab, geo.n_groups, st);
  return e == cudaSuccess ? DSV_OK : DSV_ERR_CUDA;
}

extern "C" dsv_status dsv_attn_mass(const float* LSE_sel, const float* LSE_all, int64_t S, int32_t P, float* mass,
                                    float* per_query, void* stream) {
  if (!LSE_sel || !LSE_all || !mass || S < 1 || P < 1 || P > kMaxProblems) return DSV_ERR_INVALID_ARG;
  if (!aligned(LSE_sel, 4) || !aligned(LSE_all, 4) || !aligned(mass, 4) || (per_query && !aligned(per_query, 4)))
    return DSV_ERR_INVALID_ARG;
  k_attn_mass<<<P, kMassThreads, 0, static_cast<cudaStream_t>(stream)>>>(LSE_sel, LSE_all, S, mass, per_query);
  return cudaGetLastError() == cudaSuccess ? DSV_OK : DSV_ERR_CUDA;
}
