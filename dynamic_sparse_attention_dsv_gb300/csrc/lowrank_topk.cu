// Fused low-rank score + per-group top-k selection and predicted-mass coverage.
//
// Follows "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video
// DiT Training" (gist.science technical summary): section 2.1 (per-head
// low-rank predictors W_lr^Q, W_lr^K approximating QK^T; critical KV = the
// keys holding 90% of the attention mass) and section 2.2 (fused low-rank
// MatMul + Top-K that never stores the S x S scores; adjacent queries grouped
// to share one key set).
//
// Score of key j for group g: s_gj = qbar_g . k_lr,j with qbar_g the group
// mean of q_lr (equal to the mean of q_lr,i . k_lr,j by linearity). Scores are
// formed tile by tile on the tensor cores (tcgen05, kind::tf32, three products
// hi*hi + hi*lo + lo*hi of a tf32 hi/lo split: about 2^-21 relative error) into
// TMEM and consumed in registers; they are never written to memory.
//
// Exact top-k per group row, ties to the lower key, in streaming passes over
// the same score tiles plus small per-row kernels:
//   MINMAX  per-row score range
//   HIST    256 (128 for r=64) linear bins over the range; the bracket kernel
//           finds the bin holding the k-th largest score, i.e. an interval
//           [lo, hi) of orderable score bits, the count of scores >= hi and
//           the count inside the interval
//   REFINE  (only rows whose interval holds more than kCandCap scores) the
//           interval's scores binned again by their next 8 (7 for r=64)
//           orderable bits; at most four (five) rounds narrow any interval to
//           at most kCandCap scores or to a single value, so no input can
//           overflow the candidate buffer. Rounds with nothing to refine exit
//           at once.
//   COLLECT marks every key scoring >= hi in a per-row bit mask and stages the
//           interval's scores as candidates (a single-valued interval marks
//           its keys in a tie mask instead)
//   resolve selects the candidates that complete each row's k (score desc,
//           key asc) by a radix select and marks them
//   compact writes each index row in ascending key order from the masks,
//           taking a single-valued interval's keys lowest first.
// Coverage reuses MINMAX: a COV pass bins every key by log-probability below
// the row maximum (count per half bin and mass per bin), bound searches over
// those tables give an interval for k_cov, a COV_FINE pass re-bins each
// group's window of coarse bins, and a final search on the combined tables
// gives k_cov. When coverage and top-k run in one call, the COV pass's half-bin
// counts give the bracket in place of the HIST pass.
#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "attn_common.cuh"

namespace dsv {

constexpr int kSelThreads = 320;   // warps 0-7 consume scores, 8 loads tiles, 9 issues MMAs
constexpr int kCandCap = 4096;     // candidates kept per group row
constexpr int kMaxChunks = 64;     // key chunks per row
// Problems per launch: as many as keep the projected keys within this budget.
// Fewer, larger launches beat keeping the projections L2-resident: the score
// passes are bound by their consumers, and every extra launch of the pass
// chain costs its ramp-up and tail.
constexpr size_t kProjBudget = 1ull << 30;

enum SelMode { kMinMax = 0, kHist = 1, kCollect = 2, kRefine = 3, kCov = 4, kCovFine = 5, kMass = 6 };

// Per-row state of the boundary interval after each bracket step.
enum RowState { kRowCollect = 0, kRowRefine = 1, kRowTied = 2 };

template <int RP>
struct SelCfg {
  static constexpr int kAtoms = RP / 32;               // 128-byte atoms per fp32 row
  static constexpr int kTileBytes = 128 * RP * 4;      // one [128][RP] fp32 tile
  static constexpr int kStages = (RP == 32) ? 2 : 1;
  static constexpr int kHistBins = (RP == 32) ? 256 : 128;
  static constexpr int kHistLog2 = (RP == 32) ? 8 : 7;
  static constexpr int kCovBins = (RP == 32) ? 128 : 64;
  static constexpr int kHistBytes = 128 * 1024 / (RP / 32);
  // Coverage bins (coarse or fine) in the histogram area: 32-bit counts
  // ([bin][row]) at 0, then 32-bit fixed-point masses ([bin][row]).
  static constexpr int kCovMassOff = kCovBins * 128 * 4;
  static_assert(2 * kCovMassOff <= kHistBytes, "coverage counts and masses fit the histogram area");
  static constexpr int kOffAlo = kTileBytes;
  static constexpr int kOffB = 2 * kTileBytes;
  static constexpr int kOffHist = kOffB + kStages * 2 * kTileBytes;
  static constexpr int kOffMisc = kOffHist + kHistBytes;
  static constexpr int kSmem = kOffMisc + 256 + 1024;  // + barriers, + alignment slack
  // MINMAX and MASS keep no histogram: a 2 KB exchange area, then the barriers,
  // so two blocks share an SM and one's start and finish overlap the other's work
  static constexpr int kOffMiscSmall = kOffHist + 2048;
  static constexpr int kSmemSmall = kOffMiscSmall + 256 + 1024;
  // all but MINMAX and MASS keep a histogram area
  __host__ __device__ static constexpr bool big(int mode) { return mode != kMinMax && mode != kMass; }
  __host__ __device__ static constexpr int smem(int mode) { return big(mode) ? kSmem : kSmemSmall; }
  __host__ __device__ static constexpr int off_misc(int mode) { return big(mode) ? kOffMisc : kOffMiscSmall; }
};

struct SelParams {
  Geometry geo;
  int32_t g_pad, n_chunks, chunk_tiles, n_tiles, n_gt;
  float scale;
  uint32_t* mmax;        // [n][g_pad] orderable max
  uint32_t* mmin;        // [n][g_pad] orderable min
  uint32_t* hist;        // HIST, REFINE, COVHIST: [n][bins][g_pad] top-k histogram
  uint32_t* cov_cnt;     // COV, COV_FINE (and fused): [n][chunks][bins][g_pad] coverage counts
  float* mass;           // COV, COV_FINE (and fused): [n][chunks][bins][g_pad] coverage masses
  const uint32_t* blo;   // [n][g_pad] boundary interval [blo, bhi) of orderable scores
  const uint32_t* bhi;
  const int32_t* rstate; // [n][g_pad] RowState
  const int32_t* tflag;  // REFINE: [n][n_gt] group tiles holding a row to refine
  uint32_t* cand_cnt;    // [n][g_pad]
  uint64_t* cand;        // [n][g_pad][kCandCap]
  uint32_t* sel_bits;    // [n][g_pad][n_tiles][4] keys scoring >= bhi, 32 keys per word
  uint32_t* eq_bits;     // same layout: keys inside a single-valued interval
  const int32_t* cwin;   // COV_FINE: [n][g_pad][4] window of coarse bins [wa, wb] and its score interval
                         // [lo, hi] as orderable bits
  // MASS (rows are single queries in group-major order):
  const uint32_t* qsel;  // [n][qn_groups][S/32] selection bitmap of each query group
  float* msum;           // [n][chunks][g_pad][2] per-row sums of exp(scale (s - max)): all keys, selected keys
  int32_t q_group, qn_groups;   // queries per group, groups per problem
  int32_t* status;
  uint64_t wait_ns;      // limit of each pipeline wait
};

__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

__device__ __forceinline__ void red_smem_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// COV bins count keys and sum their probabilities with 32-bit integer adds.
// Bin b of a row holds log-probabilities u in [b w, (b+1) w) below the row
// maximum, so each key adds q = exp(b w - u) in (exp(-w), 1] as 16.16 fixed
// point (relative precision 2^-17 whatever the probability's size); the bin's
// sum is scaled back by exp(-b w) afterwards. Integer sums are exact and
// order-independent. The counts are kept per half bin, two 16-bit counts to a
// word (low half: the bin's upper half in score, high half: its lower half),
// which gives the top-k bracket twice the coarse resolution at no extra
// shared memory. A chunk holds at most kCovMaxTiles * 128 (< 65536) keys of a
// row, so neither a half count nor the fixed-point sum overflows.
__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Bin of x >= 0 (x < 2^22): x - 1/2 rounded to the nearest integer by adding
// 1.5 * 2^23 and reading the integer bits (no float-to-int conversion, which
// issues at a quarter of the add rate). Equals floor(x) except at exact
// integers (ties to even); the map is monotone, and every pass that compares
// bins computes them with this same arithmetic, so they agree bit for bit.
constexpr float kRoundMagic = 12582912.f;   // 1.5 * 2^23
__device__ __forceinline__ float bin_round(float x) { return __fadd_rn(__fsub_rn(x, 0.5f), kRoundMagic); }
__device__ __forceinline__ int bin_of(float t, int nb) {
  return min(nb - 1, (int)(__float_as_uint(t) - __float_as_uint(kRoundMagic)));
}

// Linear bin of score s over [lo, lo + nb/inv_w); identical arithmetic in every
// place that uses it (no contraction), so the passes agree bit for bit. It is
// monotone in s: every step (subtract, multiply by inv_w >= 0, round, read the
// bits) preserves order.
__device__ __forceinline__ int lin_bin(float s, float lo, float inv_w, int nb) {
  return bin_of(bin_round(__fmul_rn(__fsub_rn(s, lo), inv_w)), nb);
}
// The histogram range of a row from its orderable score bounds.
__device__ __forceinline__ void lin_range(uint32_t mmin_ord, uint32_t mmax_ord, int nb, float* lo, float* inv_w) {
  *lo = ord2f(mmin_ord);
  const float hi = ord2f(mmax_ord);
  *inv_w = hi > *lo ? (float)nb / __fsub_rn(hi, *lo) : 0.f;
}

// Coverage's coarse bin of score s: log-probability below the row maximum
// u = scale (cmax - s), coordinate x = u inv_w, bin round(x - 1/2) clamped.
// One definition for the COV and COV_FINE passes and the window search, so
// they agree bit for bit; non-increasing in s.
__device__ __forceinline__ float cov_coord(float s, float cmax, float scale, float inv_w) {
  return __fmul_rn(__fmul_rn(scale, __fsub_rn(cmax, s)), inv_w);
}
// Coarse bin of coordinate x and its offset inside the bin (in [0, 1], more
// when clamped to the last bin); the half bin is 2 bin + (offset >= 1/2).
// Monotone in x, and the same arithmetic everywhere.
__device__ __forceinline__ int cov_bin(float x, int nb, float* frac) {
  const float t = bin_round(x);
  *frac = x - fminf(t - kRoundMagic, (float)(nb - 1));
  return bin_of(t, nb);
}
__device__ __forceinline__ void cov_row_scale(uint32_t mmax_ord, uint32_t mmin_ord, float scale, int nb, float* cmax,
                                              float* inv_w, float* w2) {
  *cmax = ord2f(mmax_ord);
  const float range = __fmul_rn(scale, __fsub_rn(*cmax, ord2f(mmin_ord)));
  *inv_w = range > 0.f ? __fdiv_rn((float)nb, range) : 0.f;
  *w2 = range > 0.f ? __fmul_rn(__fdiv_rn(range, (float)nb), 1.4426950408889634f) : 0.f;
}

// ---------------------------------------------------------------------------
// Score-tile pipeline with a per-mode consumer.
// grid = (group tiles, key chunks, problems); block = 320 threads.
// Two blocks per SM, except COV_FINE: its histogram area leaves room for one
// block, so its registers are not capped for two.
template <int RP, int MODE>
__global__ void __launch_bounds__(kSelThreads, MODE == kCovFine ? 1 : 2)
    k_select(const __grid_constant__ CUtensorMap map_qhi, const __grid_constant__ CUtensorMap map_qlo,
             const __grid_constant__ CUtensorMap map_khi, const __grid_constant__ CUtensorMap map_klo,
             const SelParams prm, const ProblemTable tab) {
  using C = SelCfg<RP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sAhi = sm;
  uint8_t* sAlo = sm + C::kOffAlo;
  uint8_t* sB = sm + C::kOffB;
  uint8_t* sHist = sm + C::kOffHist;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::off_misc(MODE));
  uint64_t* a_full = bars;
  uint64_t* b_full = bars + 1;            // [kStages]
  uint64_t* b_empty = bars + 3;           // [kStages]
  uint64_t* s_full = bars + 5;            // [2]
  uint64_t* s_empty = bars + 7;           // [2]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 10);
  uint64_t* mma_done = bars + 11;         // every MMA issued has completed (unwind)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gtile = blockIdx.x, chunk = blockIdx.y, lp = blockIdx.z;
  const int t0 = chunk * prm.chunk_tiles;
  const int nt = min(prm.chunk_tiles, prm.n_tiles - t0);
  const int S = prm.geo.S;
  // REFINE: group tiles without a row to refine leave before touching TMEM
  if constexpr (MODE == kRefine) {
    if (prm.tflag[lp * prm.n_gt + gtile] == 0) return;
  }

  if (warp == 9) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(a_full, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(b_full + i, 1);
      mbar_init(b_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(s_empty + i, 8);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nt > 0) {
      prefetch_tmap(&map_khi);
      prefetch_tmap(&map_klo);
      const int ya = lp * prm.g_pad + gtile * 128;
      mbar_arrive_expect_tx(a_full, 2 * C::kTileBytes);
      for (int a = 0; a < C::kAtoms; ++a) {
        tma_load_2d(sAhi + a * 16384, &map_qhi, a_full, a * 32, ya);
        tma_load_2d(sAlo + a * 16384, &map_qlo, a_full, a * 32, ya);
      }
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int s = i % C::kStages;
        if (i >= C::kStages && !mbar_wait(b_empty + s, ((i / C::kStages) - 1) & 1, prm.wait_ns)) {
          raise_status(prm.status, DSV_ERR_TIMEOUT);
          break;
        }
        uint8_t* bh = sB + s * 2 * C::kTileBytes;
        uint8_t* bl = bh + C::kTileBytes;
        const int yb = lp * S + (t0 + i) * 128;
        mbar_arrive_expect_tx(b_full + s, 2 * C::kTileBytes);
        for (int a = 0; a < C::kAtoms; ++a) {
          tma_load_2d(bh + a * 16384, &map_khi, b_full + s, a * 32, yb);
          tma_load_2d(bl + a * 16384, &map_klo, b_full + s, a * 32, yb);
        }
        issued = i + 1;
      }
      // the block leaves only once every copy it started has landed
      mbar_wait(a_full, 0, kDrainLimitNs);
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait(b_full + i % C::kStages, (i / C::kStages) & 1, kDrainLimitNs);
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idesc = instr_desc(128, 128, 2, 0, 0);
      const uint64_t dah0 = smem_desc(smem_u32(sAhi), 16, 1024), dal0 = smem_desc(smem_u32(sAlo), 16, 1024);
      bool ok = mbar_wait(a_full, 0, prm.wait_ns);
      for (int i = 0; ok && i < nt; ++i) {
        const int s = i % C::kStages, b = i & 1;
        if (!mbar_wait(b_full + s, (i / C::kStages) & 1, prm.wait_ns)) { ok = false; break; }
        if (i >= 2 && !mbar_wait(s_empty + b, ((i >> 1) - 1) & 1, prm.wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tbase + b * 128;
        const uint64_t ah = opaque(dah0), al = opaque(dal0);
        const uint64_t bh = smem_desc(smem_u32(sB + s * 2 * C::kTileBytes), 16, 1024);
        const uint64_t bl = desc_at(bh, C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < RP / 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_tf32_ss(d, desc_at(ah, off), desc_at(bh, off), idesc, kk > 0);
          mma_tf32_ss(d, desc_at(ah, off), desc_at(bl, off), idesc, 1);
          mma_tf32_ss(d, desc_at(al, off), desc_at(bh, off), idesc, 1);
        }
        mma_commit(b_empty + s);
        mma_commit(s_full + b);
      }
      if (!ok) raise_status(prm.status, DSV_ERR_TIMEOUT);
      // every MMA issued completes before TMEM is released
      mma_commit(mma_done);
      mbar_wait(mma_done, 0, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------- score consumers
    constexpr bool kCovPart = MODE == kCov;        // coverage coarse bins
    constexpr bool kFinePart = MODE == kCovFine;   // coverage fine bins
    constexpr bool kHistPart = MODE == kHist;      // top-k linear histogram
    constexpr bool kCollectPart = MODE == kCollect;
    constexpr bool kCovLike = kCovPart || kFinePart;
    constexpr int NBc = C::kCovBins;
    constexpr int NBh = C::kHistBins;
    const int q = warp & 3, half = warp >> 2;
    const int row = q * 32 + lane;
    const int g = gtile * 128 + row;
    const bool valid = g < prm.geo.n_groups;
    const int rid = lp * prm.g_pad + g;
    const uint32_t taddr_lane = tbase + ((uint32_t)(q * 32) << 16);

    float h_lo = 0.f, h_inv = 0.f, inv_w = 0.f, cmax = 0.f;
    float mx = -INFINITY, mn = INFINITY;
    // COLLECT stages candidates per (row, half) in the histogram area,
    // flushing kStage at a time
    constexpr int kStage = C::kHistBytes / (256 * 8);
    uint64_t* stage = reinterpret_cast<uint64_t*>(sHist) + (size_t)(half * 128 + row) * kStage;
    int n_st = 0;
    const uint32_t hist_base = smem_u32(sHist);
    const uint32_t cmass_base = hist_base + C::kCovMassOff;

    // COLLECT: scores >= t_above are selected, [t_in, t_above) is the boundary
    // interval; REFINE: the interval [olo, olo + owid) of orderable scores,
    // binned by (o - olo) >> oshift
    float t_in = INFINITY, t_above = INFINITY;
    uint32_t olo = 0, owid = 0, oshift = 0;
    int state = kRowCollect;
    if constexpr (kHistPart) lin_range(prm.mmin[rid], prm.mmax[rid], NBh, &h_lo, &h_inv);
    if constexpr (kCollectPart || MODE == kRefine) {
      if (valid) {
        olo = prm.blo[rid];
        const uint32_t ohi = prm.bhi[rid];
        state = prm.rstate[rid];
        t_in = ord2f(olo);
        t_above = ord2f(ohi);
        owid = ohi - olo;
        const int bits = owid > 1u ? 32 - __clz(owid - 1u) : 0;
        oshift = (uint32_t)max(0, bits - C::kHistLog2);
      }
      if (MODE == kRefine && state != kRowRefine) owid = 0;   // this row takes no part
    }
    // MASS: this row's maximum score, the scale in log2 units, its group's
    // selection words and the running sums
    float m_sc = 0.f, m_all = 0.f, m_sel = 0.f;
    const uint32_t* m_bits = nullptr;
    if constexpr (MODE == kMass) {
      cmax = ord2f(prm.mmax[rid]);
      m_sc = prm.scale * 1.4426950408889634f;
      const int gq = min(g, prm.geo.S - 1) / prm.q_group;
      m_bits = prm.qsel + ((size_t)lp * prm.qn_groups + gq) * (size_t)(prm.geo.S / 32);
    }
    float w2 = 0.f;   // coverage: coarse bin width in log2 units
    // fine bins: the row's window of coarse bins [wa, wb], NBc fine bins over
    // it (fine coordinate (x - wa) * fscale, fine width fw2 in log2 units)
    int wa = NBc, wb = -1;
    float fscale = 0.f, fw2 = 0.f;
    float f_lo = INFINITY, f_hi = -INFINITY;   // the window's scores: [f_lo, f_hi]
    if constexpr (kCovLike) cov_row_scale(prm.mmax[rid], prm.mmin[rid], prm.scale, NBc, &cmax, &inv_w, &w2);
    if constexpr (kFinePart) {
      if (valid) {
        const int4 wv = *reinterpret_cast<const int4*>(prm.cwin + 4 * (size_t)rid);
        wa = wv.x;
        wb = wv.y;
        f_lo = ord2f((uint32_t)wv.z);
        f_hi = ord2f((uint32_t)wv.w);
      }
      const int nw = wb - wa + 1;
      fscale = nw > 0 ? (float)NBc / (float)nw : 0.f;
      fw2 = nw > 0 ? w2 * (float)nw / (float)NBc : 0.f;
    }
    if constexpr (C::big(MODE) && MODE != kCollect) {
      // zero this CTA's private histograms
      uint32_t* h = reinterpret_cast<uint32_t*>(sHist);
      for (int i = tid; i < C::kHistBytes / 4; i += 256) h[i] = 0;
      epi_barrier();
    }
    // writes the staged candidates of this (row, half) with one slot reservation
    auto flush = [&](int n) {
      const uint32_t slot0 = atomicAdd(prm.cand_cnt + rid, (uint32_t)n);
      for (int i = 0; i < n; ++i)
        if (slot0 + i < (uint32_t)kCandCap) prm.cand[(size_t)rid * kCandCap + slot0 + i] = stage[i];
    };

    for (int i = 0; i < nt; ++i) {
      const int b = i & 1;
      if (!mbar_wait_warp(s_full + b, (i >> 1) & 1, prm.wait_ns)) {
        if (lane == 0) raise_status(prm.status, DSV_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const int key0 = (t0 + i) * 128;
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(taddr_lane + b * 128 + half * 64, r0);
        tmem_ld32(taddr_lane + b * 128 + half * 64 + 32, r1);
        tmem_ld_wait(r0);
        reg_fence(r1);
        const int kb = key0 + half * 64;
        uint64_t selm = 0;   // MASS: selected columns of this half-tile
        if constexpr (MODE == kMass) selm = *reinterpret_cast<const uint64_t*>(m_bits + kb / 32);
        uint32_t gm_lo = 0, gm_hi = 0;   // COLLECT: columns scoring >= t_above
        uint32_t cm_lo = 0, cm_hi = 0;   // COLLECT: columns inside the boundary interval
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float s = __uint_as_float(e < 32 ? r0[e] : r1[e - 32]) + 0.0f;
          if constexpr (MODE == kMinMax) {
            mx = fmaxf(mx, s);
            mn = fminf(mn, s);
          }
          if constexpr (MODE == kMass) {
            const float ev = ex2_fast(__fmul_rn(__fsub_rn(s, cmax), m_sc));   // exp(scale (s - max)) in (0, 1]
            m_all += ev;
            m_sel += ((selm >> e) & 1ull) ? ev : 0.f;
          }
          if constexpr (kCovPart) {
            // coarse coordinate x and bin of the key's log-probability below
            // the row maximum; q = exp(b w - u) in (exp(-w), 1], as 16.16
            // fixed point through the float bits
            const float x = cov_coord(s, cmax, prm.scale, inv_w);
            float frac;
            const int bin = cov_bin(x, NBc, &frac);
            const float qv = ex2_fast(-frac * w2);
            const uint32_t qf = __float_as_uint(fmaf(qv, 65536.f, 8388608.f)) - __float_as_uint(8388608.f);
            // the count goes to the half bin: low half word below the middle, high half above
            red_smem_u32(hist_base + (uint32_t)(bin * 128 + row) * 4u, frac >= 0.5f ? 65536u : 1u);
            red_smem_u32(cmass_base + (uint32_t)(bin * 128 + row) * 4u, qf);
          }
          if constexpr (kFinePart) {
            // the window's keys, by two compares against its exact score
            // interval (the coarse binning is monotone); binned after the tile
            const bool in = s >= f_lo && s <= f_hi;
            if (e < 32) cm_lo |= (uint32_t)in << e;
            else cm_hi |= (uint32_t)in << (e - 32);
          }
          if constexpr (kHistPart) {
            const int bin = lin_bin(s, h_lo, h_inv, NBh);
            red_smem_u32(hist_base + (uint32_t)(bin * 128 + row) * 4u, 1u);
          }
          if constexpr (kCollectPart) {
            // branch-free here; the rare candidates are handled after the loop.
            // The thresholds are exact floats of the interval's orderable
            // bounds, so the float compares equal the orderable ones
            const bool above = s >= t_above, in = s >= t_in && !above;
            if (e < 32) {
              gm_lo |= (uint32_t)above << e;
              cm_lo |= (uint32_t)in << e;
            } else {
              gm_hi |= (uint32_t)above << (e - 32);
              cm_hi |= (uint32_t)in << (e - 32);
            }
          }
          if constexpr (MODE == kRefine) {
            const uint32_t dlt = f2ord(s) - olo;   // wraps above 2^31 for scores below the interval
            if (dlt < owid) red_smem_u32(hist_base + (uint32_t)((dlt >> oshift) * 128 + row) * 4u, 1u);
          }
        }
        if constexpr (kFinePart) {
          // one short loop per window key: its score picked out of r0/r1 by a
          // select chain, its fine bin (NBc bins over the window's width) and
          // q = exp(fb fw - u') in (exp(-fw), 1] added in shared memory
          uint64_t fm = valid ? ((uint64_t)cm_hi << 32 | cm_lo) : 0ull;
#pragma unroll 1
          while (fm) {
            const int e = __ffsll((long long)fm) - 1;
            fm &= fm - 1;
            const int u = e & 31;
            const bool hi = e >= 32;
            uint32_t v = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) v = (u == i) ? (hi ? r1[i] : r0[i]) : v;
            const float x = cov_coord(__uint_as_float(v) + 0.0f, cmax, prm.scale, inv_w);
            const float y = fmaxf(__fmul_rn(__fsub_rn(x, (float)wa), fscale), 0.f);
            const float ty = bin_round(y);
            const int fb = bin_of(ty, NBc);
            const float fy = y - fminf(ty - kRoundMagic, (float)(NBc - 1));   // in [0, 1], more when clamped
            const float qv = ex2_fast(-fy * fw2);
            const uint32_t qf = __float_as_uint(fmaf(qv, 65536.f, 8388608.f)) - __float_as_uint(8388608.f);
            red_smem_u32(hist_base + (uint32_t)(fb * 128 + row) * 4u, 1u);
            red_smem_u32(cmass_base + (uint32_t)(fb * 128 + row) * 4u, qf);
          }
        }
        if constexpr (kCollectPart) {
          if (valid) {
            const size_t wi = ((size_t)rid * prm.n_tiles + (t0 + i)) * 4 + half * 2;
            *reinterpret_cast<uint2*>(prm.sel_bits + wi) = make_uint2(gm_lo, gm_hi);
            // a single-valued interval: its keys are taken lowest first by the compaction
            if (state == kRowTied) *reinterpret_cast<uint2*>(prm.eq_bits + wi) = make_uint2(cm_lo, cm_hi);
          }
          // one short loop per candidate: pick the score out of r0/r1 with a
          // select chain (no dynamically indexed registers), stage the key
          uint64_t cm = (valid && state == kRowCollect) ? ((uint64_t)cm_hi << 32 | cm_lo) : 0ull;
#pragma unroll 1
          while (cm) {
            const int e = __ffsll((long long)cm) - 1;
            cm &= cm - 1;
            const int u = e & 31;
            const bool hi = e >= 32;
            uint32_t v = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) v = (u == i) ? (hi ? r1[i] : r0[i]) : v;
            const float sv = __uint_as_float(v) + 0.0f;
            if (n_st == kStage) {
              flush(kStage);
              n_st = 0;
            }
            stage[n_st++] = ((uint64_t)(~f2ord(sv)) << 32) | (uint32_t)(kb + e);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty + b);
    }

    // ----------------------------------------------------- per-row results
    if constexpr (kCollectPart) {
      if (valid && n_st > 0) flush(n_st);
    }
    if constexpr (MODE == kMass) {
      float* ex = reinterpret_cast<float*>(sHist);   // [2][2][128] exchange of the two halves' sums
      ex[(half * 2 + 0) * 128 + row] = m_all;
      ex[(half * 2 + 1) * 128 + row] = m_sel;
      epi_barrier();
      if (half == 0 && valid) {
        const size_t o = (((size_t)lp * prm.n_chunks + chunk) * prm.g_pad + g) * 2;
        prm.msum[o] = m_all + ex[(2 + 0) * 128 + row];
        prm.msum[o + 1] = m_sel + ex[(2 + 1) * 128 + row];
      }
    }
    if constexpr (MODE == kMinMax) {
      float* ex = reinterpret_cast<float*>(sHist);   // [2][2][128], the histogram area is unused here
      ex[(half * 2 + 0) * 128 + row] = mx;
      ex[(half * 2 + 1) * 128 + row] = mn;
      epi_barrier();
      if (half == 0 && valid && nt > 0) {
        const float m2 = fmaxf(mx, ex[(2 + 0) * 128 + row]);
        const float n2 = fminf(mn, ex[(2 + 1) * 128 + row]);
        atomicMax(prm.mmax + rid, f2ord(m2));
        atomicMin(prm.mmin + rid, f2ord(n2));
      }
    }
    if constexpr (C::big(MODE) && MODE != kCollect) epi_barrier();
    if constexpr (kCovLike) {
      const uint32_t* h = reinterpret_cast<const uint32_t*>(sHist);
      const uint32_t* m = reinterpret_cast<const uint32_t*>(sHist + C::kCovMassOff);
      // a bin's probabilities were summed relative to its upper edge
      const float edge0 = kFinePart ? (float)wa * w2 : 0.f;
      const float step = kFinePart ? fw2 : w2;
      for (int bin = half * (NBc / 2); bin < (half + 1) * (NBc / 2); ++bin) {
        const size_t o = (((size_t)lp * prm.n_chunks + chunk) * NBc + bin) * prm.g_pad + g;
        prm.cov_cnt[o] = h[bin * 128 + row];
        prm.mass[o] = (float)m[bin * 128 + row] * (1.f / 65536.f) * ex2_fast(-(edge0 + (float)bin * step));
      }
    }
    if constexpr (kHistPart || MODE == kRefine) {
      const uint32_t* h = reinterpret_cast<const uint32_t*>(sHist);
      for (int bin = half * (NBh / 2); bin < (half + 1) * (NBh / 2); ++bin) {
        const uint32_t v = h[bin * 128 + row];
        if (v) atomicAdd(prm.hist + ((size_t)lp * NBh + bin) * prm.g_pad + g, v);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tbase, 256);
}

// ---------------------------------------------------------------------------
// Low-rank projections.
// k_lr of every key, split into tf32 hi and lo parts; rows padded to RP.
// One 128-key tile per block on the tensor cores: TMA brings the K tile
// (128-byte swizzled atoms), the block writes W^T (RP rows of d, zero rows
// past r) in the same K-major layout, one thread issues the d/16 MMAs
// (128 x RP x 16, bf16 in, fp32 accumulation in TMEM; bf16 products are exact
// in fp32), and each thread reads its key's row back and stores hi/lo.
template <int RP>
struct ProjCfg {
  static constexpr int kATile = 128 * 128 * 2;        // K tile, d <= 128
  static constexpr int kOffB = kATile;                // W^T: RP rows x d
  static constexpr int kOffBar = kOffB + RP * 128 * 2;
  static constexpr int kSmem = kOffBar + 64 + 1024;   // + barriers, + alignment slack
};

template <int RP>
__global__ void __launch_bounds__(128) k_key_proj(const __grid_constant__ CUtensorMap kmap,
                                                  const __nv_bfloat16* __restrict__ Wk, int R, int64_t H, int d,
                                                  int S, float* __restrict__ khi, float* __restrict__ klo,
                                                  int32_t* status, uint64_t wait_ns, const ProblemTable tab) {
  using C = ProjCfg<RP>;
  extern __shared__ uint8_t proj_smem[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(proj_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = sm;
  uint8_t* sB = sm + C::kOffB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* a_full = bars;
  uint64_t* d_full = bars + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  const int lp = blockIdx.y, p = tab.p[lp], h = p % H;
  const int tid = threadIdx.x, warp = tid >> 5, j0 = blockIdx.x * 128;
  if (warp == 0) {
    tmem_alloc(tslot, RP);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(a_full, 1);
    mbar_init(d_full, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(a_full, 128 * d * 2);
    for (int a = 0; a < d / 64; ++a) tma_load_2d(sA + a * 16384, &kmap, a_full, a * 64, p * S + j0);
  }
  // W^T into the swizzled K-major B layout: element (n, c) of row n = column n of W
  const __nv_bfloat16* W = Wk + (size_t)h * d * R;
  for (int i = tid; i < RP * d; i += 128) {
    const int c = i / RP, n = i % RP;   // consecutive threads read consecutive W columns
    const __nv_bfloat16 v = n < R ? W[c * R + n] : __float2bfloat16(0.f);
    const int cc = c & 63;
    *reinterpret_cast<__nv_bfloat16*>(sB + (c >> 6) * (RP * 128) + n * 128 + ((((cc >> 3) ^ (n & 7))) << 4) +
                                      (cc & 7) * 2) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  bool ok = true, issued = false;
  if (tid == 0) {
    ok = mbar_wait(a_full, 0, wait_ns);
    if (ok) {
      issued = true;
      constexpr uint32_t idesc = instr_desc(128, RP, 1, 0, 0);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int kk = 0; kk < d / 16; ++kk) {
        const uint32_t offa = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t offb = (kk >> 2) * (RP * 128) + (kk & 3) * 32;
        mma_f16_ss(tbase, smem_desc(a0 + offa, 16, 1024), smem_desc(b0 + offb, 16, 1024), idesc, kk > 0);
      }
      mma_commit(d_full);
    } else {
      raise_status(status, DSV_ERR_TIMEOUT);
    }
  }
  // every thread waits for the accumulator (the issuing thread's failure shows as a timeout here too)
  ok = mbar_wait_warp(d_full, 0, wait_ns);
  if (ok) {
    tc_fence_after();
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    const size_t o = ((size_t)lp * S + j0 + tid) * RP;
#pragma unroll
    for (int c32 = 0; c32 < RP / 32; ++c32) {
      uint32_t v[32];
      tmem_ld32(lane_addr + c32 * 32, v);
      tmem_ld_wait(v);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t hv[8], lv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = __uint_as_float(v[c8 * 8 + e]);
          const float hi = tf32_rna(x);
          hv[e] = __float_as_uint(hi);
          lv[e] = __float_as_uint(tf32_rna(x - hi));
        }
        st_global_v8(khi + o + c32 * 32 + c8 * 8, hv);
        st_global_v8(klo + o + c32 * 32 + c8 * 8, lv);
      }
    }
  } else if ((tid & 31) == 0) {
    raise_status(status, DSV_ERR_TIMEOUT);
  }
  if (tid == 0) {   // the tile's copy and MMAs complete before the block leaves
    mbar_wait(a_full, 0, kDrainLimitNs);
    if (issued) mbar_wait(d_full, 0, kDrainLimitNs);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, RP);
}

// qbar_g = (mean over the group's queries of Q_i) . W_lr^Q, split into tf32
// hi and lo parts. One block per (group, problem).
template <int R>
__global__ void __launch_bounds__(128) k_group_mean_proj(const __nv_bfloat16* __restrict__ Q,
                                                         const __nv_bfloat16* __restrict__ Wq, int64_t H, int d,
                                                         Geometry geo, int g_pad, float* __restrict__ qhi,
                                                         float* __restrict__ qlo, const ProblemTable tab) {
  constexpr int RP = R < 32 ? 32 : R;
  __shared__ float part[128 * 8];
  __shared__ float mean[128];
  const int g = blockIdx.x, lp = blockIdx.y, p = tab.p[lp], h = p % H;
  const int tid = threadIdx.x;
  const int lanes_per_row = d / 8, rows_per_pass = 128 / lanes_per_row;
  const int col8 = tid % lanes_per_row, rsub = tid / lanes_per_row;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  const __nv_bfloat16* Qp = Q + (size_t)p * geo.S * d;
  for (int i = rsub; i < geo.G; i += rows_per_pass) {
    const int tok = token_of(geo, g, i);
    const uint4 v = *reinterpret_cast<const uint4*>(Qp + (size_t)tok * d + col8 * 8);
    const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __bfloat162float(x[e]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) part[tid * 8 + e] = acc[e];
  __syncthreads();
  if (tid < d) {
    const int c8 = tid / 8, e = tid % 8;
    float s = 0.f;
    for (int rs = 0; rs < rows_per_pass; ++rs) s += part[(rs * lanes_per_row + c8) * 8 + e];
    mean[tid] = s / (float)geo.G;
  }
  __syncthreads();
  if (tid < RP) {
    float v = 0.f;
    if (tid < R) {
      const __nv_bfloat16* W = Wq + (size_t)h * d * R;
      for (int c = 0; c < d; ++c) v = fmaf(mean[c], __bfloat162float(W[c * R + tid]), v);
    }
    const float hi = tf32_rna(v);
    qhi[((size_t)lp * g_pad + g) * RP + tid] = hi;
    qlo[((size_t)lp * g_pad + g) * RP + tid] = tf32_rna(v - hi);
  }
}

// ---------------------------------------------------------------------------
// Per-query predicted mass (the share of each query's own predicted softmax
// mass that its group's selected keys carry).
//
// q_lr of every query, rows in group-major order (row g*G + member), split
// into tf32 hi/lo parts like k_lr: one 128-row tile (one group of 128, or
// two groups of 64, each brought in as one TMA box over the latent cube) per
// block, the d/16 MMAs (128 x RP x 16, bf16 in, fp32 in TMEM), then hi/lo.
template <int RP>
__global__ void __launch_bounds__(128) k_query_proj(const __grid_constant__ CUtensorMap qcube,
                                                    const __nv_bfloat16* __restrict__ Wq, int R, int64_t H, int d,
                                                    Geometry geo, float* __restrict__ qhi, float* __restrict__ qlo,
                                                    int32_t* status, uint64_t wait_ns, const ProblemTable tab) {
  using C = ProjCfg<RP>;
  extern __shared__ uint8_t qproj_smem[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qproj_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = sm;
  uint8_t* sB = sm + C::kOffB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* a_full = bars;
  uint64_t* d_full = bars + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  const int lp = blockIdx.y, p = tab.p[lp], h = p % H;
  const int tid = threadIdx.x, warp = tid >> 5, r0 = blockIdx.x * 128;
  const int S = geo.S;
  if (warp == 0) {
    tmem_alloc(tslot, RP);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(a_full, 1);
    mbar_init(d_full, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(a_full, 128 * d * 2);
    for (int gi = 0; gi < 128 / geo.G; ++gi) {
      const int g = r0 / geo.G + gi;
      const int ct = g / (geo.ncy * geo.ncx), cy = (g / geo.ncx) % geo.ncy, cx = g % geo.ncx;
      for (int a = 0; a < d / 64; ++a)
        tma_load_4d(sA + a * 16384 + gi * geo.G * 128, &qcube, a_full, a * 64, cx * geo.gx, cy * geo.gy,
                    p * geo.T + ct * geo.gt);
    }
  }
  const __nv_bfloat16* W = Wq + (size_t)h * d * R;
  for (int i = tid; i < RP * d; i += 128) {
    const int c = i / RP, n = i % RP;
    const __nv_bfloat16 v = n < R ? W[c * R + n] : __float2bfloat16(0.f);
    const int cc = c & 63;
    *reinterpret_cast<__nv_bfloat16*>(sB + (c >> 6) * (RP * 128) + n * 128 + ((((cc >> 3) ^ (n & 7))) << 4) +
                                      (cc & 7) * 2) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  bool ok = true, issued = false;
  if (tid == 0) {
    ok = mbar_wait(a_full, 0, wait_ns);
    if (ok) {
      issued = true;
      constexpr uint32_t idesc = instr_desc(128, RP, 1, 0, 0);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int kk = 0; kk < d / 16; ++kk) {
        const uint32_t offa = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t offb = (kk >> 2) * (RP * 128) + (kk & 3) * 32;
        mma_f16_ss(tbase, smem_desc(a0 + offa, 16, 1024), smem_desc(b0 + offb, 16, 1024), idesc, kk > 0);
      }
      mma_commit(d_full);
    } else {
      raise_status(status, DSV_ERR_TIMEOUT);
    }
  }
  ok = mbar_wait_warp(d_full, 0, wait_ns);
  if (ok) {
    tc_fence_after();
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    const size_t o = ((size_t)lp * S + r0 + tid) * RP;
#pragma unroll
    for (int c32 = 0; c32 < RP / 32; ++c32) {
      uint32_t v[32];
      tmem_ld32(lane_addr + c32 * 32, v);
      tmem_ld_wait(v);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t hv[8], lv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = __uint_as_float(v[c8 * 8 + e]);
          const float hi = tf32_rna(x);
          hv[e] = __float_as_uint(hi);
          lv[e] = __float_as_uint(tf32_rna(x - hi));
        }
        st_global_v8(qhi + o + c32 * 32 + c8 * 8, hv);
        st_global_v8(qlo + o + c32 * 32 + c8 * 8, lv);
      }
    }
  } else if ((tid & 31) == 0) {
    raise_status(status, DSV_ERR_TIMEOUT);
  }
  if (tid == 0) {   // the tile's copies and MMAs complete before the block leaves
    mbar_wait(a_full, 0, kDrainLimitNs);
    if (issued) mbar_wait(d_full, 0, kDrainLimitNs);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, RP);
}

// Selection bitmap of each query group (bit j of row (p, g): key j is in the
// group's index set); a dense problem (offset -1) selects every key. One
// block per (group, problem), built in shared memory (S/32 words). Keys
// outside [0, S) are ignored.
__global__ void __launch_bounds__(256) k_idx_bitmap(const int32_t* __restrict__ idx, int S, int n_groups,
                                                    uint32_t* bits, const ProblemTable tab) {
  extern __shared__ uint32_t sbits[];
  const int g = blockIdx.x, lp = blockIdx.y, tid = threadIdx.x;
  const int nw = S / 32;
  const bool dense = tab.off[lp] < 0;
  for (int i = tid; i < nw; i += blockDim.x) sbits[i] = dense ? ~0u : 0u;
  __syncthreads();
  if (!dense) {
    const int k = tab.k[lp];
    const int32_t* row = idx + tab.off[lp] + (int64_t)g * k;
    for (int i = tid; i < k; i += blockDim.x) {
      const int j = __ldg(row + i);
      if (j >= 0 && j < S) atomicOr(sbits + (j >> 5), 1u << (j & 31));
    }
  }
  __syncthreads();
  uint32_t* out = bits + ((size_t)lp * n_groups + g) * nw;
  for (int i = tid; i < nw; i += blockDim.x) out[i] = sbits[i];
}

// Per query: the share m = (sum over selected keys) / (sum over all keys) of
// exp(scale (s - max)), the chunks' partial sums added in chunk order in
// fp64; written at the query's token position (optional) and summed per
// block of 256 queries in a fixed tree for the per-problem mean.
constexpr int kMassThreadsR = 256;
__global__ void __launch_bounds__(kMassThreadsR) k_mass_reduce(const float* __restrict__ msum, int n_chunks,
                                                               Geometry geo, float* per_query, double* block_sums,
                                                               const ProblemTable tab) {
  __shared__ double part[kMassThreadsR];
  const int lp = blockIdx.y, tid = threadIdx.x;
  const int r = blockIdx.x * kMassThreadsR + tid;   // row in group-major order
  double m = 0.0;
  if (r < geo.S) {
    double a = 0.0, sel = 0.0;
    for (int c = 0; c < n_chunks; ++c) {
      const size_t o = (((size_t)lp * n_chunks + c) * geo.S + r) * 2;
      a += (double)msum[o];
      sel += (double)msum[o + 1];
    }
    m = a > 0.0 ? sel / a : 0.0;
    if (per_query) per_query[(int64_t)tab.p[lp] * geo.S + token_of(geo, r / geo.G, r % geo.G)] = (float)m;
  }
  part[tid] = m;
  __syncthreads();
  for (int w = kMassThreadsR / 2; w > 0; w >>= 1) {
    if (tid < w) part[tid] += part[tid + w];
    __syncthreads();
  }
  if (tid == 0) block_sums[(size_t)lp * gridDim.x + blockIdx.x] = part[0];
}

// Per problem: the mean over its S queries, block sums added in block order.
__global__ void k_mass_mean(const double* block_sums, int nblk, int S, float* mass, const ProblemTable tab) {
  const int lp = blockIdx.x;
  if (threadIdx.x != 0) return;
  double acc = 0.0;
  for (int b = 0; b < nblk; ++b) acc += block_sums[(size_t)lp * nblk + b];
  mass[tab.p[lp]] = (float)(acc / (double)S);
}

// ---------------------------------------------------------------------------
// Bracket: per row, the bin holding the k-th largest score.
// Least score (as an orderable key in [o_lo, o_hi]) whose bin is at least
// `target`; o_hi when no score up to the row maximum reaches it.
__device__ uint32_t least_with_bin(int target, uint32_t o_lo, uint32_t o_hi, float lo, float inv_w, int nb) {
  uint32_t a = o_lo, b = o_hi;   // answer in [a, b]; the bin of ord2f(b) is >= target or b = o_hi
  while (a < b) {
    const uint32_t m = a + (b - a) / 2;
    if (lin_bin(ord2f(m) + 0.0f, lo, inv_w, nb) >= target) b = m;
    else a = m + 1;
  }
  return a;
}

// State of a row whose k-th score lies in [lo, hi) with `count` scores there:
// a single value is resolved by key order, a small interval by selecting among its
// candidates, a larger one by another REFINE round.
__device__ __forceinline__ int row_state(uint32_t lo, uint32_t hi, uint32_t count) {
  if (hi - lo <= 1u) return kRowTied;
  return count <= (uint32_t)kCandCap ? kRowCollect : kRowRefine;
}

// Finds the bin b of the row's histogram (nb bins, stride g_pad) where the
// count of scores from the top first reaches k, given `above` scores above
// bin nb-1. Returns b (or -1), with *above_out the scores above bin b.
__device__ __forceinline__ int find_kth_bin(const uint32_t* h, int nb, int g_pad, int k, int above, int* above_out) {
  for (int top = nb - 1; top >= 0; top -= 8) {
    uint32_t c[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) c[e] = top - e >= 0 ? __ldg(h + (size_t)(top - e) * g_pad) : 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (top - e < 0) break;
      if (above + (int)c[e] >= k) {
        *above_out = above;
        return top - e;
      }
      above += (int)c[e];
    }
  }
  *above_out = above;
  return -1;
}

// One thread per row. The row's boundary interval from the linear histogram:
// [least score of bin b*, least score of bin b*+1) in orderable bits, the
// count of scores at or above its upper end and the count inside it. A row to
// refine has its histogram zeroed (for the first REFINE round) and flags its
// group tile.
__global__ void k_bracket(uint32_t* hist, int nb, int g_pad, int n_groups, int n_gt, const uint32_t* __restrict__ mmin,
                          const uint32_t* __restrict__ mmax, uint32_t* blo, uint32_t* bhi, int32_t* nabove,
                          uint32_t* bcount, int32_t* rstate, int32_t* tflag, int32_t* status,
                          const ProblemTable tab) {
  const int lp = blockIdx.y, g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n_groups) return;
  const int k = tab.k[lp];
  uint32_t* h = hist + (size_t)lp * nb * g_pad + g;
  int above = 0;
  int b = find_kth_bin(h, nb, g_pad, k, 0, &above);
  if (b < 0) {   // fewer than k scores: cannot happen for 1 <= k <= S
    raise_status_if_clear(status, DSV_ERR_CANDIDATES);
    b = 0;
  }
  const uint32_t count = h[(size_t)b * g_pad];
  const int rid = lp * g_pad + g;
  // every score lies in [min, max] of its row; past the maximum a threshold
  // is the next float up (never reached)
  float lo, inv_w;
  lin_range(mmin[rid], mmax[rid], nb, &lo, &inv_w);
  const uint32_t o_lo = mmin[rid], o_hi = mmax[rid] + 1u;
  const uint32_t l = least_with_bin(b, o_lo, o_hi, lo, inv_w, nb);
  const uint32_t u = least_with_bin(b + 1, o_lo, o_hi, lo, inv_w, nb);
  blo[rid] = l;
  bhi[rid] = u;
  nabove[rid] = above;
  bcount[rid] = count;
  const int st = row_state(l, u, count);
  rstate[rid] = st;
  if (st == kRowRefine) {
    for (int i = 0; i < nb; ++i) h[(size_t)i * g_pad] = 0u;
    tflag[lp * n_gt + g / 128] = 1;
  }
}

// After a REFINE round: the interval's sub-bin b (width 2^shift in orderable
// bits) holding the k-th score becomes the row's interval. Each round takes
// log2(nb) more bits, so an interval is a single value after at most
// ceil(32 / log2(nb)) rounds.
__global__ void k_refine_bracket(uint32_t* hist, int nb, int log2nb, int g_pad, int n_groups, int n_gt,
                                 uint32_t* blo, uint32_t* bhi, int32_t* nabove, uint32_t* bcount, int32_t* rstate,
                                 const int32_t* tflag, int32_t* tflag_next, int32_t* status, const ProblemTable tab) {
  const int lp = blockIdx.y, g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n_groups || tflag[lp * n_gt + g / 128] == 0) return;
  const int rid = lp * g_pad + g;
  if (rstate[rid] != kRowRefine) return;
  const int k = tab.k[lp];
  uint32_t* h = hist + (size_t)lp * nb * g_pad + g;
  const uint32_t lo = blo[rid], hi = bhi[rid], wid = hi - lo;
  const int bits = 32 - __clz(wid - 1u);   // wid >= 2 here
  const int shift = max(0, bits - log2nb);
  int above = 0;
  const int b = find_kth_bin(h, nb, g_pad, k, nabove[rid], &above);
  if (b < 0) {   // the sub-bins hold fewer scores than the interval did: inconsistent
    raise_status_if_clear(status, DSV_ERR_CANDIDATES);
    rstate[rid] = kRowTied;
    nabove[rid] = k;
    return;
  }
  const uint32_t count = h[(size_t)b * g_pad];
  const uint32_t l = lo + ((uint32_t)b << shift);
  const uint64_t end = (uint64_t)lo + ((uint64_t)(b + 1) << shift);
  const uint32_t u = end < (uint64_t)hi ? (uint32_t)end : hi;
  blo[rid] = l;
  bhi[rid] = u;
  nabove[rid] = above;
  bcount[rid] = count;
  const int st = row_state(l, u, count);
  rstate[rid] = st;
  if (st == kRowRefine) {
    for (int i = 0; i < nb; ++i) h[(size_t)i * g_pad] = 0u;
    tflag_next[lp * n_gt + g / 128] = 1;
  }
}

// Resolve: a row whose interval holds at most kCandCap candidates marks the
// first k - above of them in (score desc, key asc) order in the row's
// selection mask. The candidates are (~score << 32 | key) words; with r the
// rank of the score below the interval's top, x = r << kb | key orders them
// the same way and is unique per candidate. A most-significant-digit radix
// select over x (11-bit digits, a shared-memory histogram per digit) finds
// the boundary: the candidates below the chosen digit are taken, those above
// dropped, and the next digit splits the rest, until the chosen digit's
// candidates are exactly the ones still needed. Single-valued intervals are
// left to the compaction.
constexpr int kResolveThreads = 512;
constexpr int kResolvePer = kCandCap / kResolveThreads;   // candidates per thread
constexpr int kDigitBits = 11;

// Block-wide exclusive prefix sum of one value per thread (kResolveThreads).
__device__ __forceinline__ uint32_t block_exclusive_sum(uint32_t v, uint32_t* warp_tot) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[wid] = inc;
  __syncthreads();
  uint32_t base = 0;
  for (int w = 0; w < wid; ++w) base += warp_tot[w];
  return base + inc - v;
}

__global__ void __launch_bounds__(kResolveThreads, 2) k_resolve(const uint64_t* __restrict__ cand,
                                                           const uint32_t* cand_cnt, const uint32_t* bhi,
                                                           const int32_t* nabove, const uint32_t* bcount,
                                                           const int32_t* rstate, int g_pad, int n_words, int S,
                                                           uint32_t* sel_bits, int32_t* status,
                                                           const ProblemTable tab) {
  constexpr int kBuckets = 1 << kDigitBits;
  __shared__ uint32_t hist[kBuckets];
  __shared__ uint32_t warp_tot[kResolveThreads / 32];
  __shared__ uint32_t s_digit, s_before;
  const int g = blockIdx.x, lp = blockIdx.y, tid = threadIdx.x;
  const int rid = lp * g_pad + g;
  const int st = rstate[rid];
  if (st == kRowTied) return;
  const int k = tab.k[lp];
  const int need = k - nabove[rid];
  const uint32_t ncand = cand_cnt[rid];
  if (st != kRowCollect || ncand != bcount[rid] || ncand > (uint32_t)kCandCap || need < 1 ||
      (uint32_t)need > ncand) {
    if (tid == 0) raise_status_if_clear(status, DSV_ERR_CANDIDATES);
    return;
  }
  uint32_t* row_bits = sel_bits + (size_t)rid * n_words;
  const uint64_t* c = cand + (size_t)rid * kCandCap;
  const int kb = 32 - __clz((uint32_t)(S - 1) | 1u);   // key bits
  const uint32_t kmask = (1u << kb) - 1u;
  if ((uint32_t)need == ncand) {   // the whole interval is taken
    for (int i = tid; i < need; i += kResolveThreads) {
      const uint32_t j = (uint32_t)c[i];
      atomicOr(row_bits + (j >> 5), 1u << (j & 31));
    }
    return;
  }
  // r = (~score of the interval's top) - (~score): 0 for the highest score
  const uint32_t top = ~(bhi[rid] - 1u);
  uint64_t x[kResolvePer];
  uint32_t live = 0;
  uint32_t rmax = 0;
#pragma unroll
  for (int e = 0; e < kResolvePer; ++e) {
    const int i = tid + e * kResolveThreads;
    x[e] = 0;
    if (i < (int)ncand) {
      const uint64_t w = c[i];
      const uint32_t r = (uint32_t)(w >> 32) - top;
      rmax = max(rmax, r);
      x[e] = ((uint64_t)r << kb) | ((uint32_t)w & kmask);
      live |= 1u << e;
    }
  }
  // the interval's width bounds r, so the select starts at the top bit of x
  const int rbits = 32 - __clz(__reduce_max_sync(0xffffffffu, rmax) | 0u);
  if ((tid & 31) == 0) warp_tot[tid >> 5] = (uint32_t)rbits;
  __syncthreads();
  int L = kb;
  for (int w = 0; w < kResolveThreads / 32; ++w) L = max(L, kb + (int)warp_tot[w]);
  __syncthreads();
  uint32_t remaining = (uint32_t)need;
  uint64_t prefix = 0;
  for (int hb = L; hb > 0; hb -= kDigitBits) {
    const int shift = hb > kDigitBits ? hb - kDigitBits : 0, bits = hb - shift;
    const uint32_t dmask = (1u << bits) - 1u;
    for (int i = tid; i < kBuckets; i += kResolveThreads) hist[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kResolvePer; ++e)
      if (((live >> e) & 1u) && (x[e] >> hb) == prefix) atomicAdd(&hist[(uint32_t)(x[e] >> shift) & dmask], 1u);
    __syncthreads();
    // the digit whose bucket holds the remaining-th live candidate
    constexpr int kPerThread = kBuckets / kResolveThreads;
    uint32_t v = 0;
#pragma unroll
    for (int q = 0; q < kPerThread; ++q) {
      const int bkt = tid * kPerThread + q;
      v += bkt < (1 << bits) ? hist[bkt] : 0u;
    }
    const uint32_t before = block_exclusive_sum(v, warp_tot);
    if (before < remaining && remaining <= before + v) {
      uint32_t acc = before;
      for (int q = 0; q < kPerThread; ++q) {
        const uint32_t h = hist[tid * kPerThread + q];
        if (acc + h >= remaining) {
          s_digit = (uint32_t)(tid * kPerThread + q);
          s_before = acc;
          break;
        }
        acc += h;
      }
    }
    __syncthreads();
    const uint32_t d = s_digit, below = s_before, at = hist[d];
    // take the live candidates below the digit; keep those at it only if
    // they are not all needed
    const bool take_at = remaining - below == at;
#pragma unroll
    for (int e = 0; e < kResolvePer; ++e) {
      if (!((live >> e) & 1u) || (x[e] >> hb) != prefix) continue;
      const uint32_t dg = (uint32_t)(x[e] >> shift) & dmask;
      if (dg < d || (dg == d && take_at)) {
        const uint32_t j = (uint32_t)x[e] & kmask;
        atomicOr(row_bits + (j >> 5), 1u << (j & 31));
      }
      if (dg != d || take_at) live &= ~(1u << e);
    }
    if (take_at) return;
    remaining -= below;
    prefix = (prefix << bits) | d;
    __syncthreads();   // hist and the shared digit are rewritten next round
  }
  if (tid == 0) raise_status_if_clear(status, DSV_ERR_CANDIDATES);   // x is unique: cannot be reached
}

// Index rows from the masks: one block per group row, its 8 warps on
// consecutive segments of the row's mask words. A row's selection is its
// selection mask, plus, when its boundary interval is a single value, the
// k - above lowest keys of its tie mask (the cut is found first: each warp
// counts its segment's ties, and the warp holding the cut walks its words).
// Each warp counts its segment's selected keys, a block scan gives each
// segment its first output position, and each warp then takes its words 32
// at a time: every lane writes its word's keys into the warp's shared staging
// area at the word's prefix position (a short loop over the set bits; the
// keys cluster, so the counts differ, but only shared stores diverge), and
// the warp copies the staged keys out with stores of 32 consecutive indices.
constexpr int kCompactWarps = 8;

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  return x;
}

// Tie-mask bits of word w that lie at or below key `cut`.
__device__ __forceinline__ uint32_t keep_upto(int w, int cut) {
  const int d = cut - w * 32;
  return d >= 31 ? ~0u : (d < 0 ? 0u : (2u << d) - 1u);
}

__global__ void __launch_bounds__(32 * kCompactWarps) k_sel_compact(const uint32_t* __restrict__ bits,
                                                                    const uint32_t* __restrict__ eq_bits,
                                                                    const int32_t* rstate, const int32_t* nabove,
                                                                    int g_pad, int n_words, int32_t* idx,
                                                                    int32_t* status, const ProblemTable tab) {
  __shared__ int seg_total[kCompactWarps];
  __shared__ int s_cut;
  __shared__ int32_t stage[kCompactWarps][32 * 32];
  const int g = blockIdx.x, lp = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = tab.k[lp];
  const int rid = lp * g_pad + g;
  int32_t* out = idx + tab.off[lp] + (int64_t)g * k;
  const uint32_t* row = bits + (size_t)rid * n_words;
  const uint32_t* eq = eq_bits + (size_t)rid * n_words;
  const int seg = ((n_words + kCompactWarps * 32 - 1) / (kCompactWarps * 32)) * 32;   // words per warp
  const int w_begin = min(n_words, warp * seg), w_end = min(n_words, w_begin + seg);
  const bool tied = rstate[rid] == kRowTied;
  if (threadIdx.x == 0) s_cut = -1;
  if (tied) {
    const int budget = k - nabove[rid];
    int ce = 0;
    for (int w = w_begin + lane; w < w_end; w += 32) ce += __popc(__ldg(eq + w));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ce += __shfl_xor_sync(0xffffffffu, ce, d);
    if (lane == 0) seg_total[warp] = ce;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += seg_total[i];
    if (before < budget && budget <= before + ce) {
      int rem = budget - before;   // >= 1: the rem-th tie of this segment is the last one taken
      for (int w0 = w_begin; w0 < w_end; w0 += 32) {
        const uint32_t m = w0 + lane < w_end ? __ldg(eq + w0 + lane) : 0u;
        const int c = __popc(m);
        const int incl = warp_incl_scan(c, lane);
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (rem <= total) {
          const uint32_t hit = __ballot_sync(0xffffffffu, incl >= rem);
          const int L = __ffs(hit) - 1;
          if (lane == L) s_cut = (w0 + L) * 32 + (int)__fns(m, 0, rem - (incl - c));
          break;
        }
        rem -= total;
      }
    }
  }
  __syncthreads();
  const int cut = s_cut;
  auto word = [&](int w) -> uint32_t {
    const uint32_t m = __ldg(row + w);
    return tied ? (m | (__ldg(eq + w) & keep_upto(w, cut))) : m;
  };
  int cnt = 0;
#pragma unroll 8
  for (int w = w_begin + lane; w < w_end; w += 32) cnt += __popc(word(w));
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, d);
  __syncthreads();   // every warp has read seg_total (tie counts) before it is reused
  if (lane == 0) seg_total[warp] = cnt;
  __syncthreads();
  int base = 0, row_total = 0;
  for (int i = 0; i < kCompactWarps; ++i) {
    base += i < warp ? seg_total[i] : 0;
    row_total += seg_total[i];
  }
  // 32 words (1024 keys) per step: each lane writes its word's selected keys
  // into the warp's staging area at its exclusive prefix, then the warp
  // copies them out in order with coalesced stores
  int32_t* st = stage[warp];
  for (int w0 = w_begin; w0 < w_end; w0 += 32) {
    const uint32_t m = w0 + lane < w_end ? word(w0 + lane) : 0u;
    const int c = __popc(m);
    const int incl = warp_incl_scan(c, lane);
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int pos = incl - c;
    const int kbase = (w0 + lane) * 32;
    for (uint32_t mm = m; mm; mm &= mm - 1u) st[pos++] = kbase + __ffs(mm) - 1;
    __syncwarp();
    for (int q = lane; q < total; q += 32) {
      const int p = base + q;
      if (p < k) out[p] = st[q];
    }
    __syncwarp();
    base += total;
  }
  if (threadIdx.x == 0 && row_total != k) raise_status_if_clear(status, DSV_ERR_CANDIDATES);
}

// Rows with k == S select every key.
__global__ void k_fill_all(int32_t* idx, int64_t off, int S, int64_t total) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x)
    idx[off + i] = (int32_t)(i % S);
}

// ---------------------------------------------------------------------------
// Coverage reduce. The COV pass gives every group row a coarse table: per
// bin of log-probability below the row maximum (width w), the count of keys
// and their exact total probability. Then:
//   k_cov_merge   (group, bin) totals over key chunks, one thread per pair
//   k_cov_scan    per group: cumulative counts and normalised masses, the
//                 bin width and 1 / (total probability)
//   bounds search the smallest k whose upper bound on C reaches the target
//                 (k_lo) and the smallest whose lower bound does (k_hi):
//                 within a bin the keys' probabilities lie between the bin's
//                 edge values, which bounds any j of them; k_cov is in
//                 [k_lo, k_hi]
//   k_cov_window  per group, the coarse bins holding its ranks k_lo..k_hi
//   COV_FINE      the window's keys again, in as many fine bins as coarse
//                 ones (count and exact probability), then merged and scanned
//   final search  k_cov in [k_lo, k_hi] on the combined table (coarse bins
//                 outside the window, fine bins inside), interpolating inside
//                 a bin as if its log-probabilities were evenly spread; the
//                 fine bins bring that error down by their count.
// Every search is a sequence of wide rounds (k_cov_eval / k_cov_pick): each
// evaluates C at up to kCovPoints values of k spread evenly over the current
// interval and keeps the sub-interval where C first reaches the target; once
// the interval holds at most kCovPoints values all are evaluated. Evaluation
// blocks take kCovGroupsPerBlock groups each and their partial sums are
// added in block order, so the result does not depend on scheduling.
// `half_cnt` non-null: the count words hold two half-bin counts (the coarse
// pass); their sums go to cum_cnt and the half counts to half_cnt
// ([problem][2 nb][g_pad]).
__global__ void k_cov_merge(const uint32_t* __restrict__ cnt, const float* __restrict__ mass, int nb, int n_chunks,
                            int g_pad, int n_groups, int32_t* cum_cnt, double* cum_mass, int32_t* half_cnt) {
  const int lp = blockIdx.z, b = blockIdx.y, g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n_groups) return;
  int c0 = 0, c1 = 0;
  double m = 0.0;
  for (int ch = 0; ch < n_chunks; ++ch) {
    const size_t o = (((size_t)lp * n_chunks + ch) * nb + b) * g_pad + g;
    const uint32_t v = cnt[o];
    if (half_cnt) {
      c0 += (int)(v & 0xffffu);
      c1 += (int)(v >> 16);
    } else {
      c0 += (int)v;
    }
    m += (double)mass[o];
  }
  const size_t rid = (size_t)lp * g_pad + g;
  cum_cnt[rid * nb + b] = c0 + c1;
  cum_mass[rid * nb + b] = m;
  if (half_cnt) {
    half_cnt[((size_t)lp * 2 * nb + 2 * b) * g_pad + g] = c0;
    half_cnt[((size_t)lp * 2 * nb + 2 * b + 1) * g_pad + g] = c1;
  }
}

// One warp per group: lane l owns bins [l*per, l*per + per) of the (at most
// 128) bins. Cumulative counts; masses cumulated and divided by `norm_total`
// (the group's total when null), scaled by `norm_scale` (a per-group factor,
// 1 when null). `width`/`zinv` (optional): the bin width in natural-log units
// and 1 / total probability.
__global__ void k_cov_scan(const uint32_t* mmax, const uint32_t* mmin, int nb, int g_pad, int n_groups, float scale,
                           int32_t* cum_cnt, double* cum_mass, float* width, float* zinv, const double* norm_scale) {
  const int lp = blockIdx.y, lane = threadIdx.x & 31;
  const int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (g >= n_groups) return;
  const size_t rid = (size_t)lp * g_pad + g;
  int32_t* cc = cum_cnt + rid * nb;
  double* cm = cum_mass + rid * nb;
  const int per = nb / 32;   // 4 (nb = 128) or 2 (nb = 64)
  int c[4] = {0, 0, 0, 0};
  double m[4] = {0.0, 0.0, 0.0, 0.0};
  int csum = 0;
  double msum = 0.0;
  for (int e = 0; e < per; ++e) {
    c[e] = cc[lane * per + e];
    m[e] = cm[lane * per + e];
    csum += c[e];
    msum += m[e];
  }
  int ci = csum;   // inclusive warp scans of the lane totals
  double mi = msum;
  for (int d = 1; d < 32; d <<= 1) {
    const int cy = __shfl_up_sync(0xffffffffu, ci, d);
    const double my = __shfl_up_sync(0xffffffffu, mi, d);
    if (lane >= d) {
      ci += cy;
      mi += my;
    }
  }
  const double total = __shfl_sync(0xffffffffu, mi, 31);
  const double f = norm_scale ? norm_scale[rid] : 1.0;
  const double inv = total > 0.0 ? f / total : 0.0;
  int crun = ci - csum;
  double mrun = mi - msum;
  for (int e = 0; e < per; ++e) {
    crun += c[e];
    mrun += m[e];
    cc[lane * per + e] = crun;
    cm[lane * per + e] = mrun * inv;
  }
  if (lane == 0 && width) width[rid] = scale * (ord2f(mmax[rid]) - ord2f(mmin[rid])) / (float)nb;
  if (lane == 0 && zinv) zinv[rid] = total > 0.0 ? (float)(1.0 / total) : 0.f;
}

constexpr int kCovPoints = 1024;
constexpr int kCovGroupsPerBlock = 16;

enum CovEval { kCovBoundLo = 0, kCovBoundHi = 1, kCovCombined = 2 };

// First index of a cumulative table (n entries) whose count reaches k.
__device__ __forceinline__ int first_reaching(const int32_t* cc, int n, int k) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (cc[mid] >= k) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

// Mass of j of a bin's n keys (bin mass mb, log-probabilities spread evenly
// over a width dw).
__device__ __forceinline__ float spread_part(float mb, int j, int n, float dw) {
  const float f = n > 0 ? (float)j / (float)n : 1.f;
  return dw > 1e-6f ? mb * (1.f - __expf(-f * dw)) / (1.f - __expf(-dw)) : mb * f;
}

// A group's tables as staged by k_cov_eval: coarse cumulative counts/masses
// over nb bins of width w; the window [wa, wb] of coarse bins and its fine
// cumulative counts/masses over nb bins (masses as shares of the group's
// total, like the coarse ones).
struct CovTables {
  const int32_t* cc;
  const float* cm;
  const int32_t* fc;
  const float* fm;
  int nb, wa, wb;
  float w, zinv;
};

// C's per-group term at k: the mass of the group's k most probable keys, as
// a lower or upper bound from the coarse bins, or interpolated on the
// combined table.
__device__ float cov_group_mass(const CovTables& t, int k, int mode) {
  const int b = first_reaching(t.cc, t.nb, k);
  const int pc = b > 0 ? t.cc[b - 1] : 0;
  const float pm = b > 0 ? t.cm[b - 1] : 0.f;
  const int n = t.cc[b] - pc, j = k - pc;
  const float mb = t.cm[b] - pm;
  if (mode != kCovCombined) {
    // every key of bin b has a probability between its edges' values
    const float pmax = __expf(-(float)b * t.w) * t.zinv, pmin = __expf(-(float)(b + 1) * t.w) * t.zinv;
    if (mode == kCovBoundLo) return pm + fmaxf((float)j * pmin, mb - (float)(n - j) * pmax);
    return pm + fminf((float)j * pmax, mb - (float)(n - j) * pmin);
  }
  if (b < t.wa || b > t.wb) return pm + spread_part(mb, j, n, t.w);
  const int base_c = t.wa > 0 ? t.cc[t.wa - 1] : 0;
  const float base_m = t.wa > 0 ? t.cm[t.wa - 1] : 0.f;
  const int kk = k - base_c;
  const int f = first_reaching(t.fc, t.nb, kk);
  const int fpc = f > 0 ? t.fc[f - 1] : 0;
  const float fpm = f > 0 ? t.fm[f - 1] : 0.f;
  const float fw = t.w * (float)(t.wb - t.wa + 1) / (float)t.nb;
  return base_m + fpm + spread_part(t.fm[f] - fpm, kk - fpc, t.fc[f] - fpc, fw);
}

// The k of point p for interval [lo, hi] (search), or the curve's point p
// (curve: k = ceil((p+1) S / n_curve)); -1 for no point.
__device__ __forceinline__ int cov_point(bool curve, int lo, int hi, int p, int S, int n_curve) {
  if (curve) return p < n_curve ? (int)(((int64_t)(p + 1) * S + n_curve - 1) / n_curve) : -1;
  const int64_t span = (int64_t)hi - lo + 1;
  if (span <= kCovPoints) return p < span ? lo + p : -1;
  return (int)(lo - 1 + ((int64_t)(p + 1) * span + kCovPoints - 1) / kCovPoints);
}

// range[2*lp .. 2*lp+1]: [lo, hi] of a search, or of the fine window when
// fine tables are read.
__global__ void k_cov_range_init(int32_t* range, const int32_t* from_lo, const int32_t* from_hi, int S, int n) {
  const int lp = blockIdx.x * blockDim.x + threadIdx.x;
  if (lp >= n) return;
  range[2 * lp] = from_lo ? from_lo[lp] : 1;
  range[2 * lp + 1] = from_hi ? from_hi[lp] : S;
}

// One thread per point; the block's kCovGroupsPerBlock group tables are
// staged in shared memory first. fine_cnt == nullptr: coarse tables only.
__global__ void __launch_bounds__(kCovPoints) k_cov_eval(int mode, bool curve, int nb, int g_pad, int n_groups,
                                                         int S, const int32_t* cum_cnt, const double* cum_mass,
                                                         const float* width, const float* zinv, const int32_t* win,
                                                         const int32_t* fine_cnt, const double* fine_mass,
                                                         const int32_t* range, int n_curve, double* partial) {
  static_assert(SelCfg<32>::kCovBins <= 128 && SelCfg<64>::kCovBins <= 128, "coverage tables hold 128 bins");
  static_assert(SelCfg<32>::kCovBins * 128 * 8 <= SelCfg<32>::kHistBytes &&
                    SelCfg<64>::kCovBins * 128 * 8 <= SelCfg<64>::kHistBytes,
                "COV counts and sums fit the histogram area");
  __shared__ int32_t s_cc[kCovGroupsPerBlock * 128], s_fc[kCovGroupsPerBlock * 128];
  __shared__ float s_cm[kCovGroupsPerBlock * 128], s_fm[kCovGroupsPerBlock * 128];
  __shared__ float s_w[kCovGroupsPerBlock], s_z[kCovGroupsPerBlock];
  __shared__ int s_wa[kCovGroupsPerBlock], s_wb[kCovGroupsPerBlock];
  const int lp = blockIdx.y, blk = blockIdx.x, nblk = gridDim.x, p = threadIdx.x;
  // blockIdx.z > 0: the second of two searches launched together (the two
  // bound searches), with its own range and partials
  if (gridDim.z > 1) {
    mode = blockIdx.z == 0 ? kCovBoundHi : kCovBoundLo;
    range += (size_t)blockIdx.z * 2 * gridDim.y;
    partial += (size_t)blockIdx.z * gridDim.y * nblk * kCovPoints;
  }
  if (!curve && range[2 * lp] < 0) return;   // this search already has its answer
  const int g0 = blk * kCovGroupsPerBlock, ng = min(n_groups - g0, kCovGroupsPerBlock);
  const size_t base = (size_t)lp * g_pad + g0;
  for (int i = p; i < ng * nb; i += blockDim.x) {
    s_cc[i] = cum_cnt[base * nb + i];
    s_cm[i] = (float)cum_mass[base * nb + i];
    s_fc[i] = fine_cnt ? fine_cnt[base * nb + i] : 0;
    s_fm[i] = fine_cnt ? (float)fine_mass[base * nb + i] : 0.f;
  }
  if (p < ng) {
    s_w[p] = width[base + p];
    s_z[p] = zinv[base + p];
    s_wa[p] = fine_cnt ? win[4 * (base + p)] : nb;   // no window: every bin is coarse
    s_wb[p] = fine_cnt ? win[4 * (base + p) + 1] : -1;
  }
  __syncthreads();
  const int k = cov_point(curve, range[2 * lp], range[2 * lp + 1], p, S, n_curve);
  double acc = 0.0;
  if (k >= 1)
    for (int g = 0; g < ng; ++g) {
      const CovTables t{s_cc + g * nb, s_cm + g * nb, s_fc + g * nb, s_fm + g * nb, nb, s_wa[g], s_wb[g], s_w[g],
                        s_z[g]};
      acc += (double)cov_group_mass(t, k, mode);
    }
  partial[((size_t)lp * nblk + blk) * kCovPoints + p] = acc;
}

// Sums the partials of each point in block order. Search: narrow range[lp]
// to the sub-interval where C first reaches the target, or, when every k of
// the interval was evaluated, write the answer to out[out_idx]. Curve: write
// the curve.
__global__ void __launch_bounds__(1024) k_cov_pick(bool curve, int nblk, int n_groups, int S, float target,
                                                   const double* partial, int32_t* range, int32_t* out,
                                                   int32_t* out2, bool out_by_problem, float* curve_out, int n_curve,
                                                   const ProblemTable tab) {
  __shared__ int first;
  const int lp = blockIdx.x, p = threadIdx.x;
  // blockIdx.y > 0: the second of two searches launched together (answer in out2)
  if (blockIdx.y > 0) {
    range += (size_t)blockIdx.y * 2 * gridDim.x;
    partial += (size_t)blockIdx.y * gridDim.x * nblk * kCovPoints;
    out = out2;
  }
  const int lo = range[2 * lp], hi = range[2 * lp + 1];
  if (!curve && lo < 0) return;   // this search already has its answer
  if (p == 0) first = kCovPoints;
  __syncthreads();  // every thread has read range before thread 0 rewrites it
  const int k = cov_point(curve, lo, hi, p, S, n_curve);
  double c = 0.0;
  for (int b = 0; b < nblk; ++b) c += partial[((size_t)lp * nblk + b) * kCovPoints + p];
  c /= (double)n_groups;
  if (curve) {
    if (k >= 1) curve_out[(size_t)tab.p[lp] * n_curve + p] = (float)c;
    return;
  }
  if (k >= 1 && c >= (double)target) atomicMin(&first, p);
  __syncthreads();
  if (p != 0) return;
  const int64_t span = (int64_t)hi - lo + 1;
  if (span <= kCovPoints) {
    // C(S) = 1 >= target up to rounding; with no qualifying point keep hi
    out[out_by_problem ? tab.p[lp] : lp] = first < kCovPoints ? lo + first : hi;
    range[2 * lp] = -1;   // later rounds of this search leave at once
    return;
  }
  const int f = first < kCovPoints ? first : kCovPoints - 1;  // answer in (k_{f-1}, k_f]
  range[2 * lp] = f > 0 ? cov_point(false, lo, hi, f - 1, S, 0) + 1 : lo;
  range[2 * lp + 1] = cov_point(false, lo, hi, f, S, 0);
}

// Per group: the coarse bins [wa, wb] holding its ranks k_lo .. k_hi, and
// the factor that makes the fine masses (shares of the window's own total)
// shares of the group's total.
// The window's scores: coarse bins are non-increasing in the score, so the
// scores whose bin lies in [wa, wb] form the interval [lo, hi] of orderable
// bits, found by binary search with the passes' own binning arithmetic
// (empty when lo > hi).
// `half` = true: the same for half bins (2 nb of them).
__device__ uint32_t least_with_cbin_at_most(int target, uint32_t o_lo, uint32_t o_hi, float cmax, float scale,
                                            float inv_w, int nb, bool half = false) {
  uint32_t a = o_lo, b = o_hi;   // answer in [a, b]; o_hi when no score reaches it
  while (a < b) {
    const uint32_t m = a + (b - a) / 2;
    float frac;
    const int bin = cov_bin(cov_coord(ord2f(m) + 0.0f, cmax, scale, inv_w), nb, &frac);
    if ((half ? 2 * bin + (frac >= 0.5f ? 1 : 0) : bin) <= target) b = m;
    else a = m + 1;
  }
  return a;
}

__global__ void k_cov_window(int nb, int g_pad, int n_groups, float scale, const uint32_t* mmax, const uint32_t* mmin,
                             const int32_t* cum_cnt, const double* cum_mass, const int32_t* k_lo, const int32_t* k_hi,
                             int32_t* win, double* fine_scale) {
  const int lp = blockIdx.y, g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n_groups) return;
  const size_t rid = (size_t)lp * g_pad + g;
  const int32_t* cc = cum_cnt + rid * nb;
  const double* cm = cum_mass + rid * nb;
  const int wa = first_reaching(cc, nb, k_lo[lp]);
  const int wb = first_reaching(cc, nb, k_hi[lp]);
  float cmax, inv_w, w2;
  cov_row_scale(mmax[rid], mmin[rid], scale, nb, &cmax, &inv_w, &w2);
  const uint32_t o_lo = mmin[rid], o_hi = mmax[rid] + 1u;
  const uint32_t lo = least_with_cbin_at_most(wb, o_lo, o_hi, cmax, scale, inv_w, nb);       // bin <= wb
  const uint32_t hi = least_with_cbin_at_most(wa - 1, o_lo, o_hi, cmax, scale, inv_w, nb);   // bin < wa
  int4 out;
  out.x = wa;
  out.y = wb;
  out.z = (int)lo;
  out.w = (int)(hi - 1u);   // the last score with bin >= wa
  *reinterpret_cast<int4*>(win + 4 * rid) = out;
  fine_scale[rid] = cm[wb] - (wa > 0 ? cm[wa - 1] : 0.0);
}

// Top-k bracket from the coverage pass's half-bin counts. Its bins are
// linear in the score over the row's [min, max], like the top-k histogram's,
// so once coverage has run, the half bin holding the k-th largest score, the
// scores above it and the scores inside it are read from that table and the
// histogram pass is not needed. Same outputs as k_bracket: the interval
// [least score of half bin h*, least score of half bin h*-1) in orderable
// bits, found with the coverage passes' own binning arithmetic.
__global__ void k_bracket_cov(int nb, int g_pad, int n_groups, int n_gt, float scale, const uint32_t* mmax,
                              const uint32_t* mmin, const int32_t* cum_cnt, const int32_t* half_cnt, uint32_t* hist,
                              int hist_nb,
                              uint32_t* blo, uint32_t* bhi, int32_t* nabove, uint32_t* bcount, int32_t* rstate,
                              int32_t* tflag, int32_t* status, const ProblemTable tab) {
  const int lp = blockIdx.y, g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n_groups) return;
  const int k = tab.k[lp];
  const size_t rid = (size_t)lp * g_pad + g;
  // the coarse bin from the cumulative coarse counts, then one of its halves
  const int32_t* cc = cum_cnt + rid * nb;
  const int b = first_reaching(cc, nb, k);
  if (cc[b] < k) raise_status_if_clear(status, DSV_ERR_CANDIDATES);   // fewer than k scores: inconsistent
  int above = b > 0 ? cc[b - 1] : 0;
  const int32_t* hc = half_cnt + (size_t)lp * 2 * nb * g_pad + g;
  const int h0 = __ldg(hc + (size_t)(2 * b) * g_pad), h1 = __ldg(hc + (size_t)(2 * b + 1) * g_pad);
  int hb = 2 * b;
  uint32_t count = (uint32_t)h0;
  if (above + h0 < k) {
    hb = 2 * b + 1;
    above += h0;
    count = (uint32_t)h1;
  }
  float cmax, inv_w, w2;
  cov_row_scale(mmax[rid], mmin[rid], scale, nb, &cmax, &inv_w, &w2);
  const uint32_t o_lo = mmin[rid], o_hi = mmax[rid] + 1u;
  const uint32_t l = least_with_cbin_at_most(hb, o_lo, o_hi, cmax, scale, inv_w, nb, true);
  const uint32_t u = least_with_cbin_at_most(hb - 1, o_lo, o_hi, cmax, scale, inv_w, nb, true);   // o_hi for hb = 0
  blo[rid] = l;
  bhi[rid] = u;
  nabove[rid] = above;
  bcount[rid] = count;
  const int st = row_state(l, u, count);
  rstate[rid] = st;
  if (st == kRowRefine) {
    uint32_t* h = hist + (size_t)lp * hist_nb * g_pad + g;
    for (int i = 0; i < hist_nb; ++i) h[(size_t)i * g_pad] = 0u;
    tflag[lp * n_gt + g / 128] = 1;
  }
}

// ---------------------------------------------------------------------------
// Host orchestration.
struct TopkPlan {
  Geometry geo;
  int RP, n_gt, g_pad, n_tiles, pc;
  int hist_bins, cov_bins;
  int max_chunks;   // key chunks of the largest launch (per-chunk arrays are sized by it)
};
constexpr int kCovMaxTiles = 65535 / 128;   // COV bin words hold at most 65535 keys of a row per chunk

static int max_chunks_of(const struct TopkPlan& pl, int P);

static TopkPlan make_plan(const dsv_shape& s, int32_t r, const dsv_group& g) {
  TopkPlan p;
  p.geo = make_geometry(s, g);
  p.RP = (r == 64) ? 64 : 32;
  p.n_gt = (p.geo.n_groups + 127) / 128;
  p.g_pad = p.n_gt * 128;
  p.n_tiles = p.geo.S / 128;
  const size_t per = (size_t)p.geo.S * p.RP * 8;
  const int P = (int)(s.B * s.H);
  p.pc = (int)std::max<size_t>(1, std::min<size_t>((size_t)P, kProjBudget / per));
  p.hist_bins = p.RP == 32 ? SelCfg<32>::kHistBins : SelCfg<64>::kHistBins;
  p.cov_bins = p.RP == 32 ? SelCfg<32>::kCovBins : SelCfg<64>::kCovBins;
  p.max_chunks = max_chunks_of(p, P);
  return p;
}

// Key chunks per row. A launch has n_gt * n_local * n_chunks blocks, each
// scoring chunk_tiles key tiles; the count minimises the launch's waves on the
// 152 SMs (one block per SM, as in the passes with the large histograms) times
// the tiles per block plus a start-up of about two tiles, so the last wave is
// not left mostly empty.
static void chunking(const TopkPlan& pl, int n_local, int* n_chunks, int* chunk_tiles, int max_tiles = 1 << 30) {
  constexpr long kSms = 152, kStartTiles = 2;
  const long base = (long)pl.n_gt * n_local;
  const int lo = std::max(1, (pl.n_tiles + max_tiles - 1) / max_tiles);
  const int hi = std::max(lo, std::min(kMaxChunks, pl.n_tiles));
  long best = -1;
  int best_ct = pl.n_tiles;
  for (int nc = lo; nc <= hi; ++nc) {
    const int ct = (pl.n_tiles + nc - 1) / nc;
    if (ct > max_tiles) continue;
    const long used = (pl.n_tiles + ct - 1) / ct;
    const long cost = ((base * used + kSms - 1) / kSms) * (ct + kStartTiles);
    if (best < 0 || cost < best) {
      best = cost;
      best_ct = ct;
    }
  }
  *chunk_tiles = best_ct;
  *n_chunks = (pl.n_tiles + best_ct - 1) / best_ct;
}

// Largest chunk count over the launches of P problems (full launches of pc
// problems and the remainder), for both the top-k and the coverage passes.
static int max_chunks_of(const TopkPlan& pl, int P) {
  int m = 1, nc, ct;
  for (int n_local : {pl.pc, P % pl.pc}) {
    if (n_local <= 0) continue;
    chunking(pl, n_local, &nc, &ct);
    m = std::max(m, nc);
    chunking(pl, n_local, &nc, &ct, kCovMaxTiles);
    m = std::max(m, nc);
  }
  return m;
}

struct TopkWs {
  float *khi, *klo, *qhi, *qlo;
  uint32_t *mmax, *mmin, *hist, *cand_cnt;
  uint32_t* cov_hist;
  float* mass;
  uint32_t *blo, *bhi, *bcount;
  int32_t *nabove, *rstate, *tflag;
  uint32_t *selb, *eqb;
  uint64_t* cand;
  int32_t* cum_cnt;
  int32_t* half_cnt;   // [n][2 * cov_bins][g_pad] half-bin counts of the coarse pass
  double* cum_mass;
  float *width, *zinv;
  int32_t *fine_cnt, *cov_win, *kwin_lo, *kwin_hi;
  double *fine_mass, *fine_scale;
  double* cov_partial;
  int32_t* cov_range;
};

// REFINE rounds: each narrows an interval by log2(bins) bits of the 32, so
// this many leave a single value.
static int refine_rounds(const TopkPlan& pl) {
  const int lg = pl.RP == 32 ? SelCfg<32>::kHistLog2 : SelCfg<64>::kHistLog2;
  return (32 + lg - 1) / lg;
}

// Carves the workspace (base == nullptr: sizing only): the projections and
// row ranges, then the top-k buffers, the coverage buffers, or both.
enum CarveMode { kCarveTopk = 1, kCarveCov = 2, kCarveBoth = 3 };
static size_t carve(void* base, const TopkPlan& pl, int mode, TopkWs* w) {
  Carver c(base);
  const size_t pc = pl.pc, S = pl.geo.S, gp = pl.g_pad, RP = pl.RP;
  w->khi = c.take<float>(pc * S * RP);
  w->klo = c.take<float>(pc * S * RP);
  w->qhi = c.take<float>(pc * gp * RP);
  w->qlo = c.take<float>(pc * gp * RP);
  w->mmax = c.take<uint32_t>(pc * gp);
  w->mmin = c.take<uint32_t>(pc * gp);
  if (mode & kCarveTopk) {
    w->hist = c.take<uint32_t>(pc * pl.hist_bins * gp);
    w->blo = c.take<uint32_t>(pc * gp);
    w->bhi = c.take<uint32_t>(pc * gp);
    w->bcount = c.take<uint32_t>(pc * gp);
    w->nabove = c.take<int32_t>(pc * gp);
    w->rstate = c.take<int32_t>(pc * gp);
    w->tflag = c.take<int32_t>((size_t)(refine_rounds(pl) + 1) * pc * pl.n_gt);
    w->cand_cnt = c.take<uint32_t>(pc * gp);
    w->cand = c.take<uint64_t>(pc * gp * kCandCap);
    w->selb = c.take<uint32_t>(pc * gp * pl.n_tiles * 4);
    w->eqb = c.take<uint32_t>(pc * gp * pl.n_tiles * 4);
  }
  if (mode & kCarveCov) {
    w->cov_hist = c.take<uint32_t>(pc * pl.max_chunks * pl.cov_bins * gp);
    w->mass = c.take<float>(pc * pl.max_chunks * pl.cov_bins * gp);
    w->cum_cnt = c.take<int32_t>(pc * gp * pl.cov_bins);
    w->half_cnt = c.take<int32_t>(pc * gp * 2 * pl.cov_bins);
    w->cum_mass = c.take<double>(pc * gp * pl.cov_bins);
    w->width = c.take<float>(pc * gp);
    w->zinv = c.take<float>(pc * gp);
    w->fine_cnt = c.take<int32_t>(pc * gp * pl.cov_bins);
    w->fine_mass = c.take<double>(pc * gp * pl.cov_bins);
    w->fine_scale = c.take<double>(pc * gp);
    w->cov_win = c.take<int32_t>(pc * gp * 4);
    w->kwin_lo = c.take<int32_t>(pc);
    w->kwin_hi = c.take<int32_t>(pc);
    // two searches can run together (the two bounds): partials and ranges for both
    w->cov_partial = c.take<double>(2 * pc * ((gp + kCovGroupsPerBlock - 1) / kCovGroupsPerBlock) * kCovPoints);
    w->cov_range = c.take<int32_t>(2 * pc * 2);
  }
  return c.used + 256;
}

template <int RP, int MODE>
static cudaError_t launch_select(dim3 grid, cudaStream_t st, const CUtensorMap* maps, const SelParams& prm,
                                 const ProblemTable& tab) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_select<RP, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SelCfg<RP>::smem(MODE));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  k_select<RP, MODE><<<grid, kSelThreads, SelCfg<RP>::smem(MODE), st>>>(maps[0], maps[1], maps[2], maps[3], prm, tab);
  return cudaGetLastError();
}

template <int MODE>
static cudaError_t select_pass(int RP, dim3 grid, cudaStream_t st, const CUtensorMap* maps, const SelParams& prm,
                               const ProblemTable& tab) {
  return RP == 32 ? launch_select<32, MODE>(grid, st, maps, prm, tab)
                  : launch_select<64, MODE>(grid, st, maps, prm, tab);
}

static cudaError_t launch_proj(int r, const void* Q, const void* K, const void* Wq, const void* Wk,
                               const dsv_shape& s, const TopkPlan& pl, const TopkWs& w, const ProblemTable& tab,
                               int32_t* status, cudaStream_t st) {
  const int n = tab.n, d = (int)s.d;
  const size_t qbytes = (size_t)n * pl.g_pad * pl.RP * sizeof(float);
  cudaError_t e = cudaMemsetAsync(w.qhi, 0, qbytes, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(w.qlo, 0, qbytes, st);
  if (e != cudaSuccess) return e;
  dim3 gk(pl.geo.S / 128, n), gq(pl.geo.n_groups, n);
  auto Qp = static_cast<const __nv_bfloat16*>(Q);
  auto Wkp = static_cast<const __nv_bfloat16*>(Wk);
  auto Wqp = static_cast<const __nv_bfloat16*>(Wq);
  static bool proj_configured = false;
  if (!proj_configured) {
    cudaFuncSetAttribute(k_key_proj<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, ProjCfg<32>::kSmem);
    cudaFuncSetAttribute(k_key_proj<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, ProjCfg<64>::kSmem);
    proj_configured = true;
  }
  // the key rows of the whole batch as a [B*H*S][d] tensor, 128-row boxes
  CUtensorMap kmap;
  if (!make_map_2d(&kmap, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d, (uint64_t)s.B * s.H * pl.geo.S, 64, 128))
    return cudaErrorInvalidValue;
  switch (r) {
    case 16:
      k_key_proj<32><<<gk, 128, ProjCfg<32>::kSmem, st>>>(kmap, Wkp, 16, s.H, d, pl.geo.S, w.khi, w.klo, status, wait_limit_ns(), tab);
      k_group_mean_proj<16><<<gq, 128, 0, st>>>(Qp, Wqp, s.H, d, pl.geo, pl.g_pad, w.qhi, w.qlo, tab);
      break;
    case 32:
      k_key_proj<32><<<gk, 128, ProjCfg<32>::kSmem, st>>>(kmap, Wkp, 32, s.H, d, pl.geo.S, w.khi, w.klo, status, wait_limit_ns(), tab);
      k_group_mean_proj<32><<<gq, 128, 0, st>>>(Qp, Wqp, s.H, d, pl.geo, pl.g_pad, w.qhi, w.qlo, tab);
      break;
    default:
      k_key_proj<64><<<gk, 128, ProjCfg<64>::kSmem, st>>>(kmap, Wkp, 64, s.H, d, pl.geo.S, w.khi, w.klo, status, wait_limit_ns(), tab);
      k_group_mean_proj<64><<<gq, 128, 0, st>>>(Qp, Wqp, s.H, d, pl.geo, pl.g_pad, w.qhi, w.qlo, tab);
      break;
  }
  return cudaGetLastError();
}

static bool make_score_maps(CUtensorMap* maps, const TopkPlan& pl, const TopkWs& w, int n) {
  const uint64_t RP = pl.RP;
  return make_map_2d(&maps[0], w.qhi, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, RP, (uint64_t)n * pl.g_pad, 32, 128) &&
         make_map_2d(&maps[1], w.qlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, RP, (uint64_t)n * pl.g_pad, 32, 128) &&
         make_map_2d(&maps[2], w.khi, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, RP, (uint64_t)n * pl.geo.S, 32, 128) &&
         make_map_2d(&maps[3], w.klo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, RP, (uint64_t)n * pl.geo.S, 32, 128);
}

static dsv_status validate_lowrank(const void* Q, const void* K, const void* Wq, const void* Wk, const dsv_shape& s,
                                   int32_t r, const dsv_group& g) {
  dsv_status v = validate_common(s, g, true);
  if (v != DSV_OK) return v;
  if (!Q || !K || !Wq || !Wk) return DSV_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(Wq, 2) || !aligned(Wk, 2)) return DSV_ERR_INVALID_ARG;
  if (r != 16 && r != 32 && r != 64) return DSV_ERR_UNSUPPORTED;
  return DSV_OK;
}

// Parameters of the score passes of one launch of problems.
static SelParams sel_params(const TopkPlan& pl, const TopkWs& w, int n_chunks, int chunk_tiles, float scale,
                            int32_t* status) {
  SelParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.geo = pl.geo;
  prm.g_pad = pl.g_pad;
  prm.n_chunks = n_chunks;
  prm.chunk_tiles = chunk_tiles;
  prm.n_tiles = pl.n_tiles;
  prm.n_gt = pl.n_gt;
  prm.scale = scale;
  prm.mmax = w.mmax;
  prm.mmin = w.mmin;
  prm.hist = w.hist;
  prm.cov_cnt = w.cov_hist;
  prm.mass = w.mass;
  prm.blo = w.blo;
  prm.bhi = w.bhi;
  prm.rstate = w.rstate;
  prm.cand_cnt = w.cand_cnt;
  prm.cand = w.cand;
  prm.sel_bits = w.selb;
  prm.eq_bits = w.eqb;
  prm.cwin = w.cov_win;
  prm.status = status;
  prm.wait_ns = wait_limit_ns();
  return prm;
}

static cudaError_t minmax_pass(const TopkPlan& pl, const TopkWs& w, const ProblemTable& tab, const CUtensorMap* maps,
                               dim3 grid, const SelParams& prm, cudaStream_t st) {
  const size_t rows = (size_t)tab.n * pl.g_pad;
  if (cudaMemsetAsync(w.mmax, 0, rows * 4, st) != cudaSuccess) return cudaErrorUnknown;
  if (cudaMemsetAsync(w.mmin, 0xFF, rows * 4, st) != cudaSuccess) return cudaErrorUnknown;
  return select_pass<kMinMax>(pl.RP, grid, st, maps, prm, tab);
}

// Top-k, once the linear histogram (nb bins) is in w.hist: the bracket and
// the REFINE rounds (group tiles with no row to refine leave at once).
// With `cov_scale` > 0 the bracket comes from the coverage pass's coarse table
// (coverage ran on these rows with that scale) instead of the histogram.
static cudaError_t topk_bracket_refine(const TopkPlan& pl, const TopkWs& w, const ProblemTable& tab,
                                       const CUtensorMap* maps, dim3 grid, SelParams prm, int nb, int32_t* status,
                                       cudaStream_t st, float cov_scale = 0.f) {
  const int n = tab.n;
  const int rounds = refine_rounds(pl);
  const int lg = pl.RP == 32 ? SelCfg<32>::kHistLog2 : SelCfg<64>::kHistLog2;
  const size_t nflag = (size_t)n * pl.n_gt;
  const dim3 rgrid(pl.n_gt, n);
  if (cov_scale > 0.f)
    k_bracket_cov<<<rgrid, 128, 0, st>>>(pl.cov_bins, pl.g_pad, pl.geo.n_groups, pl.n_gt, cov_scale, w.mmax, w.mmin,
                                         w.cum_cnt, w.half_cnt, w.hist, pl.hist_bins, w.blo, w.bhi, w.nabove, w.bcount,
                                         w.rstate,
                                         w.tflag, status, tab);
  else
    k_bracket<<<rgrid, 128, 0, st>>>(w.hist, nb, pl.g_pad, pl.geo.n_groups, pl.n_gt, w.mmin, w.mmax, w.blo, w.bhi,
                                     w.nabove, w.bcount, w.rstate, w.tflag, status, tab);
  if (cudaGetLastError() != cudaSuccess) return cudaErrorUnknown;
  for (int r = 0; r < rounds; ++r) {
    prm.tflag = w.tflag + r * nflag;
    if (select_pass<kRefine>(pl.RP, grid, st, maps, prm, tab) != cudaSuccess) return cudaErrorUnknown;
    k_refine_bracket<<<rgrid, 128, 0, st>>>(w.hist, pl.hist_bins, lg, pl.g_pad, pl.geo.n_groups, pl.n_gt, w.blo,
                                            w.bhi, w.nabove, w.bcount, w.rstate, w.tflag + r * nflag,
                                            w.tflag + (r + 1) * nflag, status, tab);
    if (cudaGetLastError() != cudaSuccess) return cudaErrorUnknown;
  }
  return cudaSuccess;
}

// Top-k, once COLLECT has run: resolve the candidates, write the index rows.
static cudaError_t topk_finish(const TopkPlan& pl, const TopkWs& w, const ProblemTable& tab, int32_t* idx,
                               int32_t* status, cudaStream_t st) {
  const int n = tab.n;
  k_resolve<<<dim3(pl.geo.n_groups, n), kResolveThreads, 0, st>>>(w.cand, w.cand_cnt, w.bhi, w.nabove, w.bcount,
                                                                    w.rstate, pl.g_pad, pl.n_tiles * 4, pl.geo.S,
                                                                    w.selb, status, tab);
  if (cudaGetLastError() != cudaSuccess) return cudaErrorUnknown;
  k_sel_compact<<<dim3(pl.geo.n_groups, n), 32 * kCompactWarps, 0, st>>>(w.selb, w.eqb, w.rstate, w.nabove, pl.g_pad,
                                                                          pl.n_tiles * 4, idx, status, tab);
  return cudaGetLastError();
}

// Memsets before the top-k histogram of one launch.
static cudaError_t topk_clear(const TopkPlan& pl, const TopkWs& w, int n, cudaStream_t st) {
  const size_t rows = (size_t)n * pl.g_pad;
  if (cudaMemsetAsync(w.hist, 0, rows * pl.hist_bins * 4, st) != cudaSuccess) return cudaErrorUnknown;
  if (cudaMemsetAsync(w.tflag, 0, (size_t)(refine_rounds(pl) + 1) * n * pl.n_gt * 4, st) != cudaSuccess)
    return cudaErrorUnknown;
  return cudaMemsetAsync(w.cand_cnt, 0, rows * 4, st);
}

// The top-k passes of one launch of problems whose projections are in the
// workspace; `minmax` = false when the row ranges are already there.
// `cov_scale` > 0: coverage has just run on the same rows with that scale,
// and its coarse table gives the bracket in place of the histogram pass.
static cudaError_t topk_passes(const TopkPlan& pl, const TopkWs& w, const ProblemTable& tab, const CUtensorMap* maps,
                               bool minmax, int32_t* idx, int32_t* status, cudaStream_t st, float cov_scale = 0.f) {
  int n_chunks, chunk_tiles;
  chunking(pl, tab.n, &n_chunks, &chunk_tiles);
  const SelParams prm = sel_params(pl, w, n_chunks, chunk_tiles, 0.f, status);
  const dim3 grid(pl.n_gt, n_chunks, tab.n);
  if (minmax && minmax_pass(pl, w, tab, maps, grid, prm, st) != cudaSuccess) return cudaErrorUnknown;
  if (topk_clear(pl, w, tab.n, st) != cudaSuccess) return cudaErrorUnknown;
  if (cov_scale <= 0.f && select_pass<kHist>(pl.RP, grid, st, maps, prm, tab) != cudaSuccess) return cudaErrorUnknown;
  if (topk_bracket_refine(pl, w, tab, maps, grid, prm, pl.hist_bins, status, st, cov_scale) != cudaSuccess)
    return cudaErrorUnknown;
  if (select_pass<kCollect>(pl.RP, grid, st, maps, prm, tab) != cudaSuccess) return cudaErrorUnknown;
  return topk_finish(pl, w, tab, idx, status, st);
}

struct CovSearch {
  int nblk, rounds;
};

static CovSearch cov_search_shape(const TopkPlan& pl) {
  CovSearch c;
  c.nblk = (pl.geo.n_groups + kCovGroupsPerBlock - 1) / kCovGroupsPerBlock;
  // rounds: the interval shrinks from S values to at most ceil(span / kCovPoints) per round
  c.rounds = 1;
  for (int64_t span = pl.geo.S; span > kCovPoints; span = (span + kCovPoints - 1) / kCovPoints) ++c.rounds;
  return c;
}

// One search (mode, answer in out) or, with `out2`, the two bound searches
// together (grid z / y selects the search; answers in out and out2).
static void cov_search(const TopkPlan& pl, const TopkWs& w, const ProblemTable& tab, int mode, bool fine,
                       float mass, int32_t* out, int32_t* out2, bool by_problem, cudaStream_t st) {
  const CovSearch cs = cov_search_shape(pl);
  const int n = tab.n, ng = pl.geo.n_groups, S = pl.geo.S, nb = pl.cov_bins;
  const int ns = out2 ? 2 : 1;
  for (int r = 0; r < cs.rounds; ++r) {
    k_cov_eval<<<dim3(cs.nblk, n, ns), kCovPoints, 0, st>>>(mode, false, nb, pl.g_pad, ng, S, w.cum_cnt,
                                                            w.cum_mass, w.width, w.zinv, w.cov_win,
                                                            fine ? w.fine_cnt : nullptr, w.fine_mass, w.cov_range, 0,
                                                            w.cov_partial);
    k_cov_pick<<<dim3(n, ns), kCovPoints, 0, st>>>(false, cs.nblk, ng, S, mass, w.cov_partial, w.cov_range, out,
                                                   out2, by_problem, nullptr, 0, tab);
  }
}

// Coverage, once the coarse pass has run: merged tables, the certified
// interval [k_lo, k_hi] from the bin-edge bounds, each group's window.
static cudaError_t cov_after_coarse(const TopkPlan& pl, const TopkWs& w, const ProblemTable& tab, int n_chunks,
                                    float scale, float mass, cudaStream_t st) {
  const int n = tab.n, nb = pl.cov_bins, ng = pl.geo.n_groups, S = pl.geo.S;
  const dim3 mgrid((ng + 127) / 128, nb, n), sgrid((ng + 7) / 8, n), wgrid((ng + 127) / 128, n);
  k_cov_merge<<<mgrid, 128, 0, st>>>(w.cov_hist, w.mass, nb, n_chunks, pl.g_pad, ng, w.cum_cnt, w.cum_mass,
                                     w.half_cnt);
  k_cov_scan<<<sgrid, 256, 0, st>>>(w.mmax, w.mmin, nb, pl.g_pad, ng, scale, w.cum_cnt, w.cum_mass, w.width, w.zinv,
                                    nullptr);
  // both bounds at once: k_lo from the upper bound, k_hi from the lower bound
  k_cov_range_init<<<2, 256, 0, st>>>(w.cov_range, nullptr, nullptr, S, 2 * n);
  cov_search(pl, w, tab, kCovBoundHi, false, mass, w.kwin_lo, w.kwin_hi, false, st);
  k_cov_window<<<wgrid, 128, 0, st>>>(nb, pl.g_pad, ng, scale, w.mmax, w.mmin, w.cum_cnt, w.cum_mass, w.kwin_lo,
                                      w.kwin_hi, w.cov_win, w.fine_scale);
  return cudaGetLastError();
}

// Coverage, once the fine pass has run: k_cov within [k_lo, k_hi] on the
// combined tables, and the curve.
static cudaError_t cov_after_fine(const TopkPlan& pl, const TopkWs& w, const ProblemTable& tab, int n_chunks,
                                  float scale, float mass, int32_t* k_cov, float* curve, int n_curve,
                                  cudaStream_t st) {
  const int n = tab.n, nb = pl.cov_bins, ng = pl.geo.n_groups, S = pl.geo.S;
  const dim3 mgrid((ng + 127) / 128, nb, n), sgrid((ng + 7) / 8, n);
  k_cov_merge<<<mgrid, 128, 0, st>>>(w.cov_hist, w.mass, nb, n_chunks, pl.g_pad, ng, w.fine_cnt, w.fine_mass,
                                     nullptr);
  k_cov_scan<<<sgrid, 256, 0, st>>>(w.mmax, w.mmin, nb, pl.g_pad, ng, scale, w.fine_cnt, w.fine_mass, nullptr,
                                    nullptr, w.fine_scale);
  k_cov_range_init<<<1, 256, 0, st>>>(w.cov_range, w.kwin_lo, w.kwin_hi, S, n);
  cov_search(pl, w, tab, kCovCombined, true, mass, k_cov, nullptr, true, st);
  if (curve) {
    const CovSearch cs = cov_search_shape(pl);
    k_cov_eval<<<dim3(cs.nblk, n), kCovPoints, 0, st>>>(kCovCombined, true, nb, pl.g_pad, ng, S, w.cum_cnt,
                                                        w.cum_mass, w.width, w.zinv, w.cov_win, w.fine_cnt,
                                                        w.fine_mass, w.cov_range, n_curve, w.cov_partial);
    k_cov_pick<<<n, kCovPoints, 0, st>>>(true, cs.nblk, ng, S, mass, w.cov_partial, w.cov_range, k_cov, nullptr,
                                          true, curve, n_curve, tab);
  }
  return cudaGetLastError();
}

// The coverage passes of one launch of problems whose projections are in the
// workspace; `minmax` = false when the row ranges are already there.
static cudaError_t cov_passes(const TopkPlan& pl, const TopkWs& w, const ProblemTable& tab, const CUtensorMap* maps,
                              bool minmax, float scale, float mass, int32_t* k_cov, float* curve, int n_curve,
                              int32_t* status, cudaStream_t st) {
  int n_chunks, chunk_tiles;
  chunking(pl, tab.n, &n_chunks, &chunk_tiles, kCovMaxTiles);
  const SelParams prm = sel_params(pl, w, n_chunks, chunk_tiles, scale, status);
  const dim3 grid(pl.n_gt, n_chunks, tab.n);
  if (minmax && minmax_pass(pl, w, tab, maps, grid, prm, st) != cudaSuccess) return cudaErrorUnknown;
  if (select_pass<kCov>(pl.RP, grid, st, maps, prm, tab) != cudaSuccess) return cudaErrorUnknown;
  if (cov_after_coarse(pl, w, tab, n_chunks, scale, mass, st) != cudaSuccess) return cudaErrorUnknown;
  if (select_pass<kCovFine>(pl.RP, grid, st, maps, prm, tab) != cudaSuccess) return cudaErrorUnknown;
  return cov_after_fine(pl, w, tab, n_chunks, scale, mass, k_cov, curve, n_curve, st);
}

}  // namespace dsv

using namespace dsv;

extern "C" size_t dsv_lowrank_topk_workspace_size(dsv_shape shape, int32_t r, dsv_group group) {
  if (validate_common(shape, group, true) != DSV_OK || (r != 16 && r != 32 && r != 64)) return 0;
  TopkPlan pl = make_plan(shape, r, group);
  TopkWs w;
  return carve(nullptr, pl, kCarveTopk, &w);
}

extern "C" size_t dsv_coverage_workspace_size(dsv_shape shape, int32_t r, dsv_group group) {
  if (validate_common(shape, group, true) != DSV_OK || (r != 16 && r != 32 && r != 64)) return 0;
  TopkPlan pl = make_plan(shape, r, group);
  TopkWs w;
  return carve(nullptr, pl, kCarveCov, &w);
}

extern "C" size_t dsv_coverage_topk_workspace_size(dsv_shape shape, int32_t r, dsv_group group) {
  if (validate_common(shape, group, true) != DSV_OK || (r != 16 && r != 32 && r != 64)) return 0;
  TopkPlan pl = make_plan(shape, r, group);
  TopkWs w;
  return carve(nullptr, pl, kCarveBoth, &w);
}

extern "C" dsv_status dsv_lowrank_topk(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr,
                                       dsv_shape shape, int32_t r, dsv_group group, const int32_t* k_per_head,
                                       const int64_t* idx_offset, int32_t* idx, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status, void* stream) {
  dsv_status v = validate_lowrank(Q, K, Wq_lr, Wk_lr, shape, r, group);
  if (v != DSV_OK) return v;
  if (!k_per_head || !idx_offset || !idx || !aligned(idx, 4)) return DSV_ERR_INVALID_ARG;
  const TopkPlan pl = make_plan(shape, r, group);
  const int P = (int)(shape.B * shape.H);
  const int S = pl.geo.S;
  for (int p = 0; p < P; ++p)
    if (idx_offset[p] >= 0 && (k_per_head[p] < 1 || k_per_head[p] > S)) return DSV_ERR_INVALID_ARG;
  TopkWs w;
  const size_t need = carve(nullptr, pl, kCarveTopk, &w);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DSV_ERR_WORKSPACE;
  carve(workspace, pl, kCarveTopk, &w);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  std::vector<int> active;
  for (int p = 0; p < P; ++p) {
    if (idx_offset[p] < 0) continue;
    if (k_per_head[p] == S) {
      const int64_t total = (int64_t)pl.geo.n_groups * S;
      k_fill_all<<<1216, 256, 0, st>>>(idx, idx_offset[p], S, total);
      if (cudaGetLastError() != cudaSuccess) return DSV_ERR_CUDA;
      continue;
    }
    active.push_back(p);
  }
  for (size_t c0 = 0; c0 < active.size(); c0 += pl.pc) {
    ProblemTable tab;
    memset(&tab, 0, sizeof(tab));
    tab.n = (int)std::min<size_t>(pl.pc, active.size() - c0);
    for (int i = 0; i < tab.n; ++i) {
      const int p = active[c0 + i];
      tab.p[i] = p;
      tab.k[i] = k_per_head[p];
      tab.off[i] = idx_offset[p];
    }
    if (launch_proj(r, Q, K, Wq_lr, Wk_lr, shape, pl, w, tab, dev_status, st) != cudaSuccess) return DSV_ERR_CUDA;
    CUtensorMap maps[4];
    if (!make_score_maps(maps, pl, w, tab.n)) return DSV_ERR_CUDA;
    if (topk_passes(pl, w, tab, maps, true, idx, dev_status, st) != cudaSuccess) return DSV_ERR_CUDA;
  }
  return DSV_OK;
}

extern "C" dsv_status dsv_coverage(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr,
                                   dsv_shape shape, int32_t r, dsv_group group, float scale, float mass,
                                   int32_t* k_cov, float* curve, int32_t n_curve, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_status, void* stream) {
  dsv_status v = validate_lowrank(Q, K, Wq_lr, Wk_lr, shape, r, group);
  if (v != DSV_OK) return v;
  if (!k_cov || !(scale > 0.f) || !(mass > 0.f && mass <= 1.f)) return DSV_ERR_INVALID_ARG;
  if (curve && (n_curve < 1 || n_curve > 1024)) return DSV_ERR_INVALID_ARG;
  const TopkPlan pl = make_plan(shape, r, group);
  if (pl.n_tiles > kMaxChunks * kCovMaxTiles) return DSV_ERR_UNSUPPORTED;
  TopkWs w;
  const size_t need = carve(nullptr, pl, kCarveCov, &w);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DSV_ERR_WORKSPACE;
  carve(workspace, pl, kCarveCov, &w);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int P = (int)(shape.B * shape.H);
  for (int c0 = 0; c0 < P; c0 += pl.pc) {
    ProblemTable tab;
    memset(&tab, 0, sizeof(tab));
    tab.n = std::min(pl.pc, P - c0);
    for (int i = 0; i < tab.n; ++i) {
      tab.p[i] = c0 + i;
      tab.k[i] = 1;
      tab.off[i] = 0;
    }
    if (launch_proj(r, Q, K, Wq_lr, Wk_lr, shape, pl, w, tab, dev_status, st) != cudaSuccess) return DSV_ERR_CUDA;
    CUtensorMap maps[4];
    if (!make_score_maps(maps, pl, w, tab.n)) return DSV_ERR_CUDA;
    if (cov_passes(pl, w, tab, maps, true, scale, mass, k_cov, curve, n_curve, dev_status, st) != cudaSuccess)
      return DSV_ERR_CUDA;
  }
  return DSV_OK;
}

extern "C" dsv_status dsv_coverage_topk(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr,
                                        dsv_shape shape, int32_t r, dsv_group group, float scale, float mass,
                                        int32_t* k_cov, float* curve, int32_t n_curve, const int32_t* k_per_head,
                                        const int64_t* idx_offset, int32_t* idx, void* workspace,
                                        size_t workspace_bytes, int32_t* dev_status, void* stream) {
  dsv_status v = validate_lowrank(Q, K, Wq_lr, Wk_lr, shape, r, group);
  if (v != DSV_OK) return v;
  if (!k_cov || !(scale > 0.f) || !(mass > 0.f && mass <= 1.f)) return DSV_ERR_INVALID_ARG;
  if (curve && (n_curve < 1 || n_curve > 1024)) return DSV_ERR_INVALID_ARG;
  if (!k_per_head || !idx_offset || !idx || !aligned(idx, 4)) return DSV_ERR_INVALID_ARG;
  const TopkPlan pl = make_plan(shape, r, group);
  if (pl.n_tiles > kMaxChunks * kCovMaxTiles) return DSV_ERR_UNSUPPORTED;
  const int P = (int)(shape.B * shape.H);
  const int S = pl.geo.S;
  bool all_selected = true;   // every problem takes a proper top-k (no dense head, no k = S)
  for (int p = 0; p < P; ++p) {
    if (idx_offset[p] >= 0 && (k_per_head[p] < 1 || k_per_head[p] > S)) return DSV_ERR_INVALID_ARG;
    all_selected = all_selected && idx_offset[p] >= 0 && k_per_head[p] < S;
  }
  TopkWs w;
  const size_t need = carve(nullptr, pl, kCarveBoth, &w);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DSV_ERR_WORKSPACE;
  if (!all_selected) {
    // problem tables differ between the two: run them one after the other
    v = dsv_coverage(Q, K, Wq_lr, Wk_lr, shape, r, group, scale, mass, k_cov, curve, n_curve, workspace,
                     workspace_bytes, dev_status, stream);
    if (v != DSV_OK) return v;
    return dsv_lowrank_topk(Q, K, Wq_lr, Wk_lr, shape, r, group, k_per_head, idx_offset, idx, workspace,
                            workspace_bytes, dev_status, stream);
  }
  carve(workspace, pl, kCarveBoth, &w);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int c0 = 0; c0 < P; c0 += pl.pc) {
    ProblemTable tab;
    memset(&tab, 0, sizeof(tab));
    tab.n = std::min(pl.pc, P - c0);
    for (int i = 0; i < tab.n; ++i) {
      tab.p[i] = c0 + i;
      tab.k[i] = k_per_head[c0 + i];
      tab.off[i] = idx_offset[c0 + i];
    }
    // one projection and one row-range pass serve both
    if (launch_proj(r, Q, K, Wq_lr, Wk_lr, shape, pl, w, tab, dev_status, st) != cudaSuccess) return DSV_ERR_CUDA;
    CUtensorMap maps[4];
    if (!make_score_maps(maps, pl, w, tab.n)) return DSV_ERR_CUDA;
    if (cov_passes(pl, w, tab, maps, true, scale, mass, k_cov, curve, n_curve, dev_status, st) != cudaSuccess)
      return DSV_ERR_CUDA;
    // the coverage pass's coarse table brackets the k-th score: no histogram pass
    if (topk_passes(pl, w, tab, maps, false, idx, dev_status, st, scale) != cudaSuccess) return DSV_ERR_CUDA;
  }
  return DSV_OK;
}

// ---------------------------------------------------------------------------
// Per-query predicted mass: workspace and launches.
namespace dsv {

struct MassWs {
  float *khi, *klo, *qhi, *qlo;
  uint32_t *mmax, *mmin, *bits;
  float* msum;
  double* bsum;
};

// The score passes of the per-query rows: one 128-query tile per row tile.
static TopkPlan query_plan(const TopkPlan& pl) {
  TopkPlan q = pl;
  q.n_gt = pl.geo.S / 128;
  q.g_pad = pl.geo.S;
  return q;
}

// Problems per launch: the key and query projections within the budget.
static int mass_problems_per_launch(const TopkPlan& pl, int P) {
  const size_t per = (size_t)pl.geo.S * pl.RP * 16;
  return (int)std::max<size_t>(1, std::min<size_t>((size_t)P, kProjBudget / per));
}

static size_t carve_mass(void* base, const TopkPlan& pl, int P, MassWs* w) {
  const TopkPlan qp = query_plan(pl);
  const int pc = mass_problems_per_launch(pl, P);
  int max_chunks = 1, nc, ct;
  for (int n_local : {pc, P % pc}) {
    if (n_local <= 0) continue;
    chunking(qp, n_local, &nc, &ct);
    max_chunks = std::max(max_chunks, nc);
  }
  Carver c(base);
  const size_t S = pl.geo.S, RP = pl.RP, n = pc;
  w->khi = c.take<float>(n * S * RP);
  w->klo = c.take<float>(n * S * RP);
  w->qhi = c.take<float>(n * S * RP);
  w->qlo = c.take<float>(n * S * RP);
  w->mmax = c.take<uint32_t>(n * S);
  w->mmin = c.take<uint32_t>(n * S);
  w->bits = c.take<uint32_t>(n * pl.geo.n_groups * (S / 32));
  w->msum = c.take<float>(n * max_chunks * S * 2);
  w->bsum = c.take<double>(n * ((S + kMassThreadsR - 1) / kMassThreadsR));
  return c.used + 256;
}

}  // namespace dsv

extern "C" size_t dsv_predicted_mass_workspace_size(dsv_shape shape, int32_t r, dsv_group group) {
  if (validate_common(shape, group, true) != DSV_OK || (r != 16 && r != 32 && r != 64)) return 0;
  const TopkPlan pl = make_plan(shape, r, group);
  MassWs w;
  return carve_mass(nullptr, pl, (int)(shape.B * shape.H), &w);
}

extern "C" dsv_status dsv_predicted_mass(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr,
                                         dsv_shape shape, int32_t r, dsv_group group, const int32_t* idx,
                                         const int32_t* k_per_head, const int64_t* idx_offset, float scale,
                                         float* mass, float* per_query, void* workspace, size_t workspace_bytes,
                                         int32_t* dev_status, void* stream) {
  dsv_status v = validate_lowrank(Q, K, Wq_lr, Wk_lr, shape, r, group);
  if (v != DSV_OK) return v;
  if (!mass || !(scale > 0.f) || !aligned(mass, 4) || (per_query && !aligned(per_query, 4)))
    return DSV_ERR_INVALID_ARG;
  if (idx && (!k_per_head || !idx_offset || !aligned(idx, 4))) return DSV_ERR_INVALID_ARG;
  const TopkPlan pl = make_plan(shape, r, group);
  const Geometry& geo = pl.geo;
  const int P = (int)(shape.B * shape.H), S = geo.S, d = (int)shape.d;
  if (S > 262144) return DSV_ERR_UNSUPPORTED;   // a group's bitmap is built in 32 KB of shared memory
  if (idx)
    for (int p = 0; p < P; ++p)
      if (idx_offset[p] >= 0 && (k_per_head[p] < 1 || k_per_head[p] > S)) return DSV_ERR_INVALID_ARG;
  MassWs w;
  const size_t need = carve_mass(nullptr, pl, P, &w);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DSV_ERR_WORKSPACE;
  carve_mass(workspace, pl, P, &w);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const TopkPlan qp = query_plan(pl);
  const int pc = mass_problems_per_launch(pl, P);
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(k_key_proj<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, ProjCfg<32>::kSmem);
    cudaFuncSetAttribute(k_key_proj<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, ProjCfg<64>::kSmem);
    cudaFuncSetAttribute(k_query_proj<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, ProjCfg<32>::kSmem);
    cudaFuncSetAttribute(k_query_proj<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, ProjCfg<64>::kSmem);
    configured = true;
  }
  CUtensorMap kmap, qcube;
  if (!make_map_2d(&kmap, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d, (uint64_t)P * S, 64, 128) ||
      !make_cube_map(&qcube, Q, geo, d, P))
    return DSV_ERR_CUDA;
  auto Wk = static_cast<const __nv_bfloat16*>(Wk_lr);
  auto Wq = static_cast<const __nv_bfloat16*>(Wq_lr);
  const uint64_t lim = wait_limit_ns();
  for (int c0 = 0; c0 < P; c0 += pc) {
    ProblemTable tab;
    memset(&tab, 0, sizeof(tab));
    tab.n = std::min(pc, P - c0);
    for (int i = 0; i < tab.n; ++i) {
      const int p = c0 + i;
      const bool dense = !idx || idx_offset[p] < 0;
      tab.p[i] = p;
      tab.k[i] = dense ? S : k_per_head[p];
      tab.off[i] = dense ? -1 : idx_offset[p];
    }
    const int n = tab.n;
    const dim3 pgrid(S / 128, n);
    if (pl.RP == 32) {
      k_key_proj<32><<<pgrid, 128, ProjCfg<32>::kSmem, st>>>(kmap, Wk, r, shape.H, d, S, w.khi, w.klo, dev_status,
                                                              lim, tab);
      k_query_proj<32><<<pgrid, 128, ProjCfg<32>::kSmem, st>>>(qcube, Wq, r, shape.H, d, geo, w.qhi, w.qlo,
                                                                dev_status, lim, tab);
    } else {
      k_key_proj<64><<<pgrid, 128, ProjCfg<64>::kSmem, st>>>(kmap, Wk, r, shape.H, d, S, w.khi, w.klo, dev_status,
                                                              lim, tab);
      k_query_proj<64><<<pgrid, 128, ProjCfg<64>::kSmem, st>>>(qcube, Wq, r, shape.H, d, geo, w.qhi, w.qlo,
                                                                dev_status, lim, tab);
    }
    k_idx_bitmap<<<dim3(geo.n_groups, n), 256, (size_t)(S / 32) * 4, st>>>(idx, S, geo.n_groups, w.bits, tab);
    if (cudaGetLastError() != cudaSuccess) return DSV_ERR_CUDA;
    const uint64_t RP = pl.RP;
    CUtensorMap maps[4];
    if (!make_map_2d(&maps[0], w.qhi, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, RP, (uint64_t)n * S, 32, 128) ||
        !make_map_2d(&maps[1], w.qlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, RP, (uint64_t)n * S, 32, 128) ||
        !make_map_2d(&maps[2], w.khi, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, RP, (uint64_t)n * S, 32, 128) ||
        !make_map_2d(&maps[3], w.klo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, RP, (uint64_t)n * S, 32, 128))
      return DSV_ERR_CUDA;
    int n_chunks, chunk_tiles;
    chunking(qp, n, &n_chunks, &chunk_tiles);
    SelParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.geo = geo;
    prm.geo.n_groups = S;   // rows of the score tiles are single queries
    prm.g_pad = S;
    prm.n_chunks = n_chunks;
    prm.chunk_tiles = chunk_tiles;
    prm.n_tiles = pl.n_tiles;
    prm.n_gt = qp.n_gt;
    prm.scale = scale;
    prm.mmax = w.mmax;
    prm.mmin = w.mmin;
    prm.qsel = w.bits;
    prm.msum = w.msum;
    prm.q_group = geo.G;
    prm.qn_groups = geo.n_groups;
    prm.status = dev_status;
    prm.wait_ns = lim;
    const dim3 grid(qp.n_gt, n_chunks, n);
    if (cudaMemsetAsync(w.mmax, 0, (size_t)n * S * 4, st) != cudaSuccess) return DSV_ERR_CUDA;
    if (cudaMemsetAsync(w.mmin, 0xFF, (size_t)n * S * 4, st) != cudaSuccess) return DSV_ERR_CUDA;
    if (select_pass<kMinMax>(pl.RP, grid, st, maps, prm, tab) != cudaSuccess) return DSV_ERR_CUDA;
    if (select_pass<kMass>(pl.RP, grid, st, maps, prm, tab) != cudaSuccess) return DSV_ERR_CUDA;
    const int nblk = (S + kMassThreadsR - 1) / kMassThreadsR;
    k_mass_reduce<<<dim3(nblk, n), kMassThreadsR, 0, st>>>(w.msum, n_chunks, geo, per_query, w.bsum, tab);
    k_mass_mean<<<n, 32, 0, st>>>(w.bsum, nblk, S, mass, tab);
    if (cudaGetLastError() != cudaSuccess) return DSV_ERR_CUDA;
  }
  return DSV_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of dsv_lowrank_topk.
//
// Some callers cannot allocate device memory at the point where they need a
// top-k: a plugin whose enqueue step may not allocate, a serving loop whose
// device memory budget is fixed at start-up, or an embedding runtime that owns
// every allocation itself. For them the scratch lives in the fixed array below,
// reserved in the library's own device image: every GPU that loads this code
// holds kStaticScratchBytes of it until the process exits.
namespace dsv {

constexpr size_t kStaticScratchBytes = 64ull << 20;   // 64 MiB
static __device__ __align__(256) uint8_t g_topk_scratch[kStaticScratchBytes];

// Unique id of the calling thread's current CUDA context, 0 when there is
// none yet or the driver cannot report it. A device reset or a context torn
// down and made again gives a new id.
static unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_topk_scratch for the current device. The host-side name
// is only a stand-in, so the address is looked up through the runtime, with
// the device current: once per device and context (the first lookup also
// loads this module there). The cached address is keyed by the context's id,
// so after a device reset the next call looks it up again instead of using an
// address of the old context; when no id can be read, every call looks it up.
static void* static_scratch_address(cudaError_t* err) {
  static std::mutex mu;
  static void* addr[128] = {};
  static unsigned long long ctx_of[128] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long id = current_context_id();
  if (!addr[dev] || id == 0 || ctx_of[dev] != id) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
    ctx_of[dev] = current_context_id();   // the lookup made the device's primary context current
  }
  return addr[dev];
}

}  // namespace dsv

extern "C" dsv_status dsv_lowrank_topk_noalloc(const void* Q, const void* K, const void* Wq_lr, const void* Wk_lr,
                                               dsv_shape shape, int32_t r, dsv_group group,
                                               const int32_t* k_per_head, const int64_t* idx_offset, int32_t* idx,
                                               int32_t* dev_status, void* stream) {
  dsv_status v = validate_lowrank(Q, K, Wq_lr, Wk_lr, shape, r, group);
  if (v != DSV_OK) return v;
  const size_t need = dsv_lowrank_topk_workspace_size(shape, r, group);
  if (need == 0) return DSV_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return DSV_ERR_WORKSPACE;   // shape needs more than the fixed scratch
  cudaError_t err = cudaSuccess;
  void* scratch = static_scratch_address(&err);
  if (!scratch) return DSV_ERR_CUDA;
  return dsv_lowrank_topk(Q, K, Wq_lr, Wk_lr, shape, r, group, k_per_head, idx_offset, idx, scratch,
                          kStaticScratchBytes, dev_status, stream);
}
