// Shared host/device definitions of libdsv: problem tables, token geometry,
// validation helpers and workspace carving.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/libdsv.h"
#include "ptx.cuh"

namespace dsv {

constexpr int kMaxProblems = 256;                     // B*H per call
constexpr uint64_t kWaitLimitNs = 2000000000ull;      // default limit of a bounded wait (2 s)
// Limit of the waits that drain copies and MMAs a block has already issued,
// after one of its pipeline waits ran out: those complete whatever the
// pipeline's state, so this one does not follow the settable limit.
constexpr uint64_t kDrainLimitNs = 2000000000ull;

// Per-problem table passed by value as a kernel parameter (3 KB).
struct ProblemTable {
  int32_t n;                     // problems in this launch
  int32_t p[kMaxProblems];       // global problem index (b*H + h)
  int32_t k[kMaxProblems];       // keys per group (S for dense)
  int64_t off[kMaxProblems];     // idx offset of row (p, 0); -1 = dense
};

// Token geometry of the latent grid and the query-group cubes.
struct Geometry {
  int32_t T, Y, X, gt, gy, gx;
  int32_t S, G, n_groups, nct, ncy, ncx;
};

__host__ __device__ inline Geometry make_geometry(const dsv_shape& s, const dsv_group& g) {
  Geometry q;
  q.T = (int32_t)s.T; q.Y = (int32_t)s.Y; q.X = (int32_t)s.X;
  q.gt = g.gt; q.gy = g.gy; q.gx = g.gx;
  q.S = q.T * q.Y * q.X;
  q.G = g.gt * g.gy * g.gx;
  q.nct = q.T / g.gt; q.ncy = q.Y / g.gy; q.ncx = q.X / g.gx;
  q.n_groups = q.nct * q.ncy * q.ncx;
  return q;
}

// Token position of member `t` (0..G-1, (t,y,x) lexicographic) of group `g`.
__host__ __device__ inline int32_t token_of(const Geometry& q, int32_t g, int32_t t) {
  const int32_t ct = g / (q.ncy * q.ncx), cy = (g / q.ncx) % q.ncy, cx = g % q.ncx;
  const int32_t a = t / (q.gy * q.gx), b = (t / q.gx) % q.gy, c = t % q.gx;
  return ((ct * q.gt + a) * q.Y + cy * q.gy + b) * q.X + cx * q.gx + c;
}

// Raises the caller's device status word (never lowers it).
__device__ __forceinline__ void raise_status(int32_t* st, int32_t code) {
  if (st) atomicMax(st, code);
}
// Raises a consistency-check failure only when nothing was raised before:
// after a wait ran out, the later kernels of the call see incomplete data,
// and the status word keeps reporting the cause.
__device__ __forceinline__ void raise_status_if_clear(int32_t* st, int32_t code) {
  if (st && atomicAdd(st, 0) == 0) atomicMax(st, code);
}

// Float -> uint32 with the same ordering (-0 and +0 must be unified first).
__host__ __device__ __forceinline__ uint32_t f2ord(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__host__ __device__ __forceinline__ float ord2f(uint32_t o) {
  uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

// ------------------------------------------------------------ host helpers
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Carves consecutive 256-byte aligned regions out of a workspace.
struct Carver {
  char* base;
  size_t used = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <class T>
  T* take(size_t count) {
    used = round_up(used, 256);
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += count * sizeof(T);
    return p;
  }
};

// Checks shape/group/pointers common to every call. Returns DSV_OK or the error.
dsv_status validate_common(const dsv_shape& s, const dsv_group& g, bool need_d_supported);

// The pipeline wait limit passed to every kernel launched from now on
// (kWaitLimitNs unless dsv_set_wait_limit_ns changed it).
uint64_t wait_limit_ns();

// Returns the driver's tensor-map encoder (resolved once).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// 2D bf16/fp32 tensor map over a row-major [rows][cols] matrix with a box of
// box_rows x box_cols and 128-byte swizzle. Returns false on failure.
bool make_map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t cols,
                 uint64_t rows, uint32_t box_cols, uint32_t box_rows);

}  // namespace dsv
