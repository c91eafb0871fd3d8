// common.cuh -- shared device helpers of the GB300 PISA selector.
//
// Fixed geometry of the library: head dim d = 64, leaf size C = 64, merge
// factor g = 2 ("Block Sparse Attention with Log-Linear Complexity", §7.3:
// d = 64, C = 64, g = 2).  A node of level l >= 1 spans 64 * 2^(l-1) tokens;
// level 0 is the raw keys.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pisa.h"

namespace pisa {

constexpr int kD = 64;          // head dimension
constexpr int kC = 64;          // leaf size (tokens)
constexpr int kLog2C = 6;
constexpr int kMaxLevels = 32;  // N <= 2^30 tokens -> at most 25 levels
constexpr int kMaxK = 32;
constexpr float kScale = 0.125f;  // 1/sqrt(64), exact in fp32
constexpr unsigned kFull = 0xffffffffu;  // all lanes of a warp

// Level geometry passed by value to kernels.  Sizes M[l] are those of the
// current sequence length; row offsets off[l] come from the capacity n_cap so
// that a decode cache keeps its layout while it grows.
struct Levels {
  int L;                         // levels that hold nodes for the current length
  int M[kMaxLevels + 1];         // M[l], l = 1..L (M[0] = tokens)
  long long off[kMaxLevels + 1]; // row offset of level l inside one (b, kv) block
  long long total;               // rows per (b, kv) block (from n_cap)
};

// M_1 = ceil(n / C), M_l = ceil(M_{l-1} / 2) = ceil(n / (C * 2^(l-1))).
__host__ __device__ inline int num_levels_for(long long n) {
  long long m = (n + kC - 1) >> kLog2C;
  int L = 1;
  while (m > 1) {
    m = (m + 1) >> 1;
    ++L;
  }
  return L;
}

__host__ __device__ inline long long level_size_for(long long n, int l) {
  if (l == 0) return n;
  const int sh = kLog2C + l - 1;  // a node of level l spans 2^sh tokens
  return (n + (1LL << sh) - 1) >> sh;
}

// First token of node i at level l (level 0: the raw key i itself).
__host__ __device__ inline long long node_start(int l, long long i) {
  return l == 0 ? i : (i << (kLog2C + l - 1));
}

// Tokens node i of level l holds when the sequence has n tokens.
__host__ __device__ inline int node_count(int l, long long i, long long n) {
  long long s = node_start(l, i);
  long long e = (i + 1) << (kLog2C + l - 1);
  if (e > n) e = n;
  return (int)(e - s);
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Unpack 8 bf16 held in a 16-byte vector into fp32 (exact).
__device__ __forceinline__ void unpack8(const uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Token-count-weighted mean of two children (exact formula, no contraction):
// parent = (m0 * n0 + m1 * n1) / (n0 + n1).  A parent with one child equals it.
// Shared by the prefill build and the decode path update so both produce the
// same bits for the same node.
// s / n correctly rounded.  When n is a power of two its reciprocal is exact and the
// product rounds the same exact quotient, so it gives the bits of the division.
__device__ __forceinline__ float div_count(float s, int n) {
  return (n & (n - 1)) == 0 ? __fmul_rn(s, __int_as_float((127 - (__ffs(n) - 1)) << 23)) : __fdiv_rn(s, (float)n);
}

__device__ __forceinline__ float merge_mean(float m0, int n0, float m1, int n1) {
  if (n1 <= 0) return m0;
  float s = __fadd_rn(__fmul_rn(m0, (float)n0), __fmul_rn(m1, (float)n1));
  return div_count(s, n0 + n1);
}

// Record a device-side error in the caller's workspace status word (first
// error wins).
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Debug builds (-DPISA_DEBUG_BOUNDS): every gathered index is range-checked on the
// device; a failed check records PISA_ERR_DEVICE_BOUNDS in the status word of the
// call (its address set by the launcher into this translation unit's copy of
// g_bounds_status) and the access is replaced by a harmless one.  Nothing traps.  In
// the default build the checks are not compiled.
#ifdef PISA_DEBUG_BOUNDS
static __device__ int* g_bounds_status;
__device__ __forceinline__ bool in_bounds(bool ok) {
  if (!ok) set_status(g_bounds_status, PISA_ERR_DEVICE_BOUNDS);
  return ok;
}
#define PISA_IN_BOUNDS(cond) (::pisa::in_bounds(cond))
#define PISA_SET_BOUNDS_STATUS(ptr, stream)                                                              \
  do {                                                                                                   \
    int* p_ = (ptr);                                                                                     \
    cudaMemcpyToSymbolAsync(::pisa::g_bounds_status, &p_, sizeof(p_), 0, cudaMemcpyHostToDevice, stream); \
  } while (0)
#else
#define PISA_IN_BOUNDS(cond) (true)
#define PISA_SET_BOUNDS_STATUS(ptr, stream) \
  do {                                      \
  } while (0)
#endif

}  // namespace pisa
