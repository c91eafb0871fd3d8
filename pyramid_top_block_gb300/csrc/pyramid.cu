// pyramid.cu -- fine-to-coarse mean pooling of the keys into the PISA pyramid.
//
// "Block Sparse Attention with Log-Linear Complexity", §3.1 Fine to coarse:
// level 1 holds leaf blocks of C tokens, each the mean of its keys; every level
// above merges g = 2 adjacent blocks; each summary equals the mean of all the
// raw keys it covers.  A ragged node (the sequence tail) is the mean over the
// tokens present, i.e. children merge with token-count weights.
//
// Data flow (HBM-bound: K is read exactly once):
//   pyramid_leaves_kernel : one CTA per group of LPB consecutive leaves.  Each
//       thread owns 8 consecutive features (one 16-byte bf16 vector) of one KV
//       head and sums that column over the leaf's tokens in token order, so a
//       warp reads whole 256-byte token rows.  The CTA then merges its LPB
//       leaves up log2(LPB) levels in shared memory.
//   pyramid_top_col_kernel: one warp per (b, kv, feature) merges the remaining
//       levels up to the root, three in each lane's registers, five by shuffles;
//   pyramid_top_kernel    : the same level by level through global memory, for
//       layouts whose merged-in-CTA level is larger (many KV heads).
// Divisions by a power-of-two count are exact multiplications (div_count), the
// same bits as the division.
#include <mutex>

#include "api.cuh"

namespace pisa {

// Largest power of two LPB with LPB * Hkv <= 32 (so LPB * Hkv * 8 <= 256 threads).
__host__ __device__ inline int leaves_per_block(int Hkv) {
  int lpb = 1;
  while (lpb * 2 * Hkv <= 32) lpb *= 2;
  return lpb;
}

__global__ void __launch_bounds__(256) pyramid_leaves_kernel(
    const __nv_bfloat16* __restrict__ keys, float* __restrict__ summ, Levels lv, long long N,
    long long n_cap, int Hkv, int lpb, int merge_levels, const int32_t* __restrict__ lens) {
  extern __shared__ float sm[];  // [lpb][Hkv][64]
  const int chunks = Hkv * 8;
  const int tid = threadIdx.x;
  const int c = tid % chunks;
  const int kv = c >> 3;
  const int c8 = c & 7;
  const int jl = tid / chunks;  // local leaf
  const int b = blockIdx.y;
  const long long leaf = (long long)blockIdx.x * lpb + jl;
  // ragged batch: sequence b holds lens[b] tokens (clamped to [0, n_cap]); nodes past its
  // own level sizes are left untouched
  if (lens) N = min((long long)max(lens[b], 0), n_cap);
  const long long M1 = level_size_for(N, 1);
  float* blk = summ + ((long long)b * Hkv + kv) * lv.total * kD;

  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (jl < lpb && leaf < M1) {
    const int cnt = node_count(1, leaf, N);
    const __nv_bfloat16* src = keys + (((long long)b * n_cap + leaf * kC) * Hkv + kv) * kD + c8 * 8;
    const long long stride = (long long)Hkv * kD;
    for (int r0 = 0; r0 < cnt; r0 += 16) {
      uint4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u)
        v[u] = (r0 + u < cnt) ? __ldg(reinterpret_cast<const uint4*>(src + (r0 + u) * stride))
                              : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        if (r0 + u < cnt) {
          float f[8];
          unpack8(v[u], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = div_count(acc[i], cnt);
    float4* dst = reinterpret_cast<float4*>(blk + (lv.off[1] + leaf) * kD + c8 * 8);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  if (jl < lpb) {
#pragma unroll
    for (int i = 0; i < 8; ++i) sm[(jl * Hkv + kv) * kD + c8 * 8 + i] = acc[i];
  }
  // In-CTA merges: level l node j (local) <- children 2j, 2j+1 of level l-1.
  for (int l = 2; l <= merge_levels + 1; ++l) {
    const int nodes = lpb >> (l - 1);
    const long long i = (long long)blockIdx.x * nodes + jl;
    const bool active = jl < nodes && i < level_size_for(N, l);
    float out[8];
    __syncthreads();
    if (active) {
      const long long c0 = 2 * i, c1 = 2 * i + 1;
      const int n0 = node_count(l - 1, c0, N);
      const int n1 = c1 < level_size_for(N, l - 1) ? node_count(l - 1, c1, N) : 0;
      const float* s0 = sm + ((2 * jl) * Hkv + kv) * kD + c8 * 8;
      const float* s1 = sm + ((2 * jl + 1) * Hkv + kv) * kD + c8 * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) out[e] = merge_mean(s0[e], n0, n1 > 0 ? s1[e] : 0.f, n1);
    }
    __syncthreads();
    if (active) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sm[(jl * Hkv + kv) * kD + c8 * 8 + e] = out[e];
      float4* dst = reinterpret_cast<float4*>(blk + (lv.off[l] + i) * kD + c8 * 8);
      dst[0] = make_float4(out[0], out[1], out[2], out[3]);
      dst[1] = make_float4(out[4], out[5], out[6], out[7]);
    }
  }
}

// Levels first_level .. L for one (b, kv) per CTA, level by level.
__global__ void __launch_bounds__(256) pyramid_top_kernel(float* __restrict__ summ, Levels lv,
                                                           long long N, int Hkv, int first_level,
                                                           const int32_t* __restrict__ lens, long long n_cap) {
  const int b = blockIdx.x / Hkv, kv = blockIdx.x % Hkv;
  if (lens) N = min((long long)max(lens[b], 0), n_cap);
  float* blk = summ + ((long long)b * Hkv + kv) * lv.total * kD;
  for (int l = first_level; l <= lv.L; ++l) {
    const long long M = level_size_for(N, l), Mc = level_size_for(N, l - 1);
    for (long long w = threadIdx.x; w < M * kD; w += blockDim.x) {
      const long long i = w / kD;
      const int e = (int)(w % kD);
      const long long c0 = 2 * i, c1 = 2 * i + 1;
      const int n0 = node_count(l - 1, c0, N);
      const int n1 = c1 < Mc ? node_count(l - 1, c1, N) : 0;
      const float m0 = blk[(lv.off[l - 1] + c0) * kD + e];
      const float m1 = n1 > 0 ? blk[(lv.off[l - 1] + c1) * kD + e] : 0.f;
      blk[(lv.off[l] + i) * kD + e] = merge_mean(m0, n0, m1, n1);
    }
    __syncthreads();
  }
}

constexpr int kTopNodes = 256;  // largest input level the column kernel below takes (32 lanes x 8 nodes)

// The same levels, one warp per (b, kv, feature): lane j holds nodes [8 j, 8 j + 8) of
// the input level (at most kTopNodes nodes) for one feature, merges them three levels
// up in its registers, then five more levels by shuffles between lanes (writing every
// node it forms).  Same merges in the same pairs, hence the same bits as the kernels
// above; a warp's chain is eight merges long instead of a CTA's thirty-one.
constexpr int kColWarps = 8;  // warps (feature columns) per CTA
__global__ void __launch_bounds__(kColWarps * 32) pyramid_top_col_kernel(float* __restrict__ summ, Levels lv,
                                                                         long long N, int Hkv, int first_level,
                                                                         const int32_t* __restrict__ lens,
                                                                         long long n_cap, int columns) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = blockIdx.x * kColWarps + warp;  // (b * Hkv + kv) * kD + feature
  if (col >= columns) return;  // warp-uniform
  const int bkv = col / kD, f = col % kD;
  const int b = bkv / Hkv;
  if (lens) N = min((long long)max(lens[b], 0), n_cap);
  float* blk = summ + (long long)bkv * lv.total * kD + f;
  const int L = lv.L;
  const int l0 = first_level - 1;  // the input level
  const long long M0 = level_size_for(N, l0);
  float v[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const long long node = 8LL * lane + u;
    v[u] = node < M0 ? blk[(lv.off[l0] + node) * kD] : 0.f;
  }
  // three levels inside the lane: 8 -> 4 -> 2 -> 1 nodes
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int l = first_level + j;
    if (l <= L) {
      const long long M = level_size_for(N, l), Mc = level_size_for(N, l - 1);
      const int cnt = 4 >> j;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i < cnt) {
          const long long node = (long long)cnt * lane + i;
          const long long c0 = 2 * node, c1 = 2 * node + 1;
          const int n0 = c0 < Mc ? node_count(l - 1, c0, N) : 0;
          const int n1 = c1 < Mc ? node_count(l - 1, c1, N) : 0;
          v[i] = merge_mean(v[2 * i], n0, v[2 * i + 1], n1);
          if (node < M) blk[(lv.off[l] + node) * kD] = v[i];
        }
      }
    }
  }
  // five levels across lanes: node lane >> (j + 1) from the lanes 2^j apart
  float x = v[0];
#pragma unroll
  for (int j = 0; j < 5; ++j) {
    const int l = first_level + 3 + j;
    const float y = __shfl_down_sync(kFull, x, 1 << j);
    if (l <= L && (lane & ((2 << j) - 1)) == 0) {
      const long long M = level_size_for(N, l), Mc = level_size_for(N, l - 1);
      const long long node = lane >> (j + 1);
      const long long c0 = 2 * node, c1 = 2 * node + 1;
      const int n0 = c0 < Mc ? node_count(l - 1, c0, N) : 0;
      const int n1 = c1 < Mc ? node_count(l - 1, c1, N) : 0;
      x = merge_mean(x, n0, y, n1);
      if (node < M) blk[(lv.off[l] + node) * kD] = x;
    }
  }
}

__global__ void fill_lengths_kernel(int32_t* lengths, int B, int value) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < B) lengths[i] = value;
}

// Host launcher (declared in api.cuh).
cudaError_t launch_build_pyramid(const __nv_bfloat16* keys, float* summ, const Levels& lv,
                                 long long N, long long n_cap, int B, int Hkv, int32_t* lengths,
                                 cudaStream_t s, bool ragged) {
  const int32_t* lens = ragged ? lengths : nullptr;  // per-sequence lengths read on the device
  const int lpb = leaves_per_block(Hkv);
  int merge_levels = 0;
  while ((1 << (merge_levels + 1)) <= lpb) ++merge_levels;
  if (merge_levels > lv.L - 1) merge_levels = lv.L - 1;
  const long long M1 = lv.M[1];
  dim3 grid((unsigned)((M1 + lpb - 1) / lpb), (unsigned)B);
  const int threads = lpb * Hkv * 8;
  const size_t smem = (size_t)lpb * Hkv * kD * sizeof(float);
  pyramid_leaves_kernel<<<grid, threads, smem, s>>>(keys, summ, lv, N, n_cap, Hkv, lpb, merge_levels, lens);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (merge_levels + 2 <= lv.L) {
    const int first = merge_levels + 2;
    if (lv.M[first - 1] <= kTopNodes && lv.L - first + 1 <= 8) {
      const int columns = B * Hkv * kD;
      pyramid_top_col_kernel<<<(columns + kColWarps - 1) / kColWarps, kColWarps * 32, 0, s>>>(summ, lv, N, Hkv, first,
                                                                                             lens, n_cap, columns);
    } else {
      pyramid_top_kernel<<<B * Hkv, 256, 0, s>>>(summ, lv, N, Hkv, first, lens, n_cap);
    }
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (lengths && !ragged) {
    fill_lengths_kernel<<<(B + 127) / 128, 128, 0, s>>>(lengths, B, (int)N);
    note_launch();
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace pisa
