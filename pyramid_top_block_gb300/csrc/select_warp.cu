// select_warp.cu -- the decode step: one warp walks the cached pyramid for the
// newest query of a sequence.  Each (b, kv, t) walk is one warp; the arithmetic
// is fp32 on the CUDA cores with bf16 inputs, fp32 summaries and fp32
// accumulation ("Block Sparse Attention with Log-Linear Complexity", §7.3: dot
// products accumulated in FP32).
#include "api.cuh"
#include "walk.cuh"

namespace pisa {

// One decode step for one (b, kv): append k_new at position n = lengths[b],
// refresh the leaf mean and its ancestor path (the decoding design keeps the
// mean pyramid cached and touches only the new token's path), then walk for
// the query at t = n over the n+1 tokens present.  Threads 0..63 own one
// feature each for the path update; warp 0 runs the walk.
template <int G>
__global__ void __launch_bounds__(64) decode_kernel(
    const __nv_bfloat16* __restrict__ q_new, const __nv_bfloat16* __restrict__ k_new,
    __nv_bfloat16* keys, float* summ, const int32_t* __restrict__ lengths, Levels cap_lv,
    long long n_cap, int Hq, int Hkv, int K, int32_t* __restrict__ idx, float* __restrict__ scores,
    int* status) {
  __shared__ __align__(16) float qs[G * kD];
  __shared__ WarpScratch scratch;
  const int b = blockIdx.x / Hkv, kv = blockIdx.x % Hkv;
  const int tid = threadIdx.x, lane = tid & 31;
  const long long p = lengths[b];
  int32_t* io = idx + (long long)blockIdx.x * K;
  float* so = scores ? scores + (long long)blockIdx.x * K : nullptr;
  if (p < 0 || p >= n_cap) {  // sequence full: leave it unchanged, report
    if (tid == 0) set_status(status, PISA_ERR_DEVICE_BOUNDS);
    if (tid < K) {
      io[tid] = -1;
      if (so) so[tid] = -INFINITY;
    }
    return;
  }
  const long long n = p + 1;
  Levels lv;
  lv.L = num_levels_for(n);
  lv.total = cap_lv.total;
  for (int l = 0; l <= lv.L; ++l) {
    lv.M[l] = (int)level_size_for(n, l);
    lv.off[l] = cap_lv.off[l];
  }
  __nv_bfloat16* keys_b = keys + (long long)b * n_cap * Hkv * kD;
  float* blk = summ + ((long long)b * Hkv + kv) * cap_lv.total * kD;
  {  // path update: feature e = tid
    const int e = tid;
    const __nv_bfloat16 kn = k_new[((long long)b * Hkv + kv) * kD + e];
    keys_b[(p * Hkv + kv) * kD + e] = kn;
    const long long leaf = p >> kLog2C;
    float acc = 0.f;
    for (long long r = leaf * kC; r <= p; ++r) acc = __fadd_rn(acc, bf2f(keys_b[(r * Hkv + kv) * kD + e]));
    float m = __fdiv_rn(acc, (float)(p - leaf * kC + 1));
    blk[(lv.off[1] + leaf) * kD + e] = m;
    long long i = leaf;
    for (int l = 2; l <= lv.L; ++l) {
      const long long child = i;
      i >>= 1;
      const long long c0 = 2 * i, c1 = 2 * i + 1;
      const int n0 = node_count(l - 1, c0, n);
      const int n1 = c1 < lv.M[l - 1] ? node_count(l - 1, c1, n) : 0;
      const float m0 = c0 == child ? m : blk[(lv.off[l - 1] + c0) * kD + e];
      const float m1 = n1 > 0 ? (c1 == child ? m : blk[(lv.off[l - 1] + c1) * kD + e]) : 0.f;
      m = merge_mean(m0, n0, m1, n1);
      blk[(lv.off[l] + i) * kD + e] = m;
    }
  }
  const __nv_bfloat16* qrow = q_new + ((long long)b * Hq + (long long)kv * G) * kD;
  for (int i = tid; i < G * kD; i += blockDim.x) qs[i] = bf2f(qrow[i]);
  __threadfence_block();
  __syncthreads();
  if (tid >= 32) return;
  int myS;
  const int nS = warp_walk_intermediate<G>(blk, lv, qs, p, K, true, scratch, lane, &myS);
  warp_leaf_select<G>(keys_b, Hkv, kv, lv, qs, p, n, K, true, nS, myS, scratch, lane, io, so);
}

__global__ void bump_lengths_kernel(int32_t* lengths, int B, long long n_cap) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B && lengths[b] >= 0 && lengths[b] < n_cap) lengths[b] += 1;
}

// ---------------------------------------------------------------- launchers

template <int G>
static cudaError_t launch_decode_G(const __nv_bfloat16* q_new, const __nv_bfloat16* k_new,
                                   __nv_bfloat16* keys, float* summ, int32_t* lengths,
                                   const Levels& cap_lv, long long n_cap, int B, int Hq, int Hkv,
                                   int K, int32_t* idx, float* scores, int* status, cudaStream_t s) {
  decode_kernel<G><<<B * Hkv, 64, 0, s>>>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, Hq, Hkv,
                                          K, idx, scores, status);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bump_lengths_kernel<<<(B + 127) / 128, 128, 0, s>>>(lengths, B, n_cap);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_decode_warp(const __nv_bfloat16* q_new, const __nv_bfloat16* k_new,
                               __nv_bfloat16* keys, float* summ, int32_t* lengths,
                               const Levels& cap_lv, long long n_cap, int B, int Hq, int Hkv, int K,
                               int32_t* idx, float* scores, int* status, cudaStream_t s) {
  switch (Hq / Hkv) {
    case 1: return launch_decode_G<1>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, s);
    case 2: return launch_decode_G<2>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, s);
    case 4: return launch_decode_G<4>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, s);
    case 8: return launch_decode_G<8>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, s);
    case 16: return launch_decode_G<16>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pisa
