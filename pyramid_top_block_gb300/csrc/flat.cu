// flat.cu -- the flat block selector, the conventional stage-1 baseline the pyramid
// walk replaces ("PISA cuts block-sparse attention selection to O(N log N) ...":
// block-sparse attention such as BSA scores all N/C key blocks for every query).
// Every eligible leaf gets the exact leaf score of "Block Sparse Attention with
// Log-Linear Complexity", Scoring: LogSumExp (raw-key LSE summed over the group's
// heads, keys after t masked when causal), and the K best are kept, ties to the
// lower index, listed ascending with -1 padding.
//
// The scores come from the same tcgen05 leaf kernel as the pyramid's leaf level:
// tiles of R = 128 / max(G, 8) consecutive query positions against every key block
// (two sibling leaves) that any of them can see, described in closed form.
#include "api.cuh"

namespace pisa {

// Tiles of one (b, kv) before query group qg.  Group qg (positions [qg R, qg R + R))
// needs key blocks p < P(qg): P = qg / u + 1 with u = 128 / R groups per block when
// causal (the block of the group's last position), M2 otherwise.
__host__ __device__ inline long long flat_tiles_before(long long qg, int u, long long M2, bool causal) {
  if (!causal) return qg * M2;
  const long long a = qg / u, rem = qg % u;
  return (long long)u * a * (a + 1) / 2 + rem * (a + 1);
}

__global__ void flat_list_kernel(uint32_t* __restrict__ list, long long N) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < N) list[t] = (uint32_t)t << 5;
}

// Tile i of (b, kv) = i / T1: {first position, rows, key block p, b * Hkv + kv}.
// total[0..1] = {0, tile count}: the leaf kernel's tile range.
__global__ void flat_desc_kernel(int4* __restrict__ desc, int* __restrict__ total, long long T1, int BH,
                                 long long N, int R, int u, long long M2, int causal) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0) {
    total[0] = 0;
    total[1] = (int)(T1 * BH);
  }
  if (i >= T1 * BH) return;
  const int bh = (int)(i / T1);
  const long long j = i % T1;
  long long qg, p;
  if (!causal) {
    qg = j / M2;
    p = j % M2;
  } else {
    // block a of u groups holds the groups with a + 1 tiles each, from u a (a + 1) / 2 on
    long long a = (long long)((sqrt(8.0 * (double)j / u + 1.0) - 1.0) * 0.5);
    while (a > 0 && (long long)u * a * (a + 1) / 2 > j) --a;
    while ((long long)u * (a + 1) * (a + 2) / 2 <= j) ++a;
    const long long r = j - (long long)u * a * (a + 1) / 2;
    qg = a * u + r / (a + 1);
    p = r % (a + 1);
  }
  const long long rows = N - qg * R < R ? N - qg * R : R;
  desc[i] = make_int4((int)(qg * R), (int)rows, (int)p, bh);
}

// Order of the Top-K: higher score first, lower index on equal scores.
__device__ __forceinline__ bool flat_better(float sa, int ia, float sb, int ib) {
  return sa > sb || (sa == sb && ia < ib);
}

// One warp per (b, kv, t): K rounds, each taking the best leaf below the previous
// winner in that order (a warp-wide argmax over the row of leaf scores).
__global__ void flat_topk_kernel(const float* __restrict__ leaf, long long jobs, long long N, long long stride,
                                 int M1, int K, int causal, int32_t* __restrict__ idx, float* __restrict__ scores) {
  const long long job = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (job >= jobs) return;
  const long long t = job % N;
  const int nc = causal ? (int)min((long long)M1, (t >> kLog2C) + 1) : M1;
  const float* row = leaf + job * stride;
  float ps = INFINITY;  // previous winner (score, index); every leaf is below (+inf, -1)
  int pi = -1;
  float my_s = -INFINITY;
  int my_i = -1;
  for (int r = 0; r < K; ++r) {
    float bs = -INFINITY;
    int bi = -1;
    for (int c = lane; c < nc; c += 32) {
      const float sc = row[c];
      if (flat_better(ps, pi, sc, c) && (bi < 0 || flat_better(sc, c, bs, bi))) {
        bs = sc;
        bi = c;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(kFull, bs, o);
      const int oi = __shfl_xor_sync(kFull, bi, o);
      if (oi >= 0 && (bi < 0 || flat_better(os, oi, bs, bi))) {
        bs = os;
        bi = oi;
      }
    }
    if (lane == r) {
      my_s = bs;
      my_i = bi;
    }
    ps = bs;
    pi = bi;
  }
  // lane r < K holds the r-th winner (or -1): write the winners in ascending leaf order
  const bool have = lane < K && my_i >= 0;
  int pos = 0;
  for (int o = 0; o < K; ++o) {
    const int oi = __shfl_sync(kFull, my_i, o);
    pos += (oi >= 0 && oi < my_i) ? 1 : 0;
  }
  const int nsel = __popc(__ballot_sync(kFull, have));
  int32_t* io = idx + job * K;
  float* so = scores ? scores + job * K : nullptr;
  if (have) {
    io[pos] = my_i;
    if (so) so[pos] = my_s;
  }
  if (lane >= nsel && lane < K) {
    io[lane] = -1;
    if (so) so[lane] = -INFINITY;
  }
}

cudaError_t launch_select_flat(const LeafTcLaunch& L, long long T1, long long stride, int* total,
                               cudaStream_t s) {
  const int G = L.Hq / L.Hkv;
  const int Gp = G < 8 ? 8 : G;
  const int R = 128 / Gp;
  const int BH = L.B * L.Hkv;
  flat_list_kernel<<<(unsigned)((L.N + 255) / 256), 256, 0, s>>>(L.list, L.N);
  note_launch();
  const long long T = T1 * BH;
  flat_desc_kernel<<<(unsigned)((T + 255) / 256), 256, 0, s>>>(L.tile_desc, total, T1, BH, L.N, R, 128 / R,
                                                               L.M2, L.causal);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  LeafTcLaunch F = L;
  F.tile_off = total;
  F.b0 = 0;
  F.b1 = 1;
  e = launch_leaf_tc_kernel(F, 1, stride, s);
  if (e != cudaSuccess) return e;
  const long long jobs = (long long)BH * L.N;
  flat_topk_kernel<<<(unsigned)((jobs * 32 + 255) / 256), 256, 0, s>>>(L.leaf_scores, jobs, L.N, stride,
                                                                       (int)level_size_for(L.N, 1), L.K, L.causal,
                                                                       L.idx, L.scores);
  note_launch();
  return cudaGetLastError();
}

long long flat_tiles_per_bh(long long N, int G, int K_unused, bool causal) {
  (void)K_unused;
  const int Gp = G < 8 ? 8 : G;
  const int R = 128 / Gp;
  const long long groups = (N + R - 1) / R;
  return flat_tiles_before(groups, 128 / R, level_size_for(N, 2), causal);
}

}  // namespace pisa
