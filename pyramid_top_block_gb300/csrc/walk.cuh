// walk.cuh -- warp-level building blocks of the coarse-to-fine Top-K walk.
//
// "Block Sparse Attention with Log-Linear Complexity", §3.2 Coarse to fine:
// selection starts at the root; each level only considers the children of the
// previous level's survivors (at most g*K candidates), keeps the K best and
// expands them; a level with at most K candidates is kept without scoring.
// "Scoring: LogSumExp": a candidate's score is log sum exp of q.kbar over its
// children's summaries (raw keys at the leaf level).  §4.1: the scores of the
// query heads that share a KV head are summed.
//
// One warp owns one (b, kv, t) walk.  Survivor lists live one entry per lane;
// candidate lists and their scores live in a per-warp shared-memory scratch of
// 2*kMaxK entries.  Top-K is a rank count: candidate i survives iff fewer than
// K candidates beat it, where j beats i when score_j > score_i, or the scores
// are equal and j has the lower node index (the lowest index wins ties).
#pragma once

#include "common.cuh"

namespace pisa {

struct WarpScratch {
  int cand[2 * kMaxK];
  float score[2 * kMaxK];
  int next[kMaxK];
};

// fp32 dot products of one fp32 summary row with the G query heads in smem.
template <int G>
__device__ __forceinline__ void dot_summary(const float* row, const float* qs, float* z) {
  float k[kD];
  const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll
  for (int j = 0; j < kD / 4; ++j) {
    float4 v = r4[j];
    k[4 * j] = v.x;
    k[4 * j + 1] = v.y;
    k[4 * j + 2] = v.z;
    k[4 * j + 3] = v.w;
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < kD; ++j) a = fmaf(qs[h * kD + j], k[j], a);
    z[h] = a * kScale;
  }
}

// fp32 dot products of one bf16 key row with the G query heads in smem.
template <int G>
__device__ __forceinline__ void dot_key(const __nv_bfloat16* row, const float* qs, float* z) {
  float k[kD];
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
#pragma unroll
  for (int j = 0; j < kD / 8; ++j) unpack8(r4[j], k + 8 * j);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < kD; ++j) a = fmaf(qs[h * kD + j], k[j], a);
    z[h] = a * kScale;
  }
}

// Head-summed LSE score of candidate c at level l >= 2: children 2c (always
// eligible when c is) and 2c+1 (if it exists and, when causal, starts <= t).
template <int G>
__device__ float score_intermediate(const float* blk, const Levels& lv, int l, long long c,
                                    const float* qs, long long t, bool causal) {
  float z0[G], z1[G];
  const long long r0 = 2 * c, r1 = 2 * c + 1;
  dot_summary<G>(blk + (lv.off[l - 1] + r0) * kD, qs, z0);
  const bool has1 = r1 < lv.M[l - 1] && (!causal || node_start(l - 1, r1) <= t);
  float sc = 0.f;
  if (has1) {
    dot_summary<G>(blk + (lv.off[l - 1] + r1) * kD, qs, z1);
#pragma unroll
    for (int h = 0; h < G; ++h) sc += lse2(z0[h], z1[h]);
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) sc += z0[h];
  }
  return sc;
}

// Exact leaf score: sum over heads of log sum exp over the raw keys of leaf c
// that lie below n_eff (n_eff = min(N, t+1) when causal).  All lanes return it.
template <int G>
__device__ float warp_leaf_score(const __nv_bfloat16* keys_b, int Hkv, int kv, long long c,
                                 long long n_eff, const float* qs, int lane) {
  const long long r0 = c * kC + lane, r1 = r0 + 32;
  const bool a0 = r0 < n_eff, a1 = r1 < n_eff;
  float z0[G], z1[G];
  if (a0) dot_key<G>(keys_b + (r0 * Hkv + kv) * kD, qs, z0);
  if (a1) dot_key<G>(keys_b + (r1 * Hkv + kv) * kD, qs, z1);
  float total = 0.f;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float m = fmaxf(a0 ? z0[h] : -INFINITY, a1 ? z1[h] : -INFINITY);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    float e = (a0 ? expf(z0[h] - m) : 0.f) + (a1 ? expf(z1[h] - m) : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(kFull, e, o);
    total += m + logf(e);
  }
  return total;
}

// Rank-count Top-K over ws.cand/score[0..nC): writes the K survivors in
// ascending candidate order to ws.next and returns the survivor held by this
// lane (lane < K).  Candidates must already be in ascending node order.
__device__ __forceinline__ void warp_topk(WarpScratch& ws, int nC, int K, int lane) {
  bool sel[2];
  unsigned m[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int ci = lane + 32 * s;
    sel[s] = false;
    if (ci < nC) {
      const float sc = ws.score[ci];
      int rank = 0;
      for (int j = 0; j < nC; ++j) {
        const float o = ws.score[j];
        rank += (o > sc) || (o == sc && j < ci);
      }
      sel[s] = rank < K;
    }
    m[s] = __ballot_sync(kFull, sel[s]);
  }
  const unsigned lt = (1u << lane) - 1u;
  const int p0 = __popc(m[0] & lt);
  const int p1 = __popc(m[0]) + __popc(m[1] & lt);
  const int c0 = ws.cand[lane];
  const int c1 = lane + 32 < nC ? ws.cand[lane + 32] : 0;
  __syncwarp();
  if (sel[0]) ws.next[p0] = c0;
  if (sel[1]) ws.next[p1] = c1;
  __syncwarp();
}

// Candidates of the next level: the children of the survivors S (lane j holds
// S[j], j < nS) that exist below M and are eligible.  Writes them ascending to
// ws.cand and returns their number.
__device__ __forceinline__ int warp_expand(WarpScratch& ws, int nS, int myS, int level, long long M,
                                           long long t, bool causal, int lane) {
  const bool v0 = lane < nS;
  const long long c1 = 2LL * myS + 1;
  const bool v1 = v0 && c1 < M && (!causal || node_start(level, c1) <= t);
  const unsigned b1 = __ballot_sync(kFull, v1);
  const int pos = lane + __popc(b1 & ((1u << lane) - 1u));
  const int nC = nS + __popc(b1);
  __syncwarp();
  if (v0) {
    ws.cand[pos] = 2 * myS;
    if (v1) ws.cand[pos + 1] = (int)c1;
  }
  __syncwarp();
  return nC;
}

// The walk over the intermediate levels L-1 .. 2 for one query.  On return,
// lanes j < nS hold the level-2 survivors S_2[j] (ascending) in *myS; when the
// tree has fewer than 3 levels S_2 is the root {0} (for a single leaf, a
// virtual level-2 parent 0 whose only child is leaf 0).
template <int G>
__device__ int warp_walk_intermediate(const float* blk, const Levels& lv, const float* qs, long long t,
                                      int K, bool causal, WarpScratch& ws, int lane, int* myS_out) {
  int nS = 1;
  int myS = 0;
  for (int l = lv.L - 1; l >= 2; --l) {
    const int nC = warp_expand(ws, nS, myS, l, lv.M[l], t, causal, lane);
    if (nC <= K) {  // at most K candidates: keep them all, unscored
      nS = nC;
      myS = lane < nC ? ws.cand[lane] : 0;
      __syncwarp();
      continue;
    }
    for (int ci = lane; ci < nC; ci += 32)
      ws.score[ci] = score_intermediate<G>(blk, lv, l, ws.cand[ci], qs, t, causal);
    __syncwarp();
    warp_topk(ws, nC, K, lane);
    nS = K;
    myS = lane < K ? ws.next[lane] : 0;
    __syncwarp();
  }
  *myS_out = myS;
  return nS;
}

// Leaf level: candidates = eligible children of S_2; score them exactly when
// there are more than K (or when scores are requested), keep the Top-K and
// write them ascending with -1 / -inf padding.
template <int G>
__device__ void warp_leaf_select(const __nv_bfloat16* keys_b, int Hkv, int kv, const Levels& lv,
                                 const float* qs, long long t, long long N, int K, bool causal,
                                 int nS, int myS, WarpScratch& ws, int lane, int32_t* idx_out,
                                 float* score_out) {
  const int nC = warp_expand(ws, nS, myS, 1, lv.M[1], t, causal, lane);
  const long long n_eff = causal ? (t + 1 < N ? t + 1 : N) : N;
  const bool need_scores = nC > K || score_out != nullptr;
  if (need_scores) {
    for (int ci = 0; ci < nC; ++ci) {
      const float sc = warp_leaf_score<G>(keys_b, Hkv, kv, ws.cand[ci], n_eff, qs, lane);
      if (lane == 0) ws.score[ci] = sc;
    }
    __syncwarp();
  }
  int nOut;
  if (nC > K) {
    warp_topk(ws, nC, K, lane);
    nOut = K;
  } else {
    if (lane < nC) ws.next[lane] = ws.cand[lane];
    nOut = nC;
    __syncwarp();
  }
  if (lane < K) {
    const int leaf = lane < nOut ? ws.next[lane] : -1;
    idx_out[lane] = leaf;
    if (score_out) {
      float sc = -INFINITY;
      if (leaf >= 0) {
        // find the candidate slot of this leaf (candidates are ascending)
        for (int ci = 0; ci < nC; ++ci)
          if (ws.cand[ci] == leaf) sc = ws.score[ci];
      }
      score_out[lane] = sc;
    }
  }
  __syncwarp();
}

}  // namespace pisa
