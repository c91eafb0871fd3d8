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
// Survivor lists live one entry per lane of one warp; candidate lists and their
// scores live in a shared-memory scratch of 2*kMaxK entries.  Top-K is a rank
// count: candidate i survives iff fewer than K candidates beat it, where j beats
// i when score_j > score_i, or the scores are equal and j has the lower node
// index (the lowest index wins ties).
#pragma once

#include "common.cuh"

namespace pisa {

struct __align__(16) WarpScratch {
  int cand[2 * kMaxK];
  float score[2 * kMaxK];
  int next[kMaxK];
};

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
      const float4* s4 = reinterpret_cast<const float4*>(ws.score);  // 4 scores per load
      for (int q4 = 0; 4 * q4 < nC; ++q4) {
        const float4 o = s4[q4];
        const int q = 4 * q4;
        rank += (q < nC && (o.x > sc || (o.x == sc && q < ci)));
        rank += (q + 1 < nC && (o.y > sc || (o.y == sc && q + 1 < ci)));
        rank += (q + 2 < nC && (o.z > sc || (o.z == sc && q + 2 < ci)));
        rank += (q + 3 < nC && (o.w > sc || (o.w == sc && q + 3 < ci)));
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

}  // namespace pisa
