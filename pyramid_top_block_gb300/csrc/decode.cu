// decode.cu -- the decode step: append one key per sequence, refresh its leaf
// and ancestor path, and walk the cached pyramid for the newest query.
// "Block Sparse Attention with Log-Linear Complexity", §5.1 (decoding keeps the
// mean pyramid cached and touches only the new token's path) and §3.2 / Scoring
// / §4.1 for the walk.  bf16 inputs, fp32 summaries (the path update on the CUDA
// cores), dot products on mma.sync with fp32 accumulation.
//
// One CTA of kDecWarps warps per (b, kv).  Threads 0..63 update the path (one
// feature each).  Warps 0..kWalkWarps - 1 then walk the intermediate levels: every
// level's candidates are scored four to a warp on mma.sync (query heads as the A
// operand, the children's fp32 summary rows as bf16 high + low B columns), every
// walking warp ranks the same scores and expands the same survivors itself, so a
// level costs one barrier of the walking warps.  The other warps are handed the
// level-2 candidates and ask their leaves' keys into L2 meanwhile; then all warps
// score the leaf candidates exactly (mma.sync, the query heads as rows and a leaf's
// 64 keys as 8 column tiles) and warp 0 ranks them.  The step is a chain of
// dependent memory round trips (the new length, the path, one per level, the leaf
// keys) on a grid of B * Hkv CTAs.
#include "api.cuh"
#include "tc.cuh"

namespace pisa {

constexpr int kDecWarps = 16;
constexpr int kWalkWarps = 4;  // warps that walk the intermediate levels
constexpr int kPfThreads = (kDecWarps - kWalkWarps + 1) * 32;  // warp 0 + the other warps, at named barrier 2

// bf16 m16n8k16 MMA with fp32 accumulation (D = A B + C).
__device__ __forceinline__ void dec_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The query heads of this (b, kv) as the A operand of q . k: rows g and g + 8 of
// the fragment are heads g and g + 8 (zero beyond G); k-step ks takes the bf16
// pairs (words) 8 j + 2 ks and 8 j + 2 ks + 1 of a row, so a lane's words of every
// k-step are one contiguous 32-byte slice of each row.
template <int G>
__device__ __forceinline__ void leaf_q_frags(const __nv_bfloat16* q_bkv, int lane, uint32_t (&A)[4][4]) {
  const int g = lane >> 2, j = lane & 3;
  uint4 h0[2] = {}, h1[2] = {};
  if (g < G) {
    const uint4* r = reinterpret_cast<const uint4*>(q_bkv + g * kD) + 2 * j;
    h0[0] = r[0];
    h0[1] = r[1];
  }
  if (g + 8 < G) {
    const uint4* r = reinterpret_cast<const uint4*>(q_bkv + (g + 8) * kD) + 2 * j;
    h1[0] = r[0];
    h1[1] = r[1];
  }
  const uint32_t w0[8] = {h0[0].x, h0[0].y, h0[0].z, h0[0].w, h0[1].x, h0[1].y, h0[1].z, h0[1].w};
  const uint32_t w1[8] = {h1[0].x, h1[0].y, h1[0].z, h1[0].w, h1[1].x, h1[1].y, h1[1].z, h1[1].w};
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    A[ks][0] = w0[2 * ks];
    A[ks][1] = w1[2 * ks];
    A[ks][2] = w0[2 * ks + 1];
    A[ks][3] = w1[2 * ks + 1];
  }
}

// Exact leaf score on the tensor cores: sum over heads of log sum exp over the raw
// keys of leaf c below n.  S[16 heads x 64 keys] = Q K^T in 8 tiles of 8 keys (the
// B operand of tile nt: key 8 nt + g, the lane's 32-byte slice of its row), fp32
// accumulation of the exact bf16 products; then per head a max / sum over the
// lane's 16 keys and the lane quad, and the head sum over g.
template <int G>
__device__ __forceinline__ float warp_leaf_mma(const __nv_bfloat16* keys_b, int Hkv, int kv, long long c, long long n,
                                               const uint32_t (&A)[4][4], int lane) {
  const int g = lane >> 2, j = lane & 3;
  if (!PISA_IN_BOUNDS(c >= 0 && c * kC < n)) c = 0;
  float z[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const long long r = c * kC + 8 * nt + g;
    uint4 k0 = make_uint4(0, 0, 0, 0), k1 = k0;
    if (r < n) {
      const uint4* kp = reinterpret_cast<const uint4*>(keys_b + (r * Hkv + kv) * kD) + 2 * j;
      k0 = kp[0];
      k1 = kp[1];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) z[nt][i] = 0.f;
    dec_mma(z[nt], A[0], k0.x, k0.y);
    dec_mma(z[nt], A[1], k0.z, k0.w);
    dec_mma(z[nt], A[2], k1.x, k1.y);
    dec_mma(z[nt], A[3], k1.z, k1.w);
  }
  // z[nt][e] = head g, key 8 nt + 2 j + e; z[nt][2 + e] = head g + 8, same key
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const bool in = c * kC + 8 * nt + 2 * j + e < n;
      z[nt][e] = in ? z[nt][e] * kScale : -INFINITY;
      z[nt][2 + e] = in ? z[nt][2 + e] * kScale : -INFINITY;
      m0 = fmaxf(m0, z[nt][e]);
      m1 = fmaxf(m1, z[nt][2 + e]);
    }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    m0 = fmaxf(m0, __shfl_xor_sync(kFull, m0, o));
    m1 = fmaxf(m1, __shfl_xor_sync(kFull, m1, o));
  }
  float e0 = 0.f, e1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      e0 += ex2_approx((z[nt][e] - m0) * 1.4426950408889634f);
      e1 += ex2_approx((z[nt][2 + e] - m1) * 1.4426950408889634f);
    }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    e0 += __shfl_xor_sync(kFull, e0, o);
    e1 += __shfl_xor_sync(kFull, e1, o);
  }
  float v = (g < G ? m0 + lg2_approx(e0) * 0.69314718055994531f : 0.f) +
            (g + 8 < G ? m1 + lg2_approx(e1) * 0.69314718055994531f : 0.f);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Scores of candidates 4 tile .. 4 tile + 3 at level l (children at level l - 1, rows1,
// M1 rows) on mma.sync: the query heads are the A operand (qa, as for the leaf scores), the
// 8 children rows the B columns (column g: child g & 1 of candidate 4 tile + (g >> 1); a
// lane takes dims 16 j .. 16 j + 15 of it, the same k order as the A fragments).  The fp32
// summaries enter as bf16 high and low parts (x = hi + lo to 16 bits), two MMAs per
// k-step.  After the MMAs lane (g, j) holds heads g and g + 8 of both children of candidate
// 4 tile + j: the two-child log-sum-exp per head, then the head sum over g.  While the rows
// are in flight the children's own children (rows2, level l - 2) are asked into L1.
template <int G>
__device__ __forceinline__ void tile_node_scores(const float* rows1, long long M1, const float* rows2, long long M2,
                                                 const int* cand, int nC, int tile, const uint32_t (&qa)[4][4],
                                                 int lane, float* sc) {
  const int g = lane >> 2, j = lane & 3;
  const int cb = 4 * tile + (g >> 1);
  const int c = cb < nC ? cand[cb] : -1;
  const long long child = 2LL * c + (g & 1);
  const bool have = c >= 0 && PISA_IN_BOUNDS(child < M1 || (g & 1));
  float4 x[4];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) x[ks] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (have && child < M1) {
    const float4* r = reinterpret_cast<const float4*>(rows1 + child * kD) + 4 * j;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) x[ks] = r[ks];
    if (rows2 != nullptr) {
      const long long gc = 2 * child + (j >> 1);
      if (gc < M2) asm volatile("prefetch.global.L1 [%0];" ::"l"(rows2 + gc * kD + (j & 1) * (kD / 2)));
    }
  }
  float dh[4] = {0.f, 0.f, 0.f, 0.f}, dl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(x[ks].x, x[ks].y), h1 = __floats2bfloat162_rn(x[ks].z, x[ks].w);
    const uint32_t u0 = *reinterpret_cast<const uint32_t*>(&h0), u1 = *reinterpret_cast<const uint32_t*>(&h1);
    const __nv_bfloat162 l0 = __floats2bfloat162_rn(x[ks].x - __uint_as_float(u0 << 16),
                                                    x[ks].y - __uint_as_float(u0 & 0xffff0000u));
    const __nv_bfloat162 l1 = __floats2bfloat162_rn(x[ks].z - __uint_as_float(u1 << 16),
                                                    x[ks].w - __uint_as_float(u1 & 0xffff0000u));
    dec_mma(dh, qa[ks], u0, u1);
    dec_mma(dl, qa[ks], *reinterpret_cast<const uint32_t*>(&l0), *reinterpret_cast<const uint32_t*>(&l1));
  }
  const int cj = 4 * tile + j;
  const int cc = cj < nC ? cand[cj] : -1;
  const bool two = cc >= 0 && 2LL * cc + 1 < M1;
  // log(e^z0 + e^z1) = max + log(1 + e^-|z0 - z1|), in base 2 on the exponential unit
  constexpr float kL2e = 1.4426950408889634f, kLn2 = 0.69314718055994531f;
  float v = 0.f;
  if (g < G) {
    const float z0 = (dh[0] + dl[0]) * kScale, z1 = (dh[1] + dl[1]) * kScale;
    v += two ? fmaxf(z0, z1) + kLn2 * lg2_approx(1.f + ex2_approx(-fabsf(z0 - z1) * kL2e)) : z0;
  }
  if (g + 8 < G) {
    const float z0 = (dh[2] + dl[2]) * kScale, z1 = (dh[3] + dl[3]) * kScale;
    v += two ? fmaxf(z0, z1) + kLn2 * lg2_approx(1.f + ex2_approx(-fabsf(z0 - z1) * kL2e)) : z0;
  }
  v += __shfl_xor_sync(kFull, v, 4);
  v += __shfl_xor_sync(kFull, v, 8);
  v += __shfl_xor_sync(kFull, v, 16);
  if (g == 0 && cj < nC) sc[cj] = v;
}

// Candidate i of nC (scores sc) survives iff fewer than K candidates beat it: j beats i
// when its score is higher, or equal with j < i (the lower node index).  sel[u] is the
// verdict for i = lane + 32 u; the scores travel by shuffles.
__device__ __forceinline__ void shuffle_rank(const float* sc, int nC, int K, int lane, bool (&sel)[2]) {
  const float x0 = lane < nC ? sc[lane] : 0.f;
  const float x1 = lane + 32 < nC ? sc[lane + 32] : 0.f;
  int r0 = 0, r1 = 0;
  const int n0 = min(nC, 32);
  // (unrolled: the shuffles of several j are in flight together)
#pragma unroll 8
  for (int j = 0; j < n0; ++j) {
    const float y = __shfl_sync(kFull, x0, j);
    r0 += (y > x0 || (y == x0 && j < lane));
    r1 += (y >= x1);  // j < 32 <= lane + 32
  }
#pragma unroll 8
  for (int j = 32; j < nC; ++j) {
    const float y = __shfl_sync(kFull, x1, j - 32);
    r0 += (y > x0);  // j >= 32 > lane
    r1 += (y > x1 || (y == x1 && j < lane + 32));
  }
  sel[0] = lane < nC && r0 < K;
  sel[1] = lane + 32 < nC && r1 < K;
}

// One decode step for one (b, kv): append k_new at position p = lengths[b],
// refresh the leaf mean and its ancestor path, then walk for the query at t = p
// over the n = p + 1 tokens present.
template <int G>
__global__ void __launch_bounds__(kDecWarps * 32) decode_kernel(
    const __nv_bfloat16* __restrict__ q_new, const __nv_bfloat16* __restrict__ k_new,
    __nv_bfloat16* keys, float* summ, int32_t* lengths, Levels cap_lv,
    long long n_cap, int Hq, int Hkv, int K, int32_t* __restrict__ idx, float* __restrict__ scores,
    int* status, int* arrivals) {
  __shared__ float sib[kMaxLevels + 1][kD];  // siblings along the new token's path
  __shared__ __align__(16) __nv_bfloat16 lk[kC * kD];  // the earlier keys of the new token's leaf
  __shared__ int dcand[kDecWarps][2 * kMaxK];   // each warp's copy of the candidate list
  __shared__ int dnext[kDecWarps][kMaxK];       // each warp's survivor compaction
  __shared__ float dscore[2][2 * kMaxK];        // candidate scores, by level parity
  __shared__ float dnext_s[kMaxK];
  __shared__ float dleaf[2 * kMaxK];  // leaf scores
  __shared__ int leaf_nc;             // leaf candidates
  __shared__ int pf_cand[2 * kMaxK];  // level-2 candidates, whose leaves' keys the other warps ask into L2
  __shared__ int pf_n;
  const int b = blockIdx.x / Hkv, kv = blockIdx.x % Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t qa[4][4];  // the walking warps' query fragments, requested before anything else
  if (warp < kWalkWarps) leaf_q_frags<G>(q_new + ((long long)b * Hq + (long long)kv * G) * kD, lane, qa);
  // the new key's feature of the path-update threads, likewise (it does not depend on the length)
  const __nv_bfloat16 kn = tid < kD ? k_new[((long long)b * Hkv + kv) * kD + tid] : __float2bfloat16(0.f);
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
  // level sizes for the n tokens present (shifts), row offsets from the capacity layout
  const int Ln = num_levels_for(n);
  auto Mof = [n](int l) -> long long { return level_size_for(n, l); };
  auto Oof = [&cap_lv](int l) -> long long { return cap_lv.off[l]; };
  __nv_bfloat16* keys_b = keys + (long long)b * n_cap * Hkv * kD;
  float* blk = summ + ((long long)b * Hkv + kv) * cap_lv.total * kD;
  const long long leaf = p >> kLog2C;
  if (tid < kD) {
    // siblings of the path nodes (levels 1..L-1), fetched together before the new token
    // changes anything they depend on: none of them is on the path
    // (all loads issued before any store, so their latencies overlap)
    const int e = tid;
    float v[kMaxLevels + 1];
#pragma unroll
    for (int l = 2; l <= kMaxLevels; ++l) {
      const long long s = (leaf >> (l - 2)) ^ 1;
      v[l] = (l <= Ln && s < Mof(l - 1)) ? blk[(Oof(l - 1) + s) * kD + e] : 0.f;
    }
#pragma unroll
    for (int l = 2; l <= kMaxLevels; ++l)
      if (l <= Ln) sib[l][e] = v[l];
  }
  {  // the leaf's earlier keys, 16 bytes per thread
    const int nprev = (int)(p - leaf * kC);  // 0..63
    for (int i = tid; i < nprev * (kD / 8); i += kDecWarps * 32) {
      const int r = i / (kD / 8), v = i % (kD / 8);
      reinterpret_cast<uint4*>(lk)[i] =
          *reinterpret_cast<const uint4*>(keys_b + ((leaf * kC + r) * Hkv + kv) * kD + 8 * v);
    }
  }
  __syncthreads();
  if (tid < kD) {
    // path update, feature e = tid: the leaf mean over its tokens in order, then the
    // count-weighted merges up to the root (the same formula as the build)
    const int e = tid;
    keys_b[(p * Hkv + kv) * kD + e] = kn;
    float acc = 0.f;  // (unrolled: the shared-memory loads run ahead of the chain of adds)
#pragma unroll 8
    for (int r = 0; r < (int)(p - leaf * kC); ++r) acc = __fadd_rn(acc, bf2f(lk[r * kD + e]));
    acc = __fadd_rn(acc, bf2f(kn));
    float m = div_count(acc, (int)(p - leaf * kC + 1));
    blk[(Oof(1) + leaf) * kD + e] = m;
    long long i = leaf;
    // (unrolled by four: the counts and addresses of the next levels are ready before
    // the chain of merges reaches them)
#pragma unroll 4
    for (int l = 2; l <= Ln; ++l) {
      const long long child = i;
      i >>= 1;
      const long long c0 = 2 * i, c1 = 2 * i + 1;
      const int n0 = node_count(l - 1, c0, n);
      const int n1 = c1 < Mof(l - 1) ? node_count(l - 1, c1, n) : 0;
      const float m0 = c0 == child ? m : sib[l][e];
      const float m1 = n1 > 0 ? (c1 == child ? m : sib[l][e]) : 0.f;
      m = merge_mean(m0, n0, m1, n1);
      blk[(Oof(l) + i) * kD + e] = m;
    }
  }
  __threadfence_block();
  __syncthreads();

  // The walk, by warps 0 .. kWalkWarps - 1.  Each holds the same survivor list (lane j:
  // the j-th survivor) and expands it into its own copy of the candidate list; the
  // candidates are scored four to a warp-tile on mma.sync, into a score array shared by
  // the walking warps and double-buffered by level parity; after one barrier of the
  // walking warps every one of them ranks the same scores and compacts the same
  // survivors.  The other warps wait for the leaf candidates.
  if (warp < kWalkWarps) {
    int* cand = dcand[warp];
    int nS = 1, myS = 0;
    int par = 0;
    int nC = 1;
    bool pf_sent = false;
    if (Ln == 1) {  // a single leaf, which is the root
      if (lane == 0) cand[0] = 0;
      __syncwarp();
    }
    for (int l = Ln - 1; l >= 1; --l) {
      {  // candidates: the children of the survivors (in decode every existing node is eligible)
        const bool v0 = lane < nS;
        const long long c1 = 2LL * myS + 1;
        const bool v1 = v0 && c1 < Mof(l);
        const unsigned b1 = __ballot_sync(kFull, v1);
        const int pos = lane + __popc(b1 & ((1u << lane) - 1u));
        nC = nS + __popc(b1);
        if (v0 && PISA_IN_BOUNDS(pos + (v1 ? 1 : 0) < 2 * kMaxK)) {
          cand[pos] = 2 * myS;
          if (v1) cand[pos + 1] = (int)c1;
        }
        __syncwarp();
      }
      if (l == 1) break;
      if (l == 2 && warp == 0) {  // hand the level-2 candidates to the warps that do not walk
        for (int i = lane; i < nC; i += 32) pf_cand[i] = cand[i];
        if (lane == 0) pf_n = nC;
        pf_sent = true;
        asm volatile("bar.arrive 2, %0;" ::"n"(kPfThreads) : "memory");
      }
      if (nC <= K) {  // kept whole, unscored
        nS = nC;
        myS = lane < nC ? cand[lane] : 0;
        __syncwarp();
        continue;
      }
      float* sc = dscore[par];
      const float* rows1 = blk + Oof(l - 1) * kD;
      const float* rows2 = l >= 3 ? blk + Oof(l - 2) * kD : nullptr;
      const long long M1 = Mof(l - 1), M2 = l >= 3 ? Mof(l - 2) : 0;
      for (int tile = warp; 4 * tile < nC; tile += kWalkWarps) {
        tile_node_scores<G>(rows1, M1, rows2, M2, cand, nC, tile, qa, lane, sc);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kWalkWarps * 32) : "memory");
      // rank count over the shared scores (candidate i survives iff fewer than K beat it; j
      // beats i when its score is higher, or equal with j < i, i.e. the lower node index)
      bool sel[2];
      shuffle_rank(sc, nC, K, lane, sel);
      unsigned m[2] = {__ballot_sync(kFull, sel[0]), __ballot_sync(kFull, sel[1])};
      int* nx = dnext[warp];
      const unsigned lt = (1u << lane) - 1u;
      if (sel[0]) nx[__popc(m[0] & lt)] = cand[lane];
      if (sel[1]) nx[__popc(m[0]) + __popc(m[1] & lt)] = cand[lane + 32];
      __syncwarp();
      nS = K;
      myS = lane < K ? nx[lane] : 0;
      __syncwarp();
      par ^= 1;
    }
    if (warp == 0) {
      if (lane == 0) leaf_nc = nC;  // warp 0's candidate list holds the leaves
      if (!pf_sent) {  // no level 2 (a tree of one or two levels): nothing to prefetch
        if (lane == 0) pf_n = 0;
        asm volatile("bar.arrive 2, %0;" ::"n"(kPfThreads) : "memory");
      }
    }
  } else {
    // the keys of the level-2 candidates' leaves go to L2 while the walking warps score level 2
    asm volatile("bar.sync 2, %0;" ::"n"(kPfThreads) : "memory");
    const int np = pf_n;
    for (int i = tid - kWalkWarps * 32; i < np * 128; i += (kDecWarps - kWalkWarps) * 32) {
      const long long r = 128LL * pf_cand[i >> 7] + (i & 127);
      if (r < n) asm volatile("prefetch.global.L2 [%0];" ::"l"(keys_b + (r * Hkv + kv) * kD));
    }
  }
  __syncthreads();
  // leaves: the children of the level-2 survivors, scored exactly when there are more than
  // K of them or when scores are requested
  const int nC = leaf_nc;
  const int* cand = dcand[0];
  float* sc = dleaf;
  if (nC > K || so != nullptr) {
    uint32_t qa[4][4];
    leaf_q_frags<G>(q_new + ((long long)b * Hq + (long long)kv * G) * kD, lane, qa);
    for (int ci = warp; ci < nC; ci += kDecWarps) {
      const float v = warp_leaf_mma<G>(keys_b, Hkv, kv, cand[ci], n, qa, lane);
      if (lane == 0) sc[ci] = v;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  bool sel[2] = {lane < nC, lane + 32 < nC};  // K or fewer leaves: all kept
  if (nC > K) shuffle_rank(sc, nC, K, lane, sel);
  unsigned m[2] = {__ballot_sync(kFull, sel[0]), __ballot_sync(kFull, sel[1])};
  const unsigned lt = (1u << lane) - 1u;
  int* nx = dnext[0];
  float* nxs = dnext_s;
  if (sel[0]) {
    nx[__popc(m[0] & lt)] = cand[lane];
    nxs[__popc(m[0] & lt)] = so ? sc[lane] : 0.f;
  }
  if (sel[1]) {
    nx[__popc(m[0]) + __popc(m[1] & lt)] = cand[lane + 32];
    nxs[__popc(m[0]) + __popc(m[1] & lt)] = so ? sc[lane + 32] : 0.f;
  }
  __syncwarp();
  const int nOut = __popc(m[0]) + __popc(m[1]);
  if (lane < K) {
    io[lane] = lane < nOut ? nx[lane] : -1;
    if (so) so[lane] = lane < nOut ? nxs[lane] : -INFINITY;
  }
  if (lane == 0) {
    // every thread of this CTA has read lengths[b] (they all passed the barrier above);
    // the last of the sequence's Hkv CTAs to get here advances it
    __threadfence();
    if (atomicAdd(arrivals + b, 1) == Hkv - 1) lengths[b] = (int32_t)(p + 1);
  }
}

// ---------------------------------------------------------------- launchers

template <int G>
static cudaError_t launch_decode_G(const __nv_bfloat16* q_new, const __nv_bfloat16* k_new,
                                   __nv_bfloat16* keys, float* summ, int32_t* lengths,
                                   const Levels& cap_lv, long long n_cap, int B, int Hq, int Hkv,
                                   int K, int32_t* idx, float* scores, int* status, int* arrivals, cudaStream_t s) {
  PISA_SET_BOUNDS_STATUS(status, s);
  decode_kernel<G><<<B * Hkv, kDecWarps * 32, 0, s>>>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, Hq, Hkv,
                                          K, idx, scores, status, arrivals);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_decode_warp(const __nv_bfloat16* q_new, const __nv_bfloat16* k_new,
                               __nv_bfloat16* keys, float* summ, int32_t* lengths,
                               const Levels& cap_lv, long long n_cap, int B, int Hq, int Hkv, int K,
                               int32_t* idx, float* scores, int* status, int* arrivals, cudaStream_t s) {
  switch (Hq / Hkv) {
    case 1: return launch_decode_G<1>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, arrivals, s);
    case 2: return launch_decode_G<2>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, arrivals, s);
    case 4: return launch_decode_G<4>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, arrivals, s);
    case 8: return launch_decode_G<8>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, arrivals, s);
    case 16: return launch_decode_G<16>(q_new, k_new, keys, summ, lengths, cap_lv, n_cap, B, Hq, Hkv, K, idx, scores, status, arrivals, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pisa
