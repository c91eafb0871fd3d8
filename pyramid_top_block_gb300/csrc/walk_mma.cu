// walk_mma.cu -- the intermediate levels of the prefill walk on tensor cores.
//
// "Block Sparse Attention with Log-Linear Complexity", §3.2 (coarse-to-fine:
// each level expands the previous survivors, keeps the Top-K of at most g*K
// candidates, keeps a level of <= K candidates unscored), "Scoring: LogSumExp"
// (a candidate's score is log sum exp of q.kbar over its children's summaries),
// §4.1 (summed over the query heads of the GQA group).
//
// Carrying the logits down the tree.  For a query head h and a node v let
// z_v = q_h . kbar_v / sqrt(d).  A node's mean is the count-weighted mean of its
// children's, n_v kbar_v = n_a kbar_a + n_b kbar_b.  With
//     Delta_v = kbar_ref - kbar_v     (ref = the child with fewer tokens, a if equal)
//     u_v     = q_h . Delta_v / sqrt(d)
// the children's logits are z_ref = z_v + u_v and z_oth = z_v - r u_v with
// r = n_ref / n_oth <= 1 (r = 1 for every node but the last of a level).  So
// the LSE over the two children is
//     log(e^{z_v + u} + e^{z_v - r u}) = z_v + max(u, -r u) + log(1 + e^{-(1+r)|u|}),
// i.e. z_v + log(2 cosh u) for equal children.  Summed over the heads of the
// group, a candidate's score is Z_v + sum_h [max(u_h, -r u_h) + log(1 + e^{-(1+r)|u_h|})]
// with Z_v = sum_h z_{v,h}, and its children's head sums are Z_v + sum_h u_h and
// Z_v - r sum_h u_h.  The walk therefore carries ONE scalar per candidate and
// needs one 16-head dot product per candidate (with its Delta row) per level;
// rounding errors add up linearly down the path.  A child that starts after
// the query (causal) leaves the single-child score Z_child.
//
// The walk starts at the highest level with more than K nodes (all levels
// above it are kept whole, without scoring): its eligible nodes are the first
// candidates, and their Z = (sum_h q_h) . kbar / sqrt(d) is one fp32 dot product.
//
// Precision.  Delta rows are stored as a pair of bf16 vectors hi + lo
// (hi = bf16(x), lo = bf16(x - hi)), ~2^-17 relative; q is bf16 and exact.
// The dot products are bf16 mma.sync.m16n8k16 in fp32: M = 16 candidates
// (their Delta rows, hi and lo), N = 8 query heads (two tiles for 16 heads),
// K = 64 features.  Thread (g, j) of the warp then holds candidates g and g+8
// for heads 2j, 2j+1 (+8), so a head sum is two shuffles inside a lane quad.
//
// Layout of a stored row (256 bytes): hi[64] then lo[64], each with its 32
// bf16 pairs permuted so that lane quad position j reads its four k-steps'
// A-fragment words as two 16-byte loads at byte offset 32 j.  Rows are stored
// pre-multiplied by log2(e)/sqrt(d), so q . row is a logit in base-2 units.
//
// Table of one (b, kv): the Delta rows of levels 2..L (levels ascending, nodes
// ascending), one zero row, then kZRows "mean rows" kbar of the nodes of the
// first scored level (zero beyond its size): q_h . kbar for every head is one
// MMA tile, which gives that level's head-summed Z.
#include <mutex>
#include <type_traits>

#include "api.cuh"
#include "tc.cuh"

namespace pisa {

constexpr int kWalkWarps = 8;    // walk_mma_kernel (K <= 32): 8 warps, 3 CTAs per SM
// walk_k8_kernel / walk_k8s_kernel (K <= 8): one CTA of 24 warps per SM, so that the
// shared-memory copy of the top levels' rows is held once per SM instead of three times
// and can cover one more level (the 496 rows of levels 9..5 at 262144 tokens).
constexpr int kWalk8Warps = 24;

struct RowOffsets {
  long long o[kMaxLevels + 2];
};
constexpr int kRowBytes = 256;
constexpr int kZRows = 2 * kMaxK;    // mean rows of the first scored level (at most 2K nodes)
constexpr float kRowScale = 0.18033688011112042f;  // log2(e) / sqrt(64)
constexpr int kCacheRowBytes = 272;  // shared-memory row stride (16-byte pad against bank conflicts)
constexpr int kCacheRows = 240;      // Delta rows of the top scored levels kept in shared memory (K <= 32 kernel)
constexpr int kCacheRows8 = 496;     // the same for the K <= 8 kernels (one CTA per SM)

// Storage position (in bf16 elements, 0..63) of feature d inside a permuted half-row.
__host__ __device__ __forceinline__ int perm_pos(int d) {
  const int P = d >> 1, ks = P >> 3, rem = P & 7, j = rem & 3, half = rem >> 2;
  return 2 * (8 * j + 2 * ks + half) + (d & 1);
}

// Which child a node's Delta row refers to: 1 when the second child exists and
// holds fewer tokens (the ragged tail), else 0.
__device__ __forceinline__ int ref_child(int l, long long v, long long Mc, long long N, int* n0, int* n1) {
  *n0 = node_count(l - 1, 2 * v, N);
  *n1 = (2 * v + 1 < Mc) ? node_count(l - 1, 2 * v + 1, N) : 0;
  return (*n1 > 0 && *n1 < *n0) ? 1 : 0;
}

// Route table: thread per (b, kv, row, feature pair).
__global__ void route_table_kernel(const float* __restrict__ summ, Levels lv, long long N, int BH,
                                   long long rows_per_bh, RowOffsets ro, int l_start,
                                   unsigned char* __restrict__ table) {
  const long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)BH * rows_per_bh * 32;
  if (w >= total) return;
  const int pr = (int)(w & 31);
  const long long row = (w >> 5) % rows_per_bh;
  const long long bh = (w >> 5) / rows_per_bh;
  const float* blk = summ + bh * lv.total * kD;
  const long long zrow0 = ro.o[lv.L + 1] + 1;
  float x[2] = {0.f, 0.f};
  if (lv.L >= 2 && row < ro.o[lv.L + 1]) {  // Delta row (the spare row after them stays zero)
    int l = 2;
    while (l < lv.L && row >= ro.o[l + 1]) ++l;
    const long long v = row - ro.o[l];
    int n0, n1;
    const int ref = ref_child(l, v, lv.M[l - 1], N, &n0, &n1);
    const float* pv = blk + (lv.off[l] + v) * kD;
    const float* pc = blk + (lv.off[l - 1] + 2 * v + ref) * kD;
    for (int e = 0; e < 2; ++e) x[e] = (pc[2 * pr + e] - pv[2 * pr + e]) * kRowScale;
  } else if (l_start >= 2 && row >= zrow0 && row - zrow0 < lv.M[l_start]) {  // mean row
    const float* pv = blk + (lv.off[l_start] + (row - zrow0)) * kD;
    for (int e = 0; e < 2; ++e) x[e] = pv[2 * pr + e] * kRowScale;
  }
  __nv_bfloat16* hi = reinterpret_cast<__nv_bfloat16*>(table + (bh * rows_per_bh + row) * kRowBytes);
  __nv_bfloat16* lo = hi + 64;
  for (int e = 0; e < 2; ++e) {
    const int d = 2 * pr + e;
    const __nv_bfloat16 h = __float2bfloat16_rn(x[e]);
    hi[perm_pos(d)] = h;
    lo[perm_pos(d)] = __float2bfloat16_rn(x[e] - __bfloat162float(h));
  }
}

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with a zero accumulator in.
__device__ __forceinline__ void mma_bf16_16816_z(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

struct WalkSmem {  // per-warp views into dynamic shared memory
  int* cand;     // [2K] node ids of the current candidates (ascending)
  float* zs;     // [2K] head-summed logit Z of each candidate
  float* su;     // [2K] head-summed u of each candidate (for its children's Z)
  float* score;  // [2K]
  int* sel;      // [K] candidate indices of the survivors (ascending)
  float* qsum;   // [64] sum over the group's heads of q (fp32)
};

// [qsum 64][score S4][cand 2K][zs 2K][su 2K][sel K] (4-byte words, S4 = 2K rounded up
// to a multiple of 4), rounded up to 16 bytes: qsum and score are read as float4 and
// stay 16-byte aligned in every warp's slice.
__host__ __device__ inline int score_slots(int K) { return (2 * K + 3) & ~3; }
__host__ __device__ inline size_t walk_smem_per_warp(int K) {
  return ((size_t)(64 + score_slots(K) + 6 * K + K) * 4 + 15) & ~(size_t)15;
}

// Children of candidate c (level l) in a sequence of n tokens: whether the
// second child exists and is eligible, which child the Delta row refers to
// and the ratio r = n_ref / n_oth.  Only the last node of a level can have
// unequal children.
struct Kids {
  bool two;    // the second child exists and is eligible
  bool ref1;   // Delta refers to the second child
  float r;
};

__device__ __forceinline__ Kids kids_of(int l, int c, int Mc, int n, int t, bool causal) {
  Kids k;
  const int c1 = 2 * c + 1;
  const bool exists = c1 < Mc;
  k.two = exists && (!causal || (c1 << (kLog2C + l - 2)) <= t);
  k.ref1 = false;
  k.r = 1.f;
  if (exists && c1 == Mc - 1) {  // possibly ragged last pair
    const int n0 = node_count(l - 1, 2 * c, n), n1 = node_count(l - 1, c1, n);
    if (n1 < n0) {
      k.ref1 = true;
      k.r = (float)n1 / (float)n0;
    }
  }
  return k;
}

// Grid: blockIdx.y = (b, kv); the CTAs of one (b, kv) take its query positions
// interleaved (t = blockIdx.x + gridDim.x * i) so causal work stays balanced.
// Each CTA first copies the Delta rows of levels [l_lo, l_start] of its (b, kv)
// (contiguous in the table) into shared memory.
__global__ void __launch_bounds__(kWalkWarps * 32, 3) walk_mma_kernel(
    const __nv_bfloat16* __restrict__ Q, const float* __restrict__ summ, const unsigned char* __restrict__ table,
    Levels lv, RowOffsets ro, long long rows_per_bh, int N, int Hq, int Hkv, int K, int causal, int l_start,
    int l_lo, int32_t* __restrict__ surv, int32_t* __restrict__ srank, int* __restrict__ count, int t0, int t1,
    int chunk_shift, int M2, int mode) {
  extern __shared__ __align__(16) unsigned char wsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, j = lane & 3;
  const int G = Hq / Hkv;
  const int C2 = 2 * K;
  const long long bh = blockIdx.y;
  // shared cache of the top levels' rows
  const int crow0 = (l_start >= 2) ? (int)ro.o[l_lo] : 0;
  const int ncache = (l_start >= 2) ? (int)(ro.o[l_start + 1] - ro.o[l_lo]) : 0;
  unsigned char* cache = wsm + (size_t)kWalkWarps * walk_smem_per_warp(K);
  {
    const uint4* src = reinterpret_cast<const uint4*>(table + (bh * rows_per_bh + crow0) * kRowBytes);
    for (int e = threadIdx.x; e < ncache * 16; e += blockDim.x)
      *reinterpret_cast<uint4*>(cache + (e >> 4) * kCacheRowBytes + (e & 15) * 16) = __ldg(src + e);
  }
  __syncthreads();
  unsigned char* base = wsm + (size_t)warp * walk_smem_per_warp(K);
  WalkSmem S;
  S.qsum = reinterpret_cast<float*>(base);
  S.score = S.qsum + 64;
  S.cand = reinterpret_cast<int*>(S.score + score_slots(K));
  S.zs = reinterpret_cast<float*>(S.cand + C2);
  S.su = S.zs + C2;
  S.sel = reinterpret_cast<int*>(S.su + C2);
  constexpr float kL2e = 1.4426950408889634f;
  constexpr float kLn2 = 0.69314718055994531f;

  for (int t = t0 + blockIdx.x + gridDim.x * warp; t < t1; t += gridDim.x * kWalkWarps) {
    const long long job = bh * N + t;
    const int kv = (int)(bh % Hkv);
    const long long b = bh / Hkv;
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(Q + ((b * N + t) * Hq + (long long)kv * G) * kD);
    {  // the warp's next query: its G head rows into L2 while this one walks
      const int tn = t + gridDim.x * kWalkWarps;
      if (tn < t1 && lane < G)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(Q + ((b * N + tn) * Hq + (long long)kv * G + lane) * kD));
    }
    int nS;  // survivors (candidate indices in S.sel) at the last processed level
    if (l_start < 2) {
      // at most K nodes at level 2: every eligible level-2 node survives unscored
      const int m2 = lv.L >= 2 ? lv.M[2] : 1;
      const int el = causal ? min(m2, (t >> (kLog2C + 1)) + 1) : m2;
      nS = el;
      if (lane < el) {
        S.cand[lane] = lane;
        S.sel[lane] = lane;
      }
    } else {
      // head-summed query (fp32), lane owns features 2*lane, 2*lane+1
      {
        float a0 = 0.f, a1 = 0.f;
        for (int h = 0; h < G; ++h) {
          const uint32_t w = __ldg(q0 + h * 32 + lane);
          a0 += __uint_as_float(w << 16);
          a1 += __uint_as_float(w & 0xffff0000u);
        }
        S.qsum[2 * lane] = a0;
        S.qsum[2 * lane + 1] = a1;
      }
      // Q^T fragments (the MMA's B operand), per k-step: [0] / [2] = words (2j, 2j+8) of
      // head g (head tile 0), [1] / [3] the same for head g + 8 (head tile 1); heads >= G are zero
      uint32_t A[4][4];
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int w0 = 8 * ks + j;
        A[ks][0] = g < G ? __ldg(q0 + g * 32 + w0) : 0u;
        A[ks][1] = g + 8 < G ? __ldg(q0 + (g + 8) * 32 + w0) : 0u;
        A[ks][2] = g < G ? __ldg(q0 + g * 32 + w0 + 4) : 0u;
        A[ks][3] = g + 8 < G ? __ldg(q0 + (g + 8) * 32 + w0 + 4) : 0u;
      }
      __syncwarp();
      // first candidates: the eligible nodes of level l_start, Z by a direct fp32 dot
      int nC;
      {
        const int ml = lv.M[l_start];
        nC = causal ? min(ml, (t >> (kLog2C + l_start - 1)) + 1) : ml;
        for (int ci = lane; ci < nC; ci += 32) {
          const float4* kr = reinterpret_cast<const float4*>(summ + (bh * lv.total + lv.off[l_start] + ci) * kD);
          const float4* qs = reinterpret_cast<const float4*>(S.qsum);
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float4 kk = __ldg(kr + e), qq = qs[e];
            acc = fmaf(qq.x, kk.x, fmaf(qq.y, kk.y, fmaf(qq.z, kk.z, fmaf(qq.w, kk.w, acc))));
          }
          S.cand[ci] = ci;
          S.zs[ci] = acc * kScale;
        }
      }
      __syncwarp();
      const unsigned char* tb = table + bh * rows_per_bh * kRowBytes;
      for (int l = l_start;; --l) {
        const bool scoring = nC > K;
        const int Mc = lv.M[l - 1];
        const unsigned char* lrow = tb + ro.o[l] * kRowBytes;
        const bool cached = l >= l_lo;
        const unsigned char* crow = cache + (ro.o[l] - crow0) * kCacheRowBytes;
        for (int mt = 0; mt * 16 < nC; ++mt) {
          // A fragments: Delta rows (hi, lo) of candidates 16mt + g and 16mt + g + 8
          const int c0i = mt * 16 + g, c1i = c0i + 8;
          uint4 h0[2], l0[2], h1[2], l1[2];
          {
            const uint4 z = make_uint4(0, 0, 0, 0);
            h0[0] = h0[1] = l0[0] = l0[1] = h1[0] = h1[1] = l1[0] = l1[1] = z;
            if (cached) {
              if (c0i < nC && PISA_IN_BOUNDS(S.cand[c0i] >= 0 && S.cand[c0i] < lv.M[l])) {
                const uint4* p = reinterpret_cast<const uint4*>(crow + S.cand[c0i] * kCacheRowBytes + 32 * j);
                h0[0] = p[0];
                h0[1] = p[1];
                l0[0] = p[8];
                l0[1] = p[9];
              }
              if (c1i < nC && PISA_IN_BOUNDS(S.cand[c1i] >= 0 && S.cand[c1i] < lv.M[l])) {
                const uint4* p = reinterpret_cast<const uint4*>(crow + S.cand[c1i] * kCacheRowBytes + 32 * j);
                h1[0] = p[0];
                h1[1] = p[1];
                l1[0] = p[8];
                l1[1] = p[9];
              }
            } else {
              if (c0i < nC && PISA_IN_BOUNDS(S.cand[c0i] >= 0 && S.cand[c0i] < lv.M[l])) {
                const uint4* p = reinterpret_cast<const uint4*>(lrow + (long long)S.cand[c0i] * kRowBytes + 32 * j);
                h0[0] = __ldg(p);
                h0[1] = __ldg(p + 1);
                l0[0] = __ldg(p + 8);
                l0[1] = __ldg(p + 9);
              }
              if (c1i < nC && PISA_IN_BOUNDS(S.cand[c1i] >= 0 && S.cand[c1i] < lv.M[l])) {
                const uint4* p = reinterpret_cast<const uint4*>(lrow + (long long)S.cand[c1i] * kRowBytes + 32 * j);
                h1[0] = __ldg(p);
                h1[1] = __ldg(p + 1);
                l1[0] = __ldg(p + 8);
                l1[1] = __ldg(p + 9);
              }
            }
          }
          // four independent accumulation chains: (head tile 0/1) x (hi/lo)
          float dh[2][4] = {}, dl[2][4] = {};
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint4& H0 = h0[ks >> 1];
            const uint4& H1 = h1[ks >> 1];
            const uint4& L0 = l0[ks >> 1];
            const uint4& L1 = l1[ks >> 1];
            const bool hiw = ks & 1;
            const uint32_t ah[4] = {hiw ? H0.z : H0.x, hiw ? H1.z : H1.x, hiw ? H0.w : H0.y, hiw ? H1.w : H1.y};
            const uint32_t al[4] = {hiw ? L0.z : L0.x, hiw ? L1.z : L1.x, hiw ? L0.w : L0.y, hiw ? L1.w : L1.y};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              mma_bf16_16816(dh[nt], ah, A[ks][nt], A[ks][nt + 2]);
              mma_bf16_16816(dl[nt], al, A[ks][nt], A[ks][nt + 2]);
            }
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ci = cc ? c1i : c0i;
            float su = 0.f, am = 0.f, pr = 1.f;
            Kids kd;
            kd.two = false;
            kd.ref1 = false;
            kd.r = 1.f;
            if (ci < nC) {
              kd = kids_of(l, S.cand[ci], Mc, N, t, causal != 0);
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  if (8 * nt + 2 * j + e < G) {
                    const float u = (dh[nt][2 * cc + e] + dl[nt][2 * cc + e]) * kLn2;
                    su += u;
                    if (scoring && kd.two) {
                      if (mode == 0) {
                        am += u >= 0.f ? u : -kd.r * u;
                        pr *= 1.f + ex2_approx(-(1.f + kd.r) * fabsf(u) * kL2e);
                      } else {
                        am += u * u;  // for the variance of the two children's logits
                      }
                    }
                  }
                }
              }
            }
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
              su += __shfl_xor_sync(kFull, su, o);
              if (scoring) {
                am += __shfl_xor_sync(kFull, am, o);
                pr *= __shfl_xor_sync(kFull, pr, o);
              }
            }
            if (j == 0 && ci < nC) {
              S.su[ci] = su;
              if (scoring) {
                const float z = S.zs[ci];
                float two_sc = am + lg2_approx(pr) * kLn2;  // LSE: z + max part + log(1 + ...)
                if (mode != 0) two_sc = 0.5f * (1.f - kd.r) * su + (mode == 2 ? 0.125f * (1.f + kd.r) * (1.f + kd.r) * am : 0.f);
                S.score[ci] = kd.two ? z + two_sc : z + (kd.ref1 ? -kd.r : 1.f) * su;
              }
            }
          }
        }
        __syncwarp();
        // survivors (candidate indices, ascending)
        if (!scoring) {
          nS = nC;
          if (lane < nC) S.sel[lane] = lane;
        } else {
          // rank keys: the score's bits made order-preserving as an unsigned, the low six bits
          // replaced by 63 - candidate index (ties, and scores within 2^-17 relative, go to the
          // lower index); slots past nC hold 0, below every key
          unsigned* keys = reinterpret_cast<unsigned*>(S.score);
          unsigned ky[2];
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {
            const int ci = lane + 32 * s2;
            ky[s2] = 0u;
            if (ci < nC) {
              const unsigned fb = __float_as_uint(S.score[ci]);
              ky[s2] = ((fb ^ ((unsigned)((int)fb >> 31) | 0x80000000u)) & ~63u) | (unsigned)(63 - ci);
            }
          }
          __syncwarp();
          const int nC4 = (nC + 3) & ~3;
          if (lane < nC4) keys[lane] = ky[0];
          if (lane + 32 < nC4) keys[lane + 32] = ky[1];
          __syncwarp();
          bool keep[2];
          unsigned m[2];
          {
            int r0 = 0, r1 = 0;
            const uint4* k4 = reinterpret_cast<const uint4*>(keys);
            for (int q4 = 0; q4 * 4 < nC; ++q4) {
              const uint4 o = k4[q4];
              r0 += (o.x > ky[0]) + (o.y > ky[0]) + (o.z > ky[0]) + (o.w > ky[0]);
              r1 += (o.x > ky[1]) + (o.y > ky[1]) + (o.z > ky[1]) + (o.w > ky[1]);
            }
            keep[0] = lane < nC && r0 < K;
            keep[1] = lane + 32 < nC && r1 < K;
            m[0] = __ballot_sync(kFull, keep[0]);
            m[1] = __ballot_sync(kFull, keep[1]);
          }
          const unsigned lt = (1u << lane) - 1u;
          if (keep[0]) S.sel[__popc(m[0] & lt)] = lane;
          if (keep[1]) S.sel[__popc(m[0]) + __popc(m[1] & lt)] = lane + 32;
          nS = K;
        }
        __syncwarp();
        if (l == 2) break;
        // next candidates: eligible children of the survivors, with their head-summed Z
        int c = 0, ci_s = 0;
        bool v1 = false;
        float z0 = 0.f, z1 = 0.f;
        if (lane < nS) {
          ci_s = S.sel[lane];
          c = S.cand[ci_s];
          const Kids kd = kids_of(l, c, Mc, N, t, causal != 0);
          v1 = kd.two;
          const float z = S.zs[ci_s], su = S.su[ci_s];
          const float zr = z + su, zo = fmaf(-kd.r, su, z);
          z0 = kd.ref1 ? zo : zr;
          z1 = kd.ref1 ? zr : zo;
        }
        const unsigned b1 = __ballot_sync(kFull, v1);
        const int pos = lane + __popc(b1 & ((1u << lane) - 1u));
        const int nN = nS + __popc(b1);
        __syncwarp();
        if (lane < nS) {
          S.cand[pos] = 2 * c;
          S.zs[pos] = z0;
          if (v1) {
            S.cand[pos + 1] = 2 * c + 1;
            S.zs[pos + 1] = z1;
          }
        }
        nC = nN;
        __syncwarp();
      }
    }
    // level-2 survivors (node ids, ascending) -> workspace, and bucket counts
    int32_t* out = surv + job * K;
    if (lane < K) {
      int p = -1;
      if (lane < nS) p = S.cand[S.sel[lane]];
      out[lane] = p;
      if (p >= 0 && PISA_IN_BOUNDS(p < M2))
        srank[job * K + lane] = atomicAdd(count + (((long long)(t >> chunk_shift) * gridDim.y + bh) * M2 + p), 1);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Walk for K <= 8: every level has at most 16 candidates, one MMA tile, and the
// whole walk stays in registers.  MMA row m holds candidate m; after the head
// sums lane (g, j) owns candidate g + 8 (j & 1) (lanes j and j ^ 2 hold
// identical copies), and survivor positions are popcounts of ballots.  Rows g
// and g + 1 of a quarter-warp's shared-memory loads are then usually two
// siblings, adjacent rows, which the 272-byte row stride puts in disjoint
// banks.  Scores are base-2 logits (the rows carry log2(e)/sqrt(d)).

// The ragged last pair of children, per level l (children at level l - 1).
struct LevelTail {
  int node[kMaxLevels + 2];  // parent whose second child holds fewer tokens than its first (-1: none)
  float nr[kMaxLevels + 2];  // -(n_second / n_first) for that parent
};

constexpr int kCandBuf = 80;  // per-warp 32-bit words: two buffers of 16 node ids + 16 Z, 16 rank keys

__device__ __forceinline__ void ld_row(const unsigned char* p, bool shared_src, uint4& h0, uint4& h1, uint4& l0,
                                       uint4& l1) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
  if (shared_src) {
    h0 = v[0];
    h1 = v[1];
    l0 = v[8];
    l1 = v[9];
  } else {
    h0 = __ldg(v);
    h1 = __ldg(v + 1);
    l0 = __ldg(v + 8);
    l1 = __ldg(v + 9);
  }
}

// q . row for the two MMA-row candidates (a: row g, b: row g + 8) and the
// lane's heads: u[nt][0..1] = candidate a, heads 8 nt + 2j + {0, 1};
// u[nt][2..3] = candidate b.
template <int NT>
__device__ __forceinline__ void tile_dots(const uint32_t (&A)[4][4], const uint4 (&ra)[4], const uint4 (&rb)[4],
                                          float (&u)[NT][4]) {
  float dh[NT][4], dl[NT][4];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    const uint4& Ha = ra[ks >> 1];
    const uint4& La = ra[2 + (ks >> 1)];
    const uint4& Hb = rb[ks >> 1];
    const uint4& Lb = rb[2 + (ks >> 1)];
    const bool hw = ks & 1;
    const uint32_t ah[4] = {hw ? Ha.z : Ha.x, hw ? Hb.z : Hb.x, hw ? Ha.w : Ha.y, hw ? Hb.w : Hb.y};
    const uint32_t al[4] = {hw ? La.z : La.x, hw ? Lb.z : Lb.x, hw ? La.w : La.y, hw ? Lb.w : Lb.y};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (ks == 0) {
        mma_bf16_16816_z(dh[nt], ah, A[ks][nt], A[ks][nt + 2]);
        mma_bf16_16816_z(dl[nt], al, A[ks][nt], A[ks][nt + 2]);
      } else {
        mma_bf16_16816(dh[nt], ah, A[ks][nt], A[ks][nt + 2]);
        mma_bf16_16816(dl[nt], al, A[ks][nt], A[ks][nt + 2]);
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) u[nt][i] = dh[nt][i] + dl[nt][i];
}

// Lane keeps candidate s of the pair (a, b) it computed partial sums for: its
// own partial plus the partner lane's (lane ^ 1 holds the other candidate).
__device__ __forceinline__ float keep_add(float pa, float pb, int s) {
  const float send = s ? pa : pb, mine = s ? pb : pa;
  return mine + __shfl_xor_sync(kFull, send, 1);
}
__device__ __forceinline__ float keep_mul(float pa, float pb, int s) {
  const float send = s ? pa : pb, mine = s ? pb : pa;
  return mine * __shfl_xor_sync(kFull, send, 1);
}

// MODE: 0 LSE over the two children (PISA), 1 their mean (PISA-1), 2 mean + variance / 2
// (PISA-2).  With children logits z + u and z - r u: mean = z + (1 - r) u / 2, variance / 2 =
// (1 + r)^2 u^2 / 8 (natural units; ln 2 (1 + r)^2 u^2 / 8 for base-2 logits u).
template <int NT, int MODE>
__global__ void __launch_bounds__(kWalk8Warps * 32, 1) walk_k8_kernel(
    const __nv_bfloat16* __restrict__ Q, const unsigned char* __restrict__ table, Levels lv, RowOffsets ro,
    LevelTail tail, long long rows_per_bh, int N, int Hq, int Hkv, int K, int causal, int l_start, int l_lo,
    int32_t* __restrict__ surv, int32_t* __restrict__ srank, int* __restrict__ count, int t0, int t1, int chunk_shift,
    int M2) {
  extern __shared__ __align__(16) unsigned char wsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, j = lane & 3, s = j & 1;
  const int oc = g + 8 * s;  // the candidate this lane owns after the head sums
  const int G = Hq / Hkv;
  const long long bh = blockIdx.y;
  const int kv = (int)(bh % Hkv);
  const long long b = bh / Hkv;
  const long long zrow0 = ro.o[lv.L + 1] + 1;
  // shared memory: [mean rows 16][Delta rows of levels l_lo..l_start][per-warp candidate buffers]
  const int crow0 = (l_start >= 2) ? (int)ro.o[l_lo] : 0;
  const int ncache = (l_start >= 2) ? (int)(ro.o[l_start + 1] - ro.o[l_lo]) : 0;
  unsigned char* czr = wsm;
  unsigned char* cdr = wsm + 16 * kCacheRowBytes;
  int* cbuf = reinterpret_cast<int*>(cdr + (size_t)ncache * kCacheRowBytes) + warp * kCandBuf;
  // per level l: {row base (byte offset in the cache, or row index in the table), M_{l-1} - 1,
  // ragged parent, -r of its children}
  __shared__ int4 lvt[kMaxLevels + 2];
  if (threadIdx.x >= 2 && threadIdx.x <= lv.L) {
    const int l = threadIdx.x;
    const bool cached = l >= l_lo && l <= l_start;
    lvt[l] = make_int4(cached ? (int)((ro.o[l] - crow0) * kCacheRowBytes) : (int)ro.o[l], lv.M[l - 1] - 1,
                       tail.node[l], __float_as_int(tail.nr[l]));
  }
  const unsigned char* tb = table + bh * rows_per_bh * kRowBytes;  // this (b, kv)'s table
  if (l_start >= 2) {
    const unsigned char* src0 = tb;
    for (int e = threadIdx.x; e < 16 * 16; e += blockDim.x)
      *reinterpret_cast<uint4*>(czr + (e >> 4) * kCacheRowBytes + (e & 15) * 16) =
          __ldg(reinterpret_cast<const uint4*>(src0 + zrow0 * kRowBytes) + e);
    for (int e = threadIdx.x; e < ncache * 16; e += blockDim.x)
      *reinterpret_cast<uint4*>(cdr + (e >> 4) * kCacheRowBytes + (e & 15) * 16) =
          __ldg(reinterpret_cast<const uint4*>(src0 + (long long)crow0 * kRowBytes) + e);
  }
  __syncthreads();
  // padded heads (>= G) get an exponent of -inf: their factor 1 + 2^arg stays 1
  float2 pad[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    pad[nt].x = (8 * nt + 2 * j < G) ? 0.f : -INFINITY;
    pad[nt].y = (8 * nt + 2 * j + 1 < G) ? 0.f : -INFINITY;
  }
  const unsigned lt = (1u << lane) - 1u;
  constexpr unsigned kLo = 0x11111111u, kHi = 0x22222222u;  // lanes owning candidates 0..7 / 8..15 (j = 0 / 1)

  for (int t = t0 + blockIdx.x + gridDim.x * warp; t < t1; t += gridDim.x * kWalk8Warps) {
    __syncwarp();  // the previous query's reads of the candidate buffers are done
    const long long job = bh * N + t;
    int32_t* out = surv + job * K;
    int32_t* rk = srank + job * K;  // a survivor's rank in its bucket: the count before it
    int* cnt = count + ((long long)(t >> chunk_shift) * gridDim.y + bh) * M2;  // chunk-major buckets
    if (l_start < 2) {
      // at most K nodes at level 2: every eligible level-2 node survives unscored
      const int m2 = lv.L >= 2 ? lv.M[2] : 1;
      const int el = causal ? min(m2, (t >> (kLog2C + 1)) + 1) : m2;
      if (lane < K) {
        const int p = lane < el ? lane : -1;
        out[lane] = p;
        if (p >= 0) rk[lane] = atomicAdd(cnt + p, 1);
      }
      continue;
    }
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(Q + ((b * N + t) * Hq + (long long)kv * G) * kD);
    {  // the warp's next query: its G head rows into L2 while this one walks
      const int tn = t + gridDim.x * kWalk8Warps;
      if (tn < t1 && lane < G)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(Q + ((b * N + tn) * Hq + (long long)kv * G + lane) * kD));
    }
    // Q^T fragments (the MMA's B operand): [ks][nt] / [ks][nt + 2] = words (8ks + j, 8ks + j + 4)
    // of head g + 8 nt; heads >= G are zero
    uint32_t A[4][4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const int w0 = 8 * ks + j;
      A[ks][0] = g < G ? __ldg(q0 + g * 32 + w0) : 0u;
      A[ks][2] = g < G ? __ldg(q0 + g * 32 + w0 + 4) : 0u;
      A[ks][1] = (NT > 1 && g + 8 < G) ? __ldg(q0 + (g + 8) * 32 + w0) : 0u;
      A[ks][3] = (NT > 1 && g + 8 < G) ? __ldg(q0 + (g + 8) * 32 + w0 + 4) : 0u;
    }
    // first candidates: the eligible nodes of level l_start; Z from the mean rows
    int nC;
    {
      const int ml = lv.M[l_start];
      nC = causal ? min(ml, (t >> (kLog2C + l_start - 1)) + 1) : ml;
    }
    int c = oc;  // node id of the owned candidate
    float Z;
    {
      uint4 ra[4], rb[4];
      // (rows of candidates >= nC are loaded too; their results are never kept)
      ld_row(czr + g * kCacheRowBytes + 32 * j, true, ra[0], ra[1], ra[2], ra[3]);
      ld_row(czr + (g + 8) * kCacheRowBytes + 32 * j, true, rb[0], rb[1], rb[2], rb[3]);
      float u[NT][4];
      tile_dots<NT>(A, ra, rb, u);
      float sa = 0.f, sb = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        sa += u[nt][0] + u[nt][1];
        sb += u[nt][2] + u[nt][3];
      }
      Z = keep_add(sa, sb, s);
      Z += __shfl_xor_sync(kFull, Z, 2);
    }
    for (int l = l_start;; --l) {
      const bool scoring = nC > K;
      const int4 lt4 = lvt[l];
      const int lim = causal ? min(lt4.y, t >> (l + 4)) : lt4.y;  // last eligible second child
      const int rag = lt4.z;
      const float rnr = __int_as_float(lt4.w);
      // rows of the two MMA-row candidates
      const int c_oth = __shfl_xor_sync(kFull, c, 1);
      const int na = s ? c_oth : c, nb = s ? c : c_oth;
      const bool va = g < nC, vb = g + 8 < nC;
      // candidates >= nC read row 0 of the level (their results are never kept)
      int ra_row = va ? na : 0, rb_row = vb ? nb : 0;
      if (!PISA_IN_BOUNDS(ra_row >= 0 && ra_row < lv.M[l] && rb_row >= 0 && rb_row < lv.M[l])) ra_row = rb_row = 0;
      uint4 ra[4], rb[4];
      if (l >= l_lo) {
        const unsigned char* base = cdr + lt4.x + 32 * j;
        ld_row(base + ra_row * kCacheRowBytes, true, ra[0], ra[1], ra[2], ra[3]);
        ld_row(base + rb_row * kCacheRowBytes, true, rb[0], rb[1], rb[2], rb[3]);
      } else {
        const unsigned char* base = tb + (long long)lt4.x * kRowBytes + 32 * j;
        ld_row(base + ra_row * kRowBytes, false, ra[0], ra[1], ra[2], ra[3]);
        ld_row(base + rb_row * kRowBytes, false, rb[0], rb[1], rb[2], rb[3]);
      }
      float u[NT][4];
      tile_dots<NT>(A, ra, rb, u);
      // per candidate of the pair: sum of u, sum of max(u, -r u), prod of (1 + 2^{-(1+r)|u|})
      float su[2], am[2], pr[2];
      const bool any_rag = MODE == 0 && rag >= 0 && __any_sync(kFull, (va && na == rag) || (vb && nb == rag));
#pragma unroll
      for (int cc = 0; cc < 2 && MODE != 0; ++cc) {  // moments: sum of u and of u^2 over the lane's heads
        unsigned long long s2 = f2_pack(0.f, 0.f), q2 = s2;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const unsigned long long u2 = f2_pack(u[nt][2 * cc], u[nt][2 * cc + 1]);
          s2 = f2_add(s2, u2);
          if (MODE == 2) q2 = f2_fma(u2, u2, q2);
        }
        float a, bb;
        f2_unpack(s2, a, bb);
        su[cc] = a + bb;
        f2_unpack(q2, a, bb);
        am[cc] = a + bb;
        pr[cc] = 1.f;
      }
#pragma unroll
      for (int cc = 0; cc < 2 && MODE == 0; ++cc) {
        unsigned long long s2 = f2_pack(0.f, 0.f), m2 = s2, p2 = f2_pack(1.f, 1.f);
        if (!any_rag) {  // r = 1: max(u, -u) = |u|, exponent -2|u|
          const unsigned long long m2c = f2_pack(-2.f, -2.f);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float ux = u[nt][2 * cc], uy = u[nt][2 * cc + 1];
            const unsigned long long u2 = f2_pack(ux, uy), a2 = f2_pack(fabsf(ux), fabsf(uy));
            s2 = f2_add(s2, u2);
            m2 = f2_add(m2, a2);
            const unsigned long long x2 = f2_fma(a2, m2c, f2_pack(pad[nt].x, pad[nt].y));
            float xx, xy;
            f2_unpack(x2, xx, xy);
            p2 = f2_fma(p2, f2_pack(ex2_approx(xx), ex2_approx(xy)), p2);
          }
        } else {
          const int nd = cc ? nb : na;
          const float nr = nd == rag ? rnr : -1.f;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float ux = u[nt][2 * cc], uy = u[nt][2 * cc + 1];
            const float tx = nr * ux, ty = nr * uy;
            const float mx = fmaxf(ux, tx), my = fmaxf(uy, ty);
            s2 = f2_add(s2, f2_pack(ux, uy));
            m2 = f2_add(m2, f2_pack(mx, my));
            const float ex = ex2_approx(fminf(ux, tx) - mx + pad[nt].x);
            const float ey = ex2_approx(fminf(uy, ty) - my + pad[nt].y);
            p2 = f2_fma(p2, f2_pack(ex, ey), p2);
          }
        }
        float a, bb;
        f2_unpack(s2, a, bb);
        su[cc] = a + bb;
        f2_unpack(m2, a, bb);
        am[cc] = a + bb;
        f2_unpack(p2, a, bb);
        pr[cc] = a * bb;
      }
      // head sums for the owned candidate
      float sum_u = keep_add(su[0], su[1], s);
      float part = 0.f;  // MODE 0: sum of the LSE excess over z; MODE 2: sum of u^2
      if (MODE == 0) part = keep_add(am[0], am[1], s) + lg2_approx(keep_mul(pr[0], pr[1], s));
      if (MODE == 2) part = keep_add(am[0], am[1], s);
      sum_u += __shfl_xor_sync(kFull, sum_u, 2);
      if (MODE != 1) part += __shfl_xor_sync(kFull, part, 2);
      const bool valid = oc < nC;
      const bool two = 2 * c + 1 <= lim;
      const bool ref1 = c == rag;
      const float nr = ref1 ? rnr : -1.f;
      bool keep = valid;
      if (scoring) {
        float two_sc = part;  // the candidate's score minus Z when both children count
        if (MODE == 1) two_sc = 0.5f * (1.f + nr) * sum_u;
        if (MODE == 2) two_sc = 0.5f * (1.f + nr) * sum_u + 0.69314718055994531f * 0.125f * (1.f - nr) * (1.f - nr) * part;
        const float sc = Z + (two ? two_sc : (ref1 ? nr : 1.f) * sum_u);
        // order-preserving integer key; the low 4 bits hold 15 - candidate (lower index wins a tie)
        const unsigned fb = __float_as_uint(sc);
        unsigned key = fb ^ ((unsigned)((int)fb >> 31) | 0x80000000u);
        key = valid ? ((key & ~15u) | (unsigned)(15 - oc)) : 0u;
        // rank = number of larger keys: lanes j < 2 count among candidates 0..7, j >= 2 among 8..15
        unsigned* keys = reinterpret_cast<unsigned*>(cbuf) + 64;
        if (j < 2) keys[oc] = key;
        __syncwarp();
        const uint4* kq = reinterpret_cast<const uint4*>(keys + 8 * (j >> 1));
        const uint4 k0 = kq[0], k1 = kq[1];
        int rank = (k0.x > key) + (k0.y > key) + (k0.z > key) + (k0.w > key) + (k1.x > key) + (k1.y > key) +
                   (k1.z > key) + (k1.w > key);
        rank += __shfl_xor_sync(kFull, rank, 2);
        keep = valid && rank < K;
      }
      // survivors before this candidate (in candidate order), and those with two children
      const unsigned bk = __ballot_sync(kFull, keep), b2 = __ballot_sync(kFull, keep && two);
      const int before = s ? __popc(bk & kLo) + __popc(bk & kHi & lt) : __popc(bk & kLo & lt);
      if (l == 2) {
        if (j < 2 && keep && PISA_IN_BOUNDS(c >= 0 && c < M2 && before < K)) {
          out[before] = c;
          rk[before] = atomicAdd(cnt + c, 1);
        }
        const int nS = __popc(bk & (kLo | kHi));
        if (lane < K && lane >= nS) out[lane] = -1;
        break;
      }
      // next candidates: the survivors' eligible children, ascending, with their Z
      {
        const float zr = Z + sum_u, zo = fmaf(nr, sum_u, Z);
        int* buf = cbuf + ((l & 1) << 5);
        if (j < 2 && keep) {
          const int pos = before + (s ? __popc(b2 & kLo) + __popc(b2 & kHi & lt) : __popc(b2 & kLo & lt));
          buf[pos] = 2 * c;
          buf[16 + pos] = __float_as_int(ref1 ? zo : zr);
          if (two) {
            buf[pos + 1] = 2 * c + 1;
            buf[16 + pos + 1] = __float_as_int(ref1 ? zr : zo);
          }
        }
        nC = __popc(bk & (kLo | kHi)) + __popc(b2 & (kLo | kHi));
        __syncwarp();
        if (oc < nC) {
          c = buf[oc];
          Z = __int_as_float(buf[16 + oc]);
        }
      }
    }
  }
}


// ---------------------------------------------------------------------------
// The K <= 8 walk for G = 16 with the operands of the MMA swapped: the query's 16
// heads are the A operand (rows g and g + 8 of the fragment, loaded once per
// query) and the candidates' rows are the B operand (n = g of each 8-candidate
// tile).  A lane's B pair for k-step ks is two adjacent words of one row in the
// table's layout, so the rows feed the MMA straight from their 16-byte loads
// (with candidates as the A operand every A quad mixes two rows and has to be
// assembled by register moves).  After the MMAs lane (g, j) holds u for heads g,
// g + 8 and candidates 8 ct + 2 j + e (ct, e in {0, 1}); the head sums run as a
// three-step butterfly over g that leaves candidate oc = 8 b4 + 2 j + b3 (bN =
// lane bit N) on the two lanes that differ in bit 2.  Same arithmetic per
// (candidate, head) as walk_k8_kernel; head sums associate differently.

// Keeps the value of candidate `hi` (if the lane bit is set) or `lo` and adds
// (or multiplies) the partner's copy of the same candidate.
__device__ __forceinline__ float bfly_add(float lo, float hi, int bit, int mask) {
  const float send = bit ? lo : hi, mine = bit ? hi : lo;
  return mine + __shfl_xor_sync(kFull, send, mask);
}

// q . row for this lane's two B rows (ra: candidate g, rb: candidate g + 8) against
// the query's heads: u[ct][0..1] = head g, candidates 8 ct + 2 j + {0, 1};
// u[ct][2..3] = head g + 8, the same candidates.  The B pair of k-step ks is the
// word pair (2 (ks & 1), +1) of ra / rb [ks >> 1] (hi) and [2 + (ks >> 1)] (lo).
__device__ __forceinline__ void tile_dots_s(const uint32_t (&A)[4][4], const uint4 (&ra)[4], const uint4 (&rb)[4],
                                            float (&u)[2][4]) {
  float dh[2][4], dl[2][4];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    const uint4& Ha = ra[ks >> 1];
    const uint4& La = ra[2 + (ks >> 1)];
    const uint4& Hb = rb[ks >> 1];
    const uint4& Lb = rb[2 + (ks >> 1)];
    const bool hw = ks & 1;
    if (ks == 0) {
      mma_bf16_16816_z(dh[0], A[ks], Ha.x, Ha.y);
      mma_bf16_16816_z(dl[0], A[ks], La.x, La.y);
      mma_bf16_16816_z(dh[1], A[ks], Hb.x, Hb.y);
      mma_bf16_16816_z(dl[1], A[ks], Lb.x, Lb.y);
    } else {
      mma_bf16_16816(dh[0], A[ks], hw ? Ha.z : Ha.x, hw ? Ha.w : Ha.y);
      mma_bf16_16816(dl[0], A[ks], hw ? La.z : La.x, hw ? La.w : La.y);
      mma_bf16_16816(dh[1], A[ks], hw ? Hb.z : Hb.x, hw ? Hb.w : Hb.y);
      mma_bf16_16816(dl[1], A[ks], hw ? Lb.z : Lb.x, hw ? Lb.w : Lb.y);
    }
  }
#pragma unroll
  for (int ct = 0; ct < 2; ++ct)
#pragma unroll
    for (int i = 0; i < 4; ++i) u[ct][i] = dh[ct][i] + dl[ct][i];
}

template <int MODE>
__global__ void __launch_bounds__(kWalk8Warps * 32, 1) walk_k8s_kernel(
    const __nv_bfloat16* __restrict__ Q, const unsigned char* __restrict__ table, Levels lv, RowOffsets ro,
    LevelTail tail, long long rows_per_bh, int N, int Hq, int Hkv, int K, int causal, int l_start, int l_lo,
    int32_t* __restrict__ surv, int32_t* __restrict__ srank, int* __restrict__ count, int t0, int t1, int chunk_shift,
    int M2) {
  extern __shared__ __align__(16) unsigned char wsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, j = lane & 3;
  const int b2 = (lane >> 2) & 1, b3 = (lane >> 3) & 1, b4 = (lane >> 4) & 1;
  const int oc = 8 * b4 + 2 * j + b3;  // the candidate this lane owns after the head sums
  // first-copy lane of candidate c: 16 (c >> 3) + 8 (c & 1) + ((c >> 1) & 3); `below` marks
  // those of the candidates before oc, kOwn all first copies (lane bit 2 clear)
  unsigned below = 0;
  for (int c = 0; c < oc; ++c) below |= 1u << (16 * (c >> 3) + 8 * (c & 1) + ((c >> 1) & 3));
  constexpr unsigned kOwn = 0x0F0F0F0Fu;
  constexpr int G = 16;  // the launcher's condition (Hq / Hkv == 16)
  const long long bh = blockIdx.y;
  const int kv = (int)(bh % Hkv);
  const long long b = bh / Hkv;
  const long long zrow0 = ro.o[lv.L + 1] + 1;
  const int crow0 = (l_start >= 2) ? (int)ro.o[l_lo] : 0;
  const int ncache = (l_start >= 2) ? (int)(ro.o[l_start + 1] - ro.o[l_lo]) : 0;
  unsigned char* czr = wsm;
  unsigned char* cdr = wsm + 16 * kCacheRowBytes;
  int* cbuf = reinterpret_cast<int*>(cdr + (size_t)ncache * kCacheRowBytes) + warp * kCandBuf;
  __shared__ int4 lvt[kMaxLevels + 2];
  if (threadIdx.x >= 2 && threadIdx.x <= lv.L) {
    const int l = threadIdx.x;
    const bool cached = l >= l_lo && l <= l_start;
    lvt[l] = make_int4(cached ? (int)((ro.o[l] - crow0) * kCacheRowBytes) : (int)ro.o[l], lv.M[l - 1] - 1,
                       tail.node[l], __float_as_int(tail.nr[l]));
  }
  const unsigned char* tb = table + bh * rows_per_bh * kRowBytes;
  if (l_start >= 2) {
    for (int e = threadIdx.x; e < 16 * 16; e += blockDim.x)
      *reinterpret_cast<uint4*>(czr + (e >> 4) * kCacheRowBytes + (e & 15) * 16) =
          __ldg(reinterpret_cast<const uint4*>(tb + zrow0 * kRowBytes) + e);
    for (int e = threadIdx.x; e < ncache * 16; e += blockDim.x)
      *reinterpret_cast<uint4*>(cdr + (e >> 4) * kCacheRowBytes + (e & 15) * 16) =
          __ldg(reinterpret_cast<const uint4*>(tb + (long long)crow0 * kRowBytes) + e);
  }
  __syncthreads();
  for (int t = t0 + blockIdx.x + gridDim.x * warp; t < t1; t += gridDim.x * kWalk8Warps) {
    __syncwarp();  // the previous query's reads of the candidate buffers are done
    const long long job = bh * N + t;
    if (l_start < 2) {
      int32_t* out = surv + job * K;
      int32_t* rk = srank + job * K;
      int* cnt = count + ((long long)(t >> chunk_shift) * gridDim.y + bh) * M2;  // chunk-major buckets
      const int m2 = lv.L >= 2 ? lv.M[2] : 1;
      const int el = causal ? min(m2, (t >> (kLog2C + 1)) + 1) : m2;
      if (lane < K) {
        const int p = lane < el ? lane : -1;
        out[lane] = p;
        if (p >= 0) rk[lane] = atomicAdd(cnt + p, 1);
      }
      continue;
    }
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(Q + ((b * N + t) * Hq + (long long)kv * G) * kD);
    {  // the warp's next query: its G head rows into L2 while this one walks
      const int tn = t + gridDim.x * kWalk8Warps;
      if (tn < t1 && lane < G)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(Q + ((b * N + tn) * Hq + (long long)kv * G + lane) * kD));
    }
    // Q as the A operand: [ks] = {head g word 8ks + j, head g + 8 same word, head g word
    // 8ks + j + 4, head g + 8 same word} (all 16 heads are real: G = 16)
    uint32_t A[4][4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const int w0 = 8 * ks + j;
      A[ks][0] = __ldg(q0 + g * 32 + w0);
      A[ks][2] = __ldg(q0 + g * 32 + w0 + 4);
      A[ks][1] = __ldg(q0 + (g + 8) * 32 + w0);
      A[ks][3] = __ldg(q0 + (g + 8) * 32 + w0 + 4);
    }
    int nC;
    {
      const int ml = lv.M[l_start];
      nC = causal ? min(ml, (t >> (kLog2C + l_start - 1)) + 1) : ml;
    }
    int c = oc;            // node id of the owned candidate
    int na = g, nb = g + 8;  // node ids of this lane's B rows (candidates g and g + 8)
    float Z;
    {
      uint4 ra[4], rb[4];
      ld_row(czr + g * kCacheRowBytes + 32 * j, true, ra[0], ra[1], ra[2], ra[3]);
      ld_row(czr + (g + 8) * kCacheRowBytes + 32 * j, true, rb[0], rb[1], rb[2], rb[3]);
      float u[2][4];
      tile_dots_s(A, ra, rb, u);
      // sum over the lane's two heads, then over g
      const float z0 = u[0][0] + u[0][2], z1 = u[0][1] + u[0][3], z2 = u[1][0] + u[1][2], z3 = u[1][1] + u[1][3];
      float ze = bfly_add(z0, z2, b4, 16), zo = bfly_add(z1, z3, b4, 16);
      Z = bfly_add(ze, zo, b3, 8);
      Z += __shfl_xor_sync(kFull, Z, 4);
    }
    for (int l = l_start;; --l) {
      const bool scoring = nC > K;
      const int4 lt4 = lvt[l];
      const int lim = causal ? min(lt4.y, t >> (l + 4)) : lt4.y;  // last eligible second child
      const int rag = lt4.z;
      const float rnr = __int_as_float(lt4.w);
      const bool va = g < nC, vb = g + 8 < nC;
      int ra_row = va ? na : 0, rb_row = vb ? nb : 0;  // (rows >= nC: never kept)
      if (!PISA_IN_BOUNDS(ra_row >= 0 && ra_row < lv.M[l] && rb_row >= 0 && rb_row < lv.M[l])) ra_row = rb_row = 0;
      uint4 ra[4], rb[4];
      if (l >= l_lo) {
        const unsigned char* base = cdr + lt4.x + 32 * j;
        ld_row(base + ra_row * kCacheRowBytes, true, ra[0], ra[1], ra[2], ra[3]);
        ld_row(base + rb_row * kCacheRowBytes, true, rb[0], rb[1], rb[2], rb[3]);
      } else {
        const unsigned char* base = tb + (long long)lt4.x * kRowBytes + 32 * j;
        ld_row(base + ra_row * kRowBytes, false, ra[0], ra[1], ra[2], ra[3]);
        ld_row(base + rb_row * kRowBytes, false, rb[0], rb[1], rb[2], rb[3]);
      }
      float u[2][4];
      tile_dots_s(A, ra, rb, u);
      // per candidate 8 ct + 2 j + e over the lane's two heads: sum of u, and the
      // LSE excess over z (MODE 0) or the sum of u^2 (MODE 2)
      float su[2][2], pt[2][2];
      const bool any_rag = MODE == 0 && rag >= 0 && __any_sync(kFull, (va && na == rag) || (vb && nb == rag));
      const int* cur = cbuf + (((l + 1) & 1) << 5);  // this level's candidate node ids
#pragma unroll
      for (int ct = 0; ct < 2; ++ct) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float ua = u[ct][e], ub = u[ct][2 + e];  // heads g and g + 8
          su[ct][e] = ua + ub;
          if (MODE == 2) pt[ct][e] = fmaf(ua, ua, ub * ub);
          if (MODE == 0 && !any_rag) {  // r = 1: max(u, -u) = |u|, exponent -2 |u|
            const float aa = fabsf(ua), ab = fabsf(ub);
            const float ea = ex2_approx(-2.f * aa), eb = ex2_approx(-2.f * ab);
            pt[ct][e] = (aa + ab) + lg2_approx(fmaf(ea, 1.f + eb, 1.f + eb));
          } else if (MODE == 0) {
            float nr = -1.f;
            {
              const int ci = 8 * ct + 2 * j + e;
              const int nd = l == l_start ? ci : cur[ci];
              if (ci < nC && nd == rag) nr = rnr;
            }
            // max(u, nr u) + log2(1 + 2^(min - max)) per head, summed over the two
            const float tax = nr * ua, tbx = nr * ub;
            const float mxa = fmaxf(ua, tax), mxb = fmaxf(ub, tbx);
            const float ea = ex2_approx(fminf(ua, tax) - mxa), eb = ex2_approx(fminf(ub, tbx) - mxb);
            pt[ct][e] = (mxa + mxb) + lg2_approx(fmaf(ea, 1.f + eb, 1.f + eb));
          }
        }
      }
      // butterfly over g: keep tile b4, then parity b3, then add the copy on lane ^ 4
      float sum_u = bfly_add(bfly_add(su[0][0], su[1][0], b4, 16), bfly_add(su[0][1], su[1][1], b4, 16), b3, 8);
      sum_u += __shfl_xor_sync(kFull, sum_u, 4);
      float part = 0.f;
      if (MODE != 1) {
        part = bfly_add(bfly_add(pt[0][0], pt[1][0], b4, 16), bfly_add(pt[0][1], pt[1][1], b4, 16), b3, 8);
        part += __shfl_xor_sync(kFull, part, 4);
      }
      const bool valid = oc < nC;
      const bool two = 2 * c + 1 <= lim;
      const bool ref1 = c == rag;
      const float nr = ref1 ? rnr : -1.f;
      bool keep = valid;
      if (scoring) {
        float two_sc = part;
        if (MODE == 1) two_sc = 0.5f * (1.f + nr) * sum_u;
        if (MODE == 2) two_sc = 0.5f * (1.f + nr) * sum_u + 0.69314718055994531f * 0.125f * (1.f - nr) * (1.f - nr) * part;
        const float sc = Z + (two ? two_sc : (ref1 ? nr : 1.f) * sum_u);
        const unsigned fb = __float_as_uint(sc);
        unsigned key = fb ^ ((unsigned)((int)fb >> 31) | 0x80000000u);
        key = valid ? ((key & ~15u) | (unsigned)(15 - oc)) : 0u;
        // rank = number of larger keys: lanes with bit 2 clear count among candidates 0..7,
        // the others among 8..15
        unsigned* keys = reinterpret_cast<unsigned*>(cbuf) + 64;
        if (b2 == 0) keys[oc] = key;
        __syncwarp();
        const uint4* kq = reinterpret_cast<const uint4*>(keys + 8 * b2);
        const uint4 k0 = kq[0], k1 = kq[1];
        int rank = (k0.x > key) + (k0.y > key) + (k0.z > key) + (k0.w > key) + (k1.x > key) + (k1.y > key) +
                   (k1.z > key) + (k1.w > key);
        rank += __shfl_xor_sync(kFull, rank, 4);
        keep = valid && rank < K;
      }
      const unsigned bk = __ballot_sync(kFull, keep), b2k = __ballot_sync(kFull, keep && two);
      const int before = __popc(bk & below);
      if (l == 2) {
        int32_t* out = surv + job * K;
        int32_t* rk = srank + job * K;
        int* cnt = count + ((long long)(t >> chunk_shift) * gridDim.y + bh) * M2;  // chunk-major buckets
        if (b2 == 0 && keep && PISA_IN_BOUNDS(c >= 0 && c < M2 && before < K)) {
          out[before] = c;
          rk[before] = atomicAdd(cnt + c, 1);
        }
        const int nS = __popc(bk & kOwn);
        if (lane < K && lane >= nS) out[lane] = -1;
        break;
      }
      {
        const float zr = Z + sum_u, zo = fmaf(nr, sum_u, Z);
        int* buf = cbuf + ((l & 1) << 5);
        if (b2 == 0 && keep && PISA_IN_BOUNDS(before + __popc(b2k & below) + (two ? 1 : 0) < 16)) {
          const int pos = before + __popc(b2k & below);
          buf[pos] = 2 * c;
          buf[16 + pos] = __float_as_int(ref1 ? zo : zr);
          if (two) {
            buf[pos + 1] = 2 * c + 1;
            buf[16 + pos + 1] = __float_as_int(ref1 ? zr : zo);
          }
        }
        nC = __popc(bk & kOwn) + __popc(b2k & kOwn);
        __syncwarp();
        if (oc < nC) {
          c = buf[oc];
          Z = __int_as_float(buf[16 + oc]);
        }
        na = g < nC ? buf[g] : 0;
        nb = g + 8 < nC ? buf[g + 8] : 0;
      }
    }
  }
}

// Host side: table size and launches.
static int walk_sm_count() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 152;
  }
  return n[dev];
}

long long route_rows_per_bh(const Levels& lv) {
  long long r = 1 + kZRows;  // the zero row and the mean rows
  for (int l = 2; l <= lv.L; ++l) r += lv.M[l];
  return r;
}

cudaError_t launch_prefill_walk_mma(const WalkLaunch& W, cudaStream_t s) {
  const Levels& lv = *W.lv;
  const long long rows = route_rows_per_bh(lv);
  const int BH = W.B * W.Hkv;
  RowOffsets ro;  // row offset of each level inside a (b, kv) table (levels 2..L ascending)
  long long o = 0;
  for (int l = 0; l < kMaxLevels + 2; ++l) ro.o[l] = 0;
  for (int l = 2; l <= lv.L; ++l) {
    ro.o[l] = o;
    o += lv.M[l];
  }
  ro.o[lv.L + 1] = o;
  // first scored level: the highest level holding more than K nodes (0: none)
  int l_start = 0;
  for (int l = lv.L; l >= 2; --l)
    if (lv.M[l] > W.K) {
      l_start = l;
      break;
    }
  cudaError_t e = cudaSuccess;
  PISA_SET_BOUNDS_STATUS(W.status, s);
  if (W.build_table) {
    const long long thr = (long long)BH * rows * 32;
    route_table_kernel<<<(unsigned)((thr + 255) / 256), 256, 0, s>>>(W.summ, lv, W.N, BH, rows, ro, l_start, W.table);
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    mark_phase(1, s);
  }
  if (W.t1 <= W.t0) return cudaSuccess;
  // the rows of levels [l_lo, l_start] (at most kCacheRows / kCacheRows8) are cached in
  // shared memory
  const bool k8 = W.K <= 8;
  const int cache_rows = k8 ? kCacheRows8 : kCacheRows;
  int l_lo = l_start + 1, crows = 0;
  while (l_start >= 2 && l_lo - 1 >= 2 && crows + lv.M[l_lo - 1] <= cache_rows) {
    --l_lo;
    crows += lv.M[l_lo];
  }
  // CTAs per (b, kv): one CTA per SM (K <= 8) or about three, over the whole grid
  const long long ctas = (k8 ? 1LL : 3LL) * walk_sm_count();
  int per_bh = (int)((ctas + BH - 1) / BH);
  if (per_bh > W.t1 - W.t0) per_bh = (int)(W.t1 - W.t0);
  if (per_bh < 1) per_bh = 1;
  dim3 grid((unsigned)per_bh, (unsigned)BH);
  const int G = W.Hq / W.Hkv;
  if (W.K <= 8) {
    LevelTail tail;
    for (int l = 0; l < kMaxLevels + 2; ++l) {
      tail.node[l] = -1;
      tail.nr[l] = -1.f;
    }
    for (int l = 2; l <= lv.L; ++l) {
      const int Mc = lv.M[l - 1];
      if (Mc >= 2 && (Mc & 1) == 0) {
        const int n0 = node_count(l - 1, Mc - 2, W.N), n1 = node_count(l - 1, Mc - 1, W.N);
        if (n1 < n0) {
          tail.node[l] = Mc / 2 - 1;
          tail.nr[l] = -((float)n1 / (float)n0);
        }
      }
    }
    const size_t smem = (size_t)(16 + crows) * kCacheRowBytes + (size_t)kWalk8Warps * kCandBuf * 4;
    auto pick = [&](auto nt) {
      constexpr int NT = decltype(nt)::value;
      return W.mode == 1 ? walk_k8_kernel<NT, 1> : W.mode == 2 ? walk_k8_kernel<NT, 2> : walk_k8_kernel<NT, 0>;
    };
    auto pick_s = [&]() {
      return W.mode == 1 ? walk_k8s_kernel<1> : W.mode == 2 ? walk_k8s_kernel<2> : walk_k8s_kernel<0>;
    };
    // G = 16: the swapped-operand walk; smaller groups (one 8-head tile) keep the
    // candidates as the A operand
    auto kern = G == 16 ? pick_s() : pick(std::integral_constant<int, 1>());
    {
      static std::mutex mu;
      static size_t attr[2][3] = {};
      std::lock_guard<std::mutex> lock(mu);
      if (smem > attr[G > 8][W.mode]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr[G > 8][W.mode] = smem;
      }
    }
    kern<<<grid, kWalk8Warps * 32, smem, s>>>(W.Q, W.table, lv, ro, tail, rows, (int)W.N, W.Hq, W.Hkv, W.K, W.causal,
                                              l_start, l_lo, W.surv, W.srank, W.count, (int)W.t0, (int)W.t1,
                                              W.chunk_shift, W.M2);
    note_launch();
    return cudaGetLastError();
  }
  const size_t smem = walk_smem_per_warp(W.K) * kWalkWarps + (size_t)crows * kCacheRowBytes;
  {  // per-warp scratch grows with K, the row cache with the tree
    static std::mutex mu;
    static size_t attr = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (smem > attr) {
      e = cudaFuncSetAttribute(walk_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr = smem;
    }
  }
  walk_mma_kernel<<<grid, kWalkWarps * 32, smem, s>>>(W.Q, W.summ, W.table, lv, ro, rows, (int)W.N, W.Hq, W.Hkv, W.K,
                                                       W.causal, l_start, l_lo, W.surv, W.srank, W.count,
                                                       (int)W.t0, (int)W.t1, W.chunk_shift, W.M2, W.mode);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pisa
