// leaf_tc.cu -- the leaf level of the prefill walk on the 5th-generation tensor
// cores, with queries clustered by the key block they need.
//
// "Block Sparse Attention with Log-Linear Complexity", "Scoring: LogSumExp"
// (at the leaf level the score of a block is the exact log-sum-exp over its raw
// keys), §4.1 (summed over the query heads of a GQA group) and §5.1 (the prefill
// kernel clusters the queries that need the same key block so that each loaded
// block is reused by all of them).
//
// After the intermediate levels every query holds <= K level-2 survivors p; its
// leaf candidates are the two children 2p, 2p+1 of each, i.e. the 128 keys
// [128p, 128p+128).  Pipeline (on one stream, for a run of whole query chunks):
//   (the walk kernel)   counts (query, survivor) pairs per bucket, a bucket being
//                       (query chunk, b * Hkv + kv, p), chunk-major so that a run
//                       of chunks owns one contiguous range of buckets and tiles;
//                       a chunk of 2^chunk_shift query positions keeps the
//                       gathered query rows L2-resident
//   leaf_scan_kernel    exclusive scans: entry offsets and tile offsets
//   leaf_scatter_kernel write each pair (t << 5 | slot) into its bucket
//   leaf_tile_desc_kernel  one descriptor per tile {first entry, rows, p, b*Hkv+kv}
//   leaf_tc_kernel      persistent, warp-specialised: per tile of R = 128/max(G,8)
//                       queries of one bucket, D[128 x 128] = Q_rows[128 x 64] x
//                       K_block[128 x 64]^T on tcgen05 (bf16 in, fp32 in TMEM),
//                       then per row two masked log-sum-exps and a sum over the
//                       group's heads
//   leaf_final(8)_kernel  Top-K of the <= 2K leaf scores per query
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "api.cuh"
#include "tc.cuh"

namespace pisa {

constexpr int kAccBufs = 4;       // TMEM accumulators of 128 fp32 columns (two pairs of tiles)
// Query-row stages (16 KB each), one per accumulator: the stages of a pair of tiles are
// free again once the pair's MMAs have completed, which acc_pair already signals.
constexpr int kLeafStages = kAccBufs;
static_assert(kAccBufs == 4, "two pair stages of two tiles each: indices are taken with masks");
constexpr int kLeafWarps = 20;    // key-block loader, MMA, 2 query-row warps, 4 epilogue warpgroups
constexpr int kEpiGroups = 4;     // epilogue warpgroups (warps 4..19)
// Warpgroup w takes tiles w, w + 4, ...: before waiting for tile k (pair k / 2) it has
// seen tile k - 4 (pair k / 2 - 2, the same pair stage) complete, so the barrier it waits
// on is exactly one phase ahead of what it saw, and it cannot run further ahead either:
// the next phase of that stage needs this tile's own release.
static_assert(kEpiGroups == kAccBufs, "the phase argument above takes one tile per accumulator and warpgroup");
constexpr int kTileBlock = 32;    // consecutive tiles handled by one CTA in a row (even: pairs never straddle)
constexpr int kTileBytes = 128 * 128;  // 128 rows of 64 bf16
constexpr int kKeyBufs = 4;       // key blocks in flight (the loader runs up to 3 blocks ahead)
constexpr size_t kLeafSmem = (size_t)(kLeafStages + kKeyBufs) * kTileBytes + 1024;

struct LeafTcParams {
  const __nv_bfloat16* Q;
  const uint32_t* list;
  const int* bucket_off;
  const int* tile_off;
  const int4* tile_desc;  // per tile: first entry, rows, level-2 survivor p, b * Hkv + kv
  int b0, b1;  // the buckets of this launch; their tiles are tile_off[b0] .. tile_off[b1] - 1
  int Hq, Hkv, G, Gp, R, K;
  long long N, n_cap;
  int M2, nchunks;
  int causal;
  float* leaf_scores;
  int* status;
  // flat mode: every query row of a tile is scored against the tile's key block and the two
  // leaf scores go to leaf_scores[(b * Hkv + kv) * N + t][2p, 2p + 1] (row stride flat_stride)
  int flat;
  long long flat_stride;
};

// Global index of this CTA's k-th tile: blocks of kTileBlock consecutive tiles,
// block j on CTA j % gridDim.x.
__device__ __forceinline__ int tile_of(int k) {
  return (blockIdx.x + gridDim.x * (k / kTileBlock)) * kTileBlock + (k % kTileBlock);
}

__device__ __forceinline__ void leaf_abort(volatile int* abort, int* status) {
  *abort = 1;
  set_status(status, PISA_ERR_DEVICE_TIMEOUT);
}

constexpr float kL2e8 = 0.18033688011112042f;  // log2(e) / sqrt(64)

// sum_{i < cnt} 2^(x_i * log2(e)/8 + nb) over one 32-column chunk of raw q.k dot
// products (nb = -ref * log2(e)/8 for the half's reference logit ref), for halves
// that some lane does not have in full (the causal edge): four scalar accumulators.
__device__ __forceinline__ float chunk_exp_sum(const float (&x)[32], int cnt, float nb) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    s0 += c < cnt ? ex2_approx(fmaf(x[c], kL2e8, nb)) : 0.f;
    s1 += c + 1 < cnt ? ex2_approx(fmaf(x[c + 1], kL2e8, nb)) : 0.f;
    s2 += c + 2 < cnt ? ex2_approx(fmaf(x[c + 2], kL2e8, nb)) : 0.f;
    s3 += c + 3 < cnt ? ex2_approx(fmaf(x[c + 3], kL2e8, nb)) : 0.f;
  }
  return (s0 + s1) + (s2 + s3);
}

// sum over one full 64-key half (two 32-column chunks x, y) of 2^(x_i log2(e)/8 + nb):
// packed f32x2 arithmetic (one fma.f32x2 and one add.f32x2 per two keys), both chunks
// into the same four pair accumulators, reduced once.
__device__ __forceinline__ float half_exp_sum_full(const float (&x)[32], const float (&y)[32], float nb) {
  const unsigned long long k2 = f2_pack(kL2e8, kL2e8), n2 = f2_pack(nb, nb);
  unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float a, b;
    f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), k2, n2), a, b);
    acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], f2_pack(ex2_approx(a), ex2_approx(b)));
  }
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float a, b;
    f2_unpack(f2_fma(f2_pack(y[c], y[c + 1]), k2, n2), a, b);
    acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], f2_pack(ex2_approx(a), ex2_approx(b)));
  }
  float p, q;
  f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), p, q);
  return p + q;
}

// Masked log-sum-exp of one 64-key half (one leaf) from two 32-column chunks.
// Exponents are taken relative to the half's first key (no max pass); if the sum
// would overflow, the reference moves up to the half's maximum and the sum is
// taken again.
struct HalfLse {
  float ref, s;
  // One 64-key half from two 32-column chunks (cnt0 + cnt1 keys, cnt0 >= 1); `full`
  // (warp-uniform) means every lane has 64: one overflow vote for the half.
  __device__ __forceinline__ void first2(const float (&x)[32], const float (&y)[32], int cnt0, int cnt1, bool full) {
    ref = x[0];
    const float nb = -ref * kL2e8;
    const float t = full ? half_exp_sum_full(x, y, nb) : chunk_exp_sum(x, cnt0, nb) + chunk_exp_sum(y, cnt1, nb);
    if (__any_sync(kFull, !(t <= 3.0e38f))) {  // rare: rescale against the half's maximum
      if (!(t <= 3.0e38f)) {
        float m = ref;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c < cnt0) m = fmaxf(m, x[c]);
          if (c < cnt1) m = fmaxf(m, y[c]);
        }
        s = chunk_exp_sum(x, cnt0, -m * kL2e8) + chunk_exp_sum(y, cnt1, -m * kL2e8);
        ref = m;
      } else {
        s = t;
      }
    } else {
      s = t;
    }
  }
  __device__ __forceinline__ float value() const {  // natural-log units
    return ref * 0.125f + lg2_approx(s) * 0.69314718055994531f;
  }
};

// The score modes' counterpart of HalfLse: mean (MODE 1) or mean + variance / 2
// (MODE 2) of the logits z = x / 8 of one 64-key half, from shifted sums
// sum (x - x0) and sum (x - x0)^2 (x0 = the half's first key) for conditioning.
template <int MODE>
struct HalfMom {
  float ref, s1, s2;
  int n;
  __device__ __forceinline__ void first(const float (&x)[32], int cnt, bool full) {
    ref = x[0];
    s1 = s2 = 0.f;
    n = 0;
    add(x, cnt, full);
  }
  __device__ __forceinline__ void add(const float (&x)[32], int cnt, bool full) {
    if (full) {
      const unsigned long long nr2 = f2_pack(-ref, -ref);
      unsigned long long a1 = 0ull, a2 = 0ull;
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const unsigned long long d2 = f2_add(f2_pack(x[c], x[c + 1]), nr2);
        a1 = f2_add(a1, d2);
        a2 = f2_fma(d2, d2, a2);
      }
      float p, q;
      f2_unpack(a1, p, q);
      s1 += p + q;
      f2_unpack(a2, p, q);
      s2 += p + q;
      n += 32;
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float dd = c < cnt ? x[c] - ref : 0.f;
        s1 += dd;
        s2 = fmaf(dd, dd, s2);
      }
      n += cnt;
    }
  }
  __device__ __forceinline__ void first2(const float (&x)[32], const float (&y)[32], int cnt0, int cnt1, bool full) {
    first(x, cnt0, full);
    add(y, cnt1, full);
  }
  __device__ __forceinline__ float value() const {  // natural-log units
    const float inv = 1.f / (float)n, m = s1 * inv;
    float v = (ref + m) * 0.125f;
    if (MODE == 2) v += 0.5f * fmaxf(s2 * inv - m * m, 0.f) * 0.015625f;
    return v;
  }
};

// Orders the uses of registers written by tcgen05.ld after the wait::ld that
// completes them.
__device__ __forceinline__ void reg_fence32(float (&x)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 8)
    asm volatile("" : "+f"(x[i]), "+f"(x[i + 1]), "+f"(x[i + 2]), "+f"(x[i + 3]), "+f"(x[i + 4]), "+f"(x[i + 5]),
                 "+f"(x[i + 6]), "+f"(x[i + 7]));
}

// MODE: 0 LSE over each leaf's keys, 1 their mean logit, 2 mean + variance / 2.
//
// Tiles are processed in pairs (k, k + 1), k even, CTA-local.  Pair P uses query-row
// stages and TMEM accumulators 2 (P & 1) and 2 (P & 1) + 1: one barrier a_pair[P & 1]
// completes when both tiles' query rows have landed, one commit after the pair's eight
// MMAs completes acc_pair[P & 1] (one commit per two tiles: the issuing thread's chain of
// waits, MMAs and commits is what bounds this kernel), and the two epilogue warpgroups
// of the pair release acc_free[P & 1] (256 arrivals).
template <int MODE>
__global__ void __launch_bounds__(kLeafWarps * 32, 1)
    leaf_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   LeafTcParams P) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  unsigned char* sA = sm;
  unsigned char* sB = sm + kLeafStages * kTileBytes;
  __shared__ uint64_t a_pair[2], b_full[kKeyBufs], b_empty[kKeyBufs];
  __shared__ uint64_t acc_pair[2], acc_free[2], mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&a_pair[s], 1);
      mbar_init(&acc_pair[s], 1);
      mbar_init(&acc_free[s], 2 * 128);
    }
    for (int s = 0; s < kKeyBufs; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc<kAccBufs * 128>(&tmem_base);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int Gp = P.Gp, G = P.G, R = P.R;
  const int first = __ldg(P.tile_off + P.b0);
  const int total = __ldg(P.tile_off + P.b1) - first;
  const int4* __restrict__ tdesc = P.tile_desc + first;
  int my_tiles = 0;
  for (int blk = blockIdx.x; blk * kTileBlock < total; blk += gridDim.x) my_tiles += min(kTileBlock, total - blk * kTileBlock);
  const int my_pairs = (my_tiles + 1) >> 1;
  bool mma_ok = true;  // the MMA thread's final wait completed (TMEM may be freed)

  if (warp <= 1) {
    // ---------------- warp 0 loads the key block (two sibling leaves, 128 keys) of every
    // run of tiles with the same (b, kv, p) into a ring of kKeyBufs buffers; warp 1 drives the
    // tensor core, a pair of tiles at a time.  Both read this CTA's tile descriptors 32 at a
    // time (kTileBlock is even, so a pair never straddles two blocks) and find the key-block
    // changes with a ballot.
    const bool mma = warp == 1;
    const uint32_t idesc = umma_idesc_bf16(128, 128);
    int nchg = 0, cur = 0, prev_p = -1, prev_bh = -1, k = 0;
    int nissued = 0;  // key blocks whose copy lane 0 of warp 0 started
    bool ok = true;
    for (int blk = blockIdx.x; ok && blk * kTileBlock < total; blk += gridDim.x) {
      const int i0 = blk * kTileBlock;
      const int n = min(kTileBlock, total - i0);
      const int4 d = lane < n ? __ldg(tdesc + i0 + lane) : make_int4(0, 0, -1, -1);
      int pp = __shfl_up_sync(kFull, d.z, 1), pb = __shfl_up_sync(kFull, d.w, 1);
      if (lane == 0) {
        pp = prev_p;
        pb = prev_bh;
      }
      const unsigned chg = __ballot_sync(kFull, lane < n && (d.z != pp || d.w != pb));
      prev_p = __shfl_sync(kFull, d.z, n - 1);
      prev_bh = __shfl_sync(kFull, d.w, n - 1);
      if (!mma) {
        for (unsigned m = chg; m && ok; m &= m - 1) {
          const int src = __ffs(m) - 1;
          const int p = __shfl_sync(kFull, d.z, src), bh = __shfl_sync(kFull, d.w, src);
          bool w = true;
          if (lane == 0) {
            const int bb = nchg % kKeyBufs;
            if (nchg >= kKeyBufs) w = mbar_wait(&b_empty[bb], ((nchg / kKeyBufs) - 1) & 1, abort);
            if (w) {
              const int pk = PISA_IN_BOUNDS(p >= 0 && p < P.M2 && 128LL * p < P.n_cap && bh >= 0) ? p : 0;
              mbar_expect_tx(&b_full[bb], kTileBytes);
              tma_load_3d(sB + bb * kTileBytes, &kmap, 0, bh % P.Hkv, (int)((bh / P.Hkv) * P.n_cap + 128LL * pk),
                          &b_full[bb]);
              ++nissued;
            }
          }
          ok = __shfl_sync(kFull, w, 0);
          ++nchg;
        }
      } else {
        // the whole warp walks the block's pairs and waits on the barriers (so that it stays
        // converged); lane 0 alone issues the MMAs and the commits.
        bool w = true;
        const uint64_t da0 = umma_desc_sw128(sA), db0 = umma_desc_sw128(sB);
        uint64_t db = db0 + (uint64_t)(cur * (kTileBytes >> 4));
        for (int m = 0; m < n && w; m += 2) {
          const unsigned pr = (unsigned)((k + m) >> 1);
          const unsigned ps = pr & 1u, ph = (pr >> 1) & 1u;
          w = mbar_wait(&a_pair[ps], ph, abort);
          w = w && (pr < 2u || mbar_wait(&acc_free[ps], ph ^ 1u, abort));
          w = __all_sync(kFull, w);
          for (int i = 0; i < 2 && w && m + i < n; ++i) {
            if ((chg >> (m + i)) & 1) {  // warp-uniform (a ballot)
              if (nchg > 0 && lane == 0) umma_commit(&b_empty[cur]);  // fires once the previous block's MMAs are done
              cur = nchg % kKeyBufs;
              db = db0 + (uint64_t)(cur * (kTileBytes >> 4));
              w = __all_sync(kFull, mbar_wait(&b_full[cur], (nchg / kKeyBufs) & 1, abort));
              ++nchg;
            }
            if (w) {
              tc_fence_after();
              if (lane == 0) {
                const unsigned s = 2 * ps + i;
                const uint64_t da = da0 + (uint64_t)(s * (kTileBytes >> 4));
                const uint32_t td = tmem + s * 128;
                umma_bf16_first(td, da, db, idesc);
#pragma unroll
                for (int kk = 1; kk < 4; ++kk) umma_bf16_acc(td, da + 2 * kk, db + 2 * kk, idesc);
              }
            }
          }
          if (w && lane == 0) umma_commit(&acc_pair[ps]);  // also frees the pair's query-row stages
          __syncwarp();
        }
        k += n;
        ok = w;
      }
    }
    if (!ok && lane == 0) leaf_abort(abort, P.status);
    if (mma && lane == 0) {
      // every MMA this thread issued has completed once mma_done fires (waited for even
      // after an abort, with a poll limit); if it never fires TMEM is not freed
      umma_commit(&mma_done);
      if (!mbar_wait(&mma_done, 0, nullptr)) {
        leaf_abort(abort, P.status);
        mma_ok = false;
      }
    }
    if (!mma && lane == 0 && *abort) {
      // after an abort, wait (bounded) for the key blocks still in flight into this CTA
      for (int c = max(0, nissued - kKeyBufs); c < nissued; ++c)
        mbar_wait(&b_full[c % kKeyBufs], (c / kKeyBufs) & 1, nullptr);
    }
  } else if (warp == 2 || warp == 3) {
    // ---------------- query-row warps: pair P's rows are loaded by warp 2 + (P & 1), one
    // TMA box {64 features, G heads, 1 token} per query (lane l: tile 2P + l / R, row l % R),
    // all completing on a_pair[P & 1].  Before refilling the stages of pair P the warp waits
    // for pair P - 2's MMAs (its own previous pair), so it is never two phases ahead.
    const int tw = warp - 2;
    const int sub = lane / R, row = lane % R;  // tile of the pair and row this lane loads
    int issued = -1;  // last pair this warp issued (for the abort drain)
    int last_bh = -1, head0 = 0;  // this lane's last (b, kv) and its first head / token row
    long long row0 = 0;
    for (int pr = tw; pr < my_pairs; pr += 2) {
      const int kt = 2 * pr + sub;
      const bool has = sub < 2 && kt < my_tiles;
      const int4 d = has ? __ldg(tdesc + tile_of(kt)) : make_int4(0, 0, 0, 0);
      const bool live = has && row < d.y;
      const uint32_t ent = live ? __ldg(P.list + d.x + row) : 0u;
      const int ps = pr & 1;
      int nrows = __reduce_add_sync(kFull, live ? 1 : 0);
      bool w = true;
      if (lane == 0) {
        if (pr >= 2) w = mbar_wait(&acc_pair[ps], ((pr >> 1) - 1) & 1, abort);
        if (w) mbar_expect_tx(&a_pair[ps], (uint32_t)(nrows * G * 128));
      }
      if (!__shfl_sync(kFull, w, 0)) {
        if (lane == 0) leaf_abort(abort, P.status);
        break;
      }
      __syncwarp();
      if (live) {
        const long long tq = PISA_IN_BOUNDS((long long)(ent >> 5) < P.N && d.w >= 0) ? (long long)(ent >> 5) : 0;
        if (d.w != last_bh) {
          last_bh = d.w;
          head0 = (d.w % P.Hkv) * G;
          row0 = (long long)(d.w / P.Hkv) * P.N;
        }
        tma_load_3d(sA + (2 * ps + sub) * kTileBytes + row * Gp * 128, &qmap, 0, head0, (int)(row0 + tq),
                    &a_pair[ps]);
      }
      issued = pr;
    }
    if (lane == 0 && *abort && issued >= 0) mbar_wait(&a_pair[issued & 1], (issued >> 1) & 1, nullptr);
  } else {
    // ---------------- epilogue (warps 4..19): warpgroup wg takes tiles wg, wg + 4, ...;
    // TMEM -> registers one key half (64 columns, one leaf) at a time -> its log-sum-exp;
    // the accumulator is released once the second half is in registers.  The head sums
    // and the store of a tile are done while the next tile's first half is being loaded.
    const int wg = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int r = row / Gp, h = row % Gp;
    float pv0 = 0.f, pv1 = 0.f;  // the previous tile's two leaf values (before the head sums)
    float* pout = nullptr;       // where they go (nullptr: nothing pending)
    int4 dn = wg < my_tiles ? __ldg(tdesc + tile_of(wg)) : make_int4(0, 0, 0, 0);
    for (int k = wg; k < my_tiles; k += kEpiGroups) {
      const int pr = k >> 1, ps = pr & 1;
      const int4 d = dn;  // this tile's descriptor (read one tile ahead)
      const bool qvalid = r < d.y;
      const uint32_t ent = qvalid ? __ldg(P.list + d.x + r) : 0u;
      if (k + kEpiGroups < my_tiles) dn = __ldg(tdesc + tile_of(k + kEpiGroups));
      const bool ok = __all_sync(kFull, mbar_wait(&acc_pair[ps], (pr >> 1) & 1, abort));
      if (!ok) {  // warp-uniform exit
        leaf_abort(abort, P.status);
        pout = nullptr;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (k & 3) * 128;
      float xa[32], xb[32];
      tmem_ld32(taddr, xa);
      tmem_ld32(taddr + 32, xb);
      // the previous tile's head sums and store, while the loads are in flight
      {
        float a0 = pv0, a1 = pv1;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
          if (o < Gp) {
            a0 += __shfl_xor_sync(kFull, a0, o);
            a1 += __shfl_xor_sync(kFull, a1, o);
          }
        }
        if (pout) {
          pout[0] = a0;
          pout[1] = a1;
        }
      }
      const int tp = d.z, tbh = d.w;
      const int t = (int)(ent >> 5);  // < 2^27
      const int qslot = ent & 31;
      const int Ni = (int)P.N;
      // keys of this tile that count for the query: [128p, n_eff)
      const int n_eff = P.causal ? min(t + 1, Ni) : Ni;
      const int l = qvalid ? max(1, min(128, n_eff - 128 * tp)) : 128;  // columns [0, l) count
      const int c0 = min(l, 32), c1 = min(max(l - 32, 0), 32), c2 = min(max(l - 64, 0), 32),
                c3 = max(l - 96, 0);
      using Acc = typename std::conditional<MODE == 0, HalfLse, HalfMom<MODE>>::type;
      Acc h0, h1;
      tmem_ld_wait();
      reg_fence32(xa);
      reg_fence32(xb);
      h0.first2(xa, xb, c0, c1, __all_sync(kFull, l >= 64));
      const bool head = qvalid && h < G;
      pv0 = head ? h0.value() : 0.f;  // (h0 is dead from here on: fewer live registers)
      tmem_ld32(taddr + 64, xa);
      tmem_ld32(taddr + 96, xb);
      tmem_ld_wait();
      reg_fence32(xa);
      reg_fence32(xb);
      tc_fence_before();
      mbar_arrive(&acc_free[ps]);
      const bool any1 = __any_sync(kFull, c2 > 0);
      if (any1) h1.first2(xa, xb, c2 > 0 ? c2 : 1, c3, __all_sync(kFull, l == 128));
      pv1 = (head && any1) ? h1.value() : 0.f;
      pout = nullptr;
      if (qvalid && h == 0 && PISA_IN_BOUNDS(t < Ni && (P.flat || qslot < P.K))) {
        const long long job = (long long)tbh * Ni + t;
        pout = P.flat ? P.leaf_scores + job * P.flat_stride + 2 * tp : P.leaf_scores + job * (2 * P.K) + 2 * qslot;
        if (l <= 64) pv1 = -INFINITY;  // the second leaf starts after the query
      }
    }
    {  // the last tile's head sums and store
      float a0 = pv0, a1 = pv1;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        if (o < Gp) {
          a0 += __shfl_xor_sync(kFull, a0, o);
          a1 += __shfl_xor_sync(kFull, a1, o);
        }
      }
      if (pout) {
        pout[0] = a0;
        pout[1] = a1;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    const bool free_ok = __shfl_sync(kFull, mma_ok, 0);
    tc_fence_after();
    if (free_ok) tmem_dealloc<kAccBufs * 128>(tmem);
  }
}

// ------------------------------------------------------------ bucketing

// Buckets are chunk-major, (query chunk, b * Hkv + kv, level-2 node p), so that the buckets
// and tiles of a run of query chunks are contiguous.

// Entries of query positions [t0, t0 + span) of (b, kv) = blockIdx.y, entry
// e = ((b * Hkv + kv) * N + t) * K + slot.  Each thread takes kScatterItems entries
// a block apart and issues all their loads before any store, so that the dependent
// round trips (survivor, then its bucket's offset) of several entries overlap.
// (Every index fits in 32 bits: the entry point rejects B * Hkv * N * K >= 2^31 - 2^20,
// which leaves room for the last block's threads past the end, and bucket counts >= 2^31.)
constexpr int kScatterThreads = 256, kScatterItems = 4;
__global__ void __launch_bounds__(kScatterThreads) leaf_scatter_kernel(
    const int32_t* __restrict__ surv, int t0, int span, int K, int N, int BH, int chunk_shift, int M2,
    const int* __restrict__ bucket_off, const int32_t* __restrict__ srank, uint32_t* __restrict__ list) {
  const int bh = blockIdx.y;
  const int nE = span * K;
  const int x0 = blockIdx.x * (kScatterThreads * kScatterItems) + threadIdx.x;
  int p[kScatterItems], r[kScatterItems], t[kScatterItems], slot[kScatterItems];
#pragma unroll
  for (int u = 0; u < kScatterItems; ++u) {
    const int x = x0 + u * kScatterThreads;
    const unsigned jt = (unsigned)x / (unsigned)K;
    slot[u] = x - (int)jt * K;
    t[u] = t0 + (int)jt;
    p[u] = -1;
    r[u] = 0;
    if (x < nE) {
      const int e = (bh * N + t[u]) * K + slot[u];
      p[u] = surv[e];
      r[u] = srank[e];
    }
  }
  int pos[kScatterItems];
#pragma unroll
  for (int u = 0; u < kScatterItems; ++u)
    pos[u] = p[u] >= 0 ? bucket_off[((t[u] >> chunk_shift) * BH + bh) * M2 + p[u]] + r[u] : -1;
#pragma unroll
  for (int u = 0; u < kScatterItems; ++u)
    if (p[u] >= 0 && PISA_IN_BOUNDS(pos[u] >= 0 && pos[u] < BH * N * K))
      list[pos[u]] = ((uint32_t)t[u] << 5) | (uint32_t)slot[u];
}

// Exclusive scans of the bucket sizes (entries) and of their tile counts
// ceil(size / R) over buckets [0, nb) of the pointers given, continuing from the
// offsets already at bucket_off[0] / tile_off[0] (zero when `first`), in two
// passes over tiles of kScanTile buckets, one CTA of 1024 threads per tile, each
// thread kScanItems consecutive buckets (coalesced): the tiles' sums, then each
// tile's scan from the carry-in plus the sums of the tiles before it.  part[0..1]
// holds the carry-in, part[2 + 2x .. 3 + 2x] the sums of tile x.
constexpr int kScanItems = 4;
constexpr int kScanTile = 1024 * kScanItems;

// Block-wide sum of two values (every thread gets both).
__device__ __forceinline__ int2 block_sum2(int a, int b, int2* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(kFull, a, o);
    b += __shfl_xor_sync(kFull, b, o);
  }
  if (lane == 0) sh[warp] = make_int2(a, b);
  __syncthreads();
  int2 v = lane < (int)(blockDim.x >> 5) ? sh[lane] : make_int2(0, 0);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(kFull, v.x, o);
    v.y += __shfl_xor_sync(kFull, v.y, o);
  }
  __syncthreads();
  return v;
}

__global__ void __launch_bounds__(1024) leaf_scan_sums_kernel(const int* __restrict__ count, int nb, int R, int first,
                                                               const int* __restrict__ bucket_off,
                                                               const int* __restrict__ tile_off, int* __restrict__ part) {
  __shared__ int2 sh[32];
  const int lgR = __ffs(R) - 1;  // R = 128 / max(G, 8) is a power of two
  const int i = blockIdx.x * kScanTile + kScanItems * threadIdx.x;
  int se = 0, st = 0;
#pragma unroll
  for (int q = 0; q < kScanItems; ++q) {
    const int c = i + q < nb ? count[i + q] : 0;
    se += c;
    st += (c + R - 1) >> lgR;
  }
  const int2 tot = block_sum2(se, st, sh);
  if (threadIdx.x == 0) {
    part[2 + 2 * blockIdx.x] = tot.x;
    part[3 + 2 * blockIdx.x] = tot.y;
    if (blockIdx.x == 0) {
      part[0] = first ? 0 : bucket_off[0];
      part[1] = first ? 0 : tile_off[0];
    }
  }
}

__global__ void __launch_bounds__(1024) leaf_scan_kernel(const int* __restrict__ count, int nb, int R,
                                                          const int* __restrict__ part, int* __restrict__ bucket_off,
                                                          int* __restrict__ tile_off) {
  __shared__ int2 sh[32];
  __shared__ int we[32], wt[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lgR = __ffs(R) - 1;
  // carry-in of this tile: the stage's carry plus the sums of the tiles before it
  int pe = 0, pt = 0;
  for (int y = tid; y < (int)blockIdx.x; y += blockDim.x) {
    pe += part[2 + 2 * y];
    pt += part[3 + 2 * y];
  }
  const int2 carry = block_sum2(pe, pt, sh);
  const int i = blockIdx.x * kScanTile + kScanItems * tid;
  int c[kScanItems];
  int se = 0, st = 0;
#pragma unroll
  for (int q = 0; q < kScanItems; ++q) {
    c[q] = i + q < nb ? count[i + q] : 0;
    se += c[q];
    st += (c[q] + R - 1) >> lgR;
  }
  int ie = se, it = st;  // inclusive scan over the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ve = __shfl_up_sync(kFull, ie, o), vt = __shfl_up_sync(kFull, it, o);
    if (lane >= o) {
      ie += ve;
      it += vt;
    }
  }
  if (lane == 31) {
    we[warp] = ie;
    wt[warp] = it;
  }
  __syncthreads();
  if (warp == 0) {  // scan of the 32 warp totals
    int xe = we[lane], xt = wt[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ve = __shfl_up_sync(kFull, xe, o), vt = __shfl_up_sync(kFull, xt, o);
      if (lane >= o) {
        xe += ve;
        xt += vt;
      }
    }
    we[lane] = xe;
    wt[lane] = xt;
  }
  __syncthreads();
  int oe = part[0] + carry.x + (warp ? we[warp - 1] : 0) + ie - se;
  int ot = part[1] + carry.y + (warp ? wt[warp - 1] : 0) + it - st;
#pragma unroll
  for (int q = 0; q < kScanItems; ++q) {
    if (i + q < nb) {
      bucket_off[i + q] = oe;
      tile_off[i + q] = ot;
    }
    oe += c[q];
    ot += (c[q] + R - 1) >> lgR;
  }
  if (blockIdx.x == gridDim.x - 1 && tid == 0) {
    bucket_off[nb] = part[0] + carry.x + we[31];
    tile_off[nb] = part[1] + carry.y + wt[31];
  }
}

// Descriptor of leaf tile i among the tiles of buckets [b0, b1): its bucket is the
// largest one whose first tile is <= i; {first entry, rows, level-2 survivor p,
// b * Hkv + kv}.  Each thread takes kDescItems tiles a block apart and runs their
// binary searches side by side (a fixed number of halvings each), so that the
// searches' dependent loads overlap.
constexpr int kDescThreads = 256, kDescItems = 4;
__global__ void __launch_bounds__(kDescThreads) leaf_tile_desc_kernel(
    const int* __restrict__ tile_off, const int* __restrict__ bucket_off, int b0, int b1, long long max_tiles, int R,
    int M2, int BH, int4* __restrict__ desc) {
  const int first = __ldg(tile_off + b0);
  const int end = min((long long)__ldg(tile_off + b1), first + max_tiles);
  const int i0 = first + blockIdx.x * (kDescThreads * kDescItems) + threadIdx.x;
  // lo = the largest bucket b in [b0, b1) with tile_off[b] <= tile: the answer stays in
  // [lo, lo + len) (tile_off[b0] <= tile), and len - half >= half keeps it there
  int lo[kDescItems];
#pragma unroll
  for (int u = 0; u < kDescItems; ++u) lo[u] = b0;
  for (int len = b1 - b0; len > 1;) {
    const int half = len >> 1;
#pragma unroll
    for (int u = 0; u < kDescItems; ++u)
      if (__ldg(tile_off + lo[u] + half) <= i0 + u * kDescThreads) lo[u] += half;
    len -= half;
  }
#pragma unroll
  for (int u = 0; u < kDescItems; ++u) {
    const int i = i0 + u * kDescThreads;
    if (i >= end) break;
    const int bkt = lo[u];
    const int e0 = __ldg(bucket_off + bkt) + (i - __ldg(tile_off + bkt)) * R;
    const int nrows = min(R, __ldg(bucket_off + bkt + 1) - e0);
    desc[i] = make_int4(e0, nrows, bkt % M2, (bkt / M2) % BH);
  }
}

// Final Top-K per (b, kv, t) over the leaf candidates (children of the level-2
// survivors, ascending); ineligible children carry -inf and are skipped.
// The same for K = 8: eight lanes per (b, kv, t), four rows per warp, (b, kv) =
// blockIdx.y.  Lane l of a row's group holds survivor slot l and its two leaves,
// candidates 2 l and 2 l + 1 (the second absent when its score is -inf); a slot
// counts only if no slot before it is empty (survivors are ascending with -1 padding
// at the end).  Each lane ranks its two candidates against the row's sixteen by
// shuffles inside its group (j beats i when its score is higher, or equal with j
// before i, the generic kernel's rule); the kept ones are written in candidate order.
constexpr int kFinal8Threads = 256, kFinal8Items = 4;  // rows per 8-lane group, a block apart
constexpr int kFinal8Rows = kFinal8Threads / 8 * kFinal8Items;  // rows per block
__global__ void __launch_bounds__(kFinal8Threads) leaf_final8_kernel(
    const int32_t* __restrict__ surv, const float* __restrict__ leaf_scores, int t0, int span, int N,
    int32_t* __restrict__ idx, float* __restrict__ scores) {
  constexpr int K = 8, kRowsPerBlock = kFinal8Threads / 8;
  const int lane = threadIdx.x & 31, sl = lane & 7, gbase = lane & ~7;
  const int row0 = blockIdx.x * (kRowsPerBlock * kFinal8Items) + (threadIdx.x >> 3);
  const long long job0 = (long long)blockIdx.y * N + t0;
  // every row's loads first, then the rows one by one (rows past the end still take
  // part in the shuffles)
  int p[kFinal8Items];
  float2 s2[kFinal8Items];
#pragma unroll
  for (int u = 0; u < kFinal8Items; ++u) {
    const int jt = row0 + u * kRowsPerBlock;
    p[u] = -1;
    s2[u] = make_float2(-INFINITY, -INFINITY);
    if (jt < span) {
      p[u] = __ldg(surv + (job0 + jt) * K + sl);
      s2[u] = __ldg(reinterpret_cast<const float2*>(leaf_scores + (job0 + jt) * 2 * K) + sl);
    }
  }
  const unsigned below = (1u << sl) - 1u;
#pragma unroll
  for (int u = 0; u < kFinal8Items; ++u) {
    const int jt = row0 + u * kRowsPerBlock;
    const unsigned dead = (__ballot_sync(kFull, p[u] < 0) >> gbase) & 0xFFu;
    const bool va = (dead & (below | (1u << sl))) == 0u;  // no empty slot up to this one
    const bool vb = va && s2[u].y != -INFINITY;
    const unsigned ma = (__ballot_sync(kFull, va) >> gbase) & 0xFFu;
    const unsigned mb = (__ballot_sync(kFull, vb) >> gbase) & 0xFFu;
    const int nC = __popc(ma) + __popc(mb);
    // absent candidates become NaN, which compares false with everything
    const float sa = va ? s2[u].x : __int_as_float(0x7fc00000), sb = vb ? s2[u].y : __int_as_float(0x7fc00000);
    int ra = 0, rb = 0;
#pragma unroll
    for (int o = 0; o < 8; ++o) {
      const float ya = __shfl_sync(kFull, sa, gbase | o), yb = __shfl_sync(kFull, sb, gbase | o);
      // candidates 2 o and 2 o + 1 against this lane's 2 sl and 2 sl + 1
      ra += (ya > sa) || (ya == sa && o < sl);
      ra += (yb > sa) || (yb == sa && o < sl);
      rb += (ya > sb) || (ya == sb && o <= sl);
      rb += (yb > sb) || (yb == sb && o < sl);
    }
    const bool ka = va && (nC <= K || ra < K), kb = vb && (nC <= K || rb < K);
    const unsigned kam = (__ballot_sync(kFull, ka) >> gbase) & 0xFFu;
    const unsigned kbm = (__ballot_sync(kFull, kb) >> gbase) & 0xFFu;
    if (jt < span) {
      const int oa = __popc(kam & below) + __popc(kbm & below);
      const int nOut = __popc(kam) + __popc(kbm);
      int32_t* io = idx + (job0 + jt) * K;
      float* so = scores ? scores + (job0 + jt) * K : nullptr;
      if (ka && oa < K) {  // (always below K unless the scores hold NaN)
        io[oa] = 2 * p[u];
        if (so) so[oa] = sa;
      }
      if (kb && oa + ka < K) {
        io[oa + ka] = 2 * p[u] + 1;
        if (so) so[oa + ka] = sb;
      }
      if (sl >= nOut) {
        io[sl] = -1;
        if (so) so[sl] = -INFINITY;
      }
    }
  }
}

// Final Top-K of the leaf stage for any K <= 32: one warp per (b, kv, t), (b, kv) =
// blockIdx.y.  Lane l holds survivor slot l and its two leaves (the second absent when
// its score is -inf: past the query or past the last token); the candidates' order is
// the walk's (node order).  Each candidate's 64-bit key, the order-preserving bits of
// its score above the complement of its position, goes to shared memory in that order:
// j beats i exactly when key j > key i (a higher score, or an equal one with j before
// i), so a lane ranks its two candidates by one unsigned compare per candidate, and the
// kept ones are written in candidate order, then -1 / -inf padding.
constexpr int kFinalWarps = 4;
__device__ __forceinline__ unsigned long long final_key(float s, int pos) {
  const unsigned b = __float_as_uint(s + 0.f);  // (-0 becomes +0: the two compare equal)
  const unsigned ord = b ^ ((unsigned)((int)b >> 31) | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned)(0xFFFFFFFFu - (unsigned)pos);
}
__global__ void __launch_bounds__(kFinalWarps * 32) leaf_final_kernel(
    const int32_t* __restrict__ surv, const float* __restrict__ leaf_scores, int t0, int span, int N, int K,
    int32_t* __restrict__ idx, float* __restrict__ scores) {
  __shared__ unsigned long long sh[kFinalWarps][2 * kMaxK];
  const int lane = threadIdx.x & 31, wb = threadIdx.x >> 5;
  const int jt = blockIdx.x * kFinalWarps + wb;
  if (jt >= span) return;  // warp-uniform
  const long long job = (long long)blockIdx.y * N + t0 + jt;
  const int p = lane < K ? __ldg(surv + job * K + lane) : -1;
  const bool va = p >= 0;
  const float2 s2 = va ? __ldg(reinterpret_cast<const float2*>(leaf_scores + job * 2 * K) + lane)
                       : make_float2(-INFINITY, -INFINITY);
  const float sa = s2.x, sb = s2.y;
  const bool vb = va && sb != -INFINITY;
  const unsigned lt = (1u << lane) - 1u;
  const unsigned ma = __ballot_sync(kFull, va), mb = __ballot_sync(kFull, vb);
  const int pa = __popc(ma & lt) + __popc(mb & lt);  // position of this lane's first leaf
  const int nC = __popc(ma) + __popc(mb);
  bool ka = va, kb = vb;
  if (nC > K) {  // warp-uniform
    unsigned long long* sw = sh[wb];
    const unsigned long long kA = final_key(sa, pa), kB = final_key(sb, pa + 1);
    if (va) sw[pa] = kA;
    if (vb) sw[pa + 1] = kB;
    __syncwarp();
    int ra = 0, rb = 0;
#pragma unroll 4
    for (int j = 0; j < nC; ++j) {
      const unsigned long long y = sw[j];
      ra += y > kA;
      rb += y > kB;
    }
    ka = va && ra < K;
    kb = vb && rb < K;
  }
  const unsigned ka_m = __ballot_sync(kFull, ka), kb_m = __ballot_sync(kFull, kb);
  const int oa = __popc(ka_m & lt) + __popc(kb_m & lt);
  const int nOut = __popc(ka_m) + __popc(kb_m);
  int32_t* io = idx + job * K;
  float* so = scores ? scores + job * K : nullptr;
  if (ka && PISA_IN_BOUNDS(oa < K)) {
    io[oa] = 2 * p;
    if (so) so[oa] = sa;
  }
  if (kb && PISA_IN_BOUNDS(oa + (ka ? 1 : 0) < K)) {
    io[oa + (ka ? 1 : 0)] = 2 * p + 1;
    if (so) so[oa + (ka ? 1 : 0)] = sb;
  }
  for (int w = nOut + lane; w < K; w += 32) {
    io[w] = -1;
    if (so) so[w] = -INFINITY;
  }
}

// ------------------------------------------------------------ host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 map over [rows][heads][64] with a box of {64, box_h, box_rows}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, long long rows, int heads, int box_h, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {128, (cuuint64_t)heads * 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_h, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int n[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 148;
  }
  return n[dev];
}

}  // namespace

// The persistent leaf kernel over the tiles described by L.tile_desc (their count is
// L.tile_off[L.nb]); flat != 0 selects the flat output layout.
cudaError_t launch_leaf_tc_kernel(const LeafTcLaunch& L, int flat, long long flat_stride, cudaStream_t s) {
  PISA_SET_BOUNDS_STATUS(L.status, s);  // (the flat selector comes here directly)
  const int G = L.Hq / L.Hkv;
  const int Gp = G < 8 ? 8 : G;
  const int R = 128 / Gp;
  CUtensorMap qmap, kmap;
  if (!make_map(&qmap, L.Q, (long long)L.B * L.N, L.Hq, G, 1) ||
      !make_map(&kmap, L.keys, (long long)L.B * L.n_cap, L.Hkv, 1, 128))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  std::call_once(attr_once, [] {
    cudaFuncSetAttribute(leaf_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLeafSmem);
    cudaFuncSetAttribute(leaf_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLeafSmem);
    cudaFuncSetAttribute(leaf_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLeafSmem);
  });
  LeafTcParams P;
  P.flat = flat;
  P.flat_stride = flat_stride;
  P.Q = L.Q;
  P.Hq = L.Hq;
  P.list = L.list;
  P.bucket_off = L.bucket_off;
  P.tile_off = L.tile_off;
  P.tile_desc = L.tile_desc;
  P.b0 = L.b0;
  P.b1 = L.b1;
  P.Hkv = L.Hkv;
  P.G = G;
  P.Gp = Gp;
  P.R = R;
  P.K = L.K;
  P.N = L.N;
  P.n_cap = L.n_cap;
  P.M2 = L.M2;
  P.nchunks = L.nchunks;
  P.causal = L.causal;
  P.leaf_scores = L.leaf_scores;
  P.status = L.status;
  auto kern = L.mode == 1 ? leaf_tc_kernel<1> : L.mode == 2 ? leaf_tc_kernel<2> : leaf_tc_kernel<0>;
  kern<<<sm_count(), kLeafWarps * 32, kLeafSmem, s>>>(qmap, kmap, P);
  note_launch();
  return cudaGetLastError();
}

// The leaf level of the prefill selection for query positions [L.t0, L.t1), whose
// buckets are [L.b0, L.b1) (whole query chunks, chunk-major buckets).
cudaError_t launch_prefill_leaf_tc(const LeafTcLaunch& L, cudaStream_t s) {
  if (L.t1 <= L.t0) return cudaSuccess;
  PISA_SET_BOUNDS_STATUS(L.status, s);
  const int BH = L.B * L.Hkv;
  const long long span = L.t1 - L.t0;
  const long long entries = (long long)BH * span * L.K;
  const int G = L.Hq / L.Hkv;
  const int Gp = G < 8 ? 8 : G;
  const int R = 128 / Gp;
  // bucket sizes were counted by the walk kernel as it wrote the survivors
  const int nbs = L.b1 - L.b0;
  const unsigned tiles = (unsigned)((nbs + kScanTile - 1) / kScanTile);
  if (tiles > 0) {
    leaf_scan_sums_kernel<<<tiles, 1024, 0, s>>>(L.count + L.b0, nbs, R, L.b0 == 0, L.bucket_off + L.b0,
                                                 L.tile_off + L.b0, L.scan_part);
    note_launch();
    leaf_scan_kernel<<<tiles, 1024, 0, s>>>(L.count + L.b0, nbs, R, L.scan_part, L.bucket_off + L.b0,
                                            L.tile_off + L.b0);
    note_launch();
  }
  constexpr int kScatterSpan = kScatterThreads * kScatterItems;
  leaf_scatter_kernel<<<dim3((unsigned)((span * L.K + kScatterSpan - 1) / kScatterSpan), BH), kScatterThreads, 0, s>>>(
      L.surv, (int)L.t0, (int)span, L.K, (int)L.N, BH, L.chunk_shift, L.M2, L.bucket_off, L.srank, L.list);
  note_launch();
  // a tile holds R >= 8 entries of one bucket: at most entries / 8 + (buckets) tiles
  const long long max_tiles = entries / 8 + (L.b1 - L.b0) + 1;
  constexpr int kDescSpan = kDescThreads * kDescItems;
  leaf_tile_desc_kernel<<<(unsigned)((max_tiles + kDescSpan - 1) / kDescSpan), kDescThreads, 0, s>>>(
      L.tile_off, L.bucket_off, L.b0, L.b1, max_tiles, R, L.M2, BH, L.tile_desc);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mark_phase(3, s);

  e = launch_leaf_tc_kernel(L, 0, 0, s);
  if (e != cudaSuccess) return e;
  mark_phase(4, s);
  if (L.K == 8)
    leaf_final8_kernel<<<dim3((unsigned)((span + kFinal8Rows - 1) / kFinal8Rows), BH), kFinal8Threads, 0, s>>>(
        L.surv, L.leaf_scores, (int)L.t0, (int)span, (int)L.N, L.idx, L.scores);
  else
    leaf_final_kernel<<<dim3((unsigned)((span + kFinalWarps - 1) / kFinalWarps), BH), kFinalWarps * 32, 0, s>>>(
        L.surv, L.leaf_scores, (int)L.t0, (int)span, (int)L.N, L.K, L.idx, L.scores);
  note_launch();
  e = cudaGetLastError();
  mark_phase(5, s);
  return e;
}

}  // namespace pisa
