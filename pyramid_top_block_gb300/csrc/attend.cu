// attend.cu -- stage two of block-sparse attention: each query attends over the
// original keys and values inside its selected blocks ("Block Sparse Attention
// with Log-Linear Complexity", Background: two stages), one softmax over all of
// them, keys after the query masked when causal.
//
// One warp per (b, t, kv): the group's G <= 16 query heads are the 16 rows of
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate).  The selected leaves are taken in
// blocks of 32 keys; each block's key and value rows (8 KB) are copied with
// cp.async into one of two shared-memory buffers (16-byte-chunk XOR swizzle) while
// the previous block is computed: S = Q K^T (ldmatrix), a running row max and sum
// in base 2 (online softmax), O += P V (P packed to bf16 straight from the S
// fragments, V through ldmatrix.trans).  Each (query, KV head) gathers its own
// leaves' rows, so the kernel is bound by the L2 gathers (16 KB per selected leaf).
#include <mutex>

#include "api.cuh"

namespace pisa {

constexpr int kAttWarps = 4;
constexpr int kAttStage = 2 * kC * kD * 2;  // two buffers of 32 key and 32 value rows, bf16: 16 KB per warp

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Byte offset of 16-byte chunk ch (0..7) of row r in a staged 64 x 128-byte matrix.
__device__ __forceinline__ uint32_t swz(int r, int ch) { return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)); }


__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  // 16-byte copy into shared memory; a false predicate copies nothing and zero-fills
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(pred ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One warp per (b, kv, t), grid-stride over all of them.  The selected leaves are
// walked in blocks of 32 keys (two per leaf); each block's key and value rows (8 KB)
// are copied into one of two shared-memory buffers with cp.async while the previous
// block is being computed.
__global__ void __launch_bounds__(kAttWarps * 32) sparse_attention_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Kc, const __nv_bfloat16* __restrict__ V,
    const int32_t* __restrict__ idx, int B, long long N, int Hq, int Hkv, int Ksel, int causal,
    float* __restrict__ out) {
  extern __shared__ __align__(128) unsigned char att_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, j = lane & 3;
  const int G = Hq / Hkv;
  unsigned char* st = att_smem + warp * kAttStage;  // two buffers of [K 32 rows][V 32 rows]
  const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(st);
  const float c2 = kScale * 1.4426950408889634f;  // logits in base 2
  const long long jobs = (long long)B * Hkv * N;
  for (long long job = (long long)blockIdx.x * kAttWarps + warp; job < jobs; job += (long long)gridDim.x * kAttWarps) {
    const long long t = job % N, bh = job / N;
    const int kv = (int)(bh % Hkv);
    const long long b = bh / Hkv;
    const long long n_eff = causal ? t + 1 : N;
    const int32_t* sel = idx + job * Ksel;
    // the blocks of 32 keys that count: leaf sel[i] contributes blocks 2 i and 2 i + 1
    // when they start before n_eff (a bit per block; at most 2 kMaxK blocks)
    unsigned long long blocks = 0;
    for (int i = lane; i < Ksel; i += 32) {
      const int leaf = __ldg(sel + i);
      const long long r0 = (long long)leaf * kC;
      if (leaf >= 0 && r0 < n_eff) {
        blocks |= 1ull << (2 * i);
        if (r0 + 32 < n_eff) blocks |= 1ull << (2 * i + 1);
      }
    }
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) blocks |= __shfl_xor_sync(kFull, blocks, x);
    auto row0_of = [&](int blk) -> long long { return (long long)__ldg(sel + (blk >> 1)) * kC + 32 * (blk & 1); };
    // copy block blk into buffer buf: 32 key rows and 32 value rows, 8 chunks of 16 bytes each
    auto issue = [&](int blk, int buf) {
      const long long r0 = row0_of(blk);
      const uint32_t dK = s0 + buf * (kAttStage / 2), dV = dK + 32 * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = lane + 32 * u;
        const int r = e >> 3, ch = e & 7;
        const bool in = r0 + r < N;
        const long long off = ((b * N + (in ? r0 + r : 0)) * Hkv + kv) * kD + ch * 8;
        cp_async16(dK + swz(r, ch), Kc + off, in);
        cp_async16(dV + swz(r, ch), V + off, in);
      }
      cp_async_commit();
    };
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(Q + ((b * N + t) * Hq + (long long)kv * G) * kD);
    uint32_t qa[4][4];  // A fragments: rows = heads g, g + 8; heads >= G are zero
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const int w0 = 8 * ks + j;
      qa[ks][0] = g < G ? __ldg(q0 + g * 32 + w0) : 0u;
      qa[ks][1] = g + 8 < G ? __ldg(q0 + (g + 8) * 32 + w0) : 0u;
      qa[ks][2] = g < G ? __ldg(q0 + g * 32 + w0 + 4) : 0u;
      qa[ks][3] = g + 8 < G ? __ldg(q0 + (g + 8) * 32 + w0 + 4) : 0u;
    }
    float o[8][4];
#pragma unroll
    for (int dn = 0; dn < 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows g and g + 8
    __syncwarp();  // the previous job's shared-memory reads are done
    int cur = blocks ? __ffsll((long long)blocks) - 1 : -1;
    if (cur >= 0) issue(cur, 0);
    int buf = 0;
    while (cur >= 0) {
      const unsigned long long rest = blocks & ~((2ull << cur) - 1ull);
      const int nxt = rest ? __ffsll((long long)rest) - 1 : -1;
      if (nxt >= 0) {
        issue(nxt, buf ^ 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncwarp();
      const uint32_t sK = s0 + buf * (kAttStage / 2), sV = sK + 32 * 128;
      const long long r0 = row0_of(cur);
      const int nv = (int)(n_eff - r0 < 32 ? n_eff - r0 : 32);  // keys of the block that count
      float sacc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
        for (int kp = 0; kp < 2; ++kp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sK + swz(8 * nt + (lane & 7), 4 * kp + (lane >> 3)), b0, b1, b2, b3);
          mma16816(sacc[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
          mma16816(sacc[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2], qa[2 * kp + 1][3], b2, b3);
        }
      }
      // online softmax in base 2: masked keys are -inf, the row maxima are quad-reduced
      float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = 8 * nt + 2 * j + (e & 1);
          const float v = col < nv ? sacc[nt][e] * c2 : -INFINITY;
          sacc[nt][e] = v;
          if (e < 2)
            bm0 = fmaxf(bm0, v);
          else
            bm1 = fmaxf(bm1, v);
        }
#pragma unroll
      for (int x = 1; x < 4; x <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, x));
        bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, x));
      }
      const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
      const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int dn = 0; dn < 8; ++dn) {
        o[dn][0] *= al0;
        o[dn][1] *= al0;
        o[dn][2] *= al1;
        o[dn][3] *= al1;
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sacc[nt][0] = exp2f(sacc[nt][0] - mn0);
        sacc[nt][1] = exp2f(sacc[nt][1] - mn0);
        sacc[nt][2] = exp2f(sacc[nt][2] - mn1);
        sacc[nt][3] = exp2f(sacc[nt][3] - mn1);
        l0 += sacc[nt][0] + sacc[nt][1];
        l1 += sacc[nt][2] + sacc[nt][3];
      }
      // O += P V: the S fragments of keys 16 kk .. 16 kk + 15 are the A fragments
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t a0 = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
        const uint32_t a1 = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
        const uint32_t a2 = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        const uint32_t a3 = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < 4; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sV + swz(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * dp + (lane >> 4)), b0, b1, b2, b3);
          mma16816(o[2 * dp], a0, a1, a2, a3, b0, b1);
          mma16816(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      __syncwarp();  // the buffer's reads are done before it is refilled
      cur = nxt;
      buf ^= 1;
    }
#pragma unroll
    for (int x = 1; x < 4; x <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, x);
      l1 += __shfl_xor_sync(kFull, l1, x);
    }
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
    float* ob = out + ((b * N + t) * Hq + (long long)kv * G) * kD;
#pragma unroll
    for (int dn = 0; dn < 8; ++dn) {
      if (g < G)
        *reinterpret_cast<float2*>(ob + g * kD + 8 * dn + 2 * j) = make_float2(o[dn][0] * i0, o[dn][1] * i0);
      if (g + 8 < G)
        *reinterpret_cast<float2*>(ob + (g + 8) * kD + 8 * dn + 2 * j) = make_float2(o[dn][2] * i1, o[dn][3] * i1);
    }
  }
}

cudaError_t launch_sparse_attention(const __nv_bfloat16* Q, const __nv_bfloat16* K, const __nv_bfloat16* V,
                                    const int32_t* idx, int B, long long N, int Hq, int Hkv, int Ksel, int causal,
                                    float* out, cudaStream_t s) {
  const size_t smem = (size_t)kAttWarps * kAttStage;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [smem] {
    attr_err = cudaFuncSetAttribute(sparse_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const long long jobs = (long long)B * Hkv * N;
  long long blocks = (jobs + kAttWarps - 1) / kAttWarps;
  if (blocks > 152LL * 24) blocks = 152LL * 24;
  sparse_attention_kernel<<<(unsigned)blocks, kAttWarps * 32, smem, s>>>(Q, K, V, idx, B, N, Hq, Hkv, Ksel, causal,
                                                                        out);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pisa
