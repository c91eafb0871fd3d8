// api.cuh -- host-side launchers shared between the C ABI layer and kernels.
#pragma once

#include "common.cuh"

namespace pisa {

// Counts kernels this library launched (a profiling aid, not synchronised with
// the device).  Every launcher calls note_launch() once per <<<>>> launch.
void note_launch(int n = 1);

// Records the caller's profiling event for phase boundary `i` of the current
// select call on stream s, if the caller attached events (no-op otherwise).
void mark_phase(int i, cudaStream_t s);

cudaError_t launch_build_pyramid(const __nv_bfloat16* keys, float* summ, const Levels& lv,
                                 long long N, long long n_cap, int B, int Hkv, int32_t* lengths,
                                 cudaStream_t s, bool ragged = false);

// Everything the leaf level of the prefill walk needs (buffers are caller
// workspace slices; see pisa_api.cu for the layout).
struct LeafTcLaunch {
  const __nv_bfloat16* Q;
  const __nv_bfloat16* keys;
  int B, Hq, Hkv, K, causal;
  long long N, n_cap;
  int M2, nchunks, chunk_shift, nb;
  long long t0, t1;  // query positions of this launch: whole query chunks (or up to N)
  int b0, b1;        // their buckets
  const int32_t* surv;
  int* count;
  const int32_t* srank;  // rank of each survivor inside its bucket (from the walk)
  int* bucket_off;
  int* tile_off;
  int* scan_part;  // 2 + 2 * ceil(buckets / 4096) ints of scan scratch
  int4* tile_desc;      // [max_tiles] {first entry, rows, level-2 survivor p, b * Hkv + kv}
  long long max_tiles;  // upper bound on the number of tiles
  uint32_t* list;
  float* leaf_scores;
  int32_t* idx;
  float* scores;
  int* status;
  int mode;  // leaf score: 0 LSE over the keys, 1 mean logit, 2 mean + variance / 2
};

cudaError_t launch_prefill_leaf_tc(const LeafTcLaunch& L, cudaStream_t s);
cudaError_t launch_leaf_tc_kernel(const LeafTcLaunch& L, int flat, long long flat_stride, cudaStream_t s);

// The flat selector (flat.cu): L.list, L.tile_desc and L.leaf_scores are its
// workspace slices; T1 tiles per (b, kv); stride = floats per (b, kv, t) score row.
cudaError_t launch_select_flat(const LeafTcLaunch& L, long long T1, long long stride, int* total, cudaStream_t s);
long long flat_tiles_per_bh(long long N, int G, int K, bool causal);

// Stage-two block-sparse attention (attend.cu).
cudaError_t launch_sparse_attention(const __nv_bfloat16* Q, const __nv_bfloat16* K, const __nv_bfloat16* V,
                                    const int32_t* idx, int B, long long N, int Hq, int Hkv, int Ksel, int causal,
                                    float* out, cudaStream_t s);

// The intermediate levels of the prefill walk (walk_mma.cu).
struct WalkLaunch {
  const __nv_bfloat16* Q;
  const float* summ;
  const Levels* lv;
  long long N;
  int B, Hq, Hkv, K, causal;
  unsigned char* table;  // route table: B*Hkv*route_rows_per_bh(lv) rows of 256 bytes
  int32_t* surv;
  int32_t* srank;  // rank of each survivor inside its bucket (the bucket count before it)
  int* count;
  int nchunks, chunk_shift, M2;  // buckets are chunk-major: ((t >> chunk_shift) * B * Hkv + b * Hkv + kv) * M2 + p
  int mode;  // block score: 0 LSE, 1 mean of the child logits, 2 mean + variance / 2
  long long t0, t1;  // the query positions walked by this launch
  bool build_table;  // build the route table first (once per pyramid state)
  int* status;       // the call's status word (debug builds record failed index checks there)
};

long long route_rows_per_bh(const Levels& lv);
// Every argument check of a prefill selection except the workspace's (the status
// pisa_select_prefill would return for these arguments with a large enough workspace).
int prefill_check_args(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int mode, const void* idx);
cudaError_t launch_selftest_wait(int* status, long long delay_cycles, cudaStream_t s);
cudaError_t launch_prefill_walk_mma(const WalkLaunch& W, cudaStream_t s);

cudaError_t launch_decode_warp(const __nv_bfloat16* q_new, const __nv_bfloat16* k_new,
                               __nv_bfloat16* keys, float* summ, int32_t* lengths,
                               const Levels& cap_lv, long long n_cap, int B, int Hq, int Hkv, int K,
                               int32_t* idx, float* scores, int* status, int* arrivals, cudaStream_t s);

}  // namespace pisa
