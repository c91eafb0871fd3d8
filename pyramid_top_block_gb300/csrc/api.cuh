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
                                 cudaStream_t s);

cudaError_t launch_prefill_warp(const __nv_bfloat16* Q, const float* summ, const __nv_bfloat16* keys,
                                const Levels& lv, long long N, long long n_cap, int B, int Hq,
                                int Hkv, int K, int causal, int32_t* surv, int32_t* idx,
                                float* scores, cudaStream_t s);

cudaError_t launch_decode_warp(const __nv_bfloat16* q_new, const __nv_bfloat16* k_new,
                               __nv_bfloat16* keys, float* summ, int32_t* lengths,
                               const Levels& cap_lv, long long n_cap, int B, int Hq, int Hkv, int K,
                               int32_t* idx, float* scores, int* status, cudaStream_t s);

}  // namespace pisa
