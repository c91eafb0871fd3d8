// noalloc.cu -- pisa_select_prefill_noalloc: the prefill selection for callers
// that cannot allocate device memory.
//
// Some callers never get to call cudaMalloc: a host framework that owns all
// device memory and hands a plugin only its input and output buffers, or a
// request path where an allocation is not allowed because it can synchronise
// the device or fail halfway through a request.  This entry point needs no
// workspace argument.  Its scratch is the file-scope device array below, of
// fixed size PISA_NOALLOC_SCRATCH_BYTES; every GPU that loads this library
// holds that array until the process exits.
//
// The array is shared by every call in the process.  It keeps whatever the
// last call left in it; the selection clears the parts that must start at zero
// (its status word) on each call, and the rest is overwritten before it is
// read.  Calls that overlap on the GPU (on different streams, or from several
// host threads without ordering) race on the array and give wrong results:
// order them on one stream.
//
// With CUDA's lazy module loading (the default) the array comes into being
// when this file's device code is first loaded on a device, which the first
// address lookup triggers: that moment may allocate device memory and
// synchronise.  pisa_noalloc_prepare() does the lookup up front.
#include <mutex>

#include "api.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PISA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PISA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PISA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PISA_OK;
}

}  // namespace

extern "C" int pisa_select_prefill_noalloc(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K,
                                           int causal, int32_t* idx, float* scores, void* stream) {
  // the same checks, in the same order, as pisa_select_prefill; then the size limit
  const int chk = pisa::prefill_check_args(Q, Hq, pyr, N, K, 0, idx);
  if (chk != PISA_OK) return chk;
  const size_t need = pisa_select_workspace_bytes(pyr->B, N, Hq, pyr->Hkv, K);
  if (need > (size_t)PISA_NOALLOC_SCRATCH_BYTES) return PISA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  const int st = scratch_address(&ws);
  if (st != PISA_OK) return st;
  return pisa_select_prefill(Q, Hq, pyr, N, K, causal, idx, scores, ws, (size_t)PISA_NOALLOC_SCRATCH_BYTES,
                             stream);
}

extern "C" int pisa_noalloc_prepare(void** scratch) {
  void* ws = nullptr;
  const int st = scratch_address(&ws);
  if (st == PISA_OK && scratch) *scratch = ws;
  return st;
}

extern "C" int pisa_noalloc_device_status(void* stream) {
  void* ws = nullptr;
  const int st = scratch_address(&ws);
  if (st != PISA_OK) return st;
  return pisa_check_device_status(ws, stream);
}
