// pisa_api.cu -- the C ABI (include/pisa.h): argument checks, workspace
// layout and launch sequencing.  No allocation, no exceptions, one stream.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include <algorithm>
#include <mutex>
#include <vector>

#include "api.cuh"

using namespace pisa;

namespace {
std::atomic<unsigned long long> g_launches{0};
cudaEvent_t g_phase_events[16];
int g_n_phase_events = 0;
}  // namespace

namespace pisa {
void note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
void mark_phase(int i, cudaStream_t s) {
  if (i >= 0 && i < g_n_phase_events && g_phase_events[i]) cudaEventRecord(g_phase_events[i], s);
}
}  // namespace pisa

namespace {

constexpr size_t kAlign = 256;
constexpr int kPrefillPhases = 5;
constexpr size_t kStatusBytes = 256;  // status word + reserved counters

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool pow2_group(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16; }

// Level geometry for a sequence of n tokens stored in a layout for n_cap.
Levels make_levels(long long n, long long n_cap) {
  Levels lv;
  std::memset(&lv, 0, sizeof(lv));
  lv.L = num_levels_for(n);
  const int Lcap = num_levels_for(n_cap);
  lv.M[0] = (int)n;
  long long off = 0;
  for (int l = 1; l <= Lcap; ++l) {
    lv.off[l] = off;
    off += level_size_for(n_cap, l);
    if (l <= lv.L) lv.M[l] = (int)level_size_for(n, l);
  }
  lv.total = off;
  return lv;
}

// Largest grid y extent of a launch: the build, walk, scatter and final Top-K index
// (b, kv) or b along y.
constexpr long long kMaxGridY = 65535;
// Entries (b, kv, t, slot) a prefill call may hold: the bucketing kernels index them, and
// their blocks' threads past the end, in 32-bit integers.
constexpr long long kMaxEntries = (1LL << 31) - (1LL << 20);

// Sizes the library handles; returns PISA_OK or the status to report.
int check_geometry(int B, long long N, int Hq, int Hkv, int d, int C, int g, int K) {
  if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || d < 1 || C < 1 || g < 1 || K < 1)
    return PISA_ERR_INVALID_ARG;
  if (Hq % Hkv) return PISA_ERR_UNSUPPORTED;
  if (d != kD || C != kC || g != 2) return PISA_ERR_UNSUPPORTED;
  if (K > kMaxK || !pow2_group(Hq / Hkv) || Hkv > 32 || (long long)B * Hkv > kMaxGridY) return PISA_ERR_UNSUPPORTED;
  if (N > (1LL << 27)) return PISA_ERR_UNSUPPORTED;
  // 32-bit entry and tile indices, with headroom for a grid's last block past the end
  if ((long long)B * Hkv * N * K >= kMaxEntries || (long long)B * N >= (1LL << 31)) return PISA_ERR_UNSUPPORTED;
  return PISA_OK;
}

int check_pyr(const pisa_pyramid* p) {
  if (!p || !p->summaries || !p->keys) return PISA_ERR_INVALID_ARG;
  if (p->B < 1 || p->Hkv < 1 || p->n_cap < 1) return PISA_ERR_INVALID_ARG;
  if (p->d != kD || p->C != kC || p->g != 2 || p->Hkv > 32) return PISA_ERR_UNSUPPORTED;
  if ((long long)p->B * p->Hkv > kMaxGridY) return PISA_ERR_UNSUPPORTED;  // grids index (b, kv) along y
  if ((reinterpret_cast<uintptr_t>(p->summaries) | reinterpret_cast<uintptr_t>(p->keys)) & 15)
    return PISA_ERR_INVALID_ARG;
  return PISA_OK;
}

// Query positions per bucketing chunk: the leaf level gathers query rows of
// one chunk at a time, so 2^shift tokens x Hq x 128 B of Q stay in L2.  The
// chunk grows with N so that there are at most 64 chunks.
int chunk_shift_for(long long N) {
  int cs = 14;
  while ((N >> cs) > 64) ++cs;
  return cs;
}

// Workspace of the prefill selection (every slice 256-byte aligned):
//   [status 256 B][count nb]                  zeroed at every call
//   [bucket_off nb+1][tile_off nb+1]           scans of the bucket sizes
//   [scan_part 2 + 2 ceil(nb/4096)]            the scan's carry-in and per-tile sums
//   [tile_desc: max_tiles int4]                first entry, rows, p, b*Hkv+kv of each leaf tile
//   [surv2: B*Hkv*N*K int32]                   level-2 survivors
//   [srank: B*Hkv*N*K int32]                   rank of each survivor inside its bucket
//   [list: B*Hkv*N*K uint32]                   (t << 5 | slot), bucket-sorted
//   [leaf_scores: B*Hkv*N*2K fp32]
//   [route table: B*Hkv*rows x 256 B]          per-node logit-step rows of the walk
// with nb = B * Hkv * nchunks * M2 buckets (chunk of queries, level-2 node).
struct PrefillWs {
  size_t status, count, srank, bucket_off, tile_off, scan_part, tile_desc, surv, list, leaf, table, total, zero_bytes;
  long long max_tiles;
  long long nb;
  int nchunks, chunk_shift, M2;
};

PrefillWs prefill_layout(int B, long long N, int Hkv, int K) {
  PrefillWs w;
  w.chunk_shift = chunk_shift_for(N);
  w.nchunks = (int)((N + (1LL << w.chunk_shift) - 1) >> w.chunk_shift);
  w.M2 = (int)level_size_for(N, 2);
  w.nb = (long long)B * Hkv * w.nchunks * w.M2;
  const size_t entries = (size_t)B * Hkv * (size_t)N * K;
  size_t o = 0;
  w.status = o;
  o += align_up(kStatusBytes);
  w.count = o;
  o += sizeof(int) * (size_t)w.nb;
  w.zero_bytes = o;
  o = align_up(o);
  w.bucket_off = o;
  o += align_up(sizeof(int) * (size_t)(w.nb + 1));
  w.tile_off = o;
  o += align_up(sizeof(int) * (size_t)(w.nb + 1));
  w.scan_part = o;  // the bucket scan's carry-in and per-4096-bucket sums
  o += align_up(sizeof(int) * (size_t)(2 + 2 * ((w.nb + 4095) / 4096)));
  // a tile holds R = 128 / max(G, 8) >= 8 queries: at most entries / 8 + nb tiles
  w.max_tiles = (long long)(entries / 8) + w.nb + 1;
  w.tile_desc = o;
  o += align_up(sizeof(int4) * (size_t)w.max_tiles);
  w.surv = o;
  o += align_up(sizeof(int32_t) * entries);
  w.srank = o;
  o += align_up(sizeof(int32_t) * entries);
  w.list = o;
  o += align_up(sizeof(uint32_t) * entries);
  w.leaf = o;
  o += align_up(sizeof(float) * 2 * entries);
  w.table = o;
  o += align_up((size_t)B * Hkv * (size_t)route_rows_per_bh(make_levels(N, N)) * 256);
  w.total = o;
  return w;
}

// Workspace of the flat selector: [status 256 B][tile count 256 B][list N uint32]
// [tile_desc T int4][leaf scores B*Hkv*N*2*M2 fp32], T = B*Hkv*T1 tiles.
struct FlatWs {
  size_t status, total, list, desc, leaf, size;
  long long T1, T, stride;
};

FlatWs flat_layout(int B, long long N, int Hq, int Hkv, int K, bool causal) {
  FlatWs w;
  w.T1 = flat_tiles_per_bh(N, Hq / Hkv, K, causal);
  w.T = w.T1 * B * Hkv;
  w.stride = 2 * level_size_for(N, 2);
  size_t o = 0;
  w.status = o;
  o += align_up(kStatusBytes);
  w.total = o;
  o += align_up(sizeof(int));
  w.list = o;
  o += align_up(sizeof(uint32_t) * (size_t)N);
  w.desc = o;
  o += align_up(sizeof(int4) * (size_t)w.T);
  w.leaf = o;
  o += align_up(sizeof(float) * (size_t)B * Hkv * (size_t)N * (size_t)w.stride);
  w.size = o;
  return w;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PISA_OK : PISA_ERR_CUDA; }

}  // namespace

extern "C" {

int pisa_num_levels(int64_t n, int C, int g) {
  if (n < 1 || C != kC || g != 2) return -1;
  return num_levels_for(n);
}

int64_t pisa_pyramid_nodes(int64_t n_cap, int C, int g) {
  if (n_cap < 1 || C != kC || g != 2) return -1;
  return make_levels(n_cap, n_cap).total;
}

int64_t pisa_level_offset(int64_t n_cap, int C, int g, int level) {
  if (n_cap < 1 || C != kC || g != 2) return -1;
  const Levels lv = make_levels(n_cap, n_cap);
  if (level < 1 || level > lv.L) return -1;
  return lv.off[level];
}

int pisa_build_pyramid(const pisa_pyramid* pyr, int64_t N, void* stream) {
  int st = check_pyr(pyr);
  if (st) return st;
  if (N < 1 || N > pyr->n_cap) return PISA_ERR_INVALID_ARG;
  if (N > (1LL << 27) || pyr->n_cap > (1LL << 27)) return PISA_ERR_UNSUPPORTED;
  const Levels lv = make_levels(N, pyr->n_cap);
  return cuda_status(launch_build_pyramid(static_cast<const __nv_bfloat16*>(pyr->keys), pyr->summaries, lv,
                                          N, pyr->n_cap, pyr->B, pyr->Hkv, pyr->lengths,
                                          static_cast<cudaStream_t>(stream)));
}

int pisa_build_pyramid_ragged(const pisa_pyramid* pyr, void* stream) {
  int st = check_pyr(pyr);
  if (st) return st;
  if (!pyr->lengths) return PISA_ERR_INVALID_ARG;
  if (pyr->n_cap > (1LL << 27)) return PISA_ERR_UNSUPPORTED;
  const Levels lv = make_levels(pyr->n_cap, pyr->n_cap);
  return cuda_status(launch_build_pyramid(static_cast<const __nv_bfloat16*>(pyr->keys), pyr->summaries, lv,
                                          pyr->n_cap, pyr->n_cap, pyr->B, pyr->Hkv, pyr->lengths,
                                          static_cast<cudaStream_t>(stream), true));
}

size_t pisa_select_workspace_bytes(int B, int64_t N, int Hq, int Hkv, int K) {
  if (check_geometry(B, N, Hq, Hkv, kD, kC, 2, K) != PISA_OK) return 0;
  return prefill_layout(B, N, Hkv, K).total;
}

// The launch descriptions of one prefill selection (buffers are workspace slices);
// the query range and bucket range are set per stage.
struct PrefillPlan {
  Levels lv;
  PrefillWs w;
  WalkLaunch W;
  LeafTcLaunch L;
};

}  // extern "C"

namespace pisa {
// Every argument check of a prefill selection except the workspace's.
int prefill_check_args(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int mode, const void* idx) {
  if (mode < 0 || mode > 2) return PISA_ERR_UNSUPPORTED;
  int st = check_pyr(pyr);
  if (st) return st;
  if (!Q || !idx) return PISA_ERR_INVALID_ARG;
  st = check_geometry(pyr->B, N, Hq, pyr->Hkv, pyr->d, pyr->C, pyr->g, K);
  if (st) return st;
  if (N > pyr->n_cap) return PISA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(Q) & 15) return PISA_ERR_INVALID_ARG;
  const PrefillWs w = prefill_layout(pyr->B, N, pyr->Hkv, K);
  if (w.nb >= (1LL << 31) || (long long)pyr->B * pyr->n_cap >= (1LL << 31)) return PISA_ERR_UNSUPPORTED;
  return PISA_OK;
}
}  // namespace pisa

extern "C" {

static int prefill_check(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int mode, const void* idx,
                         const void* ws, size_t ws_bytes) {
  const int st = prefill_check_args(Q, Hq, pyr, N, K, mode, idx);
  if (st) return st;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return PISA_ERR_INVALID_ARG;
  if (ws_bytes < prefill_layout(pyr->B, N, pyr->Hkv, K).total) return PISA_ERR_WORKSPACE_TOO_SMALL;
  return PISA_OK;
}

static void prefill_plan(PrefillPlan& P, const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int causal,
                         int32_t* idx, float* scores, void* ws, int mode) {
  P.lv = make_levels(N, pyr->n_cap);
  P.w = prefill_layout(pyr->B, N, pyr->Hkv, K);
  const PrefillWs& w = P.w;
  char* base = static_cast<char*>(ws);
  int32_t* surv = reinterpret_cast<int32_t*>(base + w.surv);
  WalkLaunch& W = P.W;
  W.Q = static_cast<const __nv_bfloat16*>(Q);
  W.summ = pyr->summaries;
  W.lv = &P.lv;
  W.N = N;
  W.B = pyr->B;
  W.Hq = Hq;
  W.Hkv = pyr->Hkv;
  W.K = K;
  W.causal = causal;
  W.table = reinterpret_cast<unsigned char*>(base + w.table);
  W.surv = surv;
  W.srank = reinterpret_cast<int32_t*>(base + w.srank);
  W.count = reinterpret_cast<int*>(base + w.count);
  W.nchunks = w.nchunks;
  W.chunk_shift = w.chunk_shift;
  W.M2 = w.M2;
  W.mode = mode;
  W.t0 = 0;
  W.t1 = N;
  W.build_table = true;
  W.status = reinterpret_cast<int*>(base + w.status);
  LeafTcLaunch& L = P.L;
  L.Q = static_cast<const __nv_bfloat16*>(Q);
  L.keys = static_cast<const __nv_bfloat16*>(pyr->keys);
  L.B = pyr->B;
  L.Hq = Hq;
  L.Hkv = pyr->Hkv;
  L.K = K;
  L.causal = causal;
  L.N = N;
  L.n_cap = pyr->n_cap;
  L.M2 = w.M2;
  L.nchunks = w.nchunks;
  L.chunk_shift = w.chunk_shift;
  L.nb = (int)w.nb;
  L.surv = surv;
  L.count = reinterpret_cast<int*>(base + w.count);
  L.srank = reinterpret_cast<int32_t*>(base + w.srank);
  L.bucket_off = reinterpret_cast<int*>(base + w.bucket_off);
  L.tile_off = reinterpret_cast<int*>(base + w.tile_off);
  L.scan_part = reinterpret_cast<int*>(base + w.scan_part);
  L.tile_desc = reinterpret_cast<int4*>(base + w.tile_desc);
  L.max_tiles = w.max_tiles;
  L.list = reinterpret_cast<uint32_t*>(base + w.list);
  L.leaf_scores = reinterpret_cast<float*>(base + w.leaf);
  L.idx = idx;
  L.scores = scores;
  L.status = reinterpret_cast<int*>(base + w.status);
  L.mode = mode;
  L.t0 = 0;
  L.t1 = N;
  L.b0 = 0;
  L.b1 = (int)w.nb;
}

// Query chunks [c0, c1) of a planned selection: walk, bucketing, leaf level, final
// Top-K.  Buckets are chunk-major, so the chunks' buckets are one contiguous range.
static cudaError_t prefill_stage(PrefillPlan& P, int c0, int c1, bool build_table, cudaStream_t s) {
  const long long BHM = (long long)P.L.B * P.L.Hkv * P.w.M2;
  const long long t0 = (long long)c0 << P.w.chunk_shift;
  const long long t1 = std::min((long long)c1 << P.w.chunk_shift, (long long)P.W.N);
  P.W.t0 = P.L.t0 = t0;
  P.W.t1 = P.L.t1 = t1;
  P.W.build_table = build_table;
  P.L.b0 = (int)(c0 * BHM);
  P.L.b1 = (int)(c1 * BHM);
  cudaError_t e = launch_prefill_walk_mma(P.W, s);
  if (e != cudaSuccess) return e;
  mark_phase(2, s);
  return launch_prefill_leaf_tc(P.L, s);
}

static int select_prefill_impl(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int causal,
                               int32_t* idx, float* scores, void* ws, size_t ws_bytes, void* stream, int mode) {
  const int st = prefill_check(Q, Hq, pyr, N, K, mode, idx, ws, ws_bytes);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PrefillPlan P;
  prefill_plan(P, Q, Hq, pyr, N, K, causal, idx, scores, ws, mode);
  cudaError_t e = cudaMemsetAsync(ws, 0, P.w.zero_bytes, s);
  if (e != cudaSuccess) return PISA_ERR_CUDA;
  mark_phase(0, s);
  return cuda_status(prefill_stage(P, 0, P.w.nchunks, true, s));
}

// Events of the host-buffer pipeline, kept per device and reused from call to call:
// a stream wait captures the event's latest record at the time of the wait, so a
// later call re-recording it cannot disturb waits already enqueued.  The lock is
// held while a call enqueues its work.
constexpr int kHostStages = 16;  // query stages the transfers are split into
static std::mutex g_host_mu;
static std::vector<cudaEvent_t> g_host_ev[64];

// `height` rows of `width` bytes: one pitched copy, or one copy per row where the
// pitch is beyond what a pitched copy accepts (or there is a single row).
static cudaError_t copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, size_t height,
                             cudaMemcpyKind kind, cudaStream_t s) {
  if (height == 1) return cudaMemcpyAsync(dst, src, width, kind, s);
  if (dpitch <= (size_t)INT32_MAX && spitch <= (size_t)INT32_MAX)
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind, s);
  for (size_t r = 0; r < height; ++r) {
    const cudaError_t e = cudaMemcpyAsync(static_cast<char*>(dst) + r * dpitch,
                                          static_cast<const char*>(src) + r * spitch, width, kind, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

static cudaEvent_t* host_events(int dev, int n) {
  std::vector<cudaEvent_t>& v = g_host_ev[dev];
  while ((int)v.size() < n) {
    cudaEvent_t ev;
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    v.push_back(ev);
  }
  return v.data();
}

int pisa_select_prefill_host(const pisa_pyramid* pyr, const void* K_host, int64_t N, const void* Q_host,
                             void* Q_dev, int Hq, int K, int causal, int32_t* idx_host, int32_t* idx_dev,
                             void* ws, size_t ws_bytes, void* stream, void* copy_stream) {
  int st = prefill_check(Q_dev, Hq, pyr, N, K, 0, idx_dev, ws, ws_bytes);
  if (st) return st;
  if (!K_host || !Q_host || !idx_host || N < 1) return PISA_ERR_INVALID_ARG;
  if (N > (1LL << 27) || pyr->n_cap > (1LL << 27)) return PISA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PISA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t c = copy_stream ? static_cast<cudaStream_t>(copy_stream) : s;
  PrefillPlan P;
  prefill_plan(P, Q_dev, Hq, pyr, N, K, causal, idx_dev, nullptr, ws, 0);
  const int nch = P.w.nchunks;
  const int per = (nch + kHostStages - 1) / kHostStages;  // query chunks per stage
  const int ns = (nch + per - 1) / per;
  const int BH = pyr->B * pyr->Hkv;
  const size_t qrow = (size_t)Hq * kD * 2, krow = (size_t)pyr->Hkv * kD * 2, irow = (size_t)K * 4;
  std::lock_guard<std::mutex> lock(g_host_mu);
  cudaEvent_t* ev = host_events(dev, 2 * ns + 2);
  if (!ev) return PISA_ERR_CUDA;
  cudaEvent_t e_keys = ev[0], e_done = ev[1 + 2 * ns];
  auto stage_t = [&](int i, long long& t0, long long& t1) {
    t0 = (long long)(i * per) << P.w.chunk_shift;
    t1 = std::min((long long)std::min((i + 1) * per, nch) << P.w.chunk_shift, (long long)N);
  };
  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
    return e == cudaSuccess;
  };
  // copy stream: the keys, then the query rows stage by stage
  ok(copy_rows(pyr->keys, (size_t)pyr->n_cap * krow, K_host, (size_t)N * krow, (size_t)N * krow, pyr->B,
               cudaMemcpyHostToDevice, c));
  ok(cudaEventRecord(e_keys, c));
  for (int i = 0; i < ns; ++i) {
    long long t0, t1;
    stage_t(i, t0, t1);
    ok(copy_rows(static_cast<char*>(Q_dev) + t0 * qrow, (size_t)N * qrow, static_cast<const char*>(Q_host) + t0 * qrow,
                 (size_t)N * qrow, (size_t)(t1 - t0) * qrow, pyr->B, cudaMemcpyHostToDevice, c));
    ok(cudaEventRecord(ev[1 + i], c));
  }
  // compute stream: pyramid and route table once the keys are in, then each stage
  // once its query rows are in
  ok(cudaStreamWaitEvent(s, e_keys, 0));
  ok(cudaMemsetAsync(ws, 0, P.w.zero_bytes, s));
  ok(launch_build_pyramid(static_cast<const __nv_bfloat16*>(pyr->keys), pyr->summaries, P.lv, N, pyr->n_cap, pyr->B,
                          pyr->Hkv, pyr->lengths, s));
  P.W.t0 = P.W.t1 = 0;
  P.W.build_table = true;
  ok(launch_prefill_walk_mma(P.W, s));
  for (int i = 0; i < ns && e == cudaSuccess; ++i) {
    ok(cudaStreamWaitEvent(s, ev[1 + i], 0));
    ok(prefill_stage(P, i * per, std::min((i + 1) * per, nch), false, s));
    ok(cudaEventRecord(ev[1 + ns + i], s));
  }
  // copy stream: each stage's indices once the stage is done; the compute stream
  // then waits for the last copy, so work queued on it after this call sees them
  for (int i = 0; i < ns && e == cudaSuccess; ++i) {
    long long t0, t1;
    stage_t(i, t0, t1);
    ok(cudaStreamWaitEvent(c, ev[1 + ns + i], 0));
    ok(copy_rows(reinterpret_cast<char*>(idx_host) + t0 * irow, (size_t)N * irow,
                 reinterpret_cast<const char*>(idx_dev) + t0 * irow, (size_t)N * irow, (size_t)(t1 - t0) * irow, BH,
                 cudaMemcpyDeviceToHost, c));
  }
  ok(cudaEventRecord(e_done, c));
  ok(cudaStreamWaitEvent(s, e_done, 0));
  return e == cudaSuccess ? PISA_OK : PISA_ERR_CUDA;
}

int pisa_select_prefill(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int causal,
                        int32_t* idx, float* scores, void* ws, size_t ws_bytes, void* stream) {
  return select_prefill_impl(Q, Hq, pyr, N, K, causal, idx, scores, ws, ws_bytes, stream, 0);
}

int pisa_select_prefill_ex(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int causal,
                           int32_t* idx, float* scores, void* ws, size_t ws_bytes, void* stream,
                           int score_mode) {
  return select_prefill_impl(Q, Hq, pyr, N, K, causal, idx, scores, ws, ws_bytes, stream, score_mode);
}

int pisa_sparse_attention(const void* Q, int Hq, const void* K, const void* V, int B, int64_t N, int Hkv,
                          const int32_t* idx, int Ksel, int causal, float* out, void* stream) {
  if (!Q || !K || !V || !idx || !out || B < 1 || N < 1 || Hkv < 1 || Hq < 1) return PISA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return PISA_ERR_INVALID_ARG;
  if (Hq % Hkv) return PISA_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if ((G & (G - 1)) || G > 16 || Ksel < 1 || Ksel > 64 || (long long)B * Hkv * N >= (1LL << 40))
    return PISA_ERR_UNSUPPORTED;
  return cuda_status(launch_sparse_attention(static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
                                             static_cast<const __nv_bfloat16*>(V), idx, B, N, Hq, Hkv, Ksel,
                                             causal != 0, out, static_cast<cudaStream_t>(stream)));
}

size_t pisa_flat_workspace_bytes(int B, int64_t N, int Hq, int Hkv, int K) {
  if (check_geometry(B, N, Hq, Hkv, kD, kC, 2, K) != PISA_OK) return 0;
  const FlatWs w = flat_layout(B, N, Hq, Hkv, K, true);
  if (w.T >= (1LL << 31)) return 0;
  return flat_layout(B, N, Hq, Hkv, K, false).size;  // the non-causal layout is the larger
}

static int select_flat_impl(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int causal,
                            int32_t* idx, float* scores, void* ws, size_t ws_bytes, void* stream, int mode) {
  if (mode < 0 || mode > 2) return PISA_ERR_UNSUPPORTED;
  int st = check_pyr(pyr);
  if (st) return st;
  if (!Q || !idx || !ws) return PISA_ERR_INVALID_ARG;
  st = check_geometry(pyr->B, N, Hq, pyr->Hkv, pyr->d, pyr->C, pyr->g, K);
  if (st) return st;
  if (N > pyr->n_cap) return PISA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(Q) & 15) || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)))
    return PISA_ERR_INVALID_ARG;
  const FlatWs w = flat_layout(pyr->B, N, Hq, pyr->Hkv, K, causal != 0);
  if (w.T >= (1LL << 31) || (long long)pyr->B * pyr->n_cap >= (1LL << 31)) return PISA_ERR_UNSUPPORTED;
  if (ws_bytes < w.size) return PISA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  if (cudaMemsetAsync(base, 0, kStatusBytes, s) != cudaSuccess) return PISA_ERR_CUDA;
  LeafTcLaunch L{};
  L.Q = static_cast<const __nv_bfloat16*>(Q);
  L.keys = static_cast<const __nv_bfloat16*>(pyr->keys);
  L.B = pyr->B;
  L.Hq = Hq;
  L.Hkv = pyr->Hkv;
  L.K = K;
  L.causal = causal != 0;
  L.N = N;
  L.n_cap = pyr->n_cap;
  L.M2 = (int)level_size_for(N, 2);
  L.list = reinterpret_cast<uint32_t*>(base + w.list);
  L.tile_desc = reinterpret_cast<int4*>(base + w.desc);
  L.leaf_scores = reinterpret_cast<float*>(base + w.leaf);
  L.idx = idx;
  L.scores = scores;
  L.status = reinterpret_cast<int*>(base + w.status);
  L.mode = mode;
  return cuda_status(launch_select_flat(L, w.T1, w.stride, reinterpret_cast<int*>(base + w.total), s));
}

int pisa_select_flat(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int causal,
                     int32_t* idx, float* scores, void* ws, size_t ws_bytes, void* stream) {
  return select_flat_impl(Q, Hq, pyr, N, K, causal, idx, scores, ws, ws_bytes, stream, 0);
}

int pisa_select_flat_ex(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int causal,
                        int32_t* idx, float* scores, void* ws, size_t ws_bytes, void* stream, int score_mode) {
  return select_flat_impl(Q, Hq, pyr, N, K, causal, idx, scores, ws, ws_bytes, stream, score_mode);
}

// Decode workspace: [status 256 B][one arrival counter per sequence], zeroed per call.
size_t pisa_decode_workspace_bytes(int B, int Hq, int Hkv, int K) {
  if (check_geometry(B, 1, Hq, Hkv, kD, kC, 2, K) != PISA_OK) return 0;
  return align_up(kStatusBytes + sizeof(int) * (size_t)B);
}

int pisa_decode_append_and_select(const void* q_new, const void* k_new, int Hq, const pisa_pyramid* pyr,
                                  int K, int32_t* idx, float* scores, void* ws, size_t ws_bytes,
                                  void* stream) {
  int st = check_pyr(pyr);
  if (st) return st;
  if (!q_new || !k_new || !idx || !ws || !pyr->lengths) return PISA_ERR_INVALID_ARG;
  st = check_geometry(pyr->B, pyr->n_cap, Hq, pyr->Hkv, pyr->d, pyr->C, pyr->g, K);
  if (st) return st;
  if (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) return PISA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q_new) & 15) return PISA_ERR_INVALID_ARG;  // read 16 bytes at a time
  const size_t zero = kStatusBytes + sizeof(int) * (size_t)pyr->B;
  if (ws_bytes < align_up(zero)) return PISA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, zero, s);
  if (e != cudaSuccess) return PISA_ERR_CUDA;
  const Levels cap_lv = make_levels(pyr->n_cap, pyr->n_cap);
  e = launch_decode_warp(static_cast<const __nv_bfloat16*>(q_new), static_cast<const __nv_bfloat16*>(k_new),
                         static_cast<__nv_bfloat16*>(pyr->keys), pyr->summaries, pyr->lengths, cap_lv,
                         pyr->n_cap, pyr->B, Hq, pyr->Hkv, K, idx, scores, static_cast<int*>(ws),
                         reinterpret_cast<int*>(static_cast<char*>(ws) + kStatusBytes), s);
  return cuda_status(e);
}

int pisa_selftest_bounded_wait(void* ws, size_t ws_bytes, int64_t delay_cycles, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return PISA_ERR_INVALID_ARG;
  if (ws_bytes < kStatusBytes) return PISA_ERR_WORKSPACE_TOO_SMALL;
  if (delay_cycles < 0 || delay_cycles > (1LL << 32)) return PISA_ERR_INVALID_ARG;  // (about 2 s at most)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kStatusBytes, s) != cudaSuccess) return PISA_ERR_CUDA;
  return cuda_status(launch_selftest_wait(static_cast<int*>(ws), delay_cycles, s));
}

int pisa_check_device_status(const void* ws, void* stream) {
  if (!ws) return PISA_ERR_INVALID_ARG;
  int h = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&h, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return PISA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PISA_ERR_CUDA;
  return h;
}

uint64_t pisa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int pisa_set_phase_events(void* const* events, int n_events) {
  if (n_events < 0 || n_events > 16 || (n_events > 0 && !events)) return PISA_ERR_INVALID_ARG;
  for (int i = 0; i < n_events; ++i) g_phase_events[i] = static_cast<cudaEvent_t>(events[i]);
  g_n_phase_events = n_events;
  return PISA_OK;
}

int pisa_prefill_phase_count(void) { return kPrefillPhases; }

int pisa_event_elapsed_ms(void* start, void* end, float* ms) {
  if (!start || !end || !ms) return PISA_ERR_INVALID_ARG;
  return cudaEventElapsedTime(ms, static_cast<cudaEvent_t>(start), static_cast<cudaEvent_t>(end)) == cudaSuccess
             ? PISA_OK
             : PISA_ERR_CUDA;
}

const char* pisa_prefill_phase_name(int i) {
  static const char* names[] = {"route_table", "walk", "bucket", "leaf", "final"};
  return (i >= 0 && i < kPrefillPhases) ? names[i] : "";
}

const char* pisa_status_string(int status) {
  switch (status) {
    case PISA_OK: return "ok";
    case PISA_ERR_INVALID_ARG: return "invalid argument";
    case PISA_ERR_UNSUPPORTED: return "unsupported size (needs d=64, C=64, g=2, K<=32, Hq/Hkv in {1,2,4,8,16})";
    case PISA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PISA_ERR_CUDA: return "CUDA runtime or launch error";
    case PISA_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait timed out";
    case PISA_ERR_DEVICE_BOUNDS: return "a kernel's bounds check failed (e.g. decode cache full)";
    default: return "unknown status";
  }
}

}  // extern "C"
