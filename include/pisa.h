/*
 * pisa.h -- C ABI of the GB300 (sm_103a) PISA pyramid Top-K block selector.
 *
 * The library computes the block-selection stage of PISA block-sparse
 * attention ("Block Sparse Attention with Log-Linear Complexity", §3.1 Fine to
 * coarse: building the pyramid; §3.2 Coarse to fine: narrowing the Top-K;
 * "Scoring: LogSumExp, and why not the mean"; §4.1 the GQA head sum; §5.1 the
 * prefill and decoding kernels).  Keys are mean-pooled into a pyramid (leaves
 * of C tokens, then merges of g up to one root); each query then walks it
 * coarse-to-fine, scoring at most g*K candidates per level by a LogSumExp over
 * their children's summaries (raw keys at the leaf level), summed over the
 * query heads of its GQA group, and keeping the Top-K.
 *
 * Conventions shared by every call
 *   - All pointers named "device" are CUDA device pointers owned by the
 *     caller; the library never allocates device memory.  Host pointers are
 *     named as such.
 *   - bf16 tensors are passed as `const void*` (IEEE bfloat16, little endian).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     is asynchronous on it; outputs are valid once the stream reaches them.
 *   - Layouts are dense, row-major, 16-byte aligned:
 *       Q       [B, N, Hq,  d]  bf16      K      [B, n_cap, Hkv, d] bf16
 *       summary [B, Hkv, pisa_pyramid_nodes(n_cap, C, g), d] fp32, levels
 *               leaf-first (level 1 = leaves, then level 2, ... root last),
 *               level sizes M_1 = ceil(n_cap/C), M_l = ceil(M_{l-1}/g).
 *     Query head h belongs to KV head h / (Hq/Hkv) (contiguous groups).
 *   - Supported sizes: d = 64, C = 64, g = 2, 1 <= K <= 32,
 *     Hq/Hkv in {1, 2, 4, 8, 16}, 1 <= Hkv <= 32, N <= 2^27,
 *     B * Hkv <= 65535, B * Hkv * N * K < 2^31 - 2^20.  Anything
 *     else returns PISA_ERR_UNSUPPORTED (or PISA_ERR_INVALID_ARG when
 *     malformed).
 *   - Readings fixed by this library where the method's description is
 *     silent: logits are q.k/sqrt(d); a ragged node (sequence tail) is the
 *     mean over the tokens present; causal eligibility of a node for query t
 *     is "first token <= t", and a child that starts after t is left out of
 *     its parent's LSE (keys after t are masked in the leaf LSE); the LSE is
 *     un-normalised; Top-K ties go to the lower node index; the output lists
 *     the selected leaves in ascending order, padded with -1.
 *   - Errors: every call returns a pisa_status.  Argument errors are caught
 *     on the host before anything is launched.  Errors raised inside a
 *     kernel (a bounded wait that timed out) are recorded in a status word at
 *     the start of the caller's workspace; read it with
 *     pisa_check_device_status().  No C++ exception crosses this ABI.
 */
#ifndef PISA_H_
#define PISA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PISA_OK = 0,
  PISA_ERR_INVALID_ARG = 1,          /* NULL pointer, negative size, N > n_cap, ... */
  PISA_ERR_UNSUPPORTED = 2,          /* a size outside the supported set above      */
  PISA_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes below the *_workspace_bytes value  */
  PISA_ERR_CUDA = 4,                 /* a CUDA runtime / launch error               */
  PISA_ERR_DEVICE_TIMEOUT = 5,       /* a kernel's bounded wait gave up             */
  PISA_ERR_DEVICE_BOUNDS = 6         /* a kernel's index check failed               */
} pisa_status;

/*
 * Pyramid descriptor (plain struct, all memory caller-owned).
 *   summaries : device fp32 [B, Hkv, pisa_pyramid_nodes(n_cap, C, g), d]
 *   keys      : device bf16 [B, n_cap, Hkv, d]; the raw keys the leaf level
 *               scores against (borrowed; decode appends into it)
 *   lengths   : device int32 [B], tokens present per sequence (decode); may
 *               be NULL for prefill-only use
 *   n_cap     : capacity in tokens; the node layout is fixed by n_cap so a
 *               decode cache never moves as it grows
 */
typedef struct {
  float* summaries;
  void* keys;
  int32_t* lengths;
  int B, Hkv, d, C, g, n_cap;
} pisa_pyramid;

/* Number of levels holding nodes for n tokens (1 for n <= C), or -1. */
int pisa_num_levels(int64_t n, int C, int g);

/* Sum over levels of the node counts for a capacity of n_cap tokens, or -1. */
int64_t pisa_pyramid_nodes(int64_t n_cap, int C, int g);

/* Row offset of level `level` (1 = leaves) inside one (b, kv) summary block. */
int64_t pisa_level_offset(int64_t n_cap, int C, int g, int level);

/*
 * pisa_build_pyramid -- fine-to-coarse mean pooling (§3.1).
 * Builds every summary of the first N tokens of each sequence from pyr->keys:
 * leaf i = mean of keys [iC, min((i+1)C, N)); a node of level l >= 2 = the
 * token-count-weighted mean of its children (= mean of all its raw keys).
 * Nodes outside the first N tokens are left untouched.  If pyr->lengths is
 * not NULL, every entry is set to N.  Requires 1 <= N <= n_cap.
 */
int pisa_build_pyramid(const pisa_pyramid* pyr, int64_t N, void* stream);

/*
 * pisa_build_pyramid_ragged -- pisa_build_pyramid for a batch of sequences of
 * different lengths (§3.1 per sequence): sequence b holds pyr->lengths[b] tokens
 * (device int32, read on the device, clamped to [0, n_cap]); its nodes are the
 * means over its own tokens, nodes past its own level sizes are left untouched.
 * Nothing is read back to the host, so the call can be captured in a CUDA graph.
 * Equal lengths give the same bits as pisa_build_pyramid.  Decode steps then
 * append to each sequence at its own length.
 */
int pisa_build_pyramid_ragged(const pisa_pyramid* pyr, void* stream);

/* Workspace bytes pisa_select_prefill needs for these sizes (0 on bad sizes). */
size_t pisa_select_workspace_bytes(int B, int64_t N, int Hq, int Hkv, int K);

/*
 * pisa_select_prefill -- coarse-to-fine Top-K walk for every query (§3.2).
 *   Q      : device bf16 [B, N, Hq, d]
 *   pyr    : a pyramid built over the same N tokens (pyr->n_cap may exceed N)
 *   K      : blocks to keep per query and KV head
 *   causal : nonzero = query t sees tokens <= t only
 *   idx    : device int32 [B, Hkv, N, K] out: selected leaf blocks, ascending,
 *            -1 where fewer than K leaves are eligible
 *   scores : device fp32 [B, Hkv, N, K] out (may be NULL): the exact leaf score
 *            (raw-key LSE summed over the group's heads) of each selected
 *            leaf; -inf in padded slots
 *   ws     : device workspace of at least pisa_select_workspace_bytes(...)
 *            bytes, 256-byte aligned; its content is scratch on entry
 */
int pisa_select_prefill(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K,
                        int causal, int32_t* idx, float* scores, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * pisa_select_prefill_host -- pisa_build_pyramid + pisa_select_prefill for inputs
 * and output in host memory, with the transfers overlapped with the selection
 * ("Block Sparse Attention with Log-Linear Complexity", §3.1 and §3.2; the
 * computation and its results are exactly those of the two device calls).  The
 * keys are copied into pyr->keys and the pyramid is built over N tokens; the
 * queries are copied into Q_dev in runs of query chunks on copy_stream while
 * `stream` runs the selection of each run as soon as its rows are in, and each
 * run's indices are copied back as soon as they are final.
 *   pyr        : device pyramid, n_cap >= N; its keys, summaries and lengths are
 *                overwritten
 *   K_host     : host bf16 [B, N, Hkv, d]   (pinned memory for overlap)
 *   Q_host     : host bf16 [B, N, Hq, d]    (pinned memory for overlap)
 *   Q_dev      : device bf16 [B, N, Hq, d] staging buffer, 16-byte aligned
 *   idx_host   : host int32 [B, Hkv, N, K] out (pinned memory for overlap)
 *   idx_dev    : device int32 [B, Hkv, N, K] staging buffer
 *   ws         : as for pisa_select_prefill
 *   copy_stream: stream for the copies (NULL: `stream`, no overlap)
 * Asynchronous: host buffers must stay valid until the work completes; work
 * enqueued on `stream` after this call is ordered after all of it, copies
 * included.  Errors as pisa_select_prefill; PISA_ERR_CUDA if a copy or an event
 * cannot be enqueued.  Calls are serialised on a library lock while they enqueue.
 */
int pisa_select_prefill_host(const pisa_pyramid* pyr, const void* K_host, int64_t N, const void* Q_host,
                             void* Q_dev, int Hq, int K, int causal, int32_t* idx_host, int32_t* idx_dev,
                             void* ws, size_t ws_bytes, void* stream, void* copy_stream);

/* Workspace bytes pisa_select_flat needs (0 on bad or unsupported sizes).  It
 * grows as N^2 / C: one fp32 score per (b, kv, query, leaf) plus the tile list. */
size_t pisa_flat_workspace_bytes(int B, int64_t N, int Hq, int Hkv, int K);

/*
 * pisa_select_flat -- the flat block selector the pyramid walk replaces: "PISA
 * cuts block-sparse attention selection to O(N log N) ..." (conventional
 * block-sparse attention such as BSA scores all N/C key blocks per query).
 * Every eligible leaf gets its exact leaf score ("Block Sparse Attention with
 * Log-Linear Complexity", Scoring: LogSumExp: raw-key LSE summed over the
 * group's heads, keys after t masked when causal) and the K best are kept
 * (ties to the lower leaf index).  Arguments, layouts, ownership and errors as
 * for pisa_select_prefill; only pyr->keys is read (the summaries are unused).
 *   idx    : device int32 [B, Hkv, N, K] out: ascending, -1 padded
 *   scores : device fp32 [B, Hkv, N, K] out (may be NULL), -inf padded
 *   ws     : at least pisa_flat_workspace_bytes(...) bytes, 256-byte aligned
 * PISA_ERR_UNSUPPORTED when the tile count reaches 2^31.
 */
int pisa_select_flat(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int causal,
                     int32_t* idx, float* scores, void* ws, size_t ws_bytes, void* stream);

/*
 * Score modes of the _ex entry points ("Block Sparse Attention with Log-Linear
 * Complexity", Scoring: LogSumExp -- the Taylor expansion of the LSE around the
 * mean of the logits, without log m, truncated at first order gives the mean
 * (the PISA-1 ablation), at second order the mean plus half the variance
 * (PISA-2)).  The mode replaces the block score at every scored level,
 * intermediate (over the children's summary logits) and leaf (over the raw-key
 * logits); the reported scores are the leaf scores under that mode.
 */
#define PISA_SCORE_LSE 0
#define PISA_SCORE_MEAN 1
#define PISA_SCORE_MEAN_HALF_VAR 2

/* pisa_select_prefill with a score mode (PISA_ERR_UNSUPPORTED for other modes). */
int pisa_select_prefill_ex(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K,
                           int causal, int32_t* idx, float* scores, void* ws, size_t ws_bytes,
                           void* stream, int score_mode);

/* pisa_select_flat with a score mode (PISA_ERR_UNSUPPORTED for other modes). */
int pisa_select_flat_ex(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K, int causal,
                        int32_t* idx, float* scores, void* ws, size_t ws_bytes, void* stream,
                        int score_mode);

/*
 * pisa_sparse_attention -- stage two of block-sparse attention ("Block Sparse
 * Attention with Log-Linear Complexity", Background: two stages): each query
 * attends over the original keys and values inside its selected blocks, one
 * softmax over all of them (scale 1/sqrt(d)), keys after the query masked when
 * causal.  Arithmetic: bf16 inputs and bf16 probabilities on the tensor cores,
 * fp32 accumulation and softmax.
 *   Q      : device bf16 [B, N, Hq, d]
 *   K, V   : device bf16 [B, N, Hkv, d] (d = 64)
 *   idx    : device int32 [B, Hkv, N, Ksel] leaf blocks (C = 64 keys) per query
 *            and KV head, as pisa_select_prefill writes them; -1 entries skipped
 *   out    : device fp32 [B, N, Hq, d] out; a query without keys gets zeros
 * 1 <= Ksel <= 64, Hq/Hkv in {1, 2, 4, 8, 16}.  No workspace.  Asynchronous on
 * stream; argument errors return before any launch.
 */
int pisa_sparse_attention(const void* Q, int Hq, const void* K, const void* V, int B, int64_t N, int Hkv,
                          const int32_t* idx, int Ksel, int causal, float* out, void* stream);

/* Workspace bytes pisa_decode_append_and_select needs (0 on bad sizes). */
size_t pisa_decode_workspace_bytes(int B, int Hq, int Hkv, int K);

/*
 * pisa_decode_append_and_select -- one decoding step ([P1]/§5.1: the decoder
 * keeps the mean pyramid cached, updates only the new token's leaf mean and its
 * ancestor path, then walks for the new query).
 *   q_new  : device bf16 [B, Hq, d], the query of the token being appended
 *            (16-byte aligned)
 *   k_new  : device bf16 [B, Hkv, d], its key
 *   pyr    : pyramid with keys [B, n_cap, Hkv, d], summaries and lengths (all
 *            required); for each b the key is written at position
 *            lengths[b], the leaf and ancestor summaries are refreshed, the
 *            walk runs for t = lengths[b] (causal), and lengths[b] grows by 1.
 *            Every lengths[b] must be < n_cap (checked on the device: a full
 *            sequence is left unchanged and flags PISA_ERR_DEVICE_BOUNDS).
 *   idx    : device int32 [B, Hkv, K] out; scores: device fp32 [B, Hkv, K] or NULL
 *   ws     : device workspace of at least pisa_decode_workspace_bytes(...) bytes
 */
int pisa_decode_append_and_select(const void* q_new, const void* k_new, int Hq,
                                  const pisa_pyramid* pyr, int K, int32_t* idx, float* scores,
                                  void* ws, size_t ws_bytes, void* stream);

/*
 * pisa_select_prefill_noalloc -- the prefill selection above for callers that
 * cannot allocate device memory: no workspace argument.  (The paper has no
 * counterpart; this is a deployment convenience of this library.)
 *
 * For callers whose host framework owns all device memory and passes them
 * only input and output buffers, or whose request path may not call
 * cudaMalloc (an allocation can synchronise the device or fail mid-request).
 * The scratch it needs is a fixed device array inside this library of
 * PISA_NOALLOC_SCRATCH_BYTES bytes (32 MiB), held by every GPU that loads the
 * library until the process exits.
 *   Arguments, outputs and layouts are those of pisa_select_prefill.
 *   Returns PISA_ERR_WORKSPACE_TOO_SMALL, launching nothing, when
 *   pisa_select_workspace_bytes(B, N, Hq, Hkv, K) exceeds that size; call
 *   that function to know in advance which sizes fit.
 *   The first call on a device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture.  It allocates nothing and calls no allocating routine.
 *   All calls share the one array: calls that overlap on the GPU (different
 *   streams, or unordered host threads) race and give wrong results.  Each
 *   call clears what must start at zero.  Kernel-side status cannot be read
 *   back for this entry point (pisa_check_device_status needs a workspace).
 */
#define PISA_NOALLOC_SCRATCH_BYTES (32u << 20)
int pisa_select_prefill_noalloc(const void* Q, int Hq, const pisa_pyramid* pyr, int64_t N, int K,
                                int causal, int32_t* idx, float* scores, void* stream);

/*
 * pisa_noalloc_prepare -- set-up for pisa_select_prefill_noalloc on the current
 * device: looks up (and caches) the scratch array's device address, loading this
 * library's device code on the device if it is not loaded yet.  Writes the address
 * to *scratch when scratch is not NULL (for diagnostics).  Returns PISA_OK or
 * PISA_ERR_CUDA.
 *
 * pisa_noalloc_device_status -- synchronises `stream` and returns the status word
 * that the kernels of the last pisa_select_prefill_noalloc call on the current
 * device left in the scratch array (PISA_OK if none), like
 * pisa_check_device_status does for a caller's workspace.
 */
int pisa_noalloc_prepare(void** scratch);
int pisa_noalloc_device_status(void* stream);

/*
 * pisa_selftest_bounded_wait -- the failure path of the kernels' bounded barrier
 * waits, exercised on the GPU without faulting it: one thread waits on an mbarrier
 * that nothing arrives on, through the same wait routine the tcgen05 kernels use,
 * while another warp of its CTA raises the CTA's abort flag after delay_cycles clock
 * cycles (0 <= delay_cycles <= 2^32); the wait gives up and the kernel records
 * PISA_ERR_DEVICE_TIMEOUT in the status word of ws (device memory, >= 256 bytes,
 * 256-byte aligned, zeroed here first) and returns.  Read it with
 * pisa_check_device_status.  Returns PISA_ERR_INVALID_ARG / _WORKSPACE_TOO_SMALL on
 * bad arguments, before anything is launched.
 */
int pisa_selftest_bounded_wait(void* ws, size_t ws_bytes, int64_t delay_cycles, void* stream);

/*
 * Synchronises `stream` and returns the status word that kernels of the last
 * select / decode call on this workspace left in `ws` (PISA_OK if none).
 */
int pisa_check_device_status(const void* ws, void* stream);

/*
 * Profiling aids (host-side, not thread-safe: call from one host thread).
 * pisa_kernel_launches: kernels this library has launched since it was loaded.
 * pisa_set_phase_events: attach n_events cudaEvent_t handles (created by the
 *   caller, passed as void*); pisa_select_prefill then records event i at the
 *   start of phase i on its stream and event pisa_prefill_phase_count() at its
 *   end.  n_events = 0 detaches.  Returns PISA_OK or PISA_ERR_INVALID_ARG.
 * pisa_prefill_phase_count / pisa_prefill_phase_name: the phases of
 *   pisa_select_prefill in launch order (static strings).
 * pisa_event_elapsed_ms: milliseconds between two recorded events (cudaEvent_t
 *   passed as void*), for events the library recorded on the caller's behalf.
 */
uint64_t pisa_kernel_launches(void);
int pisa_event_elapsed_ms(void* start, void* end, float* ms);
int pisa_set_phase_events(void* const* events, int n_events);
int pisa_prefill_phase_count(void);
const char* pisa_prefill_phase_name(int phase);

/* Static, human-readable text for a pisa_status value. */
const char* pisa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PISA_H_ */
