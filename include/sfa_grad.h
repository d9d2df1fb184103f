/*
 * sfa_grad.h -- C ABI of the GB300 (sm_103a) top-k sparse flash-attention
 * backward library (libsfa.so), plus the companion forward that produces the
 * backward's saved inputs.
 *
 * Operation (aclnnSparseFlashAttentionGrad doc, section 功能说明 and stages
 * 阶段1-3): every query token t carries K int32 indices into its KV sequence;
 * index r selects keys r .. r + sparseBlockSize - 1.  With
 *   x_j  = scale * ([q || qRope]_t . [k || kRope]_j)            (per head)
 *   P_j  = exp(x_j - softmaxMax) / softmaxSum                   (masked keys: 0)
 *   Dsum = rowsum(dOut_t * out_t)                               (FlashSoftmaxGrad)
 *   dP_j = dOut_t . v_j,     dS_j = P_j (dP_j - Dsum)
 * the outputs are
 *   [dQ || dQRope]_t  = scale * sum_j dS_j [k || kRope]_j
 *   [dK || dKRope]_j += scale * dS_j [q || qRope]_t,     dV_j += P_j dOut_t
 * summed over every head and every (token, slot) that selects key j.
 * softmaxMax is the max of the scaled scores x over the selected keys and
 * softmaxSum = sum_j exp(x_j - softmaxMax) (the MindSpore
 * flash_attention_bwd.py page, compute_Pij, uses exactly these two saved
 * statistics).
 *
 * Conventions
 *  - Two phases, as on the documentation page (函数原型): ask for the workspace
 *    size, allocate it, then call.  The caller owns every buffer; the library
 *    allocates no memory, keeps no state between calls and is thread-safe
 *    (sfa_grad_host creates two streams and a few events per call).
 *  - All tensor pointers are DEVICE pointers to contiguous row-major data
 *    (16-byte aligned), except those of sfa_grad_host (host buffers).  Shapes use the page's names (参数说明 table):
 *      BSND: q, dOut, out (B,S1,N1,D); k, v (B,S2,1,D); indices (B,S1,1,K);
 *            softmaxMax/Sum (B,1,S1,N1); qRope (B,S1,N1,Dr); kRope (B,S2,1,Dr)
 *      TND:  q, dOut, out (T1,N1,D); k, v (T2,1,D); indices (T1,1,K);
 *            softmaxMax/Sum (1,T1,N1); actualSeqLengths{Query,Kv} int32 (B,)
 *            of per-batch lengths summing to T1 / T2.
 *    Outputs have the shape and dtype of the matching input and are fully
 *    overwritten (never accumulated into).
 *  - Calls are asynchronous on `stream`; a SFA_OK return means the work was
 *    enqueued.  Device-side problems (TND lengths that are negative or do not
 *    sum to T1/T2, an internal pipeline wait that timed out) are recorded in
 *    an error word inside the workspace, readable with sfa_read_device_error.
 *  - Indices need no host inspection: negative, out-of-range and (sparseMode
 *    3) future positions are masked and contribute nothing; duplicates count
 *    once per occurrence.
 *  - With deterministic = 0 the key-side sums use fp32 atomics (order varies
 *    run to run, as on the page: "默认非确定性实现"); with deterministic = 1
 *    they are reduced in a fixed order and the outputs are bitwise
 *    reproducible (约束说明, 确定性计算).
 */
#ifndef SFA_GRAD_H_
#define SFA_GRAD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes: the page's 返回值 table (aclnn status values). */
typedef enum {
  SFA_OK = 0,
  SFA_ERR_NULLPTR = 161001,       /* a required pointer is null */
  SFA_ERR_PARAM_INVALID = 161002, /* dtype / layout enum out of range, workspace too small */
  SFA_ERR_RUNTIME = 361001,       /* a CUDA launch or runtime call failed */
  SFA_ERR_SHAPE = 561002          /* a size or attribute outside the supported range */
} sfa_status;

typedef enum { SFA_DTYPE_BF16 = 0, SFA_DTYPE_FP16 = 1 } sfa_dtype;
typedef enum { SFA_LAYOUT_BSND = 0, SFA_LAYOUT_TND = 1 } sfa_layout;

/* Device error word values (sfa_read_device_error). */
#define SFA_DEVERR_NONE 0
#define SFA_DEVERR_TIMEOUT 1  /* a kernel abandoned a pipeline wait after the wall-clock limit (no hang) */
#define SFA_DEVERR_SEQLENS 2  /* TND lengths negative or not summing to T1/T2: every key was masked */

/*
 * Problem description (replaces the page's aclTensor shape metadata and the
 * scalar attributes of the first-phase call).
 *   layout             SFA_LAYOUT_BSND or SFA_LAYOUT_TND ("layout")
 *   dtype              element type of q, k, v, dOut, out, rope tensors and outputs
 *   B                  batch count (TND: number of actual-length entries)
 *   S1, S2             BSND query / kv sequence lengths (ignored for TND)
 *   T1, T2             TND total query / kv tokens (ignored for BSND)
 *   N1                 query heads, 1..128 (G = N1 / N2)
 *   N2                 kv heads; must be 1 (the op is MQA)
 *   D                  head dim; must be 512
 *   Dr                 rope dim: 64, or 0 when the rope tensors are absent
 *   K                  indices per query token (>= 1)
 *   scale              scaleValue (suggested 1/sqrt(d))
 *   sparse_block_size  1, 8, 16, 32 or 64 keys per index
 *   sparse_mode        0 (no mask) or 3 (rightDownCausal)
 *   deterministic      0 or 1
 *   wait_limit_us      0: every pipeline wait inside the kernels gives up
 *                      after 2 s; > 0: after this many microseconds.  A wait
 *                      that gives up makes its kernel wind down (no hang) and
 *                      records SFA_DEVERR_TIMEOUT; the outputs are then
 *                      incomplete.  A test hook for that path: ordinary
 *                      callers leave it 0.  Negative values are
 *                      SFA_ERR_PARAM_INVALID.
 */
typedef struct sfa_params {
  int32_t layout;
  int32_t dtype;
  int64_t B, S1, S2, T1, T2;
  int64_t N1, N2, D, Dr, K;
  double scale;
  int64_t sparse_block_size;
  int64_t sparse_mode;
  int32_t deterministic;
  int32_t wait_limit_us;
} sfa_params;

/*
 * Phase 1 (aclnnSparseFlashAttentionGradGetWorkspaceSize): validates *p and
 * writes the device workspace size in bytes to *bytes.
 * Errors: SFA_ERR_NULLPTR (p or bytes null), SFA_ERR_PARAM_INVALID (dtype,
 * layout or deterministic out of range, negative wait_limit_us), SFA_ERR_SHAPE (N2 != 1, D != 512, Dr not in {0,64},
 * N1 not in 1..128, sparse_mode not in {0,3}, block size not in
 * {1,8,16,32,64}, K < 1, negative sizes, non-finite scale, sizes overflowing
 * 32-bit row counts).
 */
sfa_status sfa_grad_workspace_size(const sfa_params* p, size_t* bytes);

/*
 * Phase 2 (aclnnSparseFlashAttentionGrad): computes dq, dk, dv, dq_rope,
 * dk_rope.  act_seq_q / act_seq_kv are device int32 arrays of length B (TND
 * only; ignored for BSND).  q_rope, k_rope, dq_rope, dk_rope are required when
 * Dr = 64 and ignored when Dr = 0.  `workspace` is a device buffer of at
 * least the phase-1 size, 256-byte aligned, owned by the caller; its contents
 * need no initialisation and are scratch after the call.  An empty query
 * (T1 = 0 or S1 = 0, 约束说明: "query为空Tensor：直接返回") returns SFA_OK after
 * zeroing dk, dv, dk_rope.  Returns SFA_ERR_NULLPTR for a missing required
 * pointer, SFA_ERR_PARAM_INVALID for a short workspace, SFA_ERR_RUNTIME when
 * a launch fails, and the phase-1 codes.
 */
sfa_status sfa_grad(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                    const void* d_out, const void* out, const float* softmax_max, const float* softmax_sum,
                    const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope, const void* k_rope,
                    void* dq, void* dk, void* dv, void* dq_rope, void* dk_rope, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * sfa_grad with per-launch timing: identical work; additionally, when
 * `events` is non-null, records events[0] on `stream` before the first
 * launch and events[i] after the i-th kernel launch (i = 1 .. n_events - 1;
 * later launches record nothing).  events[] are caller-created cudaEvent_t
 * handles.  The launch order is the one sfa_grad_plan_info describes.
 */
sfa_status sfa_grad_profile(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                            const void* d_out, const void* out, const float* softmax_max, const float* softmax_sum,
                            const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope,
                            const void* k_rope, void* dq, void* dk, void* dv, void* dq_rope, void* dk_rope,
                            void* workspace, size_t workspace_bytes, void* stream, void** events, int32_t n_events);

/*
 * Static plan of one sfa_grad call: *chunk_tokens = query tokens processed
 * per chunk of the staging buffers, *kernel_launches = number of kernels the
 * call launches, in the order sfa_grad_plan_names lists them.  Either output
 * pointer may be null.
 */
sfa_status sfa_grad_plan_info(const sfa_params* p, int64_t* chunk_tokens, int64_t* kernel_launches);

/*
 * Names of the kernels one sfa_grad call launches, in launch order (the
 * intervals the events of sfa_grad_profile delimit): "batch_prefix" (TND),
 * "meta", "dsum", then per token chunk either
 *   "rowtab", "sdp", "kvq" (row table of the chunk's slots, scores per token,
 *   then combined key-side and query-side contractions), or
 *   "blk_count", "blk_scan", "blk_scatter", "sdpb", "kvb", "dqb" (block-sparse
 *   indices whose blocks many tokens select: pairs grouped by block start,
 *   scores per block for packs of its tokens, key side accumulated per block,
 *   then dQ per token with the features on the MMA's rows; with
 *   deterministic = 1 the grouping is followed by "blk_sort" and
 *   "blk_sort_long", each group's pairs in ascending (token, index) order
 *   (groups of up to 1024 pairs, then longer ones), and "kvb" is launched
 *   sparse_block_size times, once per block-start residue modulo the block
 *   size), or
 *   with deterministic = 1 and single-key or rarely shared indices "rowtab",
 *   "sdp", "det_count", "det_scan", "det_scatter", "det_sort",
 *   "det_sort_long" (entries sorted by kv row, then token and slot), "kvq"
 *   (the key side stored as per-pair partial rows, with the query side),
 *   "det_reduce";
 * finally "cast".  Writes at most `capacity` pointers to static strings into
 * names[] (names may be null when capacity is 0) and the total count into
 * *count (may be null).  Host only; validates *p like
 * sfa_grad_workspace_size.
 */
sfa_status sfa_grad_plan_names(const sfa_params* p, const char** names, int32_t capacity, int32_t* count);

/*
 * Companion forward that produces the backward's saved inputs (the page lists
 * out, softmaxMax and softmaxSum as inputs of the backward; it does not
 * specify the forward).  out = sum_j P_j v_j with P and the statistics defined
 * as above; a row with no valid key gets out = 0, softmaxMax = -inf,
 * softmaxSum = 0.  Same conventions, shapes and error codes as sfa_grad
 * (p->deterministic is ignored: the forward is always deterministic).  The
 * keys are scored once: P is formed relative to the max of each group of 32
 * selected slots (or of each selected block) and rescaled to the final
 * statistics in the input type, so each P entry carries up to three roundings
 * to the input type before the P.V product (accumulated in fp32); the
 * statistics are fp32.
 */
sfa_status sfa_fwd_workspace_size(const sfa_params* p, size_t* bytes);
sfa_status sfa_fwd(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                   const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope, const void* k_rope,
                   void* out, float* softmax_max, float* softmax_sum, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * Index decode as the kernels see it (功能说明 gather with block expansion,
 * Mask table for sparseMode 3): writes, for every query token t and every
 * expanded slot s < K * sparse_block_size, the global kv row the slot reads
 * (BSND: b * S2 + key; TND: kv segment start + key) or -1 when the slot is
 * masked.  rows_out: device int32 (T1, K * sparse_block_size).  Needs the same
 * workspace as sfa_grad.
 */
sfa_status sfa_decode_keys(const sfa_params* p, const int32_t* indices, const int32_t* act_seq_q,
                           const int32_t* act_seq_kv, int32_t* rows_out, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Synchronises `stream` and copies the workspace error word (SFA_DEVERR_*) to
 * *code, then clears it.  Returns SFA_ERR_RUNTIME if the copy fails.
 */
sfa_status sfa_read_device_error(void* workspace, void* stream, int32_t* code);

/*
 * Allocation-free backward, for callers that cannot allocate device memory:
 * for example a plugin whose host framework's memory pool owns the whole
 * device, code running while a stream is captured into a CUDA graph, or a
 * path that must not risk the device-wide synchronisation cudaMalloc/cudaFree
 * can cause.  (The pages have no counterpart: their second phase always takes
 * a caller-allocated workspace.)
 *
 * Same arguments and results as sfa_grad without the workspace: the scratch
 * is a static device array of SFA_NOALLOC_SCRATCH_BYTES inside the library,
 * held by every GPU that loads the library until the process exits.  Problems
 * whose sfa_grad_workspace_size exceeds it are rejected with SFA_ERR_SHAPE
 * (detail in sfa_last_error_message).  The first call on a device looks up
 * the array's device address; make that first call before any stream
 * capture.  The looked-up address belongs to the device's context, so the
 * library must not be used across cudaDeviceReset.  All calls share the
 * array: calls whose GPU work overlaps (other streams or threads) race and
 * must be serialised by the caller.  Calls no cudaMalloc/cudaFree or
 * allocating routine.  Device-side problems (SFA_DEVERR_*) are recorded in the
 * scratch; read them with sfa_noalloc_read_device_error.
 */
#define SFA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
sfa_status sfa_grad_noalloc(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                            const void* d_out, const void* out, const float* softmax_max, const float* softmax_sum,
                            const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope,
                            const void* k_rope, void* dq, void* dk, void* dv, void* dq_rope, void* dk_rope,
                            void* stream);

/*
 * The device error word of sfa_grad_noalloc's static scratch on the current
 * device: synchronises `stream`, copies the word (SFA_DEVERR_*) to *code and
 * clears it, like sfa_read_device_error does for a caller's workspace.  Call
 * it on the stream of the noalloc calls it should cover.  Returns
 * SFA_ERR_NULLPTR for a null code and SFA_ERR_RUNTIME (with
 * sfa_last_error_message) when the device or the scratch address cannot be
 * determined or the copy fails.  (No counterpart on the pages.)
 */
sfa_status sfa_noalloc_read_device_error(void* stream, int32_t* code);

/*
 * sfa_grad from host buffers, with the copies overlapped with the kernels.
 * Same arguments, shapes and results as sfa_grad, except that every tensor
 * argument (the inputs, act_seq_q / act_seq_kv and the five outputs) is a
 * HOST pointer.  Page-locked (pinned) memory makes the copies asynchronous so
 * that they overlap the kernels; pageable memory works, but its copies are
 * synchronous.  `workspace` is a DEVICE buffer of at least
 * sfa_grad_host_workspace_size bytes (256-byte aligned, caller-owned): the
 * backward's workspace followed by device copies of the inputs and outputs.
 *
 * The call splits the query tokens into chunks: the first of 128 tokens,
 * each next one larger by a factor estimated from the shape (how much longer
 * a token's kernels run than its inputs take to copy, 1.25 to 8, e.g. 1.25
 * for MLA), and halving again towards the end.  On two streams it creates,
 * it copies k, v, kRope and the lengths, then each chunk's query-side rows
 * (q, qRope, dOut, out, softmaxMax, softmaxSum, indices) to the device, one
 * chunk ahead of the kernels.  Chunk c's kernels start when its rows have
 * landed, and its dQ / dQRope rows are copied back while chunk c + 1
 * computes; dK / dV / dKRope follow the final cast.  All of it is
 * ordered after earlier work on `stream`, and `stream` waits for the last
 * copy: the host outputs are complete, and the host inputs free, once
 * `stream` has been synchronised.  The two streams and the events are
 * released at the end of the call (the runtime frees them once their work is
 * done); not for use while `stream` is being captured into a graph.  With
 * deterministic = 1 the outputs are bitwise reproducible from call to call;
 * their last bits can differ from sfa_grad's, whose token chunks may be
 * larger (the fixed order of the key-side sums is chunk, token, slot).
 * Errors: those of sfa_grad (the workspace size is checked against
 * sfa_grad_host_workspace_size).  When an error is returned after copies
 * were queued, the call first waits for them, so none still reads or writes
 * the caller's host buffers.
 */
sfa_status sfa_grad_host_workspace_size(const sfa_params* p, size_t* bytes);
sfa_status sfa_grad_host(const sfa_params* p, const void* q, const void* k, const void* v, const int32_t* indices,
                         const void* d_out, const void* out, const float* softmax_max, const float* softmax_sum,
                         const int32_t* act_seq_q, const int32_t* act_seq_kv, const void* q_rope, const void* k_rope,
                         void* dq, void* dk, void* dv, void* dq_rope, void* dk_rope, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Human-readable detail of the most recent SFA_ERR_RUNTIME returned on the
 * calling thread (the failing CUDA call's error text and location), or of a
 * size rejection by sfa_grad_noalloc; empty if none.  The pointer stays valid
 * until the thread's next library call.
 */
const char* sfa_last_error_message(void);

/* Static description of a status code. */
const char* sfa_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* SFA_GRAD_H_ */
