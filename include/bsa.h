/*
 * bsa.h - C ABI of libbsa: block-sparse attention backward (and its companion
 * forward) on NVIDIA GB300 (sm_103a).
 *
 * The interface follows the two-stage call of the aclnnBlockSparseAttentionGrad
 * page ("CANN/ops-transformer块稀疏注意力梯度算子", section 函数原型, function
 * prototype): a first call checks the arguments and returns the workspace size
 * and an executor, a second call runs the computation on a stream. Argument
 * names, order and meaning follow that page's parameter table (section 参数说明);
 * status codes follow its return-code table (section 返回值).
 *
 * Conventions shared by every call:
 *   - Tensors are described by bsa_tensor: a DEVICE pointer plus dtype, shape
 *     and strides (in elements). The library never takes ownership of them; the
 *     caller keeps them alive until the stream has finished the run call.
 *   - Integer arrays (block shape, sequence lengths) are HOST memory, read and
 *     copied during the first-stage call; the caller may free them afterwards.
 *   - Executors are host objects. A run call (bsa_grad / bsa_fwd) consumes and
 *     frees its executor whether it succeeds or not; bsa_executor_destroy frees
 *     one that will never be run.
 *   - Run calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream). Device-side failures (a bounded wait that gave up) are
 *     recorded in the workspace and reported by bsa_check_status.
 *   - Every call returns a bsa_status; on failure bsa_last_error() returns a
 *     one-line explanation (thread-local, valid until the next call).
 *   - No call allocates device memory: scratch lives in the caller's workspace
 *     (bsa_mask_compact_noalloc: in an array built into the library).
 */
#ifndef BSA_H_
#define BSA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes (page: 返回值 table; 361001/561002 as on the aclnn return-code
 * list used by the related CompressorGrad page, section 返回值). */
typedef enum {
  BSA_OK = 0,
  BSA_ERR_PARAM_NULLPTR = 161001, /* a required pointer is NULL                      */
  BSA_ERR_PARAM_INVALID = 161002, /* dtype, layout, shape or value not supported    */
  BSA_ERR_RUNTIME = 361001,       /* a CUDA call or kernel launch failed            */
  BSA_ERR_INNER = 561002          /* a kernel recorded an internal failure          */
} bsa_status;

/* Element types. Inputs/outputs are F16 or BF16, softmaxLse is F32, the block
 * mask is one byte per block (BOOL or UINT8: nonzero = the block takes part). */
typedef enum { BSA_F16 = 1, BSA_BF16 = 2, BSA_F32 = 3, BSA_U8 = 4 } bsa_dtype;

typedef struct {
  void* data;        /* device pointer, 16-byte aligned for q/k/v/dout        */
  int32_t dtype;     /* bsa_dtype                                              */
  int32_t ndim;      /* 1..4                                                   */
  int64_t shape[4];  /* first ndim entries used                                */
  int64_t stride[4]; /* in elements; first ndim entries used                   */
} bsa_tensor;

typedef struct bsa_executor bsa_executor; /* opaque, host side */

/* bsa_grad_workspace_size - first stage of the backward.
 * Page: aclnnBlockSparseAttentionGradGetWorkspaceSize, parameter table and
 * formulas (计算公式): D = rowsum(dout*attentionOut), dP = dout*V^T,
 * dS = P*(dP - D), dV = P^T*dout, dQ = scale*dS*K, dK = scale*dS^T*Q with
 * P = exp(scale*Q*K^T - softmaxLse) recomputed on the selected blocks only.
 *
 *   dout, query, attention_out : [B,N1,Sq,D] (q_layout "BNSD") or [Tq,N1,D]
 *                                ("TND"); F16/BF16, all one dtype, contiguous.
 *   key, value                 : [B,N2,Skv,D] or [Tkv,N2,D]; same dtype, contiguous.
 *   softmax_lse                : F32, [B,N1,Sq,1] / [B,N1,Sq] or [Tq,N1,1] /
 *                                [Tq,N1]; natural-log logsumexp of the scaled
 *                                scores of each query row, used as given.
 *   block_sparse_mask          : one byte per block, [B,N1,ceil(Sq/bx),ceil(Skv/by)]
 *                                (TND: Sq/Skv = the longest sequence), contiguous.
 *                                NULL = every token pair takes part (dense);
 *                                the block shape is then ignored. Bits of blocks
 *                                that start at or beyond a sequence's actual
 *                                length are ignored.
 *   atten_mask                 : token mask, the atten_mask of the formula
 *                                S = Mask(scale*Q*K^T, atten_mask) (parameter table
 *                                row attenMaskOptional; polarity as on the
 *                                FlashAttentionScore page: nonzero = the pair is
 *                                masked out). NULL = none. Otherwise a 2-D
 *                                BOOL/UINT8 device matrix of at least [maxSq, maxSkv]
 *                                rows x columns, any positive strides, shared by
 *                                every batch and head and indexed by the query /
 *                                key positions counted from each sequence's start.
 *   block_shape, block_shape_len : host int64 [bx, by, ...]; NULL or len 0 =
 *                                {128, 128}; at least 2 entries, extra entries are
 *                                ignored. The library supports bx, by in {64, 128}.
 *   actual_seq_lengths(_kv), n_seq(_kv) : host int64 per-batch valid token counts.
 *                                Required for TND (sum must equal Tq/Tkv);
 *                                optional for BNSD (NULL = Sq/Skv; rows past the
 *                                length are padding: ignored on input, 0 on output).
 *   q_layout, kv_layout        : "BNSD" or "TND"; must be equal.
 *   num_key_value_heads        : N2; N1 % N2 == 0; query head h uses key head
 *                                h / (N1/N2), and dK/dV sum over the group.
 *   mask_type                  : 0 = no token mask (atten_mask NULL); 1 = apply
 *                                atten_mask. Other values are rejected.
 *   pre_tokens, next_tokens    : sliding window (parameter table rows preTokens /
 *                                nextTokens; window edges as on the
 *                                FlashAttentionScore page, 参数说明): query s and
 *                                key t of one sequence, both counted from that
 *                                sequence's first token, take part only if
 *                                s - pre_tokens <= t <= s + next_tokens (on top of
 *                                the block mask). 2147483647 for both = no window;
 *                                next_tokens = 0 = causal (top-left aligned).
 *                                pre_tokens + next_tokens must be >= 0.
 *   scale_value                : the scale (typically D^-0.5).
 *   dq, dk, dv                 : outputs with the shapes of query/key/value, same
 *                                dtype; any strides (non-contiguous allowed).
 *   D (head dim) must be 64 or 128.
 *   workspace_size, executor   : out. The workspace must be device memory of at
 *                                least *workspace_size bytes, 256-byte aligned.
 * Returns 161001 for a NULL required pointer (or TND without sequence lengths),
 * 161002 for anything else unsupported, BSA_OK otherwise. */
bsa_status bsa_grad_workspace_size(
    const bsa_tensor* dout, const bsa_tensor* query, const bsa_tensor* key,
    const bsa_tensor* value, const bsa_tensor* attention_out, const bsa_tensor* softmax_lse,
    const bsa_tensor* block_sparse_mask, const bsa_tensor* atten_mask,
    const int64_t* block_shape, int64_t block_shape_len,
    const int64_t* actual_seq_lengths, int64_t n_seq,
    const int64_t* actual_seq_lengths_kv, int64_t n_seq_kv,
    const char* q_layout, const char* kv_layout, int64_t num_key_value_heads,
    int64_t mask_type, double scale_value, int64_t pre_tokens, int64_t next_tokens,
    const bsa_tensor* dq, const bsa_tensor* dk, const bsa_tensor* dv,
    uint64_t* workspace_size, bsa_executor** executor);

/* bsa_grad - second stage of the backward (page: aclnnBlockSparseAttentionGrad).
 * Launches, on `stream`: mask compaction, the D/lse preprocess, the tcgen05
 * backward kernel, and the dQ/dK/dV finalize kernels. Consumes the executor.
 * Returns 161001 if workspace/executor is NULL, 161002 if workspace_size is
 * smaller than required, 361001 if a launch fails. */
bsa_status bsa_grad(void* workspace, uint64_t workspace_size, bsa_executor* executor,
                    void* stream);

/* bsa_fwd_workspace_size / bsa_fwd - companion forward: Out = softmax(scale*Q*K^T
 * over the selected blocks) * V and softmaxLse = natural-log logsumexp of the
 * scaled selected scores (page formulas 计算公式, forward part; online-softmax
 * update as in the FlashAttentionScore page, section 实现原理). Arguments as in
 * bsa_grad_workspace_size (atten_mask / mask_type and pre_tokens / next_tokens:
 * the same token mask and sliding window). Query rows with no selected key that
 * the window and the token mask keep (and BNSD padding rows)
 * get Out = 0 and lse = -inf. Out has the dtype of query, lse is F32. */
bsa_status bsa_fwd_workspace_size(
    const bsa_tensor* query, const bsa_tensor* key, const bsa_tensor* value,
    const bsa_tensor* block_sparse_mask, const bsa_tensor* atten_mask,
    const int64_t* block_shape, int64_t block_shape_len,
    const int64_t* actual_seq_lengths, int64_t n_seq,
    const int64_t* actual_seq_lengths_kv, int64_t n_seq_kv,
    const char* q_layout, const char* kv_layout, int64_t num_key_value_heads,
    int64_t mask_type, double scale_value, int64_t pre_tokens, int64_t next_tokens,
    const bsa_tensor* attention_out, const bsa_tensor* softmax_lse,
    uint64_t* workspace_size, bsa_executor** executor);

bsa_status bsa_fwd(void* workspace, uint64_t workspace_size, bsa_executor* executor,
                   void* stream);

/* Measurement hook (the pages have no counterpart): asks the run call of
 * `executor` to record `event_before` on its stream just before the main
 * tensor-core kernel (backward or forward) and `event_after` just after it.
 * Both are caller-created cudaEvent_t handles (NULL = do not record). */
bsa_status bsa_executor_set_timing_events(bsa_executor* executor, void* event_before,
                                          void* event_after);

/* Test of the failure path (the pages have no counterpart): with enable != 0 the
 * backward kernel of this executor's run waits once on a barrier nothing
 * completes. The wait gives up after its bound (about 1 s), every warp unwinds,
 * the run's outputs are invalid and bsa_check_status returns 561002; the CUDA
 * context stays usable. Backward executors only. */
bsa_status bsa_executor_set_wait_test(bsa_executor* executor, int32_t enable);

/* Deterministic dQ (backward executors only). With enable != 0 the run
 * computes dQ in a separate query-tile pass: every query tile walks its
 * selected key tiles in ascending order and accumulates dS*K in the tensor
 * memory of one CTA, so dQ, dK and dV are bitwise identical from run to run
 * (the default path sums dQ with fp32 reduce-adds whose order varies, so only
 * its rounding differs between runs). Costs about 40 % more tensor-core work
 * (S and dP are computed twice) and no fp32 dQ accumulator traffic.
 * Determinism as a documented property of a backward op: the CompressorGrad
 * page, section 确定性计算; pairing with PyTorch: the
 * aclnnBlockSparseAttentionGrad page, section 约束说明. */
bsa_status bsa_executor_set_deterministic(bsa_executor* executor, int32_t enable);

/* Key blocks of 64 tokens (backward executors only). With enable != 0, a run
 * whose blockShape is [bx, 64] with head dim 128 and neither sliding window nor
 * token mask computes the five products of every selected 64-key block as one
 * query-major step (S = Q K_h^T with N = 64 keys; dV_h^T, dK_h^T accumulated
 * with the head dimension on the tensor-memory lanes), one pass per key block
 * of a 128-key tile, so an unselected half of a tile is never loaded or
 * multiplied: the tensor-core work equals the algorithmic work (blockShape row
 * of the aclnnBlockSparseAttentionGrad parameter table: bx and by need not be
 * equal). Off by default: 64-wide products run at a lower rate per FLOP on
 * the tensor cores and every block sends its own dQ partial, so on GB300 the
 * default path (128 x 128 tiles with the unselected half masked) is faster
 * even when most tiles hold only one selected block. Ignored when the run does
 * not meet the conditions above; results equal the default path's up to
 * rounding order. */
bsa_status bsa_executor_set_key_block64(bsa_executor* executor, int32_t enable);

/* Frees an executor that was never passed to a run call. NULL is a no-op. */
bsa_status bsa_executor_destroy(bsa_executor* executor);

/* bsa_mask_compact_workspace_size / bsa_mask_compact - the compaction step on
 * its own (page: blockSparseMaskOptional row of the parameter table). For each
 * (b, h) (slot b*N+h): CSR row_ptr [B*N*(Mq+1)] + col_idx (selected key blocks
 * of each query block, ascending) and CSC col_ptr [B*N*(Mk+1)] + row_idx
 * (query blocks selecting each key block, ascending). Pointers use one global
 * numbering (slot s starts at the nnz of slots < s). Blocks that start at or
 * beyond the per-batch lengths (host int64 arrays, NULL = the full Mq*bx /
 * Mk*by) are dropped. All four outputs are int32 DEVICE arrays; col_idx and
 * row_idx must hold B*N*Mq*Mk entries (the dense bound). */
bsa_status bsa_mask_compact_workspace_size(const bsa_tensor* block_sparse_mask, int64_t bx,
                                           int64_t by, uint64_t* workspace_size);
bsa_status bsa_mask_compact(const bsa_tensor* block_sparse_mask, int64_t bx, int64_t by,
                            const int64_t* actual_seq_lengths, int64_t n_seq,
                            const int64_t* actual_seq_lengths_kv, int64_t n_seq_kv,
                            int32_t* row_ptr, int32_t* col_idx, int32_t* col_ptr,
                            int32_t* row_idx, void* workspace, uint64_t workspace_size,
                            void* stream);

/* bsa_mask_compact_noalloc - the compaction of bsa_mask_compact for callers that
 * cannot allocate device memory (a caller-owned pool that forbids new
 * allocations, an embedded runtime without a device allocator, a fixed memory
 * budget). The pages have no counterpart of this call. Same arguments and
 * outputs as bsa_mask_compact minus the workspace: the scratch is a 4 MiB array
 * built into the library (held by every GPU that loads it until exit); the call
 * allocates no device memory. Rejects with 161002 masks whose scratch
 * (4*(2*B + B*N*(Mq+1) + B*N*(Mk+1)) bytes, each part rounded up to 256) does not
 * fit, and B > 1024. All calls share the array and it keeps the last call's
 * contents: calls that overlap on the GPU race. The first call on a device
 * looks up the array's address (with that device current); make it before any
 * stream capture. The lookup is repeated when the device's context has
 * changed (e.g. after cudaDeviceReset). The sequence lengths travel as kernel
 * parameters, so the host arrays may be reused once the call returns.
 * Asynchronous on `stream`. */
bsa_status bsa_mask_compact_noalloc(const bsa_tensor* block_sparse_mask, int64_t bx, int64_t by,
                                    const int64_t* actual_seq_lengths, int64_t n_seq,
                                    const int64_t* actual_seq_lengths_kv, int64_t n_seq_kv,
                                    int32_t* row_ptr, int32_t* col_idx, int32_t* col_ptr,
                                    int32_t* row_idx, void* stream);

/* Synchronizes `stream`, then reads the error word a run call left at the start
 * of `workspace`: BSA_OK, or BSA_ERR_INNER if a kernel gave up a bounded wait
 * (the outputs are then not valid). 361001 if the CUDA calls fail.
 * Bounds-check build (the same ABI, libbsa_checks.so, kernels compiled with
 * BSA_CHECKS=1): the kernels also validate the work items and list entries they
 * read; an index outside its array is dropped and reported here as
 * BSA_ERR_INNER with code 13 in word 6 and the id of the failed check in word 9
 * (1 work item, 2 list entry, 3 item position, 4 entry position, 5 finalize
 * tile). In that variant only, the environment switch BSA_CHECK_TEST=1 makes the
 * next bsa_grad plant one out-of-range entry (the test of these checks).
 * Logging (the pages' call example logs through LOG_PRINT; here an environment
 * switch): with BSA_LOG set to anything but "0", this call prints the backward
 * work-list counts of the workspace (active tiles, work items, split columns),
 * bsa_grad_workspace_size the plan and bsa_grad the kernels and dQ mode it
 * launches, one line each on stderr. */
bsa_status bsa_check_status(const void* workspace, void* stream);

/* The same error words without a host synchronization: enqueues on `stream` a
 * copy of the first 8 int32 words of `workspace` into `host_words` (caller-owned
 * host memory of at least 32 bytes; page-locked memory keeps the copy
 * asynchronous). Once the stream has passed the copy, host_words[0] != 0 means
 * a kernel of the preceding run gave up a bounded wait (host_words[6] holds the
 * code of the first failed wait). 161001 for NULL pointers, 361001 if the copy
 * cannot be enqueued. */
bsa_status bsa_status_async(const void* workspace, int32_t* host_words, void* stream);

/* One-line description of the last failure in this thread ("" if none). */
const char* bsa_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int32_t bsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H_ */
