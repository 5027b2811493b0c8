/*
 * bdlm.h - C ABI of the GB300 (sm_103a) BDLM attention library.
 *
 * The library computes core attention softmax(QK^T)V ("Efficient Long-context
 * Language Model Training by Core Attention Disaggregation", abstract), its
 * backward, and the log-sum-exp merge of partial results, under the mask of
 * block diffusion LM training ("Block Parallelism For Efficient Distributed
 * Long-Context Diffusion Language Model Training", abstract; rit.work CSBP
 * post, first section):
 *
 *   each sequence is [clean n rows | corrupted n rows], cut into blocks of B;
 *   a clean row of block b sees the clean rows of blocks <= b;
 *   a corrupted row of block b sees the clean rows of blocks < b and every
 *   corrupted row of its own block b; clean rows never see corrupted rows.
 *
 * Conventions shared by every call
 *   - Tensors are dense, row-major, 16-byte aligned device buffers:
 *       q, o, dO, dq : bf16 [Lq, H, d]       k, v, dk, dv : bf16 [Lk, Hk, d]
 *       lse          : fp32 [H, Lq]          (natural log of sum_j exp(scale*q.k_j))
 *   - Query head h reads kv head h / (H / Hk).
 *   - d is 64 or 128; H % Hk == 0; 1 <= B <= 1024; every document's clean
 *     length n is positive. Blocks are cut from the start of each half, so
 *     when B does not divide n the last block of each half holds n mod B rows
 *     (a BLOCK_GROUP call still gives that block B rows: see bdlm_partial).
 *   - The caller owns every buffer, including the workspace. The library never
 *     allocates or frees device memory and never synchronises, except in
 *     bdlm_read_error. Every call is asynchronous on `stream` (NULL = the
 *     legacy default stream) and runs on the current CUDA device.
 *   - Arguments that can be checked on the host are checked before any launch;
 *     on failure the call returns a status and launches nothing. Problems found
 *     on the device (a malformed cu_seqlens, a wait that timed out) are written
 *     to an error word inside the workspace, read with bdlm_read_error.
 *   - Not thread-safe per workspace: two calls that share a workspace must be
 *     ordered on one stream.
 *   - The compute calls (forward, backward, merge, task lists) only launch
 *     kernels on `stream`, with every host-side value (task records, partial
 *     pointer lists, tensor maps) in kernel parameters, so they can be
 *     captured into a CUDA graph and replayed on new contents of the same
 *     buffers. (bdlm_read_error synchronises and cannot be captured.)
 */
#ifndef BDLM_H
#define BDLM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BDLM_API __attribute__((visibility("default")))
#else
#define BDLM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bdlm_stream_t; /* the same type as cudaStream_t */

enum bdlm_status {
    BDLM_OK = 0,
    BDLM_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned buffer       */
    BDLM_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d = 96)         */
    BDLM_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required      */
    BDLM_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed               */
    BDLM_ERR_TIMEOUT = 5,      /* device: a bounded wait ran out                  */
    BDLM_ERR_DEVICE_CHECK = 6  /* device: cu_seqlens or block list is malformed   */
};

enum bdlm_dtype { BDLM_BF16 = 0, BDLM_F32 = 1 };

enum bdlm_part_kind {
    BDLM_PART_NONE = 0,        /* full BDLM attention                             */
    BDLM_PART_KEY_WINDOW = 1,  /* keys restricted to one contiguous window        */
    BDLM_PART_BLOCK_GROUP = 2  /* queries restricted to a list of corrupted blocks*/
};

enum bdlm_part_flags {
    BDLM_PART_ACCUMULATE = 1   /* KEY_WINDOW forward: merge into the running o, lse */
};

/*
 * Restriction of one call (single sequence only; cu_seqlens == NULL).
 *
 * BDLM_PART_KEY_WINDOW - partial attention against one shard of the keys, as
 *   each rank computes it under context-sharded block parallelism (Block
 *   Parallelism abstract; rit.work CSBP post, CSBP paragraph). k and v hold
 *   exactly the keys at sequence positions [key_lo, key_hi) (Lk = key_hi -
 *   key_lo rows); q holds all L rows. A clean shard is a window inside [0, n);
 *   the local corrupted keys are the window [n, 2n). Query rows with no visible
 *   key in the window get o = 0 and lse = -inf.
 *
 * BDLM_PART_BLOCK_GROUP - the corrupted target blocks owned by one rank under
 *   block parallelism (rit.work CSBP post, block-parallelism paragraph). q
 *   holds the corrupted rows of the listed blocks, B rows each, in list order
 *   (Lq = n_q_blocks * B). k and v hold the n clean rows followed by the same
 *   blocks' corrupted rows in the same order (Lk = n + n_q_blocks * B).
 *   q_blocks is a DEVICE array of distinct block ids in [0, ceil(n / B)).
 *   When B does not divide n, the last block (id ceil(n / B) - 1) holds
 *   n mod B rows; listed, it still takes B rows of q (and of k, v), and the
 *   rows past the half's end are padding: they see no key, no row sees them,
 *   their o is 0, lse -inf and their gradients 0. Fill them with finite
 *   values (zeros), since masked products still read them.
 *
 * flags (forward only):
 *   BDLM_PART_ACCUMULATE - KEY_WINDOW only. o and lse already hold the merged
 *   result of earlier windows of the same query rows (disjoint key sets), and
 *   this call merges its window into them in place with log-sum-exp weights,
 *   in fp32 ("Block Parallelism ..." abstract: sharding the clean sequence
 *   keeps the result; rit.work CSBP post, CSBP paragraph): lse = ln(e^lse +
 *   e^lse_w), o = (e^lse o + e^lse_w o_w) / (e^lse + e^lse_w). Rows that see no
 *   key of the window are left unchanged; rows whose running lse is -inf take
 *   the window's result (their o is not read). The first window of a sequence
 *   is an ordinary call without the flag. This replaces storing every window's
 *   partial and one bdlm_lse_merge call.
 * q_lo, q_hi (KEY_WINDOW only): a token-level task (Core Attention
 *   Disaggregation abstract: attention over token-level shards). q, o, lse
 *   (and for the backward dO, dq) hold only the rows at sequence positions
 *   [q_lo, q_hi), Lq = q_hi - q_lo, e.g. one rank's own rows against one
 *   gathered clean shard; q_hi = 0 selects all L rows. The backward's dk, dv
 *   are then the window keys' gradients from these rows only.
 * o_dtype: BDLM_BF16 (0, default) or BDLM_F32 - the element type of o for a
 *   KEY_WINDOW or BLOCK_GROUP forward (fp32 keeps a running merge from being
 *   rounded at every window). Full attention and the backward take bf16 o.
 */
typedef struct {
    int32_t kind;            /* enum bdlm_part_kind                               */
    int32_t n_q_blocks;      /* BLOCK_GROUP: number of listed blocks              */
    int64_t key_lo, key_hi;  /* KEY_WINDOW: sequence positions, 0<=lo<hi<=L       */
    const int32_t* q_blocks; /* BLOCK_GROUP: device int32 [n_q_blocks]            */
    int32_t flags;           /* enum bdlm_part_flags (0 = none)                   */
    int32_t o_dtype;         /* enum bdlm_dtype of o (forward partials)           */
    int64_t q_lo, q_hi;      /* KEY_WINDOW: q holds positions [q_lo, q_hi); 0,0 = all L rows */
} bdlm_partial;

/* Workspace sizes (bytes) for one call with L query rows, H heads, head dim d
 * and n_docs packed documents (1 for a single sequence). Returns 0 for sizes
 * the library does not support. The workspace must be 256-byte aligned. */
BDLM_API size_t bdlm_attn_fwd_workspace_bytes(int64_t L, int32_t heads, int32_t head_dim, int32_t n_docs);
BDLM_API size_t bdlm_attn_bwd_workspace_bytes(int64_t L, int32_t heads, int32_t head_dim, int32_t n_docs);

/*
 * Forward: o = softmax(scale * q k^T under the BDLM mask) v, lse per row.
 *
 *   L          rows of the full concatenation: 2n for one sequence, or
 *              cu_seqlens[n_docs] for packed documents (each document is
 *              [clean n_d | corrupted n_d]). With BLOCK_GROUP, L = 2n still
 *              names the sequence and q holds only the group's rows.
 *   block      B, the diffusion block size.
 *   cu_seqlens NULL for one sequence, else a DEVICE int32 [n_docs + 1] of
 *              document offsets (0, ..., L); checked on the device
 *              (BDLM_ERR_DEVICE_CHECK through bdlm_read_error).
 *   softmax_scale  <= 0 selects 1/sqrt(d).
 *   part       NULL or kind NONE for full attention; see bdlm_partial.
 *   workspace  >= bdlm_attn_fwd_workspace_bytes(L, heads, head_dim, n_docs).
 * Writes o [Lq, H, d] bf16 and lse [H, Lq] fp32.
 */
BDLM_API int bdlm_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                  int64_t L, int32_t block, int32_t heads, int32_t kv_heads, int32_t head_dim,
                  const int32_t* cu_seqlens, int32_t n_docs, float softmax_scale,
                  const bdlm_partial* part, void* workspace, size_t workspace_bytes,
                  bdlm_stream_t stream);

/*
 * bdlm_attn_fwd_noalloc - the forward for callers that cannot allocate device
 * memory where they call it: plugins whose host framework owns every device
 * allocation, services that forbid allocation after start-up. (The paper has
 * no counterpart; this is a library convenience.)
 *
 * Same arguments and results as bdlm_attn_fwd, minus the workspace: the
 * forward's scratch (tile table, work counter, device error word) lives in a
 * fixed 4 MiB array inside the library, which every GPU that loads the
 * library holds until the process exits. That bounds the call size: when
 * bdlm_attn_fwd_workspace_bytes(L, heads, head_dim, n_docs) exceeds 4 MiB
 * (about 2.5 million rows for one sequence) the call returns
 * BDLM_ERR_WORKSPACE and launches nothing; use bdlm_attn_fwd then.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current). The address is kept together with the
 * CUDA context it belongs to and looked up again when the device's current
 * context changes (e.g. after cudaDeviceReset).
 * Every call on a device shares the one array and each call clears the parts
 * that must start at zero; calls whose execution overlaps on the GPU (other
 * streams, or other host threads) race on it, so order them.
 * Device-detected errors (a malformed cu_seqlens or block list, a wait that
 * timed out) land in the shared array, where they leave o and lse unwritten;
 * bdlm_read_error(NULL, stream) returns the error word of the last call on
 * the current device.
 */
BDLM_API int bdlm_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                  int64_t L, int32_t block, int32_t heads, int32_t kv_heads, int32_t head_dim,
                  const int32_t* cu_seqlens, int32_t n_docs, float softmax_scale,
                  const bdlm_partial* part, bdlm_stream_t stream);

/*
 * Token-level task lists ("Efficient Long-context Language Model Training by
 * Core Attention Disaggregation", abstract: core attention is stateless and
 * composes over fused batches of token-level shards of arbitrary lengths).
 *
 * A task is the query rows at positions [q_lo, q_hi) of one sequence against
 * that sequence's keys at positions [key_lo, key_hi), under the sequence's
 * BDLM mask. The sequence is [clean n | corrupted n] at rows [seq_start,
 * seq_start + 2n) of q, k and v, which hold all L rows. The tasks of one list
 * may come from different sequences of different lengths (B need not divide
 * n) and may cut one sequence's rows and keys in any way.
 */
typedef struct {
    int64_t seq_start;       /* first row of the task's sequence in q, k, v       */
    int64_t n;               /* its clean length: rows [seq_start, seq_start + 2n) */
    int64_t q_lo, q_hi;      /* query positions, 0 <= q_lo < q_hi <= 2n            */
    int64_t key_lo, key_hi;  /* key positions, 0 <= key_lo < key_hi <= 2n          */
    int32_t slot;            /* output slot, 0 <= slot < n_slots                   */
    int32_t reserved;        /* must be 0                                          */
} bdlm_task;

/* Workspace (bytes, 256-byte aligned) of a task-list forward over this HOST
 * task array; 0 if n_tasks is outside [1, 65536] or a task has an empty or
 * negative query range or a non-positive n. */
BDLM_API size_t bdlm_attn_fwd_tasks_workspace_bytes(const bdlm_task* tasks, int32_t n_tasks);

/*
 * bdlm_attn_fwd_tasks - the partial forward of every task of a list, in one
 * attention launch (after a prologue that takes the tasks to the device as
 * kernel parameters and orders their tiles: heaviest first, and among tiles
 * of equal cost earlier tasks first).
 *
 *   q, k, v    bf16 [L, H, d], [L, Hk, d]: every row.
 *   o          n_slots consecutive [L, H, d] arrays of o_dtype (BDLM_BF16 or
 *              BDLM_F32).
 *   lse        n_slots consecutive fp32 [H, L] arrays.
 *   tasks      HOST array of n_tasks tasks (1 .. 65536), read during the call;
 *              it may be reused or freed when the call returns.
 *   n_slots    1 .. 1024.
 *   workspace  >= bdlm_attn_fwd_tasks_workspace_bytes(tasks, n_tasks).
 *
 * Task t writes o[slot_t] and lse[slot_t] at rows seq_start + [q_lo, q_hi):
 * the partial result of those rows against the task's keys (o = 0 and
 * lse = -inf for rows that see none of them). Rows that no task of a slot
 * covers are left as they were. Tasks that split one row's keys go to
 * different slots, and bdlm_lse_merge over the slots (with lse = -inf set
 * beforehand where a slot has no task) combines them. Tasks of one slot must
 * not share query rows, since they would write the same outputs: such a list
 * returns BDLM_ERR_INVALID_ARG, as does a task whose sequence does not lie in
 * [0, L), whose ranges break the bounds above, or whose reserved field is not
 * 0.
 */
BDLM_API int bdlm_attn_fwd_tasks(const void* q, const void* k, const void* v, void* o, float* lse,
                  int64_t L, int32_t block, int32_t heads, int32_t kv_heads, int32_t head_dim,
                  float softmax_scale, const bdlm_task* tasks, int32_t n_tasks, int32_t n_slots,
                  int32_t o_dtype, void* workspace, size_t workspace_bytes, bdlm_stream_t stream);

/* Workspace (bytes, 256-byte aligned) of a task-list backward over this HOST
 * task array with L rows, H heads and head dim d; 0 if the list or a task is
 * malformed as for bdlm_attn_fwd_tasks_workspace_bytes (or has an empty key
 * window), or the sizes are unsupported. */
BDLM_API size_t bdlm_attn_bwd_tasks_workspace_bytes(const bdlm_task* tasks, int32_t n_tasks, int64_t L,
                  int32_t heads, int32_t head_dim);

/*
 * bdlm_attn_bwd_tasks - the backward of every task of a list, in one launch of
 * the backward's main kernel (after the task upload and the prologue, and
 * with the same preprocess and dq-convert kernels as bdlm_attn_bwd). Each
 * task's backward is taken with the FULL softmax of its rows, as for a
 * KEY_WINDOW backward: o and lse hold, for every row a task covers, the merge
 * over all the keys the row sees (e.g. the bdlm_lse_merge of the forward's
 * slots), and D = rowsum(dO * o).
 *
 *   q, o, dO   bf16 [L, H, d]; lse fp32 [H, L]; k, v bf16 [L, Hk, d].
 *   dq         bf16 [L, H, d]: the sum over the tasks of each task's dq share
 *              (its rows' gradient through its keys); 0 on rows no task covers.
 *              Over tasks that split each row's keys, it is the full dq.
 *   dk, dv     n_slots consecutive bf16 [L, Hk, d] arrays: task t writes the
 *              gradients of its window's keys from its rows into slot t (zeros
 *              for keys that none of its rows sees); keys that no task of a
 *              slot covers are left as they were. Summed over the slots, the
 *              tasks of a partition of every sequence's rows x keys give the
 *              full dk, dv.
 * Tasks of one slot must not share keys (they would write the same dk, dv
 * rows): such a list returns BDLM_ERR_INVALID_ARG, as do the per-task checks
 * of bdlm_attn_fwd_tasks. Tasks of one slot may share query rows.
 */
BDLM_API int bdlm_attn_bwd_tasks(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv,
                  int64_t L, int32_t block, int32_t heads, int32_t kv_heads, int32_t head_dim,
                  float softmax_scale, const bdlm_task* tasks, int32_t n_tasks, int32_t n_slots,
                  void* workspace, size_t workspace_bytes, bdlm_stream_t stream);

/*
 * Backward: given q, k, v, the forward's o and lse, and the upstream gradient
 * dO, writes dq [Lq, H, d], dk [Lk, Hk, d], dv [Lk, Hk, d] (bf16), the
 * gradients of softmax(QK^T)V under the BDLM mask ("Efficient Long-context
 * Language Model Training by Core Attention Disaggregation", abstract, for
 * core attention; the mask as for bdlm_attn_fwd). dk and dv sum the
 * contributions of all H/Hk query heads that share a kv head. The workspace
 * (>= bdlm_attn_bwd_workspace_bytes(L, ...)) holds D = rowsum(dO * o) and an
 * fp32 dq accumulator; its contents need no initialisation.
 *
 *   part NULL / NONE  the full attention; Lq = Lk = L.
 *   KEY_WINDOW        one clean-K/V shard (or the local corrupted keys) under
 *                     context-sharded block parallelism (Block Parallelism
 *                     abstract; rit.work CSBP post, CSBP paragraph): k, v hold
 *                     the keys at positions [key_lo, key_hi); q, dO hold all L
 *                     rows; o and lse are the MERGED (full) forward results,
 *                     not the shard's partial ones. Writes this window's share
 *                     of dq (summed over a partition of the keys, the shares
 *                     give the full dq) and the window keys' complete dk, dv.
 *   BLOCK_GROUP       one rank's corrupted target blocks (same layout as the
 *                     forward; o, lse from the group's forward). dq is complete
 *                     for the group's rows and dk, dv for its corrupted keys;
 *                     for the clean keys dk, dv hold the group's share only
 *                     (the shares of all groups plus the clean rows' own sum
 *                     to the full gradient). The block list must be strictly
 *                     ascending here (BDLM_ERR_DEVICE_CHECK otherwise, with
 *                     the offending list index). Clean keys that no listed
 *                     block sees get zero gradients.
 */
BDLM_API int bdlm_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv,
                  int64_t L, int32_t block, int32_t heads, int32_t kv_heads, int32_t head_dim,
                  const int32_t* cu_seqlens, int32_t n_docs, float softmax_scale,
                  const bdlm_partial* part, void* workspace, size_t workspace_bytes,
                  bdlm_stream_t stream);

/*
 * LSE merge of n_partials results computed against disjoint key sets (the
 * per-shard combination under context-sharded block parallelism):
 *   m = max_p lse_p over finite values, w_p = exp(lse_p - m) (0 for -inf),
 *   lse = m + ln sum_p w_p,  o = sum_p w_p o_p / sum_p w_p.
 * A row whose partials are all -inf gets o = 0, lse = -inf; a -inf partial is
 * skipped by selection, so whatever its o_p holds never reaches the output.
 *
 *   partials   HOST array of n_partials DEVICE pointers, each [rows, H, d] of
 *              partial_dtype (BDLM_BF16 or BDLM_F32).
 *   lses       HOST array of n_partials DEVICE pointers, each fp32 [H, rows].
 *   o, lse     outputs: bf16 [rows, H, d], fp32 [H, rows]; may not alias inputs.
 *   1 <= n_partials <= 64; d is 64 or 128.
 */
BDLM_API int bdlm_lse_merge(const void* const* partials, const float* const* lses, int32_t n_partials,
                   int32_t partial_dtype, int64_t rows, int32_t heads, int32_t head_dim,
                   void* o, float* lse, bdlm_stream_t stream);

/* Synchronises `stream`, then returns the device error word of the last call
 * that used `workspace` (BDLM_OK, BDLM_ERR_TIMEOUT or BDLM_ERR_DEVICE_CHECK),
 * or BDLM_ERR_CUDA if the stream reports a CUDA error. workspace == NULL
 * reads the fixed scratch of bdlm_attn_fwd_noalloc on the current device. */
BDLM_API int bdlm_read_error(const void* workspace, bdlm_stream_t stream);

/* Human-readable name of a status code (static storage). */
BDLM_API const char* bdlm_status_string(int status);

/* Number of kernels the last successful bdlm_* call on this host thread
 * launched (for launch accounting in benchmarks). */
BDLM_API int bdlm_last_launch_count(void);

/*
 * Self-test of the device failure path: launches one CTA that waits, with the
 * same bounded mbarrier wait every tensor-core kernel uses, for a barrier
 * phase that nothing completes. The wait gives up after wait_ns (clamped to
 * [1 ms, 2 s]), writes BDLM_ERR_TIMEOUT to the workspace error word and the
 * kernel returns; nothing faults and the context stays usable. The workspace
 * needs 256 bytes (its header); bdlm_read_error then returns
 * BDLM_ERR_TIMEOUT. Returns BDLM_ERR_WORKSPACE for a missing or small
 * workspace.
 */
BDLM_API int bdlm_selftest_timeout(void* workspace, size_t workspace_bytes, uint32_t wait_ns,
                  bdlm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BDLM_H */
