/*
 * msa.h -- C ABI of the MiniMax Sparse Attention (MSA) forward pass on GB300
 * (sm_103a).  Plain pointers and sizes only: no C++ or framework types cross
 * this boundary.
 *
 * The method ("MiniMax Sparse Attention: let each query pick its own blocks",
 * section "The mechanism, precisely", and the same page's Figure 1):
 *   Index Branch: per GQA group g, one index-query head; one index-key head
 *     shared by all groups.  For query i at key position pos(i):
 *       s[g,i,j] = Q_idx[i,g,:] . K_idx[j,:]             (fp32, j <= pos(i))
 *       P[g,i,b] = max over keys j of block b, j <= pos(i), of s[g,i,j]
 *       sel(i,g) = {local block pos(i)/B} U top-(k-1) of the other causal
 *                  blocks by (P descending, block index ascending)
 *   Main Branch: every query head h of group g attends, with exact softmax,
 *     to the tokens j <= pos(i) of the blocks in sel(i,g) only.
 * Deployed values: block B = 128, k = 16 (a 2,048-token budget per query);
 * 64 query heads over 4 KV heads, head dim 128 (the atlas record of the
 * report, summary paragraph).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Batches are packed variable-length sequences.  Sequence s owns query rows
 * [cu_seqlens_q[s], cu_seqlens_q[s+1]) and key rows [cu_seqlens_k[s],
 * cu_seqlens_k[s+1]).  Its queries are the LAST q_len positions of the
 * sequence: query t sits at key position pos = kv_len - q_len + t
 * (bottom-right causal alignment; a decode step is q_len = 1).  Query head h
 * belongs to group h / (num_q_heads / num_kv_heads).
 *
 * Tensors (all row-major and contiguous, all DEVICE memory of the current
 * CUDA device, owned by the caller):
 *   q      [total_q, num_q_heads,  head_dim]   bf16
 *   k, v   [total_k, num_kv_heads, head_dim]   bf16
 *   q_idx  [total_q, num_kv_heads, index_dim]  bf16
 *   k_idx  [total_k, index_dim]                bf16
 *   idx    [total_q, num_kv_heads, topk]       int32  selected blocks, ascending,
 *                                                     -1 padding at the tail
 *   o      [total_q, num_q_heads,  head_dim]   bf16
 *   lse    [total_q, num_q_heads]              fp32   natural-log sum of exp of the
 *                                                     scaled logits
 * Every tensor pointer must be 16-byte aligned; the workspace 256-byte aligned.
 *
 * Supported shapes: head_dim = 128, block_size = 128, index_dim in {64, 128},
 * 1 <= topk <= 16, num_kv_heads dividing 128, group size num_q_heads /
 * num_kv_heads a power of two in [8, 128]; decode batches also need
 * num_kv_heads <= 8 and a group size of 16.  Other values return
 * MSA_ERR_UNSUPPORTED.
 *
 * Execution: every call validates its arguments on the host, then enqueues
 * kernels on `stream` and returns without synchronising.  Nothing is
 * allocated or freed: the caller provides a workspace of at least
 * msa_workspace_size() bytes, which the call overwrites.  Two calls that run
 * at the same time must not share a workspace.  On any non-OK status nothing
 * has been enqueued, except MSA_ERR_CUDA, which reports a launch failure.
 * Errors that only the device can see (cu_seqlens that contradict the host
 * sizes, a kernel wait that timed out) make the kernels skip their work and
 * set flags that msa_read_device_status() returns.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st *msa_stream_t;

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = -1,  /* null pointer, negative size, inconsistent sizes */
  MSA_ERR_UNSUPPORTED = -2,  /* valid but outside the supported shapes above */
  MSA_ERR_ALIGNMENT = -3,    /* a pointer is not aligned as required */
  MSA_ERR_WORKSPACE = -4,    /* workspace missing or smaller than required */
  MSA_ERR_CUDA = -5,         /* a CUDA call or kernel launch failed */
  MSA_ERR_DEVICE = -6        /* no usable sm_103 device is current */
} msa_status_t;

/* Device-side error flags (msa_read_device_status). */
#define MSA_DEVICE_TIMEOUT 1u        /* a kernel wait exceeded its time limit */
#define MSA_DEVICE_BAD_SEQLENS 2u    /* cu_seqlens disagree with the host sizes */
#define MSA_DEVICE_BAD_INDEX 4u      /* a computed index failed its check (checked builds), or a block-table
                                        entry of msa_forward_decode_paged named a page outside the cache */

typedef struct msa_problem {
  int32_t num_seqs;              /* >= 1 */
  const int32_t *cu_seqlens_q;   /* device [num_seqs + 1], cu[0] = 0, nondecreasing */
  const int32_t *cu_seqlens_k;   /* device [num_seqs + 1], kv_len >= q_len per sequence */
  int32_t total_q;               /* = cu_seqlens_q[num_seqs] */
  int32_t total_k;               /* = cu_seqlens_k[num_seqs] */
  int32_t max_seqlen_q;          /* >= every q_len (host bound used for sizing) */
  int32_t max_seqlen_k;          /* >= every kv_len */
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;              /* 128 */
  int32_t index_dim;             /* 64 or 128 */
  int32_t block_size;            /* 128 */
  int32_t topk;                  /* 1..16, counts the local block */
  float softmax_scale;           /* <= 0 selects 1/sqrt(head_dim) */
} msa_problem_t;

typedef enum msa_op {
  MSA_OP_INDEX_POOL = 1,         /* msa_index_pool */
  MSA_OP_INDEX_TOPK = 2,         /* msa_index_topk */
  MSA_OP_SPARSE_ATTN_PREFILL = 3,/* msa_sparse_attn_prefill */
  MSA_OP_SPARSE_ATTN_DECODE = 4, /* msa_sparse_attn_decode */
  MSA_OP_FORWARD = 5,            /* msa_forward */
  MSA_OP_TOPK_POOLED = 6         /* msa_topk_pooled */
} msa_op_t;

/* Workspace bytes that `op` needs for `problem` (host-only; no CUDA call).
 * Returns MSA_ERR_INVALID_ARG / MSA_ERR_UNSUPPORTED as the op itself would. */
msa_status_t msa_workspace_size(const msa_problem_t *problem, msa_op_t op, size_t *bytes);

/* Index Branch, scoring and pooling only ("The mechanism, precisely": scores
 * Q_idx . K_idx^T max-pooled to blocks).  Writes pooled[r * pooled_stride + b]
 * for query/group row r = i * num_kv_heads + g and causal block
 * b <= pos(i) / block_size (the local block pools only keys j <= pos(i));
 * entries past the causal end are left untouched.  pooled_stride >= the
 * largest number of causal blocks, ceil(max_seqlen_k / block_size). */
msa_status_t msa_index_pool(const msa_problem_t *problem, const void *q_idx, const void *k_idx,
                            float *pooled, int64_t pooled_stride, void *workspace,
                            size_t workspace_bytes, msa_stream_t stream);

/* Top-k over precomputed pooled rows (same layout as msa_index_pool), local
 * block forced in: idx[r][0..topk) = ascending set, -1 padded.  Ranking:
 * pooled score descending, equal scores to the lower block index, +0 == -0. */
msa_status_t msa_topk_pooled(const msa_problem_t *problem, const float *pooled,
                             int64_t pooled_stride, int32_t *idx, void *workspace,
                             size_t workspace_bytes, msa_stream_t stream);

/* Index Branch: scores, block max-pool and top-k with the local block forced
 * ("The mechanism, precisely", first bullet).  Writes idx.  Prefill batches
 * (max_seqlen_q > 1) use the tensor-core scoring kernel with the top-k fused
 * into its epilogue; decode batches (max_seqlen_q == 1) a streaming scan. */
msa_status_t msa_index_topk(const msa_problem_t *problem, const void *q_idx, const void *k_idx,
                            int32_t *idx, void *workspace, size_t workspace_bytes,
                            msa_stream_t stream);

/* Main Branch for prefill ("The mechanism, precisely", second bullet): exact
 * softmax attention over the blocks in idx (any ascending, -1 padded set that
 * contains only causal blocks; every row must contain at least one block).
 * Writes o and lse. */
msa_status_t msa_sparse_attn_prefill(const msa_problem_t *problem, const void *q, const void *k,
                                     const void *v, const int32_t *idx, void *o, float *lse,
                                     void *workspace, size_t workspace_bytes,
                                     msa_stream_t stream);

/* Main Branch for decode batches (every q_len == 1): split over the selected
 * blocks, then a log-sum-exp combine.  Same arguments as the prefill call. */
msa_status_t msa_sparse_attn_decode(const msa_problem_t *problem, const void *q, const void *k,
                                    const void *v, const int32_t *idx, void *o, float *lse,
                                    void *workspace, size_t workspace_bytes,
                                    msa_stream_t stream);

/* Size of the device array behind msa_sparse_attn_decode_static (32 MiB). */
#define MSA_STATIC_SCRATCH_BYTES (32u << 20)

/* msa_sparse_attn_decode for callers that cannot allocate device memory: no
 * workspace argument; the scratch lives in a fixed device array of
 * MSA_STATIC_SCRATCH_BYTES that this library declares (every GPU that loads
 * the library holds it until the process exits).  The method's pages have no
 * counterpart to this call; it exists for code that runs where cudaMalloc is
 * not available or not allowed -- a host framework that hands out only its
 * own pre-allocated tensors, an allocator-free serving loop, a process whose
 * memory pool is already fully reserved -- and that would otherwise have no
 * way to provide the workspace.
 * Arguments, layouts and results are those of msa_sparse_attn_decode.  The
 * call allocates and frees nothing.  Batches whose scratch would exceed the
 * array (about 120 decode sequences at 64 query / 4 KV heads and topk 16)
 * return MSA_ERR_WORKSPACE, and msa_last_error_detail() states the bytes
 * needed and available.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current) and caches
 * it; make that first call before any stream capture.  Every call uses the
 * same array and leaves its contents behind (each call clears what must start
 * at zero), so calls whose kernels may overlap on the GPU -- on different
 * streams, or from several host threads -- race and must be serialised by the
 * caller. */
msa_status_t msa_sparse_attn_decode_static(const msa_problem_t *problem, const void *q,
                                           const void *k, const void *v, const int32_t *idx,
                                           void *o, float *lse, msa_stream_t stream);

/* Both branches: msa_index_topk then the matching Main Branch call.  Writes
 * idx (the selection), o and lse. */
msa_status_t msa_forward(const msa_problem_t *problem, const void *q, const void *k,
                         const void *v, const void *q_idx, const void *k_idx, int32_t *idx,
                         void *o, float *lse, void *workspace, size_t workspace_bytes,
                         msa_stream_t stream);

/* msa_forward for a decode batch whose cache is paged: the same operation
 * ("MiniMax Sparse Attention: let each query pick its own blocks", section
 * "The mechanism, precisely": index scores over the cached keys, block
 * max-pool, top-k with the local block forced, exact attention over the
 * selected blocks), with K, V and K_idx read from pages of 128 tokens -- one
 * key block each -- instead of packed rows.  The pages describe no paged
 * layout; this is the decode call in the form a serving cache keeps it.
 *   problem     as for msa_forward, every sequence with q_len = 1;
 *               cu_seqlens_k gives the cached lengths (its offsets are not
 *               used as row positions here).
 *   k_cache, v_cache  [num_pages * 128, Hkv, 128] bf16; k_idx_cache
 *               [num_pages * 128, d_idx] bf16.  Row 128 * p + t of a cache is
 *               token t of page p.
 *   block_table int32 [num_seqs, max_blocks_per_seq], device: key block b of
 *               sequence s (tokens 128 b .. 128 b + 127) is page
 *               block_table[s * max_blocks_per_seq + b]; entries past a
 *               sequence's last block are not read.  4-byte aligned.
 *   max_blocks_per_seq  row stride of block_table; at least
 *               ceil(max_seqlen_k / 128).
 *   num_pages   pages in each cache; num_pages * 128 < 2^31.
 *   idx, o, lse, workspace, stream  as for msa_forward (workspace size: op
 *               MSA_OP_FORWARD of the same problem).
 * A block-table entry outside [0, num_pages) is not dereferenced: its block
 * reads as zeros and the workspace status gets MSA_DEVICE_BAD_INDEX (read it
 * with msa_read_device_status).  Host-side argument errors return before any
 * launch, as for msa_forward. */
msa_status_t msa_forward_decode_paged(const msa_problem_t *problem, const void *q, const void *k_cache,
                                      const void *v_cache, const void *q_idx, const void *k_idx_cache,
                                      const int32_t *block_table, int32_t max_blocks_per_seq,
                                      int64_t num_pages, int32_t *idx, void *o, float *lse,
                                      void *workspace, size_t workspace_bytes, msa_stream_t stream);

/* Waits for `stream`, then returns in *flags the MSA_DEVICE_* bits that the
 * last call on this workspace raised (0 = none).  The only synchronising call. */
msa_status_t msa_read_device_status(const void *workspace, uint32_t *flags, msa_stream_t stream);

/* Stages of a call, for msa_set_stage_events. */
#define MSA_STAGE_PLAN 0      /* cu_seqlens validation, per-sequence facts, work lists */
#define MSA_STAGE_INDEX 1     /* index scores + block max-pool (+ fused top-k in prefill) */
#define MSA_STAGE_TOPK 2      /* top-k over pooled rows (decode, msa_topk_pooled) */
#define MSA_STAGE_SCHEDULE 3  /* inversion of the selection into per-block work items */
#define MSA_STAGE_ATTN 4      /* Main Branch partial attention */
#define MSA_STAGE_COMBINE 5   /* log-sum-exp merge of the partials into o and lse */
#define MSA_NUM_STAGES 6

/* Optional per-stage timing for the calling host thread.  `events` holds
 * 2 * MSA_NUM_STAGES cudaEvent_t handles created by the caller; while set,
 * every call records events[2*s] on its stream just before stage s and
 * events[2*s + 1] just after it (stages a call does not run are not
 * recorded).  Pass NULL to stop.  Recording adds no synchronisation. */
msa_status_t msa_set_stage_events(void *const *events);

/* Number of kernels this library has enqueued since the process started
 * (all host threads; memsets included).  A diagnostic for launch accounting. */
int64_t msa_kernel_launch_count(void);

/* For the calling host thread: a description of the CUDA failure behind the
 * last MSA_ERR_CUDA (stage and CUDA error name) -- or of the scratch shortfall
 * behind an MSA_ERR_WORKSPACE from msa_sparse_attn_decode_static -- or "". */
const char *msa_last_error_detail(void);

/* Static description of a status code. */
const char *msa_status_string(msa_status_t status);

/* ABI version of this header (bumped on incompatible changes). */
int32_t msa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
