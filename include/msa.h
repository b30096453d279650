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
 * 1 <= topk <= 64, num_kv_heads dividing 128, group size num_q_heads /
 * num_kv_heads a power of two in [8, 128], total_q < 2^25; decode batches
 * also need num_kv_heads <= 8.  Other values return MSA_ERR_UNSUPPORTED.
 *
 * Size of a prefill call: the workspace holds one partial output per (query,
 * group, selected block) until the combine, so it grows with total_q * topk:
 * about total_q * num_q_heads * topk * 264 bytes, plus total_k * num_kv_heads
 * * 256 bytes (an fp16 copy of V) and the schedule (msa_workspace_size gives
 * the exact figure).  At 64 query / 4 KV heads and topk 16 that is about 270 KB
 * per query row: 35 GB for a 131,072-query prefill, so one call on a 288 GB
 * GB300 takes up to roughly 1M query rows with nothing else resident.  Longer
 * prefills go in chunks of queries (each call's sequences with q_len <
 * kv_len: the queries are the last q_len positions), which select and attend
 * exactly as one call would.
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
 *
 * CUDA graphs: since a call neither allocates nor synchronises, it may be
 * enqueued on a stream that is being captured.  The graph keeps the pointers
 * and sizes of the captured call (its workspace and outputs included) and
 * reads the inputs' contents at each replay; the decode chain's dependent
 * launches become programmatic edges.  Make one call of each entry point
 * before the first capture (one-time driver look-ups happen on that call).
 * msa_read_device_status() synchronises and is not capturable.
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
                                        entry of msa_forward_decode_paged(_fp8)(_index) named a page outside
                                        the cache */

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
  int32_t topk;                  /* 1..64, counts the local block */
  float softmax_scale;           /* <= 0 selects 1/sqrt(head_dim) */
} msa_problem_t;

typedef enum msa_op {
  MSA_OP_INDEX_POOL = 1,         /* msa_index_pool */
  MSA_OP_INDEX_TOPK = 2,         /* msa_index_topk */
  MSA_OP_SPARSE_ATTN_PREFILL = 3,/* msa_sparse_attn_prefill */
  MSA_OP_SPARSE_ATTN_DECODE = 4, /* msa_sparse_attn_decode */
  MSA_OP_FORWARD = 5,            /* msa_forward */
  MSA_OP_TOPK_POOLED = 6,        /* msa_topk_pooled */
  MSA_OP_QUANTIZE_KV_FP8 = 7,    /* msa_quantize_kv_fp8 */
  MSA_OP_SPARSE_ATTN_PREFILL_FP8 = 8, /* msa_sparse_attn_prefill_fp8 */
  MSA_OP_SPARSE_ATTN_DECODE_FP8 = 9,  /* msa_sparse_attn_decode_fp8 */
  MSA_OP_FORWARD_FP8 = 10,       /* msa_forward_fp8 */
  MSA_OP_INDEX_PROLOGUE = 11,    /* msa_index_prologue */
  MSA_OP_QUANTIZE_INDEX_FP8 = 12 /* msa_quantize_index_fp8 */
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

/* Main Branch for decode batches (every q_len == 1): "MiniMax Sparse
 * Attention: let each query pick its own blocks", section "The mechanism,
 * precisely", second bullet -- exact attention of the one new query of each
 * sequence (at pos = kv_len - 1) over the blocks in idx; the groundtruth.day
 * article on the llama.cpp merge ("Key facts") gives the effect: about 2,048
 * KV tokens read per decode step whatever the context length.  Split over the
 * selected blocks (one partial result per (sequence, group, block)), then a
 * log-sum-exp combine.  Same arguments and results as the prefill call. */
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
 * it; make that first call before any stream capture.  The cached address
 * belongs to the context it was looked up in: after a device reset (a new
 * primary context) the next call looks it up again.  Every call uses the
 * same array and leaves its contents behind (each call clears what must start
 * at zero), so calls whose kernels may overlap on the GPU -- on different
 * streams, or from several host threads -- race and must be serialised by the
 * caller.  Device-side errors of a call (MSA_DEVICE_* flags) are kept in the
 * array's header: read them with msa_read_device_status(NULL, ...). */
msa_status_t msa_sparse_attn_decode_static(const msa_problem_t *problem, const void *q,
                                           const void *k, const void *v, const int32_t *idx,
                                           void *o, float *lse, msa_stream_t stream);

/* The whole MSA layer forward ("MiniMax Sparse Attention: let each query pick
 * its own blocks", section "The mechanism, precisely", both bullets, and
 * Figure 1: Index Branch -> top-k block indices -> Main Branch):
 * msa_index_topk, then msa_sparse_attn_prefill, or msa_sparse_attn_decode when
 * every q_len is 1, on one workspace (size: op MSA_OP_FORWARD).  Writes idx
 * (the selection), o and lse. */
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

/* Index prologue: hidden states -> index heads ("MiniMax Sparse Attention:
 * let each query pick its own blocks", Figure 1: the Index Branch takes the
 * hidden states through a linear projection, a norm and RoPE to the index
 * query and key heads; the atlas record gives d_model 3072 and a RoPE
 * dimension of 64 on 128-dim heads, and names no norm).  For every new token
 * (query row i at key position pos(i)):
 *   y_h = W_q[h] x_i (h < num_kv_heads), y_k = W_k x_i      (fp32 accumulation)
 *   z = y / sqrt(mean(y^2) + 1e-6) * gamma   per head (gamma_q for the index
 *       query heads, gamma_k for the key head)
 *   RoPE on dims 0..63: pairs (j, j + 32) rotated by pos(i) * 10000^(-j/32)
 *   Q_idx[i, h, :] = z_h;  K_idx[k_start + pos(i), :] = z_k   (bf16)
 * so a prefill writes its tokens' rows of the index-key cache and a decode
 * step appends one row per sequence.
 *   x        [total_q, d_model] bf16; d_model a multiple of 64 (at most 65536)
 *   w_q      [num_kv_heads * 128, d_model] bf16 (a linear layer's weight)
 *   w_k      [128, d_model] bf16
 *   gamma_q, gamma_k  [128] bf16
 *   q_idx    [total_q, num_kv_heads, 128] bf16 (written)
 *   k_idx    [total_k, 128] bf16 (the new tokens' rows written, others kept)
 * Needs index_dim = 128 (else MSA_ERR_UNSUPPORTED); workspace: op
 * MSA_OP_INDEX_PROLOGUE.  Pointers 16-byte aligned (gamma 2-byte). */
msa_status_t msa_index_prologue(const msa_problem_t *problem, const void *x, int32_t d_model, const void *w_q,
                                const void *w_k, const void *gamma_q, const void *gamma_k, void *q_idx,
                                void *k_idx, void *workspace, size_t workspace_bytes, msa_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8 K and V.  The atlas record of the report (provenance of section 4.2)
 * says the kernels handle fp8 as well and gives no format; this library reads
 * it as OCP E4M3 codes ("E4M3FN": bias 7, 3 mantissa bits, largest finite
 * 448, no infinities) with one fp32 scale per (key block of 128 tokens of a
 * sequence, KV head), for K and for V separately:
 *   scale = max |x| over the block's rows of that head / 448 (1 when 0),
 *   code  = round-to-nearest-even(x / scale) in fp32, saturated to +-448,
 *   value = code * scale.
 *   k8, v8            [total_k, num_kv_heads, 128] uint8 codes, 16-byte aligned
 *   k_scale, v_scale  [n_key_blocks, num_kv_heads] fp32, 4-byte aligned, where
 *                     n_key_blocks = sum over sequences of ceil(kv_len / 128)
 *                     (at most total_k / 128 + num_seqs); key block b of
 *                     sequence s is row (key blocks of sequences 0..s-1) + b.
 * The Index Branch reads bf16 Q_idx / K_idx here (a quantized index selects
 * other blocks; the fp8 index below is a separate option).  The fp8 Main
 * Branch computes exactly the bf16 one over the dequantized values
 * (value = code * scale); results differ from bf16 K/V by the quantization.
 * Decode reads the codes directly (half the K/V bytes); prefill widens them
 * once per call into exact 16-bit copies in the workspace.  A paged decode
 * cache (msa_forward_decode_paged_fp8) has one scale row per page instead:
 * k_scale / v_scale [num_pages, num_kv_heads]; msa_quantize_kv_fp8 produces
 * exactly that layout when given the page pool as one sequence of
 * num_pages * 128 keys (each page is then one key block).
 * ------------------------------------------------------------------------ */

/* bf16 K and V -> E4M3 codes and scales as above (msa_workspace_size op
 * MSA_OP_QUANTIZE_KV_FP8).  Only the rows of the sequences' key blocks are
 * written. */
msa_status_t msa_quantize_kv_fp8(const msa_problem_t *problem, const void *k, const void *v, void *k8, void *v8,
                                 float *k_scale, float *v_scale, void *workspace, size_t workspace_bytes,
                                 msa_stream_t stream);

/* msa_sparse_attn_prefill over fp8 K and V (op MSA_OP_SPARSE_ATTN_PREFILL_FP8). */
msa_status_t msa_sparse_attn_prefill_fp8(const msa_problem_t *problem, const void *q, const void *k8,
                                         const void *v8, const float *k_scale, const float *v_scale,
                                         const int32_t *idx, void *o, float *lse, void *workspace,
                                         size_t workspace_bytes, msa_stream_t stream);

/* msa_sparse_attn_decode over fp8 K and V (op MSA_OP_SPARSE_ATTN_DECODE_FP8). */
msa_status_t msa_sparse_attn_decode_fp8(const msa_problem_t *problem, const void *q, const void *k8,
                                        const void *v8, const float *k_scale, const float *v_scale,
                                        const int32_t *idx, void *o, float *lse, void *workspace,
                                        size_t workspace_bytes, msa_stream_t stream);

/* msa_forward with fp8 K and V for the Main Branch and bf16 Q_idx / K_idx for
 * the Index Branch (op MSA_OP_FORWARD_FP8). */
msa_status_t msa_forward_fp8(const msa_problem_t *problem, const void *q, const void *k8, const void *v8,
                             const float *k_scale, const float *v_scale, const void *q_idx, const void *k_idx,
                             int32_t *idx, void *o, float *lse, void *workspace, size_t workspace_bytes,
                             msa_stream_t stream);

/* msa_forward_decode_paged with fp8 K and V caches (op MSA_OP_FORWARD_FP8):
 * k8_cache, v8_cache [num_pages * 128, num_kv_heads, 128] E4M3 codes, and
 * k_scale, v_scale [num_pages, num_kv_heads] fp32, one row per page (see
 * above); the Index Branch reads the bf16 k_idx_cache as in
 * msa_forward_decode_paged.  Arguments, block table, errors and the device
 * flag for a page outside the cache as for msa_forward_decode_paged. */
msa_status_t msa_forward_decode_paged_fp8(const msa_problem_t *problem, const void *q, const void *k8_cache,
                                          const void *v8_cache, const float *k_scale, const float *v_scale,
                                          const void *q_idx, const void *k_idx_cache, const int32_t *block_table,
                                          int32_t max_blocks_per_seq, int64_t num_pages, int32_t *idx, void *o,
                                          float *lse, void *workspace, size_t workspace_bytes,
                                          msa_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8 index (the same provenance as fp8 K/V above; the report also warns that
 * quantizing the index changes which blocks are selected, so this is an
 * option beside the bf16 Index Branch, and its selections are those of the
 * method applied to the dequantized index inputs, not to the bf16 ones).
 * Q_idx and K_idx as E4M3 codes (index_dim 128 only) with the rounding of
 * msa_quantize_kv_fp8 (scale = max |x| / 448, 1 when 0; code = RNE(x / scale)
 * in fp32, saturated):
 *   q_idx8       [total_q, num_kv_heads, 128] uint8, 16-byte aligned
 *   q_idx_scale  [total_q, num_kv_heads] fp32: one scale per (query row, group)
 *   k_idx8       [total_k, 128] uint8, 16-byte aligned
 *   k_idx_scale  [n_key_blocks] fp32: one scale per key block of 128 tokens of
 *                a sequence, block b of sequence s at row (key blocks of
 *                sequences 0..s-1) + b, as for k_scale above.
 * A token score is the fp32 dot product of the two code rows (the tensor
 * cores multiply E4M3 codes exactly and sum in fp32) and a block's pooled
 * score is the block's maximum times q_idx_scale * k_idx_scale: scales must be
 * positive and finite (msa_quantize_index_fp8 gives such), so the maximum of
 * the scaled scores is the scaled maximum.  Half the index bytes of bf16: the
 * decode index scan, which streams every cached key, reads half as much.
 * ------------------------------------------------------------------------ */

/* bf16 Q_idx and/or K_idx -> E4M3 codes and scales as above (workspace op
 * MSA_OP_QUANTIZE_INDEX_FP8).  Either input may be NULL to skip that side (for
 * example a decode step that quantizes only its new queries); the outputs of
 * a given side are then not touched.  Only the rows of the sequences' key
 * blocks are written. */
msa_status_t msa_quantize_index_fp8(const msa_problem_t *problem, const void *q_idx, const void *k_idx,
                                    void *q_idx8, float *q_idx_scale, void *k_idx8, float *k_idx_scale,
                                    void *workspace, size_t workspace_bytes, msa_stream_t stream);

/* msa_index_pool over fp8 index inputs (workspace op MSA_OP_INDEX_POOL). */
msa_status_t msa_index_pool_fp8(const msa_problem_t *problem, const void *q_idx8, const float *q_idx_scale,
                                const void *k_idx8, const float *k_idx_scale, float *pooled,
                                int64_t pooled_stride, void *workspace, size_t workspace_bytes,
                                msa_stream_t stream);

/* msa_index_topk over fp8 index inputs (workspace op MSA_OP_INDEX_TOPK):
 * prefill and decode batches, the same selection rule. */
msa_status_t msa_index_topk_fp8(const msa_problem_t *problem, const void *q_idx8, const float *q_idx_scale,
                                const void *k_idx8, const float *k_idx_scale, int32_t *idx, void *workspace,
                                size_t workspace_bytes, msa_stream_t stream);

/* msa_forward_fp8 with the Index Branch on fp8 inputs as well (workspace op
 * MSA_OP_FORWARD_FP8): every K, V, Q_idx and K_idx read is an E4M3 code. */
msa_status_t msa_forward_fp8_index(const msa_problem_t *problem, const void *q, const void *k8, const void *v8,
                                   const float *k_scale, const float *v_scale, const void *q_idx8,
                                   const float *q_idx_scale, const void *k_idx8, const float *k_idx_scale,
                                   int32_t *idx, void *o, float *lse, void *workspace, size_t workspace_bytes,
                                   msa_stream_t stream);

/* msa_forward_decode_paged_fp8 with the index-key cache in fp8 as well
 * (workspace op MSA_OP_FORWARD_FP8): k_idx8_cache [num_pages * 128, 128] E4M3
 * codes with k_idx_scale [num_pages], one scale per page (msa_quantize_index_fp8
 * gives that layout for the page pool taken as one sequence of num_pages * 128
 * keys), and q_idx8 / q_idx_scale for the batch's queries.  Block table,
 * errors and the device flag for a page outside the cache as for
 * msa_forward_decode_paged. */
msa_status_t msa_forward_decode_paged_fp8_index(const msa_problem_t *problem, const void *q, const void *k8_cache,
                                                const void *v8_cache, const float *k_scale, const float *v_scale,
                                                const void *q_idx8, const float *q_idx_scale,
                                                const void *k_idx8_cache, const float *k_idx_scale,
                                                const int32_t *block_table, int32_t max_blocks_per_seq,
                                                int64_t num_pages, int32_t *idx, void *o, float *lse,
                                                void *workspace, size_t workspace_bytes, msa_stream_t stream);

/* Waits for `stream`, then returns in *flags the MSA_DEVICE_* bits that the
 * last call on this workspace raised (0 = none).  workspace = NULL reads the
 * flags of the last msa_sparse_attn_decode_static call on the current device.
 * The only synchronising call. */
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
