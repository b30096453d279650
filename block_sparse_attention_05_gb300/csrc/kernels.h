// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace msa {

struct WsHeader;
struct SeqInfo;

// Adds n to the library's count of enqueued kernels (msa_kernel_launch_count).
void note_launches(int n);

// Launches `kernel` with programmatic dependent launch allowed (see griddep_wait in common.cuh): the kernel
// must call griddep_wait() before it touches memory of the kernel before it on the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- planning
struct PlanParams {
  int num_seqs;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k, max_q, max_k;
  int qt;               // queries per index-scoring tile (0: build no tile list)
  int max_nb;           // ceil(max_k / 128)
  SeqInfo* seq;         // [num_seqs]
  int32_t* blk_off;     // [num_seqs + 1] exclusive prefix of key blocks
  int32_t* tile_base;   // [num_seqs + 1] scratch
  int32_t* hist;        // [max_nb + 2] scratch
  int32_t* cursor;      // [max_nb + 2] scratch
  int2* tiles;          // [max_tiles] (seq, first query) sorted by descending cost
  WsHeader* hdr;
};
cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);

// Device-wide exclusive scan of n int32 values; out has n + 1 entries (the
// last is the total).  If total_dst != nullptr the total is also stored there.
// tmp needs scan_tmp_ints(n) int32 elements.
int scan_tmp_ints(int n);
cudaError_t launch_exclusive_scan(const int32_t* in, int32_t* out, int n, int32_t* tmp, uint32_t* total_dst,
                                  const WsHeader* hdr, cudaStream_t stream);

// ---------------------------------------------------------------- index branch
struct IndexParams {
  const SeqInfo* seq;
  const int2* tiles;
  WsHeader* hdr;
  int hkv, d_idx, topk, qt;
  float* pooled;
  int64_t pooled_stride;
  int32_t* idx;
  // fp8 index (launch with fp8 = true; tq / tk then map E4M3 codes, d_idx 128): Q_idx scales [total_q * hkv],
  // K_idx scales [n_key_blocks], first key block of each sequence
  const float* q_scale;
  const float* k_scale;
  const int32_t* blk_off;
};
size_t index_score_smem_bytes(bool fp8);
cudaError_t launch_index_score(const CUtensorMap& tq, const CUtensorMap& tk, const IndexParams& p, bool fused,
                               bool fp8, int grid, cudaStream_t stream);

// Top-k over pooled rows r = i * hkv + g (rows of queries, or of decode
// sequences when every q_len is 1).
struct TopkParams {
  int num_seqs, total_q, hkv, topk, max_nb;
  bool one_query_per_seq;  // every sequence has exactly one query (a decode batch): query i is sequence i
  const int32_t* cu_q;
  const SeqInfo* seq;
  const float* pooled;
  int64_t pooled_stride;
  int32_t* idx;
  WsHeader* hdr;
};
cudaError_t launch_topk_pooled(const TopkParams& p, int max_nb, cudaStream_t stream);

// Decode index scan: pooled scores of the single query of each sequence.
struct DecodeScanParams {
  int num_seqs, hkv, d_idx;
  const SeqInfo* seq;
  const __nv_bfloat16* q_idx;   // [num_seqs, hkv, d_idx]
  // fp8 index (launch with fp8 = true; tk then maps E4M3 codes, d_idx 128): Q_idx codes and scales
  // [num_seqs * hkv], K_idx scales per key block (packed: first block of each sequence in blk_off) or per page
  const uint8_t* q_idx8;
  const float* q_scale;
  const float* k_scale;
  const int32_t* blk_off;
  float* pooled;                // [num_seqs * hkv, pooled_stride]
  int64_t pooled_stride;
  int units_per_seq;            // work units per sequence
  int blocks_per_unit;
  long long total_k;            // rows of K_idx (for checked builds)
  WsHeader* hdr;
  // Paged cache (optional): key block b of sequence s is page block_table[s * bt_stride + b] of 128 rows;
  // null: packed rows starting at the sequence's k_start.
  const int32_t* block_table;
  int bt_stride;
  long long n_pages;
};
size_t decode_scan_smem_bytes();
cudaError_t launch_decode_scan(const CUtensorMap& tk, const DecodeScanParams& p, bool fp8, int grid,
                               cudaStream_t stream);

// ---------------------------------------------------------------- main branch
// Partial results of one (query, group, slot): G rows of 128 16-bit values + G
// lse + G log weights.  The true partial output (normalised within the block)
// is o * exp(ow - lse): the decode kernel stores it as is in bf16 (ow = lse),
// the prefill kernel in fp16 over V scaled by 2^-e, whose magnitude stays below
// 2^14 (ow = lse + e ln 2; for fp8 V, ow = lse + ln of the V scale): fp16's 11
// significant bits keep the partial's rounding well under the output's own
// bf16 rounding.
struct PartialBuffers {
  uint16_t* o;        // [total_q, hkv, topk, G, 128]: fp16 (prefill) or bf16 (decode)
  float* lse;         // [total_q, hkv, topk, G]
  float* ow;          // [total_q, hkv, topk, G]
};

// fp16 copy of V for the prefill Main Branch: V * 2^-v_scale_shift(max |V|).
// Two launches: max |V| into hdr->vmax_bits (zeroed by the caller), then the copy.
cudaError_t launch_v_prep(const __nv_bfloat16* v, __half* v16, long long n_elems, WsHeader* hdr, int sms,
                          cudaStream_t stream);

// Main Branch work item: at most this many tiles (of qpt <= 16 queries each).
constexpr int kTilesPerChunk = 16;

// A schedule entry packs one incidence as (query << kSlotBits) | slot (slot < topk <= 64).
constexpr int kSlotBits = 6;
constexpr int kSlotMask = (1 << kSlotBits) - 1;

struct ScheduleParams {
  int num_seqs, total_q, hkv, topk, window, total_blocks, n_windows, qpc;
  const int32_t* cu_q;
  const SeqInfo* seq;
  const int32_t* blk_off;
  const int32_t* idx;
  int32_t* count;         // [n_buckets]
  int32_t* bucket_start;  // [n_buckets + 1]
  int32_t* cursor;        // [n_buckets]
  int32_t* nchunk;        // [n_buckets]
  int32_t* chunk_start;   // [n_buckets + 1]
  int32_t* entries;       // [total_q * hkv * topk]: (query << kSlotBits) | slot
  int4* chunks;           // [max_chunks] (begin, count, g | block << 8, seq)
  int32_t* scan_tmp;
  WsHeader* hdr;
  long long n_buckets;
};
cudaError_t launch_schedule(const ScheduleParams& p, cudaStream_t stream);

struct AttnParams {
  const __nv_bfloat16* q;  // [total_q, hq, 128] (also behind tm_q; read directly for L2 prefetches)
  const SeqInfo* seq;
  const int4* chunks;
  const int32_t* entries;
  PartialBuffers part;
  WsHeader* hdr;
  int hkv, group, topk, qpt;
  float scale_log2;       // softmax scale * log2(e)
  // fp8 K/V (tk / tv then map the 16-bit copies of the codes): scales [n_key_blocks, hkv], first key block of
  // each sequence; null for bf16 K/V
  const float* k_scale;
  const float* v_scale;
  const int32_t* blk_off;
};
size_t sparse_attn_smem_bytes();
cudaError_t launch_sparse_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const AttnParams& p, int grid, cudaStream_t stream);

struct DecodeAttnParams {
  int num_seqs, hkv, group, topk;
  int sms;                 // persistent grid size
  const SeqInfo* seq;
  const int32_t* idx;      // [num_seqs, hkv, topk]
  PartialBuffers part;     // Q [num_seqs, hq, 128] comes through a tensor map (min(G, 16) heads x 64 dims boxes)
  float scale_log2;
  WsHeader* hdr;
  const int32_t* block_table;  // as in DecodeScanParams
  int bt_stride;
  long long n_pages;
  // fp8 K/V (launch with fp8 = true; tk / tv then map E4M3 codes): scales [n_key_blocks, hkv] and the first key
  // block of each sequence
  const float* k_scale;
  const float* v_scale;
  const int32_t* blk_off;
};
size_t decode_attn_smem_bytes();
cudaError_t launch_decode_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeAttnParams& p, bool fp8, cudaStream_t stream);

// ---------------------------------------------------------------- index prologue
// Hidden states -> Q_idx and the new tokens' K_idx rows (projection, RMSNorm, RoPE on dims 0..63).
struct PrologueParams {
  int num_seqs, total_q, hkv, d_model;
  const int32_t* cu_q;
  const SeqInfo* seq;
  const __nv_bfloat16* gamma_q;  // [128]
  const __nv_bfloat16* gamma_k;  // [128]
  __nv_bfloat16* q_idx;          // [total_q, hkv, 128]
  __nv_bfloat16* k_idx;          // [total_k, 128]: row k_start + pos(i) of token i
  float rope_turns_hi[32];       // theta_j / (2 pi) = hi + lo, theta_j = 10000^(-j/32)
  float rope_turns_lo[32];
  WsHeader* hdr;
};
size_t index_prologue_smem_bytes();
cudaError_t launch_index_prologue(const CUtensorMap& tx, const CUtensorMap& twq, const CUtensorMap& twk,
                                  const PrologueParams& p, int sms, cudaStream_t stream);

// ---------------------------------------------------------------- fp8 K/V
// Quantization of bf16 K and V to E4M3 codes with one scale per (key block, KV head).
struct QuantParams {
  int num_seqs, hkv;
  const SeqInfo* seq;
  const int32_t* blk_off;       // [num_seqs + 1] first key block of each sequence (plan)
  const __nv_bfloat16* k;       // [total_k, hkv, 128]
  const __nv_bfloat16* v;
  uint8_t* k8;                  // [total_k, hkv, 128] E4M3 codes
  uint8_t* v8;
  float* k_scale;               // [n_key_blocks, hkv]
  float* v_scale;
  WsHeader* hdr;
};
cudaError_t launch_quantize_kv_fp8(const QuantParams& p, long long max_blocks, cudaStream_t stream);
// Quantization of the index inputs to E4M3 codes: K_idx with one scale per key block of a sequence, Q_idx with
// one per (query row, group); either side may be skipped (null input).  d_idx 128.
struct IndexQuantParams {
  int num_seqs, hkv, total_q;
  const SeqInfo* seq;
  const int32_t* blk_off;
  const __nv_bfloat16* q_idx;   // [total_q, hkv, 128] or null
  const __nv_bfloat16* k_idx;   // [total_k, 128] or null
  uint8_t* q8;
  float* q_scale;               // [total_q * hkv]
  uint8_t* k8;
  float* k_scale;               // [n_key_blocks]
  long long key_ctas;           // CTAs of the grid that take key blocks (the rest take query rows)
  WsHeader* hdr;
};
cudaError_t launch_quantize_index_fp8(const IndexQuantParams& p, cudaStream_t stream);
// 16-bit copies of fp8 K (bf16) and V (fp16) for the prefill Main Branch; exact.
cudaError_t launch_kv8_widen(const uint8_t* k8, const uint8_t* v8, __nv_bfloat16* k16, __half* v16,
                             long long n_elems, const WsHeader* hdr, int sms, cudaStream_t stream);

struct CombineParams {
  int total_q, hq, hkv, group, topk, num_seqs;
  bool one_query_per_seq;  // as in TopkParams
  int sms;  // grid: two CTAs per SM, grid-stride over the (query, head pair) items
  const int32_t* cu_q;
  const SeqInfo* seq;
  const int32_t* idx;
  PartialBuffers part;
  __nv_bfloat16* o;
  float* lse;
  WsHeader* hdr;
};
// f16_partials: the partial outputs are fp16 (prefill) rather than bf16 (decode).
cudaError_t launch_combine(const CombineParams& p, bool f16_partials, cudaStream_t stream);

}  // namespace msa
