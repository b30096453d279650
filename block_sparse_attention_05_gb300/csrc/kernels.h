// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

struct WsHeader;
struct SeqInfo;

// Adds n to the library's count of enqueued kernels (msa_kernel_launch_count).
void note_launches(int n);

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
};
size_t index_score_smem_bytes();
cudaError_t launch_index_score(const CUtensorMap& tq, const CUtensorMap& tk, const IndexParams& p, bool fused,
                               int grid, cudaStream_t stream);

// Top-k over pooled rows r = i * hkv + g (rows of queries, or of decode
// sequences when every q_len is 1).
struct TopkParams {
  int num_seqs, total_q, hkv, topk, max_nb;
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
cudaError_t launch_decode_scan(const CUtensorMap& tk, const DecodeScanParams& p, int grid, cudaStream_t stream);

// ---------------------------------------------------------------- main branch
// Partial results of one (query, group, slot): G rows of 128 bf16 + G lse + G
// log weights.  The true partial output (normalised within the block) is
// o * exp(ow - lse): the decode kernel stores it as is (ow = lse), the prefill
// kernel over V scaled by 2^-e (ow = lse + e ln 2).
struct PartialBuffers {
  __nv_bfloat16* o;   // [total_q, hkv, topk, G, 128]
  float* lse;         // [total_q, hkv, topk, G]
  float* ow;          // [total_q, hkv, topk, G]
};

// fp16 copy of V for the prefill Main Branch: V * 2^-v_scale_shift(max |V|).
// Two launches: max |V| into hdr->vmax_bits (zeroed by the caller), then the copy.
cudaError_t launch_v_prep(const __nv_bfloat16* v, __half* v16, long long n_elems, WsHeader* hdr, int sms,
                          cudaStream_t stream);

// Main Branch work item: at most this many tiles (of qpt <= 16 queries each).
constexpr int kTilesPerChunk = 16;

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
  int32_t* entries;       // [total_q * hkv * topk]
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
};
size_t sparse_attn_smem_bytes();
cudaError_t launch_sparse_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const AttnParams& p, int grid, cudaStream_t stream);

struct DecodeAttnParams {
  int num_seqs, hkv, group, topk;
  int sms;                 // persistent grid size
  const SeqInfo* seq;
  const int32_t* idx;      // [num_seqs, hkv, topk]
  PartialBuffers part;     // Q [num_seqs, hq, 128] comes through a tensor map (16 heads x 64 dims boxes)
  float scale_log2;
  WsHeader* hdr;
  const int32_t* block_table;  // as in DecodeScanParams
  int bt_stride;
  long long n_pages;
};
size_t decode_attn_smem_bytes();
cudaError_t launch_decode_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeAttnParams& p, cudaStream_t stream);

struct CombineParams {
  int total_q, hq, hkv, group, topk, num_seqs;
  int sms;  // grid: two CTAs per SM, grid-stride over the (query, head pair) items
  const int32_t* cu_q;
  const SeqInfo* seq;
  const int32_t* idx;
  PartialBuffers part;
  __nv_bfloat16* o;
  float* lse;
  WsHeader* hdr;
};
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);

}  // namespace msa
