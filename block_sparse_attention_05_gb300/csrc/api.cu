// api.cu -- the C ABI declared in include/msa.h: argument validation (all on
// the host, before any CUDA call), workspace layout, TMA tensor maps and the
// launch sequence of each entry point.  The library never allocates, frees or
// synchronises (except msa_read_device_status, which is documented to).
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "msa.h"

namespace msa {

namespace {
std::atomic<int64_t> g_launches{0};
thread_local cudaEvent_t t_stage_events[2 * MSA_NUM_STAGES];
thread_local bool t_stage_events_on = false;
thread_local int t_stage = -1;
thread_local char t_error_detail[256] = "";
const char* const kStageNames[MSA_NUM_STAGES] = {"plan", "index", "topk", "schedule", "attn", "combine"};
}  // namespace

void note_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {

// Records the caller's stage events (if any) around one stage of a call.
struct StageScope {
  int stage;
  cudaStream_t stream;
  StageScope(int s, cudaStream_t st) : stage(s), stream(st) {
    t_stage = s;
    if (t_stage_events_on) cudaEventRecord(t_stage_events[2 * stage], stream);
  }
  ~StageScope() {
    if (t_stage_events_on) cudaEventRecord(t_stage_events[2 * stage + 1], stream);
  }
};

constexpr size_t kAlign = 256;
constexpr int kWindow = 4096;       // queries per scheduling window

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

struct Derived {
  int S, T, N, hq, hkv, G, d_idx, topk, max_q, max_k, max_nb, qt, qpt, qpc, total_blocks, n_windows;
  long long max_tiles, n_buckets, max_chunks, n_inc;
  bool decode;
  float scale;
};

struct Layout {
  size_t hdr, seq, blk_off, tile_base, hist, cursor, tiles, pooled, count, bstart, bcursor, nchunk, cstart,
      entries, chunks, scan_tmp, v16, k16, part_o, part_lse, part_ow, total;
};

msa_status_t derive(const msa_problem_t* p, Derived& d) {
  if (!p) return MSA_ERR_INVALID_ARG;
  if (p->num_seqs < 1 || !p->cu_seqlens_q || !p->cu_seqlens_k) return MSA_ERR_INVALID_ARG;
  if (p->total_q < 0 || p->total_k < 0 || p->max_seqlen_q < 0 || p->max_seqlen_k < 0) return MSA_ERR_INVALID_ARG;
  if (p->max_seqlen_q > p->total_q || p->max_seqlen_k > p->total_k) return MSA_ERR_INVALID_ARG;
  if (p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->num_q_heads % p->num_kv_heads) return MSA_ERR_INVALID_ARG;
  if (p->topk <= 0 || p->head_dim <= 0 || p->index_dim <= 0 || p->block_size <= 0) return MSA_ERR_INVALID_ARG;
  if (!(p->softmax_scale == p->softmax_scale)) return MSA_ERR_INVALID_ARG;  // NaN
  if (p->head_dim != 128 || p->block_size != 128) return MSA_ERR_UNSUPPORTED;
  if (p->index_dim != 64 && p->index_dim != 128) return MSA_ERR_UNSUPPORTED;
  if (p->topk > 64) return MSA_ERR_UNSUPPORTED;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (!is_pow2(G) || G < 8 || G > 128) return MSA_ERR_UNSUPPORTED;
  if (128 % p->num_kv_heads) return MSA_ERR_UNSUPPORTED;
  d.S = p->num_seqs;
  d.T = p->total_q;
  d.N = p->total_k;
  d.hq = p->num_q_heads;
  d.hkv = p->num_kv_heads;
  d.G = G;
  d.d_idx = p->index_dim;
  d.topk = p->topk;
  d.max_q = p->max_seqlen_q;
  d.max_k = p->max_seqlen_k;
  d.max_nb = (p->max_seqlen_k + 127) / 128;
  if (d.max_nb < 1) d.max_nb = 1;
  d.qt = 128 / d.hkv;  // index work item: 128 rows of Q_idx
  d.qpt = 128 / G;
  d.qpc = d.qpt * kTilesPerChunk;
  d.total_blocks = (p->total_k + 127) / 128 + d.S;
  d.n_windows = (p->total_q + kWindow - 1) / kWindow;
  if (d.n_windows < 1) d.n_windows = 1;
  d.max_tiles = static_cast<long long>(p->total_q) / d.qt + d.S;
  d.n_inc = static_cast<long long>(p->total_q) * d.hkv * d.topk;
  d.n_buckets = static_cast<long long>(d.n_windows) * d.total_blocks * d.hkv;
  d.max_chunks = (d.n_inc + d.qpc - 1) / d.qpc + d.n_buckets;
  d.decode = (p->max_seqlen_q <= 1);
  d.scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / std::sqrt(static_cast<float>(p->head_dim));
  // schedule entries hold (query << kSlotBits) | slot in an int32
  if (d.n_buckets > 0x7FFFFFFFLL || d.n_inc > (1LL << 31) || p->total_q >= (1 << (31 - kSlotBits)))
    return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

bool op_is_forward(msa_op_t op) { return op == MSA_OP_FORWARD || op == MSA_OP_FORWARD_FP8; }
bool op_uses_index_prefill(msa_op_t op, const Derived& d) {
  return op == MSA_OP_INDEX_POOL || ((op == MSA_OP_INDEX_TOPK || op_is_forward(op)) && !d.decode);
}
bool op_uses_decode_index(msa_op_t op, const Derived& d) {
  return (op == MSA_OP_INDEX_TOPK || op_is_forward(op)) && d.decode;
}
// The index epilogue keeps a top-(k-1) register list per row for k up to this;
// larger k pool the scores into the workspace and select with a separate kernel.
constexpr int kFusedTopkMax = 16;
bool op_uses_pooled_prefill(msa_op_t op, const Derived& d) {
  return (op == MSA_OP_INDEX_TOPK || op_is_forward(op)) && !d.decode && d.topk > kFusedTopkMax;
}
bool op_uses_prefill_attn(msa_op_t op, const Derived& d) {
  return op == MSA_OP_SPARSE_ATTN_PREFILL || op == MSA_OP_SPARSE_ATTN_PREFILL_FP8 || (op_is_forward(op) && !d.decode);
}
bool op_uses_decode_attn(msa_op_t op, const Derived& d) {
  return op == MSA_OP_SPARSE_ATTN_DECODE || op == MSA_OP_SPARSE_ATTN_DECODE_FP8 || (op_is_forward(op) && d.decode);
}
bool op_is_fp8(msa_op_t op) {
  return op == MSA_OP_SPARSE_ATTN_PREFILL_FP8 || op == MSA_OP_SPARSE_ATTN_DECODE_FP8 || op == MSA_OP_FORWARD_FP8;
}

Layout layout(const Derived& d, msa_op_t op) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  L.hdr = take(sizeof(WsHeader));
  L.seq = take(sizeof(SeqInfo) * d.S);
  L.blk_off = take(sizeof(int32_t) * (d.S + 1));
  L.tile_base = take(sizeof(int32_t) * (d.S + 1));
  L.hist = take(sizeof(int32_t) * (d.max_nb + 2));
  L.cursor = take(sizeof(int32_t) * (d.max_nb + 2));
  if (op_uses_index_prefill(op, d)) L.tiles = take(sizeof(int2) * d.max_tiles);
  if (op_uses_decode_index(op, d) || op_uses_pooled_prefill(op, d))
    L.pooled = take(sizeof(float) * static_cast<size_t>(d.T) * d.hkv * d.max_nb);
  if (op_uses_prefill_attn(op, d)) {
    L.count = take(sizeof(int32_t) * d.n_buckets);
    L.bstart = take(sizeof(int32_t) * (d.n_buckets + 1));
    L.bcursor = take(sizeof(int32_t) * d.n_buckets);
    L.nchunk = take(sizeof(int32_t) * d.n_buckets);
    L.cstart = take(sizeof(int32_t) * (d.n_buckets + 1));
    L.entries = take(sizeof(int32_t) * (d.n_inc > 0 ? d.n_inc : 1));
    L.chunks = take(sizeof(int4) * (d.max_chunks > 0 ? d.max_chunks : 1));
    L.scan_tmp = take(sizeof(int32_t) * scan_tmp_ints(static_cast<int>(d.n_buckets)));
    L.v16 = take(sizeof(__half) * static_cast<size_t>(d.N) * d.hkv * kHeadDim);
    if (op_is_fp8(op)) L.k16 = take(sizeof(__nv_bfloat16) * static_cast<size_t>(d.N) * d.hkv * kHeadDim);
  }
  if (op_uses_prefill_attn(op, d) || op_uses_decode_attn(op, d)) {
    L.part_o = take(sizeof(uint16_t) * static_cast<size_t>(d.n_inc) * d.G * kHeadDim);
    L.part_lse = take(sizeof(float) * static_cast<size_t>(d.n_inc) * d.G);
    L.part_ow = take(sizeof(float) * static_cast<size_t>(d.n_inc) * d.G);
  }
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- device facts
struct DeviceFacts {
  int sms = 0;
  bool ok = false;
};

msa_status_t device_facts(DeviceFacts& f) {
  static std::mutex mu;
  static DeviceFacts cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MSA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev].ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MSA_ERR_DEVICE;
    if (major != 10 || minor != 3) return MSA_ERR_DEVICE;
    cache[dev].sms = sms;
    cache[dev].ok = true;
  }
  f = cache[dev];
  return MSA_OK;
}

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// bf16 tensor of `rank` dims (innermost first), 128-byte swizzle, zero fill.
bool make_map(CUtensorMap& m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
              const cuuint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(&m, dtype, rank, const_cast<void*>(ptr), dims, strides_bytes, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    std::snprintf(t_error_detail, sizeof t_error_detail, "tensor map encode failed (CUresult %d, rank %d)",
                  static_cast<int>(r), rank);
  return r == CUDA_SUCCESS;
}

// [rows, cols] row-major, box = 64 columns x box_rows rows
bool map_2d(CUtensorMap& m, const void* ptr, long long rows, int cols, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  return make_map(m, ptr, 2, dims, strides, box);
}

// [n, heads, 128] row-major, box = 64 dims x box_heads heads x box_rows rows
bool map_3d(CUtensorMap& m, const void* ptr, long long n, int heads, int box_heads, int box_rows,
            CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(n > 0 ? n : 1)};
  cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(heads) * 256};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(box_rows)};
  return make_map(m, ptr, 3, dims, strides, box, dtype);
}

// E4M3 codes [rows, cols] (one byte each), box = 128 codes x box_rows rows
bool map_2d_u8(CUtensorMap& m, const void* ptr, long long rows, int cols, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  return make_map(m, ptr, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// E4M3 codes [n, heads, 128] (one byte each), box = 128 codes x 1 head x 128 rows
bool map_3d_u8(CUtensorMap& m, const void* ptr, long long n, int heads) {
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(n > 0 ? n : 1)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(heads) * 128};
  cuuint32_t box[3] = {128, 1, 128};
  return make_map(m, ptr, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// Q [n, hq, 128] seen per (query, group) with the group's G heads split into
// 8-row groups and each row into its two 64-dim halves: dims {64 dims, 8 heads,
// 2 halves, G / 8 row groups, n * hkv query-groups}.  One box = one query's
// group, landing as [row group][half][8 rows][128 B] (128-byte swizzle).
bool map_q_groups(CUtensorMap& m, const void* ptr, long long n, int hkv, int G) {
  const long long nqg = n * hkv;
  cuuint64_t dims[5] = {64, 8, 2, static_cast<cuuint64_t>(G / 8), static_cast<cuuint64_t>(nqg > 0 ? nqg : 1)};
  cuuint64_t strides[4] = {256, 128, 8 * 256, static_cast<cuuint64_t>(G) * 256};
  cuuint32_t box[5] = {64, 8, 2, static_cast<cuuint32_t>(G / 8), 1};
  return make_map(m, ptr, 5, dims, strides, box);
}

// ---------------------------------------------------------------- common prologue
struct Ctx {
  Derived d;
  Layout L;
  DeviceFacts dev;
  WsHeader* hdr;
  SeqInfo* seq;
  cudaStream_t stream;
  void* ws;
  // decode from a paged cache (msa_forward_decode_paged): null block_table = packed rows
  const int32_t* block_table = nullptr;
  int bt_stride = 0;
  long long n_pages = 0;
  // fp8 K/V: k and v are E4M3 codes with these scales [n_key_blocks, hkv]
  bool fp8 = false;
  const float* k_scale = nullptr;
  const float* v_scale = nullptr;
  // fp8 index: q_idx and k_idx are E4M3 codes with these scales ([total_q * hkv] and [n_key_blocks])
  bool fp8_index = false;
  const float* q_idx_scale = nullptr;
  const float* k_idx_scale = nullptr;
  long long cache_rows() const { return block_table ? n_pages * 128 : d.N; }
};

msa_status_t begin(const msa_problem_t* p, msa_op_t op, void* ws, size_t ws_bytes, msa_stream_t stream,
                   Ctx& c) {
  t_stage = -1;
  t_error_detail[0] = 0;
  msa_status_t st = derive(p, c.d);
  if (st != MSA_OK) return st;
  if ((op == MSA_OP_SPARSE_ATTN_DECODE || op == MSA_OP_SPARSE_ATTN_DECODE_FP8) && !c.d.decode)
    return MSA_ERR_INVALID_ARG;
  // decode batches: exactly one query per sequence
  if ((op_uses_decode_index(op, c.d) || op_uses_decode_attn(op, c.d)) && c.d.T != c.d.S) return MSA_ERR_INVALID_ARG;
  if (op_uses_decode_index(op, c.d) && c.d.hkv > 8) return MSA_ERR_UNSUPPORTED;
  c.L = layout(c.d, op);
  if (!ws || ws_bytes < c.L.total) return MSA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return MSA_ERR_ALIGNMENT;
  st = device_facts(c.dev);
  if (st != MSA_OK) return st;
  c.ws = ws;
  c.hdr = at<WsHeader>(ws, c.L.hdr);
  c.seq = at<SeqInfo>(ws, c.L.seq);
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  return MSA_OK;
}

// total_q == num_seqs with every q_len <= 1 means exactly one query per sequence, so query i belongs to
// sequence i (cu_seqlens that say otherwise fail the plan kernel's check, and every later kernel skips).
bool one_query_per_seq(const Derived& d) { return d.T == d.S && d.max_q <= 1; }

msa_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MSA_OK;
  std::snprintf(t_error_detail, sizeof t_error_detail, "stage %s: %s (%d)",
                t_stage >= 0 ? kStageNames[t_stage] : "setup", cudaGetErrorName(e), static_cast<int>(e));
  return MSA_ERR_CUDA;
}

msa_status_t run_plan(const msa_problem_t* p, Ctx& c, int qt) {
  StageScope scope(MSA_STAGE_PLAN, c.stream);
  PlanParams pp{};
  pp.num_seqs = c.d.S;
  pp.cu_q = p->cu_seqlens_q;
  pp.cu_k = p->cu_seqlens_k;
  pp.total_q = c.d.T;
  pp.total_k = c.d.N;
  pp.max_q = c.d.max_q;
  pp.max_k = c.d.max_k;
  pp.qt = qt;
  pp.max_nb = c.d.max_nb;
  pp.seq = c.seq;
  pp.blk_off = at<int32_t>(c.ws, c.L.blk_off);
  pp.tile_base = at<int32_t>(c.ws, c.L.tile_base);
  pp.hist = at<int32_t>(c.ws, c.L.hist);
  pp.cursor = at<int32_t>(c.ws, c.L.cursor);
  pp.tiles = qt > 0 ? at<int2>(c.ws, c.L.tiles) : nullptr;
  pp.hdr = c.hdr;
  return cuda_status(launch_plan(pp, c.stream));
}

msa_status_t run_index_prefill(const msa_problem_t* p, Ctx& c, const void* q_idx, const void* k_idx, bool fused,
                               float* pooled, int64_t pooled_stride, int32_t* idx) {
  if (c.d.T == 0) return MSA_OK;
  CUtensorMap tq, tk;
  const long long q_rows = static_cast<long long>(c.d.T) * c.d.hkv;
  // index scoring loads two key blocks per box
  if (c.fp8_index ? (!map_2d_u8(tq, q_idx, q_rows, c.d.d_idx, 128) || !map_2d_u8(tk, k_idx, c.d.N, c.d.d_idx, 256))
                  : (!map_2d(tq, q_idx, q_rows, c.d.d_idx, 128) || !map_2d(tk, k_idx, c.d.N, c.d.d_idx, 256)))
    return MSA_ERR_CUDA;
  IndexParams ip{};
  ip.q_scale = c.q_idx_scale;
  ip.k_scale = c.k_idx_scale;
  ip.blk_off = at<int32_t>(c.ws, c.L.blk_off);
  ip.seq = c.seq;
  ip.tiles = at<int2>(c.ws, c.L.tiles);
  ip.hdr = c.hdr;
  ip.hkv = c.d.hkv;
  ip.d_idx = c.d.d_idx;
  ip.topk = c.d.topk;
  ip.qt = c.d.qt;
  ip.pooled = pooled;
  ip.pooled_stride = pooled_stride;
  ip.idx = idx;
  long long grid = c.d.max_tiles;
  if (grid > c.dev.sms) grid = c.dev.sms;
  if (grid < 1) grid = 1;
  StageScope scope(MSA_STAGE_INDEX, c.stream);
  return cuda_status(launch_index_score(tq, tk, ip, fused, c.fp8_index, static_cast<int>(grid), c.stream));
  (void)p;
}

msa_status_t run_topk_pooled(const msa_problem_t* p, Ctx& c, const float* pooled, int64_t stride, int32_t* idx) {
  TopkParams tp{};
  tp.num_seqs = c.d.S;
  tp.total_q = c.d.T;
  tp.hkv = c.d.hkv;
  tp.topk = c.d.topk;
  tp.max_nb = static_cast<int>(stride < c.d.max_nb ? stride : c.d.max_nb);
  tp.one_query_per_seq = one_query_per_seq(c.d);
  tp.cu_q = p->cu_seqlens_q;
  tp.seq = c.seq;
  tp.pooled = pooled;
  tp.pooled_stride = stride;
  tp.idx = idx;
  tp.hdr = c.hdr;
  StageScope scope(MSA_STAGE_TOPK, c.stream);
  return cuda_status(launch_topk_pooled(tp, c.d.max_nb, c.stream));
}

msa_status_t run_index_decode(const msa_problem_t* p, Ctx& c, const void* q_idx, const void* k_idx, int32_t* idx) {
  if (c.d.T == 0) return MSA_OK;
  CUtensorMap tk;
  if (c.fp8_index ? !map_2d_u8(tk, k_idx, c.cache_rows(), c.d.d_idx, 128)
                  : !map_2d(tk, k_idx, c.cache_rows(), c.d.d_idx, 128))
    return MSA_ERR_CUDA;
  float* pooled = at<float>(c.ws, c.L.pooled);
  DecodeScanParams sp{};
  sp.num_seqs = c.d.S;
  sp.hkv = c.d.hkv;
  sp.d_idx = c.d.d_idx;
  sp.seq = c.seq;
  if (c.fp8_index) {
    sp.q_idx8 = static_cast<const uint8_t*>(q_idx);
    sp.q_scale = c.q_idx_scale;
    sp.k_scale = c.k_idx_scale;
  } else {
    sp.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  }
  sp.blk_off = at<int32_t>(c.ws, c.L.blk_off);
  sp.pooled = pooled;
  sp.pooled_stride = c.d.max_nb;
  // Work units of consecutive key blocks, dealt to the CTAs in turn; every sequence gets ups units (the
  // ones past a shorter sequence's end are skipped).  bf16 keys: about 4 units per SM in total, at least 16
  // blocks each.  E4M3 codes: 4 blocks (64 KB) per unit, so that the CTAs read the stream close together;
  // it measured 5 % faster per all-fp8 decode step (decode_1m 0.1815 against 0.1913 ms, decode_128k 0.238
  // against 0.251), while bf16 keys moved within 1 % either way.  Small units only while the sequences'
  // lengths are close (the skipped units at most about as many as the real ones): a batch of one long
  // cache and many short ones keeps the few large units.
  const long long key_blocks = (static_cast<long long>(c.d.N) + kBlock - 1) / kBlock;  // at most the real ones
  const bool small_units = c.fp8_index && static_cast<long long>(c.d.S) * c.d.max_nb <= 2 * key_blocks;
  int ups, bpu;
  if (small_units) {
    bpu = 4;
    ups = (c.d.max_nb + bpu - 1) / bpu;
  } else {
    const long long want_units = 4LL * c.dev.sms;
    ups = static_cast<int>((want_units + c.d.S - 1) / c.d.S);
    if (ups < 1) ups = 1;
    bpu = (c.d.max_nb + ups - 1) / ups;
    if (bpu < 16) bpu = 16;
    ups = (c.d.max_nb + bpu - 1) / bpu;
  }
  sp.units_per_seq = ups;
  sp.blocks_per_unit = bpu;
  sp.total_k = c.cache_rows();
  sp.hdr = c.hdr;
  sp.block_table = c.block_table;
  sp.bt_stride = c.bt_stride;
  sp.n_pages = c.n_pages;
  long long units = static_cast<long long>(c.d.S) * ups;
  int grid = static_cast<int>(units < c.dev.sms ? units : c.dev.sms);
  if (grid < 1) grid = 1;
  msa_status_t st;
  {
    StageScope scope(MSA_STAGE_INDEX, c.stream);
    st = cuda_status(launch_decode_scan(tk, sp, c.fp8_index, grid, c.stream));
  }
  if (st != MSA_OK) return st;
  return run_topk_pooled(p, c, pooled, c.d.max_nb, idx);
}

// Index Branch of a prefill batch: scores, max-pool and top-k in one kernel
// (k <= kFusedTopkMax), or pooled scores into the workspace, then top-k.
msa_status_t run_index_select_prefill(const msa_problem_t* p, Ctx& c, const void* q_idx, const void* k_idx,
                                      int32_t* idx) {
  if (c.d.topk <= kFusedTopkMax) return run_index_prefill(p, c, q_idx, k_idx, true, nullptr, 0, idx);
  if (c.d.T == 0) return MSA_OK;
  float* pooled = at<float>(c.ws, c.L.pooled);
  msa_status_t st = run_index_prefill(p, c, q_idx, k_idx, false, pooled, c.d.max_nb, nullptr);
  if (st != MSA_OK) return st;
  return run_topk_pooled(p, c, pooled, c.d.max_nb, idx);
}

PartialBuffers partials(Ctx& c) {
  PartialBuffers pb;
  pb.o = at<uint16_t>(c.ws, c.L.part_o);
  pb.lse = at<float>(c.ws, c.L.part_lse);
  pb.ow = at<float>(c.ws, c.L.part_ow);
  return pb;
}

msa_status_t run_combine(const msa_problem_t* p, Ctx& c, const int32_t* idx, void* o, float* lse,
                         bool f16_partials) {
  CombineParams cp{};
  cp.total_q = c.d.T;
  cp.hq = c.d.hq;
  cp.hkv = c.d.hkv;
  cp.group = c.d.G;
  cp.topk = c.d.topk;
  cp.num_seqs = c.d.S;
  cp.one_query_per_seq = one_query_per_seq(c.d);
  cp.sms = c.dev.sms;
  cp.cu_q = p->cu_seqlens_q;
  cp.seq = c.seq;
  cp.idx = idx;
  cp.part = partials(c);
  cp.o = static_cast<__nv_bfloat16*>(o);
  cp.lse = lse;
  cp.hdr = c.hdr;
  StageScope scope(MSA_STAGE_COMBINE, c.stream);
  return cuda_status(launch_combine(cp, f16_partials, c.stream));
}

msa_status_t run_attn_prefill(const msa_problem_t* p, Ctx& c, const void* q, const void* k, const void* v,
                              const int32_t* idx, void* o, float* lse) {
  if (c.d.T == 0) return MSA_OK;
  ScheduleParams sp{};
  sp.num_seqs = c.d.S;
  sp.total_q = c.d.T;
  sp.hkv = c.d.hkv;
  sp.topk = c.d.topk;
  sp.window = kWindow;
  sp.total_blocks = c.d.total_blocks;
  sp.n_windows = c.d.n_windows;
  sp.qpc = c.d.qpc;
  sp.cu_q = p->cu_seqlens_q;
  sp.seq = c.seq;
  sp.blk_off = at<int32_t>(c.ws, c.L.blk_off);
  sp.idx = idx;
  sp.count = at<int32_t>(c.ws, c.L.count);
  sp.bucket_start = at<int32_t>(c.ws, c.L.bstart);
  sp.cursor = at<int32_t>(c.ws, c.L.bcursor);
  sp.nchunk = at<int32_t>(c.ws, c.L.nchunk);
  sp.chunk_start = at<int32_t>(c.ws, c.L.cstart);
  sp.entries = at<int32_t>(c.ws, c.L.entries);
  sp.chunks = at<int4>(c.ws, c.L.chunks);
  sp.scan_tmp = at<int32_t>(c.ws, c.L.scan_tmp);
  sp.hdr = c.hdr;
  sp.n_buckets = c.d.n_buckets;
  msa_status_t st;
  {
    StageScope scope(MSA_STAGE_SCHEDULE, c.stream);
    st = cuda_status(launch_schedule(sp, c.stream));
  }
  if (st != MSA_OK) return st;

  __half* v16 = at<__half>(c.ws, c.L.v16);
  // fp8 K/V: the Main Branch reads exact 16-bit copies of the codes (K bf16, V fp16)
  __nv_bfloat16* k16 = c.fp8 ? at<__nv_bfloat16>(c.ws, c.L.k16) : nullptr;
  CUtensorMap tq, tk, tv;
  if (!map_q_groups(tq, q, c.d.T, c.d.hkv, c.d.G) || !map_3d(tk, c.fp8 ? k16 : k, c.d.N, c.d.hkv, 1, 128) ||
      !map_3d(tv, v16, c.d.N, c.d.hkv, 1, 128, CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
    return MSA_ERR_CUDA;
  AttnParams ap{};
  ap.q = static_cast<const __nv_bfloat16*>(q);
  ap.seq = c.seq;
  ap.chunks = sp.chunks;
  ap.entries = sp.entries;
  ap.part = partials(c);
  ap.hdr = c.hdr;
  ap.hkv = c.d.hkv;
  ap.group = c.d.G;
  ap.topk = c.d.topk;
  ap.qpt = c.d.qpt;
  ap.scale_log2 = c.d.scale * 1.4426950408889634f;
  ap.k_scale = c.k_scale;
  ap.v_scale = c.v_scale;
  ap.blk_off = at<int32_t>(c.ws, c.L.blk_off);
  {
    StageScope scope(MSA_STAGE_ATTN, c.stream);
    const long long n_elems = static_cast<long long>(c.d.N) * c.d.hkv * kHeadDim;
    if (c.fp8)
      st = cuda_status(launch_kv8_widen(static_cast<const uint8_t*>(k), static_cast<const uint8_t*>(v), k16, v16,
                                        n_elems, c.hdr, c.dev.sms, c.stream));
    else
      st = cuda_status(launch_v_prep(static_cast<const __nv_bfloat16*>(v), v16, n_elems, c.hdr, c.dev.sms,
                                     c.stream));
    if (st == MSA_OK) st = cuda_status(launch_sparse_attn(tq, tk, tv, ap, c.dev.sms, c.stream));
  }
  if (st != MSA_OK) return st;
  return run_combine(p, c, idx, o, lse, true);
}

msa_status_t run_attn_decode(const msa_problem_t* p, Ctx& c, const void* q, const void* k, const void* v,
                             const int32_t* idx, void* o, float* lse) {
  if (c.d.T == 0) return MSA_OK;
  CUtensorMap tq, tk, tv;
  if (!map_3d(tq, q, c.d.T, c.d.hq, c.d.G < 16 ? c.d.G : 16, 1)) return MSA_ERR_CUDA;
  if (c.fp8 ? (!map_3d_u8(tk, k, c.cache_rows(), c.d.hkv) || !map_3d_u8(tv, v, c.cache_rows(), c.d.hkv))
            : (!map_3d(tk, k, c.cache_rows(), c.d.hkv, 1, 128) || !map_3d(tv, v, c.cache_rows(), c.d.hkv, 1, 128)))
    return MSA_ERR_CUDA;
  DecodeAttnParams dp{};
  dp.num_seqs = c.d.S;
  dp.hkv = c.d.hkv;
  dp.group = c.d.G;
  dp.topk = c.d.topk;
  dp.seq = c.seq;
  dp.idx = idx;
  dp.part = partials(c);
  dp.scale_log2 = c.d.scale * 1.4426950408889634f;
  dp.hdr = c.hdr;
  dp.sms = c.dev.sms;
  dp.block_table = c.block_table;
  dp.bt_stride = c.bt_stride;
  dp.n_pages = c.n_pages;
  dp.k_scale = c.k_scale;
  dp.v_scale = c.v_scale;
  dp.blk_off = at<int32_t>(c.ws, c.L.blk_off);
  msa_status_t st;
  {
    StageScope scope(MSA_STAGE_ATTN, c.stream);
    st = cuda_status(launch_decode_attn(tq, tk, tv, dp, c.fp8, c.stream));
  }
  if (st != MSA_OK) return st;
  return run_combine(p, c, idx, o, lse, false);
}

}  // namespace
}  // namespace msa

// ----------------------------------------------------------------------------
// Fixed device scratch for msa_sparse_attn_decode_static: the workspace that
// msa_sparse_attn_decode takes from its caller lives here instead.  Every GPU
// that loads this library holds these bytes until the process exits.
// ----------------------------------------------------------------------------
static __device__ __align__(256) uint8_t msa_static_scratch[MSA_STATIC_SCRATCH_BYTES];

namespace msa {
namespace {

// Identifier of the calling thread's current CUDA context (unique for the
// life of the process, never reused), or 0 when it cannot be read.
unsigned long long current_context_id() {
  using GetCtx = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCtx get_ctx = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_ctx = reinterpret_cast<GetCtx>(a);
      get_id = reinterpret_cast<GetId>(b);
    }
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_ctx || !get_id || get_ctx(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of msa_static_scratch on the current device.  In host code
// the array's name only stands in for the symbol, so the address is looked up
// with that device current and cached per device, together with the context it
// belongs to: after a device reset (a new primary context) it is looked up
// again.
msa_status_t static_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MSA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (!addr[dev] || (ctx != 0 && ctx != ctx_of[dev])) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, msa_static_scratch);
    if (e != cudaSuccess || !ptr) {
      std::snprintf(t_error_detail, sizeof t_error_detail, "cudaGetSymbolAddress of the static scratch: %s (%d)",
                    cudaGetErrorName(e), static_cast<int>(e));
      return MSA_ERR_CUDA;
    }
    addr[dev] = ptr;
    ctx_of[dev] = ctx;
  }
  *out = addr[dev];
  return MSA_OK;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" {

int32_t msa_abi_version(void) { return 1; }

msa_status_t msa_set_stage_events(void* const* events) {
  if (!events) {
    t_stage_events_on = false;
    return MSA_OK;
  }
  for (int i = 0; i < 2 * MSA_NUM_STAGES; ++i) {
    if (!events[i]) return MSA_ERR_INVALID_ARG;
    t_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
  }
  t_stage_events_on = true;
  return MSA_OK;
}

int64_t msa_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* msa_last_error_detail(void) { return t_error_detail; }

const char* msa_status_string(msa_status_t s) {
  switch (s) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case MSA_ERR_ALIGNMENT: return "misaligned pointer";
    case MSA_ERR_WORKSPACE: return "workspace missing or too small";
    case MSA_ERR_CUDA: return "CUDA call or kernel launch failed";
    case MSA_ERR_DEVICE: return "no usable sm_103 device";
  }
  return "unknown status";
}

msa_status_t msa_workspace_size(const msa_problem_t* problem, msa_op_t op, size_t* bytes) {
  if (!bytes) return MSA_ERR_INVALID_ARG;
  if (op < MSA_OP_INDEX_POOL || op > MSA_OP_QUANTIZE_INDEX_FP8) return MSA_ERR_INVALID_ARG;
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  *bytes = layout(d, op).total;
  return MSA_OK;
}

msa_status_t msa_index_pool(const msa_problem_t* problem, const void* q_idx, const void* k_idx, float* pooled,
                            int64_t pooled_stride, void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if (!q_idx || !k_idx || !pooled) return MSA_ERR_INVALID_ARG;
  if (pooled_stride < d.max_nb) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(pooled)) return MSA_ERR_ALIGNMENT;
  Ctx c;
  if ((st = begin(problem, MSA_OP_INDEX_POOL, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  if ((st = run_plan(problem, c, c.d.qt)) != MSA_OK) return st;
  return run_index_prefill(problem, c, q_idx, k_idx, false, pooled, pooled_stride, nullptr);
}

msa_status_t msa_topk_pooled(const msa_problem_t* problem, const float* pooled, int64_t pooled_stride,
                             int32_t* idx, void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if (!pooled || !idx) return MSA_ERR_INVALID_ARG;
  if (pooled_stride < d.max_nb) return MSA_ERR_INVALID_ARG;
  if (!aligned16(pooled) || !aligned16(idx)) return MSA_ERR_ALIGNMENT;
  Ctx c;
  if ((st = begin(problem, MSA_OP_TOPK_POOLED, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  if (c.d.T == 0) return MSA_OK;
  return run_topk_pooled(problem, c, pooled, pooled_stride, idx);
}

msa_status_t msa_index_topk(const msa_problem_t* problem, const void* q_idx, const void* k_idx, int32_t* idx,
                            void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if (!q_idx || !k_idx || !idx) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(idx)) return MSA_ERR_ALIGNMENT;
  Ctx c;
  if ((st = begin(problem, MSA_OP_INDEX_TOPK, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  if (c.d.decode) {
    if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
    return run_index_decode(problem, c, q_idx, k_idx, idx);
  }
  if ((st = run_plan(problem, c, c.d.qt)) != MSA_OK) return st;
  return run_index_select_prefill(problem, c, q_idx, k_idx, idx);
}

static msa_status_t check_attn_args(const void* q, const void* k, const void* v, const int32_t* idx,
                                    const void* o, const float* lse) {
  if (!q || !k || !v || !idx || !o || !lse) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(idx) || !aligned16(o) || !aligned16(lse))
    return MSA_ERR_ALIGNMENT;
  return MSA_OK;
}

msa_status_t msa_sparse_attn_prefill(const msa_problem_t* problem, const void* q, const void* k, const void* v,
                                     const int32_t* idx, void* o, float* lse, void* workspace,
                                     size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_attn_args(q, k, v, idx, o, lse)) != MSA_OK) return st;
  Ctx c;
  if ((st = begin(problem, MSA_OP_SPARSE_ATTN_PREFILL, workspace, workspace_bytes, stream, c)) != MSA_OK)
    return st;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  return run_attn_prefill(problem, c, q, k, v, idx, o, lse);
}

msa_status_t msa_sparse_attn_decode(const msa_problem_t* problem, const void* q, const void* k, const void* v,
                                    const int32_t* idx, void* o, float* lse, void* workspace,
                                    size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_attn_args(q, k, v, idx, o, lse)) != MSA_OK) return st;
  Ctx c;
  if ((st = begin(problem, MSA_OP_SPARSE_ATTN_DECODE, workspace, workspace_bytes, stream, c)) != MSA_OK)
    return st;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  return run_attn_decode(problem, c, q, k, v, idx, o, lse);
}

msa_status_t msa_sparse_attn_decode_static(const msa_problem_t* problem, const void* q, const void* k,
                                           const void* v, const int32_t* idx, void* o, float* lse,
                                           msa_stream_t stream) {
  t_error_detail[0] = 0;
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_attn_args(q, k, v, idx, o, lse)) != MSA_OK) return st;
  const size_t need = layout(d, MSA_OP_SPARSE_ATTN_DECODE).total;
  if (need > MSA_STATIC_SCRATCH_BYTES) {
    std::snprintf(t_error_detail, sizeof t_error_detail,
                  "this batch needs %zu bytes of scratch; the static buffer holds %zu", need,
                  static_cast<size_t>(MSA_STATIC_SCRATCH_BYTES));
    return MSA_ERR_WORKSPACE;
  }
  DeviceFacts dev;
  if ((st = device_facts(dev)) != MSA_OK) return st;
  void* scratch = nullptr;
  if ((st = static_scratch_address(&scratch)) != MSA_OK) return st;
  Ctx c;
  if ((st = begin(problem, MSA_OP_SPARSE_ATTN_DECODE, scratch, MSA_STATIC_SCRATCH_BYTES, stream, c)) != MSA_OK)
    return st;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;  // clears the scratch header first
  return run_attn_decode(problem, c, q, k, v, idx, o, lse);
}

msa_status_t msa_forward(const msa_problem_t* problem, const void* q, const void* k, const void* v,
                         const void* q_idx, const void* k_idx, int32_t* idx, void* o, float* lse,
                         void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_attn_args(q, k, v, idx, o, lse)) != MSA_OK) return st;
  if (!q_idx || !k_idx) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx)) return MSA_ERR_ALIGNMENT;
  Ctx c;
  if ((st = begin(problem, MSA_OP_FORWARD, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  if (c.d.decode) {
    if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
    if ((st = run_index_decode(problem, c, q_idx, k_idx, idx)) != MSA_OK) return st;
    return run_attn_decode(problem, c, q, k, v, idx, o, lse);
  }
  if ((st = run_plan(problem, c, c.d.qt)) != MSA_OK) return st;
  if ((st = run_index_select_prefill(problem, c, q_idx, k_idx, idx)) != MSA_OK) return st;
  return run_attn_prefill(problem, c, q, k, v, idx, o, lse);
}

msa_status_t msa_forward_decode_paged(const msa_problem_t* problem, const void* q, const void* k_cache,
                                      const void* v_cache, const void* q_idx, const void* k_idx_cache,
                                      const int32_t* block_table, int32_t max_blocks_per_seq, int64_t num_pages,
                                      int32_t* idx, void* o, float* lse, void* workspace, size_t workspace_bytes,
                                      msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if (!d.decode) return MSA_ERR_INVALID_ARG;  // one query per sequence
  if ((st = check_attn_args(q, k_cache, v_cache, idx, o, lse)) != MSA_OK) return st;
  if (!q_idx || !k_idx_cache || !block_table) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx_cache) || (reinterpret_cast<uintptr_t>(block_table) & 3u))
    return MSA_ERR_ALIGNMENT;
  if (num_pages < 1 || num_pages * 128 >= (1LL << 31)) return MSA_ERR_INVALID_ARG;
  if (max_blocks_per_seq < d.max_nb) return MSA_ERR_INVALID_ARG;  // a row must hold every block of the longest sequence
  Ctx c;
  if ((st = begin(problem, MSA_OP_FORWARD, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  c.block_table = block_table;
  c.bt_stride = max_blocks_per_seq;
  c.n_pages = num_pages;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  if ((st = run_index_decode(problem, c, q_idx, k_idx_cache, idx)) != MSA_OK) return st;
  return run_attn_decode(problem, c, q, k_cache, v_cache, idx, o, lse);
}

// ---------------------------------------------------------------- index prologue
msa_status_t msa_index_prologue(const msa_problem_t* problem, const void* x, int32_t d_model, const void* w_q,
                                const void* w_k, const void* gamma_q, const void* gamma_k, void* q_idx,
                                void* k_idx, void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if (!x || !w_q || !w_k || !gamma_q || !gamma_k || !q_idx || !k_idx) return MSA_ERR_INVALID_ARG;
  if (d_model <= 0) return MSA_ERR_INVALID_ARG;
  if (d.d_idx != 128 || d_model % 64 || d_model > (1 << 16)) return MSA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w_q) || !aligned16(w_k) || !aligned16(q_idx) || !aligned16(k_idx) ||
      (reinterpret_cast<uintptr_t>(gamma_q) & 1u) || (reinterpret_cast<uintptr_t>(gamma_k) & 1u))
    return MSA_ERR_ALIGNMENT;
  Ctx c;
  if ((st = begin(problem, MSA_OP_INDEX_PROLOGUE, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  if (c.d.T == 0) return MSA_OK;
  CUtensorMap tx, twq, twk;
  if (!map_2d(tx, x, c.d.T, d_model, 128) || !map_2d(twq, w_q, static_cast<long long>(c.d.hkv) * 128, d_model, 128) ||
      !map_2d(twk, w_k, 128, d_model, 64))  // the key head is loaded in 64-row halves (one per CTA of a pair)
    return MSA_ERR_CUDA;
  PrologueParams pp{};
  pp.num_seqs = c.d.S;
  pp.total_q = c.d.T;
  pp.hkv = c.d.hkv;
  pp.d_model = d_model;
  pp.cu_q = problem->cu_seqlens_q;
  pp.seq = c.seq;
  pp.gamma_q = static_cast<const __nv_bfloat16*>(gamma_q);
  pp.gamma_k = static_cast<const __nv_bfloat16*>(gamma_k);
  pp.q_idx = static_cast<__nv_bfloat16*>(q_idx);
  pp.k_idx = static_cast<__nv_bfloat16*>(k_idx);
  for (int j = 0; j < 32; ++j) {
    const double turns = std::pow(10000.0, -j / 32.0) / (2.0 * 3.14159265358979323846);
    pp.rope_turns_hi[j] = static_cast<float>(turns);
    pp.rope_turns_lo[j] = static_cast<float>(turns - static_cast<double>(pp.rope_turns_hi[j]));
  }
  pp.hdr = c.hdr;
  StageScope scope(MSA_STAGE_INDEX, c.stream);
  return cuda_status(launch_index_prologue(tx, twq, twk, pp, c.dev.sms, c.stream));
}

// ---------------------------------------------------------------- fp8 K/V
static msa_status_t check_fp8_args(const void* k8, const void* v8, const float* k_scale, const float* v_scale) {
  if (!k8 || !v8 || !k_scale || !v_scale) return MSA_ERR_INVALID_ARG;
  if (!aligned16(k8) || !aligned16(v8) || (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
      (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return MSA_ERR_ALIGNMENT;
  return MSA_OK;
}

msa_status_t msa_quantize_kv_fp8(const msa_problem_t* problem, const void* k, const void* v, void* k8, void* v8,
                                 float* k_scale, float* v_scale, void* workspace, size_t workspace_bytes,
                                 msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if (!k || !v) return MSA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return MSA_ERR_ALIGNMENT;
  if ((st = check_fp8_args(k8, v8, k_scale, v_scale)) != MSA_OK) return st;
  Ctx c;
  if ((st = begin(problem, MSA_OP_QUANTIZE_KV_FP8, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  QuantParams qp{};
  qp.num_seqs = c.d.S;
  qp.hkv = c.d.hkv;
  qp.seq = c.seq;
  qp.blk_off = at<int32_t>(c.ws, c.L.blk_off);
  qp.k = static_cast<const __nv_bfloat16*>(k);
  qp.v = static_cast<const __nv_bfloat16*>(v);
  qp.k8 = static_cast<uint8_t*>(k8);
  qp.v8 = static_cast<uint8_t*>(v8);
  qp.k_scale = k_scale;
  qp.v_scale = v_scale;
  qp.hdr = c.hdr;
  return cuda_status(launch_quantize_kv_fp8(qp, c.d.N > 0 ? c.d.total_blocks : 0, c.stream));
}

msa_status_t msa_sparse_attn_prefill_fp8(const msa_problem_t* problem, const void* q, const void* k8,
                                         const void* v8, const float* k_scale, const float* v_scale,
                                         const int32_t* idx, void* o, float* lse, void* workspace,
                                         size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_attn_args(q, k8, v8, idx, o, lse)) != MSA_OK) return st;
  if ((st = check_fp8_args(k8, v8, k_scale, v_scale)) != MSA_OK) return st;
  Ctx c;
  if ((st = begin(problem, MSA_OP_SPARSE_ATTN_PREFILL_FP8, workspace, workspace_bytes, stream, c)) != MSA_OK)
    return st;
  c.fp8 = true;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  return run_attn_prefill(problem, c, q, k8, v8, idx, o, lse);
}

msa_status_t msa_sparse_attn_decode_fp8(const msa_problem_t* problem, const void* q, const void* k8,
                                        const void* v8, const float* k_scale, const float* v_scale,
                                        const int32_t* idx, void* o, float* lse, void* workspace,
                                        size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_attn_args(q, k8, v8, idx, o, lse)) != MSA_OK) return st;
  if ((st = check_fp8_args(k8, v8, k_scale, v_scale)) != MSA_OK) return st;
  Ctx c;
  if ((st = begin(problem, MSA_OP_SPARSE_ATTN_DECODE_FP8, workspace, workspace_bytes, stream, c)) != MSA_OK)
    return st;
  c.fp8 = true;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  return run_attn_decode(problem, c, q, k8, v8, idx, o, lse);
}

msa_status_t msa_forward_fp8(const msa_problem_t* problem, const void* q, const void* k8, const void* v8,
                             const float* k_scale, const float* v_scale, const void* q_idx, const void* k_idx,
                             int32_t* idx, void* o, float* lse, void* workspace, size_t workspace_bytes,
                             msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_attn_args(q, k8, v8, idx, o, lse)) != MSA_OK) return st;
  if ((st = check_fp8_args(k8, v8, k_scale, v_scale)) != MSA_OK) return st;
  if (!q_idx || !k_idx) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx)) return MSA_ERR_ALIGNMENT;
  Ctx c;
  if ((st = begin(problem, MSA_OP_FORWARD_FP8, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  c.fp8 = true;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  if (c.d.decode) {
    if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
    if ((st = run_index_decode(problem, c, q_idx, k_idx, idx)) != MSA_OK) return st;
    return run_attn_decode(problem, c, q, k8, v8, idx, o, lse);
  }
  if ((st = run_plan(problem, c, c.d.qt)) != MSA_OK) return st;
  if ((st = run_index_select_prefill(problem, c, q_idx, k_idx, idx)) != MSA_OK) return st;
  return run_attn_prefill(problem, c, q, k8, v8, idx, o, lse);
}

msa_status_t msa_forward_decode_paged_fp8(const msa_problem_t* problem, const void* q, const void* k8_cache,
                                          const void* v8_cache, const float* k_scale, const float* v_scale,
                                          const void* q_idx, const void* k_idx_cache, const int32_t* block_table,
                                          int32_t max_blocks_per_seq, int64_t num_pages, int32_t* idx, void* o,
                                          float* lse, void* workspace, size_t workspace_bytes,
                                          msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if (!d.decode) return MSA_ERR_INVALID_ARG;  // one query per sequence
  if ((st = check_attn_args(q, k8_cache, v8_cache, idx, o, lse)) != MSA_OK) return st;
  if ((st = check_fp8_args(k8_cache, v8_cache, k_scale, v_scale)) != MSA_OK) return st;
  if (!q_idx || !k_idx_cache || !block_table) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx_cache) || (reinterpret_cast<uintptr_t>(block_table) & 3u))
    return MSA_ERR_ALIGNMENT;
  if (num_pages < 1 || num_pages * 128 >= (1LL << 31)) return MSA_ERR_INVALID_ARG;
  if (max_blocks_per_seq < d.max_nb) return MSA_ERR_INVALID_ARG;  // a row must hold every block of the longest sequence
  Ctx c;
  if ((st = begin(problem, MSA_OP_FORWARD_FP8, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  c.fp8 = true;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  c.block_table = block_table;
  c.bt_stride = max_blocks_per_seq;
  c.n_pages = num_pages;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  if ((st = run_index_decode(problem, c, q_idx, k_idx_cache, idx)) != MSA_OK) return st;
  return run_attn_decode(problem, c, q, k8_cache, v8_cache, idx, o, lse);
}

// ---------------------------------------------------------------- fp8 index
static msa_status_t check_fp8_index_args(const Derived& d, const void* q8, const float* q_scale, const void* k8,
                                         const float* k_scale) {
  if (!q8 || !q_scale || !k8 || !k_scale) return MSA_ERR_INVALID_ARG;
  if (d.d_idx != 128) return MSA_ERR_UNSUPPORTED;
  if (!aligned16(q8) || !aligned16(k8) || (reinterpret_cast<uintptr_t>(q_scale) & 3u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u))
    return MSA_ERR_ALIGNMENT;
  return MSA_OK;
}

static void use_fp8_index(Ctx& c, const float* q_scale, const float* k_scale) {
  c.fp8_index = true;
  c.q_idx_scale = q_scale;
  c.k_idx_scale = k_scale;
}

msa_status_t msa_quantize_index_fp8(const msa_problem_t* problem, const void* q_idx, const void* k_idx,
                                    void* q_idx8, float* q_idx_scale, void* k_idx8, float* k_idx_scale,
                                    void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if (!q_idx && !k_idx) return MSA_ERR_INVALID_ARG;
  if ((q_idx && (!q_idx8 || !q_idx_scale)) || (k_idx && (!k_idx8 || !k_idx_scale))) return MSA_ERR_INVALID_ARG;
  if (d.d_idx != 128) return MSA_ERR_UNSUPPORTED;
  if ((q_idx && (!aligned16(q_idx) || !aligned16(q_idx8) || (reinterpret_cast<uintptr_t>(q_idx_scale) & 3u))) ||
      (k_idx && (!aligned16(k_idx) || !aligned16(k_idx8) || (reinterpret_cast<uintptr_t>(k_idx_scale) & 3u))))
    return MSA_ERR_ALIGNMENT;
  Ctx c;
  if ((st = begin(problem, MSA_OP_QUANTIZE_INDEX_FP8, workspace, workspace_bytes, stream, c)) != MSA_OK)
    return st;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  IndexQuantParams qp{};
  qp.num_seqs = c.d.S;
  qp.hkv = c.d.hkv;
  qp.total_q = c.d.T;
  qp.seq = c.seq;
  qp.blk_off = at<int32_t>(c.ws, c.L.blk_off);
  qp.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  qp.k_idx = static_cast<const __nv_bfloat16*>(k_idx);
  qp.q8 = static_cast<uint8_t*>(q_idx8);
  qp.q_scale = q_idx_scale;
  qp.k8 = static_cast<uint8_t*>(k_idx8);
  qp.k_scale = k_idx_scale;
  qp.key_ctas = (k_idx && c.d.N > 0) ? c.d.total_blocks : 0;
  qp.hdr = c.hdr;
  return cuda_status(launch_quantize_index_fp8(qp, c.stream));
}

msa_status_t msa_index_pool_fp8(const msa_problem_t* problem, const void* q_idx8, const float* q_idx_scale,
                                const void* k_idx8, const float* k_idx_scale, float* pooled, int64_t pooled_stride,
                                void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_fp8_index_args(d, q_idx8, q_idx_scale, k_idx8, k_idx_scale)) != MSA_OK) return st;
  if (!pooled) return MSA_ERR_INVALID_ARG;
  if (pooled_stride < d.max_nb) return MSA_ERR_INVALID_ARG;
  if (!aligned16(pooled)) return MSA_ERR_ALIGNMENT;
  Ctx c;
  if ((st = begin(problem, MSA_OP_INDEX_POOL, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  use_fp8_index(c, q_idx_scale, k_idx_scale);
  if ((st = run_plan(problem, c, c.d.qt)) != MSA_OK) return st;
  return run_index_prefill(problem, c, q_idx8, k_idx8, false, pooled, pooled_stride, nullptr);
}

msa_status_t msa_index_topk_fp8(const msa_problem_t* problem, const void* q_idx8, const float* q_idx_scale,
                                const void* k_idx8, const float* k_idx_scale, int32_t* idx, void* workspace,
                                size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_fp8_index_args(d, q_idx8, q_idx_scale, k_idx8, k_idx_scale)) != MSA_OK) return st;
  if (!idx) return MSA_ERR_INVALID_ARG;
  if (!aligned16(idx)) return MSA_ERR_ALIGNMENT;
  Ctx c;
  if ((st = begin(problem, MSA_OP_INDEX_TOPK, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  use_fp8_index(c, q_idx_scale, k_idx_scale);
  if (c.d.decode) {
    if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
    return run_index_decode(problem, c, q_idx8, k_idx8, idx);
  }
  if ((st = run_plan(problem, c, c.d.qt)) != MSA_OK) return st;
  return run_index_select_prefill(problem, c, q_idx8, k_idx8, idx);
}

msa_status_t msa_forward_fp8_index(const msa_problem_t* problem, const void* q, const void* k8, const void* v8,
                                   const float* k_scale, const float* v_scale, const void* q_idx8,
                                   const float* q_idx_scale, const void* k_idx8, const float* k_idx_scale,
                                   int32_t* idx, void* o, float* lse, void* workspace, size_t workspace_bytes,
                                   msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if ((st = check_attn_args(q, k8, v8, idx, o, lse)) != MSA_OK) return st;
  if ((st = check_fp8_args(k8, v8, k_scale, v_scale)) != MSA_OK) return st;
  if ((st = check_fp8_index_args(d, q_idx8, q_idx_scale, k_idx8, k_idx_scale)) != MSA_OK) return st;
  Ctx c;
  if ((st = begin(problem, MSA_OP_FORWARD_FP8, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  c.fp8 = true;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  use_fp8_index(c, q_idx_scale, k_idx_scale);
  if (c.d.decode) {
    if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
    if ((st = run_index_decode(problem, c, q_idx8, k_idx8, idx)) != MSA_OK) return st;
    return run_attn_decode(problem, c, q, k8, v8, idx, o, lse);
  }
  if ((st = run_plan(problem, c, c.d.qt)) != MSA_OK) return st;
  if ((st = run_index_select_prefill(problem, c, q_idx8, k_idx8, idx)) != MSA_OK) return st;
  return run_attn_prefill(problem, c, q, k8, v8, idx, o, lse);
}

msa_status_t msa_forward_decode_paged_fp8_index(const msa_problem_t* problem, const void* q, const void* k8_cache,
                                                const void* v8_cache, const float* k_scale, const float* v_scale,
                                                const void* q_idx8, const float* q_idx_scale,
                                                const void* k_idx8_cache, const float* k_idx_scale,
                                                const int32_t* block_table, int32_t max_blocks_per_seq,
                                                int64_t num_pages, int32_t* idx, void* o, float* lse, void* workspace,
                                                size_t workspace_bytes, msa_stream_t stream) {
  Derived d;
  msa_status_t st = derive(problem, d);
  if (st != MSA_OK) return st;
  if (!d.decode) return MSA_ERR_INVALID_ARG;  // one query per sequence
  if ((st = check_attn_args(q, k8_cache, v8_cache, idx, o, lse)) != MSA_OK) return st;
  if ((st = check_fp8_args(k8_cache, v8_cache, k_scale, v_scale)) != MSA_OK) return st;
  if ((st = check_fp8_index_args(d, q_idx8, q_idx_scale, k_idx8_cache, k_idx_scale)) != MSA_OK) return st;
  if (!block_table) return MSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(block_table) & 3u) return MSA_ERR_ALIGNMENT;
  if (num_pages < 1 || num_pages * 128 >= (1LL << 31)) return MSA_ERR_INVALID_ARG;
  if (max_blocks_per_seq < d.max_nb) return MSA_ERR_INVALID_ARG;  // a row must hold every block of the longest sequence
  Ctx c;
  if ((st = begin(problem, MSA_OP_FORWARD_FP8, workspace, workspace_bytes, stream, c)) != MSA_OK) return st;
  c.fp8 = true;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  use_fp8_index(c, q_idx_scale, k_idx_scale);
  c.block_table = block_table;
  c.bt_stride = max_blocks_per_seq;
  c.n_pages = num_pages;
  if ((st = run_plan(problem, c, 0)) != MSA_OK) return st;
  if ((st = run_index_decode(problem, c, q_idx8, k_idx8_cache, idx)) != MSA_OK) return st;
  return run_attn_decode(problem, c, q, k8_cache, v8_cache, idx, o, lse);
}

msa_status_t msa_read_device_status(const void* workspace, uint32_t* flags, msa_stream_t stream) {
  if (!flags) return MSA_ERR_INVALID_ARG;
  t_error_detail[0] = 0;
  if (!workspace) {  // the fixed scratch of msa_sparse_attn_decode_static on the current device
    void* scratch = nullptr;
    const msa_status_t st = static_scratch_address(&scratch);
    if (st != MSA_OK) return st;
    workspace = scratch;
  }
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return MSA_ERR_ALIGNMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MSA_ERR_CUDA;
  *flags = v;
  return MSA_OK;
}

}  // extern "C"
