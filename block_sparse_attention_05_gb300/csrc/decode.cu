// decode.cu -- decode batches (one new query per sequence).
//
// Index scan: for each sequence, the index scores of its single query against
// every cached index key, max-pooled per 128-token block ("MiniMax Sparse
// Attention: let each query pick its own blocks", section "The mechanism,
// precisely"; the groundtruth.day article on the llama.cpp merge notes that
// selection runs in decode too and that decode then reads about 2,048 KV
// tokens whatever the context length).  The scan streams K_idx once and is
// bound by HBM bandwidth, so it is built for bytes in flight: a persistent
// grid, a TMA producer keeping a ring of 128-key tiles full (6 stages of bf16
// keys, or 12 of E4M3 codes for an fp8 index: the same bytes), and six
// consumer warps.  The 4 group queries against 16 keys are one small mma.sync
// (m16n8k16, or m16n8k32 for E4M3: keys x d_idx times d_idx x groups) -- it
// keeps the instruction count per byte low so the issue slots never limit the
// stream.
//
// Attention: persistent CTAs (two per SM) over the (sequence, group, selected
// block, 16-head slice) items: a producer thread streams each item's Q rows,
// K block and V block by TMA, four warps compute it (16 heads of the group as
// the M = 16 rows of mma.sync tiles, 32 keys per warp) and merge in shared
// memory, then write a normalised partial output and its LSE per slot.  combine.cu merges the
// slots (split-KV with a log-sum-exp combine).
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

// Six consumer warps: block j of a CTA's stream goes to stage j % stages and
// is consumed by warp j % 6; the stage count is a multiple of 6, so every stage
// has a single consumer that takes its fills in order (a parity wait is only
// sound when the waiter already consumed the stage's previous fill).  A stage
// holds one key block: 128 keys x up to 128 dims, bf16 (32 KB), or x 128 E4M3
// codes (16 KB) for an fp8 index; the fp8 ring has twice the stages (two per
// consumer), so the same bytes are in flight per SM.
template <bool FP8>
struct ScanCfg {
  static constexpr int kStages = FP8 ? 12 : 6;
  static constexpr int kConsumers = 6;
  static constexpr int kThreads = 32 * (kConsumers + 1);
  static constexpr int kTile = FP8 ? 128 * 128 : 128 * 128 * 2;
  static constexpr size_t kSmem = 1024 + kStages * kTile + 256;
  static_assert(kStages % kConsumers == 0, "each stage needs a single consumer warp");
};
constexpr int kScanMaxStages = 12;

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D = A(16x32, row) * B(32x8, col) + D, E4M3 inputs, fp32 accumulate.  The
// fragments hold four codes per register where the bf16 shape holds two
// values: a 16-byte row chunk is k 0..15 here, so the same ldmatrix loads
// feed it.
__device__ __forceinline__ void mma_16832_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of (row, 8-element chunk) in a TMA 128-byte-swizzled tile whose
// 64-column halves are 16 KB apart.
__device__ __forceinline__ uint32_t sw128_off(int row, int chunk) {
  return (chunk >> 3) * 16384 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

struct ScanSmem {
  uint64_t full[kScanMaxStages], empty[kScanMaxStages];
  int srow[kScanMaxStages];  // fp8: the K_idx scale row of the block in each stage (written with its fill)
  int abort_flag;
};

// The work of one CTA: units u = blockIdx.x + j * gridDim.x; unit u covers
// blocks [c * bpu, min((c + 1) * bpu, nb)) of sequence u / ups, whose first
// key row k0 and block count nb are cached here (loaded when the sequence
// changes, not once per unit or block).
struct ScanCursor {
  int u, b, b_end, s, k0;
  int cs = -1, nb = 0;  // the sequence whose facts are cached
};

__device__ __forceinline__ bool scan_next(const DecodeScanParams& p, ScanCursor& c) {
  while (true) {
    if (c.b < c.b_end) return true;
    c.u += gridDim.x;
    if (c.u >= p.num_seqs * p.units_per_seq) return false;
    c.s = c.u / p.units_per_seq;
    const int unit = c.u % p.units_per_seq;
    if (c.s != c.cs) {
      const SeqInfo si = p.seq[c.s];
      c.cs = c.s;
      c.nb = (si.kv_len + kBlock - 1) / kBlock;
      c.k0 = si.k_start;
    }
    c.b = unit * p.blocks_per_unit;
    c.b_end = min(c.nb, c.b + p.blocks_per_unit);
  }
}

}  // namespace

// FP8: K_idx holds E4M3 codes (d_idx 128, one 128-byte row per key) with one
// scale per key block, Q_idx codes with one scale per (sequence, group); the
// pooled score is the block's maximum code dot product times both scales.
template <bool FP8>
__global__ void __launch_bounds__(ScanCfg<FP8>::kThreads, 1)
    decode_scan_kernel(const __grid_constant__ CUtensorMap tm_k, DecodeScanParams p) {
  using Cfg = ScanCfg<FP8>;
  constexpr int kScanStages = Cfg::kStages, kScanConsumers = Cfg::kConsumers, kScanTile = Cfg::kTile;
  extern __shared__ uint8_t smem_raw[];
  WsHeader* hdr = p.hdr;
  griddep_wait();  // sequence facts and the header come from the plan kernel
  if (hdr->status & kFlagBadSeqlens) return;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  ScanSmem& sm = *reinterpret_cast<ScanSmem*>(base + kScanStages * kScanTile);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kchunks = FP8 ? 1 : p.d_idx >> 6;
  const uint32_t tile_tx = 128u * p.d_idx * (FP8 ? 1u : 2u);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kScanStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
  }
  __syncthreads();
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == kScanConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ScanCursor c{static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x), 0, 0, 0, 0};
      uint32_t it = 0;
      int blk0_s = -1, blk0 = 0;  // fp8, packed: first key block of sequence blk0_s
      while (scan_next(p, c)) {
        const int st = it % kScanStages;
        if (it >= kScanStages && !mbar_wait(&sm.empty[st], ((it / kScanStages) - 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 301);
          break;
        }
        const int row = key_block_row(p.block_table, p.bt_stride, p.n_pages, c.k0, c.s, c.b, hdr);
        index_ok(hdr, c.s, p.num_seqs, 401);
        index_ok(hdr, row, p.total_k, 402);
        if constexpr (FP8) {
          // the block's K_idx scale row, handed to the consumer with the fill (the consumer then loads the
          // scale under its MMAs): per key block of the sequence (packed) or the page (paged; a page outside
          // the cache, already flagged, reads page 0's)
          if (p.block_table) {
            const int pg = row >> 7;
            sm.srow[st] = pg < p.n_pages ? pg : 0;
          } else {
            if (c.s != blk0_s) {
              blk0_s = c.s;
              blk0 = p.blk_off[c.s];
            }
            sm.srow[st] = blk0 + c.b;
          }
        }
        mbar_arrive_expect_tx(&sm.full[st], tile_tx);
        for (int ch = 0; ch < kchunks; ++ch)
          tma_load_2d(base + st * kScanTile + ch * 16384, &tm_k, &sm.full[st], ch * 64, row);
        ++c.b;
        ++it;
      }
      for (int s = 0; s < kScanStages; ++s)
        if (it > static_cast<uint32_t>(s)) {
          const uint32_t last = ((it - 1 - s) / kScanStages) * kScanStages + s;
          mbar_wait(&sm.full[s], (last / kScanStages) & 1, nullptr);
        }
    }
  } else {
    // ------------------------------------------------------------ consumers
    ScanCursor c{static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x), 0, 0, 0, 0};
    uint32_t it = 0;
    int cur_s = -1;
    uint32_t qf[8][2];
    int pos = 0;
    float qs0 = 1.f, qs1 = 1.f;               // fp8: Q_idx scales of groups 2 lane, 2 lane + 1 (lanes 0..3)
    const int gq = lane >> 2;                 // B-fragment column = group
    while (scan_next(p, c)) {
      const int st = it % kScanStages;
      const int b = c.b;
      ++c.b;
      const uint32_t my = it;
      ++it;
      if ((my % kScanConsumers) != static_cast<uint32_t>(warp)) continue;
      if (c.s != cur_s) {
        cur_s = c.s;
        const SeqInfo si = p.seq[cur_s];
        pos = si.kv_len - 1;
        const int64_t qbase = (static_cast<int64_t>(cur_s) * p.hkv + gq) * p.d_idx;
        const bool q_ok = gq >= p.hkv || index_ok(hdr, qbase + p.d_idx - 1,
                                                  static_cast<long long>(p.num_seqs) * p.hkv * p.d_idx, 403);
        if constexpr (FP8) {
          // m16n8k32 B fragment: codes k = 4 (lane % 4) .. + 3 and 16 + 4 (lane % 4) .. + 3 of each 32
          const uint8_t* qrow = p.q_idx8 + qbase;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            qf[ks][0] = qf[ks][1] = 0u;
            if (q_ok && gq < p.hkv && ks < 4) {
              const int d0 = ks * 32 + (lane & 3) * 4;
              qf[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + d0);
              qf[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + d0 + 16);
            }
          }
          const int g0 = 2 * lane;
          qs0 = (lane < 4 && g0 < p.hkv) ? p.q_scale[static_cast<int64_t>(cur_s) * p.hkv + g0] : 1.f;
          qs1 = (lane < 4 && g0 + 1 < p.hkv) ? p.q_scale[static_cast<int64_t>(cur_s) * p.hkv + g0 + 1] : 1.f;
        } else {
          const __nv_bfloat16* qrow = p.q_idx + qbase;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            qf[ks][0] = qf[ks][1] = 0u;
            if (q_ok && gq < p.hkv && ks * 16 < p.d_idx) {
              const int d0 = ks * 16 + (lane & 3) * 2;
              qf[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + d0);
              qf[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + d0 + 8);
            }
          }
        }
      }
      if (!mbar_wait_warp(&sm.full[st], (my / kScanStages) & 1, abort_flag)) {
        report_timeout(abort_flag, hdr, 311);
        break;
      }
      float k_sc = 1.f;  // fp8: the block's K_idx scale, loaded before the MMAs that hide its latency
      if constexpr (FP8) {
        if (lane < 4) k_sc = p.k_scale[sm.srow[st]];
      }
      const uint32_t tile = smem_u32(base + st * kScanTile);
      float mx0 = -INFINITY, mx1 = -INFINITY;
      const int key_base = b * kBlock;
      const int mtx = lane >> 3, mr = lane & 7;
#pragma unroll
      for (int sub = 0; sub < 8; ++sub) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int arow = sub * 16 + (mtx & 1) * 8 + mr;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          if (FP8 ? ks < 4 : ks * 16 < p.d_idx) {
            uint32_t a[4];
            ldmatrix_x4(tile + sw128_off(arow, ks * 2 + (mtx >> 1)), a[0], a[1], a[2], a[3]);
            if constexpr (FP8)
              mma_16832_e4m3(acc, a, qf[ks][0], qf[ks][1]);
            else
              mma_16816(acc, a, qf[ks][0], qf[ks][1]);
          }
        }
        const int k0 = key_base + sub * 16 + (lane >> 2);
        if (k0 <= pos) {
          mx0 = fmaxf(mx0, acc[0]);
          mx1 = fmaxf(mx1, acc[1]);
        }
        if (k0 + 8 <= pos) {
          mx0 = fmaxf(mx0, acc[2]);
          mx1 = fmaxf(mx1, acc[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[st]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
      }
      if (FP8 && lane < 4) {  // scales are positive: scaling the maximum is the maximum of the scaled scores
        mx0 *= qs0 * k_sc;
        mx1 *= qs1 * k_sc;
      }
      if (lane < 4) {
        const int g0 = lane * 2;
        const long long rows = static_cast<long long>(p.num_seqs) * p.hkv;
        const long long at0 = (static_cast<long long>(cur_s) * p.hkv + g0) * p.pooled_stride + b;
        float* out = p.pooled + static_cast<int64_t>(cur_s) * p.hkv * p.pooled_stride + b;
        if (g0 < p.hkv && index_ok(hdr, at0, rows * p.pooled_stride, 404) && index_ok(hdr, b, p.pooled_stride, 405))
          out[static_cast<int64_t>(g0) * p.pooled_stride] = mx0;
        if (g0 + 1 < p.hkv && index_ok(hdr, at0 + p.pooled_stride, rows * p.pooled_stride, 406))
          out[static_cast<int64_t>(g0 + 1) * p.pooled_stride] = mx1;
      }
    }
  }
  __syncthreads();
}

size_t decode_scan_smem_bytes() { return ScanCfg<false>::kSmem; }

template <bool FP8>
static cudaError_t launch_scan(const CUtensorMap& tk, const DecodeScanParams& p, int grid, cudaStream_t stream) {
  using Cfg = ScanCfg<FP8>;
  cudaError_t e = cudaFuncSetAttribute(decode_scan_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cfg::kSmem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_scan_kernel<FP8>, dim3(grid), dim3(Cfg::kThreads), Cfg::kSmem, stream, tk, p);
  note_launches(1);
  return e;
}

cudaError_t launch_decode_scan(const CUtensorMap& tk, const DecodeScanParams& p, bool fp8, int grid,
                               cudaStream_t stream) {
  return fp8 ? launch_scan<true>(tk, p, grid, stream) : launch_scan<false>(tk, p, grid, stream);
}

// ----------------------------------------------------------------------------
// decode attention
// ----------------------------------------------------------------------------
namespace {

constexpr int kDecThreads = 128;  // compute warps; one more warp streams Q, K and V
// Row stride (floats) of the merge slices: 8 floats of padding put the 8 rows a
// warp's float2 stores touch at once on distinct banks.
constexpr int kOsumStride = 128 + 8;
// Per CTA (two per SM): K and V buffers (32 KB each), the item's Q (4 KB),
// the merge slices and per-warp (max, sum), the item hand-over, barriers.
// fp8 K/V: the E4M3 codes of the item's K and V blocks (16 KB each) land in
// the second half of the K and V buffers and are widened there in place.
constexpr size_t kDecSmemBytes = 1024 + 65536 + 4096 + 4 * 16 * kOsumStride * sizeof(float) +
                                 4 * 16 * 2 * sizeof(float) + 32 + (4 + 5) * 8 + 16;

// Widens one 128-byte row of E4M3 codes (TMA 128-byte swizzled, 16-byte chunks
// XOR row % 8, at tile + 16 KB) into row `row` of the bf16 tile in the layout
// the bf16 loads give (64-dim halves 16 KB apart, 128-byte swizzle).  The
// codes sit where the tile's second half goes: row `row` of the widened
// second half overwrites exactly the 128 bytes of that row's codes, so the
// whole code row is read before anything is written, and each row belongs to
// one thread.  Exact: an E4M3 value has 4 significant bits and fits bf16's
// exponent range.
__device__ __forceinline__ void widen_e4m3_row(uint8_t* tile, int row) {
  const uint8_t* src = tile + 16384;
  uint4 wr[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) wr[c] = *reinterpret_cast<const uint4*>(src + row * 128 + ((c ^ (row & 7)) << 4));
  uint8_t* dst = tile;
#pragma unroll
  for (int c = 0; c < 8; ++c) {  // codes 16c .. 16c + 15
    const uint4 w = wr[c];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __nv_fp8x2_storage_t pr = static_cast<__nv_fp8x2_storage_t>((ws[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
      const __half2 h = *reinterpret_cast<const __half2*>(&hr);
      const __nv_bfloat162 b = __floats2bfloat162_rn(__low2float(h), __high2float(h));
      o[j] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(dst + sw128_off(row, 2 * c)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(dst + sw128_off(row, 2 * c + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// (a, b) -> bf16 pair hi and bf16 pair lo with a ~= hi.x + lo.x, b ~= hi.y + lo.y
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16x2(a - __low2float(h), b - __high2float(h));
}

}  // namespace

// Persistent: two CTAs per SM, each owning the items (sequence, group, slot)
// item = blockIdx.x + j * gridDim.x.  Warp 4 (one thread) walks them, skips
// empty slots, and for each valid item hands the compute warps its output
// slot and causal limit through shared memory and loads its Q rows (16 heads,
// 4 KB) with its K block (32 KB) on one barrier and its V block (32 KB) on
// another.  K and V have a buffer and a pair of barriers each, so the next
// item's Q and K are loaded as soon as this item's S = Q K^T is done (under
// the softmax, P V and the merge) and its V as soon as P V is done; the
// compute warps issue no global loads.  After the last item an arrival
// without bytes on the K barrier, with slot -1, ends the compute warps.
// Per item: 16 heads x 128 keys; each compute warp takes 32 keys (S = Q K^T
// and O_w = P V with mma.sync m16n8k16, P split into bf16 hi + lo), then the
// four warps merge through shared memory (each writes its scaled partial to
// its own slice, then every element is summed over the four slices: no
// shared-memory atomics).
struct DecodeItem {
  long long sel;  // (sequence * hkv + group) * topk + slot, or -1 after the last item
  int lim;        // last visible key of the block (kv_len - 1 - block * 128)
  int hs;         // head slice: heads 16 hs .. 16 hs + 15 of the group
  float sk, sv;   // fp8 K/V: the block's scales (1 for bf16 K/V)
  int pad[2];
};

// Byte offset of (row, 8-element chunk) in the 16-row Q tile: 128-byte
// swizzle, 64-column halves 2 KB apart.
__device__ __forceinline__ uint32_t q_off(int row, int chunk) {
  return (chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// FP8: K and V are E4M3 codes with per-(key block, KV head) scales (tm_k and
// tm_v map the codes); the logits take the K scale and the partial output the
// V scale.
template <bool FP8>
__global__ void __launch_bounds__(kDecThreads + 32)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, DecodeAttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  WsHeader* hdr = p.hdr;
  griddep_wait();  // the selection comes from the top-k kernel
  if (hdr->status & kFlagBadSeqlens) return;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = base;                                                    // K 32 KB | V 32 KB
  uint8_t* qbuf = base + 65536;                                            // Q 16 heads x 128 (4 KB)
  float* osum = reinterpret_cast<float*>(base + 65536 + 4096);             // [4 warps][16 heads][kOsumStride]
  float* red = osum + 4 * 16 * kOsumStride;                                // [4 warps][16 heads][m, l]
  DecodeItem* info = reinterpret_cast<DecodeItem*>(red + 4 * 16 * 2);
  uint64_t* full = reinterpret_cast<uint64_t*>(info + 1);                  // [0] Q + K landed, [1] V landed
  uint64_t* empty = full + 2;                                              // [0] K read, [1] V read
  // per item: red written, partial sums added, merged output read; fp8: K and V codes widened
  uint64_t* mrg = empty + 2;
  int* abort_flag = reinterpret_cast<int*>(mrg + 5);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  // a group's heads are taken 16 at a time (G >= 16: G / 16 head slices per (sequence, group, slot));
  // with G = 8 the tile's last 8 rows are zeros and nothing of theirs is stored
  const int nhs = G >= 16 ? G / 16 : 1;
  const int rows = G >= 16 ? 16 : G;
  const long long n_items = static_cast<long long>(p.num_seqs) * p.hkv * p.topk * nhs;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);  // one arrival per compute warp
    }
    for (int i = 0; i < 5; ++i) mbar_init(&mrg[i], 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (rows < 16) {  // Q rows 8..15 of both 64-dim halves (the loads fill rows 0..7 only)
    for (int i = threadIdx.x; i < 64; i += blockDim.x) {
      reinterpret_cast<uint4*>(qbuf + 1024)[i] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(qbuf + 3072)[i] = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();

  // the block of an item, or -1 for an empty slot (no partial; the combine skips it)
  auto item_block = [&](long long it, int& s, int& g, int& b) {
    const int slot = static_cast<int>(it % p.topk);
    g = static_cast<int>((it / p.topk) % p.hkv);
    s = static_cast<int>(it / (static_cast<long long>(p.topk) * p.hkv));
    b = p.idx[it];  // it == (s * hkv + g) * topk + slot
    const SeqInfo si = p.seq[s];
    if (b < 0 || b > ((si.kv_len - 1) >> 7)) b = -1;
    (void)slot;
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t nk = 0, nv = 0;  // Q + K and V fills issued
      bool stopped = false, ended = false;
      for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
        const long long it = item / nhs;  // (sequence, group, slot)
        const int hs = static_cast<int>(item % nhs);
        int s, g, b;
        item_block(it, s, g, b);
        if (b < 0) continue;
        const int krow = key_block_row(p.block_table, p.bt_stride, p.n_pages, p.seq[s].k_start, s, b, hdr);
        // Q and K of this item once the compute warps have read the previous item's, then V likewise
        if (nk >= 1 && !mbar_wait(&empty[0], (nk - 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 322);
          stopped = true;
          break;
        }
        info->sel = it;
        info->hs = hs;
        info->lim = p.seq[s].kv_len - 1 - b * kBlock;
        info->sk = 1.f;
        info->sv = 1.f;
        if constexpr (FP8) {
          // the block's scales: per key block of the sequence (packed) or per page (paged; a page outside the
          // cache, already flagged, reads page 0's)
          const long long pg = krow >> 7;
          const long long srow =
              (p.block_table ? (pg < p.n_pages ? pg : 0) : static_cast<long long>(p.blk_off[s]) + b) * p.hkv + g;
          info->sk = p.k_scale[srow];
          info->sv = p.v_scale[srow];
        }
        mbar_arrive_expect_tx(&full[0], (FP8 ? 16384 : 32768) + rows * 256);
        tma_load_3d(qbuf, &tm_q, &full[0], 0, g * G + hs * 16, s);
        tma_load_3d(qbuf + 2048, &tm_q, &full[0], 64, g * G + hs * 16, s);
        if constexpr (FP8) {
          tma_load_3d(ring + 16384, &tm_k, &full[0], 0, g, krow);
        } else {
          tma_load_3d(ring, &tm_k, &full[0], 0, g, krow);
          tma_load_3d(ring + 16384, &tm_k, &full[0], 64, g, krow);
        }
        ++nk;
        if (nv >= 1 && !mbar_wait(&empty[1], (nv - 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 323);
          stopped = true;
          break;
        }
        if constexpr (FP8) {
          mbar_arrive_expect_tx(&full[1], 16384);
          tma_load_3d(ring + 49152, &tm_v, &full[1], 0, g, krow);
        } else {
          mbar_arrive_expect_tx(&full[1], 32768);
          tma_load_3d(ring + 32768, &tm_v, &full[1], 0, g, krow);
          tma_load_3d(ring + 49152, &tm_v, &full[1], 64, g, krow);
        }
        ++nv;
      }
      if (!stopped) {
        // no more items: one more phase of the K barrier, without bytes, carries slot -1
        if (nk >= 1 && !mbar_wait(&empty[0], (nk - 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 325);
        } else {
          info->sel = -1;
          mbar_arrive(&full[0]);
          ended = true;  // every Q + K fill has been read, so it has landed
        }
      }
      // let every issued copy land before the CTA exits
      if (!ended && nk >= 1) mbar_wait(&full[0], (nk - 1) & 1, nullptr);
      if (nv >= 1) mbar_wait(&full[1], (nv - 1) & 1, nullptr);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  // The four warps merge each item through shared memory; they meet at three
  // mbarriers per item (bounded waits, so a timeout in one warp ends the others).
  auto meet = [&](int k, uint32_t item_no) -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(&mrg[k]);
    if (!mbar_wait_warp(&mrg[k], item_no & 1, abort_flag)) {
      if (lane == 0) report_timeout(abort_flag, hdr, 330 + k);
      return false;
    }
    return true;
  };
  const volatile DecodeItem* vinfo = info;
  uint32_t n = 0;
  while (true) {
    if (!mbar_wait_warp(&full[0], n & 1, abort_flag)) {
      if (lane == 0) report_timeout(abort_flag, hdr, 321);
      break;
    }
    const long long sel = vinfo->sel;
    const int lim = vinfo->lim;
    const int hs = vinfo->hs;
    const float sk = vinfo->sk, sv = vinfo->sv;
    if (sel < 0) break;
    if constexpr (FP8) {
      widen_e4m3_row(ring, threadIdx.x);
      if (!meet(3, n)) break;
    }
    const float scale_log2 = p.scale_log2 * sk;
    const uint32_t kt = smem_u32(ring), vt = kt + 32768, qt = smem_u32(qbuf);
    const int mtx = lane >> 3, mr = lane & 7;
    // Q fragments (16 heads x 128 dims) for the m16n8k16 A operand
    uint32_t qa[8][4];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      ldmatrix_x4(qt + q_off((mtx & 1) * 8 + mr, k * 2 + (mtx >> 1)), qa[k][0], qa[k][1], qa[k][2], qa[k][3]);

    // S = Q K^T for this warp's 32 keys: 4 n-tiles of 8 keys
    float sacc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) sacc[nt][j] = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
#pragma unroll
      for (int ntp = 0; ntp < 2; ++ntp) {
        // matrices: (keys nt, d lo), (keys nt, d hi), (keys nt+1, d lo), (keys nt+1, d hi)
        const int key = warp * 32 + (ntp * 2 + (mtx >> 1)) * 8 + mr;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kt + sw128_off(key, k * 2 + (mtx & 1)), b0, b1, b2, b3);
        mma_16816(sacc[ntp * 2], qa[k], b0, b1);
        mma_16816(sacc[ntp * 2 + 1], qa[k], b2, b3);
      }
    }
    // this warp is done with Q, K and the item hand-over: the producer may load the next item's
    // (fp8: into the K buffer this CTA's threads wrote, hence the proxy fence)
    if constexpr (FP8) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[0]);
    // masked, scaled logits; per-head max and sum over this warp's keys
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int c0 = warp * 32 + nt * 8 + (lane & 3) * 2;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + (j & 1);
        const float x = (c <= lim) ? sacc[nt][j] * scale_log2 : -INFINITY;
        sacc[nt][j] = x;
      }
      m0 = fmaxf(m0, fmaxf(sacc[nt][0], sacc[nt][1]));
      m1 = fmaxf(m1, fmaxf(sacc[nt][2], sacc[nt][3]));
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, o));
      m1 = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, o));
    }
    const float r0 = (m0 == -INFINITY) ? 0.f : m0, r1 = (m1 == -INFINITY) ? 0.f : m1;
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      sacc[nt][0] = exp2f(sacc[nt][0] - r0);
      sacc[nt][1] = exp2f(sacc[nt][1] - r0);
      sacc[nt][2] = exp2f(sacc[nt][2] - r1);
      sacc[nt][3] = exp2f(sacc[nt][3] - r1);
      l0 += sacc[nt][0] + sacc[nt][1];
      l1 += sacc[nt][2] + sacc[nt][3];
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, o);
      l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
    }
    if (!mbar_wait_warp(&full[1], n & 1, abort_flag)) {
      if (lane == 0) report_timeout(abort_flag, hdr, 324);
      break;
    }
    if constexpr (FP8) {
      widen_e4m3_row(ring + 32768, threadIdx.x);
      if (!meet(4, n)) break;
    }
    // O_w = P V over the warp's 32 keys: 2 k-steps of 16 keys, 16 n-tiles of 8 dims
    float oacc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) oacc[nt][j] = 0.f;
#pragma unroll
    for (int kj = 0; kj < 2; ++kj) {
      // P = hi + lo (both bf16): ~16 significant bits for the PV product
      uint32_t pa[4], pl[4];
      split_bf16x2(sacc[2 * kj][0], sacc[2 * kj][1], pa[0], pl[0]);
      split_bf16x2(sacc[2 * kj][2], sacc[2 * kj][3], pa[1], pl[1]);
      split_bf16x2(sacc[2 * kj + 1][0], sacc[2 * kj + 1][1], pa[2], pl[2]);
      split_bf16x2(sacc[2 * kj + 1][2], sacc[2 * kj + 1][3], pa[3], pl[3]);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        // matrices: (keys lo, d 16dp..+7), (keys hi, same d), (keys lo, d +8..15), (keys hi, d +8..15)
        const int key = warp * 32 + kj * 16 + (mtx & 1) * 8 + mr;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vt + sw128_off(key, dp * 2 + (mtx >> 1)), b0, b1, b2, b3);
        mma_16816(oacc[2 * dp], pa, b0, b1);
        mma_16816(oacc[2 * dp + 1], pa, b2, b3);
        mma_16816(oacc[2 * dp], pl, b0, b1);
        mma_16816(oacc[2 * dp + 1], pl, b2, b3);
      }
    }
    // this warp is done with V
    if constexpr (FP8) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[1]);
    ++n;
    // merge the four warps: rescale to the common max, sum, normalise
    const int h0 = lane >> 2;
    if ((lane & 3) == 0) {
      red[(warp * 16 + h0) * 2 + 0] = m0;
      red[(warp * 16 + h0) * 2 + 1] = l0;
      red[(warp * 16 + h0 + 8) * 2 + 0] = m1;
      red[(warp * 16 + h0 + 8) * 2 + 1] = l1;
    }
    if (!meet(0, n - 1)) break;
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      M0 = fmaxf(M0, red[(w * 16 + h0) * 2]);
      M1 = fmaxf(M1, red[(w * 16 + h0 + 8) * 2]);
    }
    const float R0 = (M0 == -INFINITY) ? 0.f : M0, R1 = (M1 == -INFINITY) ? 0.f : M1;
    float L0 = 0.f, L1 = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw0 = red[(w * 16 + h0) * 2], mw1 = red[(w * 16 + h0 + 8) * 2];
      L0 += (mw0 == -INFINITY) ? 0.f : red[(w * 16 + h0) * 2 + 1] * exp2f(mw0 - R0);
      L1 += (mw1 == -INFINITY) ? 0.f : red[(w * 16 + h0 + 8) * 2 + 1] * exp2f(mw1 - R1);
    }
    // the V scale (fp8) multiplies the normalised partial
    const float f0 = (m0 == -INFINITY || L0 == 0.f) ? 0.f : exp2f(m0 - R0) / L0 * sv;
    const float f1 = (m1 == -INFINITY || L1 == 0.f) ? 0.f : exp2f(m1 - R1) / L1 * sv;
    // each warp's scaled partial into its own slice, then a 4-way sum per element
    float* mine = osum + warp * 16 * kOsumStride;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int d = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2*>(&mine[h0 * kOsumStride + d]) = make_float2(oacc[nt][0] * f0, oacc[nt][1] * f0);
      *reinterpret_cast<float2*>(&mine[(h0 + 8) * kOsumStride + d]) =
          make_float2(oacc[nt][2] * f1, oacc[nt][3] * f1);
    }
    if (!meet(1, n - 1)) break;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.part.o) + (sel * G + hs * 16) * kHeadDim;
    for (int i = threadIdx.x * 8; i < rows * 128; i += kDecThreads * 8) {
      const int at = (i >> 7) * kOsumStride + (i & 127);  // head i / 128, column i % 128
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; j += 4) {
        float4 a = *reinterpret_cast<const float4*>(&osum[at + j]);
#pragma unroll
        for (int w = 1; w < 4; ++w) {
          const float4 b4 = *reinterpret_cast<const float4*>(&osum[w * 16 * kOsumStride + at + j]);
          a.x += b4.x;
          a.y += b4.y;
          a.z += b4.z;
          a.w += b4.w;
        }
        acc[j] = a.x;
        acc[j + 1] = a.y;
        acc[j + 2] = a.z;
        acc[j + 3] = a.w;
      }
      uint4 v;
      v.x = pack_bf16x2(acc[0], acc[1]);
      v.y = pack_bf16x2(acc[2], acc[3]);
      v.z = pack_bf16x2(acc[4], acc[5]);
      v.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(out + i) = v;
    }
    if (threadIdx.x < rows) {
      const int h = threadIdx.x;
      float M = -INFINITY;
      for (int w = 0; w < 4; ++w) M = fmaxf(M, red[(w * 16 + h) * 2]);
      float L = 0.f;
      for (int w = 0; w < 4; ++w) {
        const float mw = red[(w * 16 + h) * 2];
        if (mw != -INFINITY) L += red[(w * 16 + h) * 2 + 1] * exp2f(mw - M);
      }
      const float lse = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * kLn2;
      p.part.lse[sel * G + hs * 16 + h] = lse;
      p.part.ow[sel * G + hs * 16 + h] = lse;  // o is stored normalised
    }
    if (!meet(2, n - 1)) break;  // red and osum are reused by the next item
  }
}

size_t decode_attn_smem_bytes() { return kDecSmemBytes; }

cudaError_t launch_decode_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeAttnParams& p, bool fp8, cudaStream_t stream) {
  const long long items = static_cast<long long>(p.num_seqs) * p.hkv * p.topk * (p.group >= 16 ? p.group / 16 : 1);
  if (items == 0) return cudaSuccess;
  // persistent: two CTAs per SM
  const long long grid = items < 2LL * p.sms ? items : 2LL * p.sms;
  const size_t smem = kDecSmemBytes;
  auto* fn = fp8 ? decode_attn_kernel<true> : decode_attn_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(fn, dim3(static_cast<unsigned>(grid)), dim3(kDecThreads + 32), smem, stream, tq, tk, tv, p);
  note_launches(1);
  return e;
}

}  // namespace msa
