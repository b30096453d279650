// prologue.cu -- index prologue: hidden states -> index query and key heads.
//
// "MiniMax Sparse Attention: let each query pick its own blocks", Figure 1:
// the Index Branch takes the hidden states through a linear projection, a norm
// and RoPE to the index query heads (one per GQA group) and the shared index
// key head.  The atlas record of the report gives d_model = 3072 and a RoPE
// dimension of 64 on 128-dim heads; the norm is not named.  This library
// reads it as: per-head RMSNorm with a learned weight (gamma_q shared by the
// index query heads, gamma_k for the key head), eps 1e-6, then rotate-half
// RoPE on the first 64 dims, pairs (j, j + 32), angle pos * 10000^(-j/32).
//
// One GEMM, X [T, d_model] x W^T with W = the hkv query heads' rows followed
// by the key head's (128 output columns each), on the tensor cores: work item
// = 128 token rows x two heads (N = 256), or, for a lone last head, 256 token
// rows x that head (two 128 x 128 MMAs sharing its weight tile, the second row
// tile staged in the unused half of the weight stage), so every item does the
// same 4.2 MFLOP per K step; K looped in 64-column blocks, A and B tiles by
// TMA (128-byte swizzle) in a 4-stage ring, tcgen05 MMAs into a
// double-buffered TMEM accumulator.  The epilogue
// warps (one TMEM lane = one token row per thread) make two passes over each
// head's 128 columns: the sum of squares, then normalisation, RoPE and the bf16
// store.  The RoPE angle is reduced to a fraction of a turn before its sine
// and cosine are taken: theta_j / 2 pi is held as a sum of two floats hi + lo,
// pos * hi is split exactly into a rounded product and its error (one fma),
// the product's integer part drops out exactly, and the small terms are added
// back -- accurate to about 1e-9 turns at positions up to millions, where an
// fp32 product pos * theta would be off by 0.06 radians.
// Token i (query row i, key position pos(i)) writes Q_idx[i, h, :] and the key
// row k_start + pos(i) of K_idx: the new tokens' rows of the index-key cache.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kProStages = 4;
constexpr int kProATile = 128 * 64 * 2;   // 128 rows x 64 bf16 = 16 KB
constexpr int kProBTile = 256 * 64 * 2;   // 256 rows x 64 bf16 = 32 KB
constexpr int kProThreads = 256;
constexpr float kRmsEps = 1e-6f;

struct ProSmem {
  uint64_t full[kProStages], empty[kProStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  float gamma[2][128];  // [0] query heads, [1] key head
};

constexpr size_t kProSmemBytes = 1024 + kProStages * (kProATile + kProBTile) + sizeof(ProSmem);

// Work items, per 256 token rows (two row tiles): the head pairs (2p, 2p + 1) of row tile 0, then those of
// row tile 1, then (n_heads odd) the lone last head over both row tiles.  Head index hkv is the key head.
// Accumulator columns 0..127 and 128..255 hold slot 0 and slot 1: the pair's two heads, or the lone head's
// two row tiles.
struct ProItem {
  int row0, h0;
  bool lone;  // one head over 256 rows (else two heads over 128 rows)
  __device__ __forceinline__ int slot_row(int u) const { return lone ? row0 + 128 * u : row0; }
  __device__ __forceinline__ int slot_head(int u) const { return lone ? h0 : h0 + u; }
};

__host__ __device__ __forceinline__ int pro_items_per_256(int hkv) {
  const int n_heads = hkv + 1;
  return 2 * (n_heads / 2) + (n_heads & 1);
}
__host__ __device__ __forceinline__ int pro_items(int total_q, int hkv) {
  return ((total_q + 255) / 256) * pro_items_per_256(hkv);
}

__device__ __forceinline__ ProItem pro_item(const PrologueParams& p, int j) {
  const int n_heads = p.hkv + 1, n_pairs = n_heads / 2, per = pro_items_per_256(p.hkv);
  const int sub = j % per;
  ProItem it;
  it.lone = sub >= 2 * n_pairs;
  it.row0 = (j / per) * 256 + (it.lone ? 0 : (sub / n_pairs) * 128);
  it.h0 = it.lone ? n_heads - 1 : (sub % n_pairs) * 2;
  return it;
}

}  // namespace

__global__ void __launch_bounds__(kProThreads, 1)
    index_prologue_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wq,
                          const __grid_constant__ CUtensorMap tm_wk, PrologueParams p) {
  extern __shared__ uint8_t smem_raw[];
  WsHeader* hdr = p.hdr;
  if (hdr->status & kFlagBadSeqlens) return;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_buf = base;                                   // kProStages x 16 KB
  uint8_t* b_buf = base + kProStages * kProATile;          // kProStages x 32 KB
  ProSmem& sm = *reinterpret_cast<ProSmem*>(base + kProStages * (kProATile + kProBTile));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = pro_items(p.total_q, p.hkv);
  const int kblocks = p.d_model / 64;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kProStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.acc_full[i], 1);
      mbar_init(&sm.acc_empty[i], 128);
    }
    mbar_init(&sm.mma_done, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_wq);
    tma_prefetch_desc(&tm_wk);
  }
  for (int d = threadIdx.x; d < 128; d += kProThreads) {
    sm.gamma[0][d] = __bfloat162float(p.gamma_q[d]);
    sm.gamma[1][d] = __bfloat162float(p.gamma_k[d]);
  }
  if (warp == 2) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
        const ProItem w = pro_item(p, j);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int st = it % kProStages;
          if (it >= kProStages && !mbar_wait(&sm.empty[st], ((it / kProStages) - 1) & 1, abort_flag)) {
            report_timeout(abort_flag, hdr, 701);
            ok = false;
            break;
          }
          // 48 KB either way: X 128 rows + two heads' weights, or X 2 x 128 rows (the second in the weight
          // stage's upper half) + one head's weights (rows past the end read as zeros and count their bytes)
          mbar_arrive_expect_tx(&sm.full[st], kProATile + kProBTile);
          tma_load_2d(a_buf + st * kProATile, &tm_x, &sm.full[st], kb * 64, w.row0);
          if (w.lone) tma_load_2d(b_buf + st * kProBTile + kProBTile / 2, &tm_x, &sm.full[st], kb * 64, w.row0 + 128);
          for (int hh = 0; hh < (w.lone ? 1 : 2); ++hh) {
            const int h = w.h0 + hh;
            uint8_t* dst = b_buf + st * kProBTile + hh * (kProBTile / 2);
            if (h < p.hkv) tma_load_2d(dst, &tm_wq, &sm.full[st], kb * 64, h * 128);
            else tma_load_2d(dst, &tm_wk, &sm.full[st], kb * 64, 0);
          }
        }
      }
      // let every issued copy land before the CTA can exit
      for (int s = 0; s < kProStages; ++s)
        if (it > static_cast<uint32_t>(s)) {
          const uint32_t last = ((it - 1 - s) / kProStages) * kProStages + s;
          mbar_wait(&sm.full[s], (last / kProStages) & 1, nullptr);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, a_iter = 0;
      bool ok = true;
      for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x, ++a_iter) {
        const ProItem w = pro_item(p, j);
        const uint32_t idesc = idesc_bf16(128, w.lone ? 128 : 256, false);
        const int ab = a_iter & 1;
        if (a_iter >= 2 && !mbar_wait(&sm.acc_empty[ab], ((a_iter >> 1) - 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 711);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int st = it % kProStages;
          if (!mbar_wait(&sm.full[st], (it / kProStages) & 1, abort_flag)) {
            report_timeout(abort_flag, hdr, 712);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aa = smem_u32(a_buf + st * kProATile), ba = smem_u32(b_buf + st * kProBTile);
          const uint32_t acc = (kb > 0) ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            umma_bf16(tmem + ab * 256, sdesc_sw128(aa + kk * 32, 16, 1024), sdesc_sw128(ba + kk * 32, 16, 1024),
                      idesc, (acc || kk > 0) ? 1u : 0u);
            if (w.lone)  // row tile 1 (its X in the weight stage's upper half) into columns 128..255
              umma_bf16(tmem + ab * 256 + 128, sdesc_sw128(ba + kProBTile / 2 + kk * 32, 16, 1024),
                        sdesc_sw128(ba + kk * 32, 16, 1024), idesc, (acc || kk > 0) ? 1u : 0u);
          }
          umma_commit(&sm.empty[st]);
        }
        if (!ok) break;
        umma_commit(&sm.acc_full[ab]);
      }
      umma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int r = (warp & 3) * 32 + lane;  // TMEM lane == token row of the tile
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    uint32_t a_iter = 0;
    for (int j = blockIdx.x; j < n_items; j += gridDim.x, ++a_iter) {
      const ProItem w = pro_item(p, j);
      const int ab = a_iter & 1;
      if (!mbar_wait_warp(&sm.acc_full[ab], (a_iter >> 1) & 1, abort_flag)) {
        report_timeout(abort_flag, hdr, 721);
        break;
      }
      tc_fence_after();
      for (int hh = 0; hh < 2; ++hh) {  // accumulator slot: its rows and head
        const int i = w.slot_row(hh) + r;
        const bool valid = i < p.total_q;
        int pos = 0;
        long long krow = 0;
        if (valid) {
          const int s = find_seq(p.cu_q, p.num_seqs, i);
          const SeqInfo si = p.seq[s];
          pos = si.kv_len - si.q_len + (i - si.q_start);
          krow = static_cast<long long>(si.k_start) + pos;
        }
        {
          const int h = w.slot_head(hh);
          const uint32_t col = lane_addr + ab * 256 + hh * 128;
          const float* gamma = sm.gamma[h < p.hkv ? 0 : 1];
          // pass 1: sum of squares of the head's 128 projections
          float ss = 0.f;
  #pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld_32cols(col + c * 32, v);
            tmem_ld_wait_regs(v);
  #pragma unroll
            for (int e = 0; e < 32; ++e) ss = fmaf(__uint_as_float(v[e]), __uint_as_float(v[e]), ss);
          }
          const float inv = 1.0f / sqrtf(ss * (1.0f / 128.0f) + kRmsEps);
          __nv_bfloat16* out = (h < p.hkv) ? p.q_idx + (static_cast<int64_t>(i) * p.hkv + h) * 128
                                           : p.k_idx + krow * 128;
          // pass 2: dims 0..63 (the RoPE pairs j, j + 32), then dims 64..127
          {
            uint32_t a[32], b[32];
            tmem_ld_32cols(col, a);
            tmem_ld_32cols(col + 32, b);
            tmem_ld_wait_regs(a);
            tmem_ld_wait_regs(b);
            uint32_t lo[16], hi[16];
  #pragma unroll
            for (int jj = 0; jj < 32; jj += 2) {
              float2 za, zb;
              float cs[2], sn[2];
  #pragma unroll
              for (int u = 0; u < 2; ++u) {
                // fraction of a turn of pos * theta_j / (2 pi), with theta_j / (2 pi) = hi + lo (two floats):
                // pos * hi = t + e exactly (fma), t - rint(t) is exact, and pos * lo is below 0.01 turns
                const float fp = static_cast<float>(pos);
                const float hi = p.rope_turns_hi[jj + u], lo = p.rope_turns_lo[jj + u];
                const float t = fp * hi;
                const float e = fmaf(fp, hi, -t);
                const float f = (t - rintf(t)) + fmaf(fp, lo, e);
                sincospif(2.0f * f, &sn[u], &cs[u]);
              }
              const float a0 = __uint_as_float(a[jj]) * inv * gamma[jj];
              const float a1 = __uint_as_float(a[jj + 1]) * inv * gamma[jj + 1];
              const float b0 = __uint_as_float(b[jj]) * inv * gamma[jj + 32];
              const float b1 = __uint_as_float(b[jj + 1]) * inv * gamma[jj + 33];
              za = make_float2(a0 * cs[0] - b0 * sn[0], a1 * cs[1] - b1 * sn[1]);
              zb = make_float2(b0 * cs[0] + a0 * sn[0], b1 * cs[1] + a1 * sn[1]);
              const __nv_bfloat162 pa = __floats2bfloat162_rn(za.x, za.y);
              const __nv_bfloat162 pb = __floats2bfloat162_rn(zb.x, zb.y);
              lo[jj >> 1] = *reinterpret_cast<const uint32_t*>(&pa);
              hi[jj >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
            }
            if (valid) {
              uint4* o4 = reinterpret_cast<uint4*>(out);
  #pragma unroll
              for (int q = 0; q < 4; ++q) {
                o4[q] = make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
                o4[4 + q] = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
              }
            }
          }
  #pragma unroll
          for (int c = 2; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld_32cols(col + c * 32, v);
            tmem_ld_wait_regs(v);
            uint32_t pk[16];
  #pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(v[e]) * inv * gamma[c * 32 + e],
                                                             __uint_as_float(v[e + 1]) * inv * gamma[c * 32 + e + 1]);
              pk[e >> 1] = *reinterpret_cast<const uint32_t*>(&t);
            }
            if (valid) {
              uint4* o4 = reinterpret_cast<uint4*>(out + c * 32);
  #pragma unroll
              for (int q = 0; q < 4; ++q) o4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acc_empty[ab]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t index_prologue_smem_bytes() { return kProSmemBytes; }

cudaError_t launch_index_prologue(const CUtensorMap& tx, const CUtensorMap& twq, const CUtensorMap& twk,
                                  const PrologueParams& p, int sms, cudaStream_t stream) {
  const long long items = pro_items(p.total_q, p.hkv);
  if (items == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(index_prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kProSmemBytes));
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  index_prologue_kernel<<<grid, kProThreads, kProSmemBytes, stream>>>(tx, twq, twk, p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
