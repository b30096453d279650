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
// by the key head's (128 output columns each), on the tensor cores, by pairs
// of CTAs (2-CTA clusters): a work item is 256 token rows x two heads (or the
// lone last head), CTA rank r taking rows 128 r .. 128 r + 127 (N = 256, or
// 128 for the lone head).  The weight rows are the same for both row tiles, so
// each CTA loads its own X rows and one half of the item's weight rows,
// multicast to both CTAs: 32 KB per K step per CTA from L2 instead of 48 (the
// single-CTA kernel was paced by that operand feed).  K is looped in 64-column
// blocks, tiles by TMA (128-byte swizzle) in a 4-stage ring whose slots a CTA
// refills only when both CTAs' MMAs have read them (each MMA warp's commit
// arrives on both CTAs' empty barriers), tcgen05 MMAs into a double-buffered
// TMEM accumulator.  The epilogue
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
constexpr int kProBTile = 256 * 64 * 2;   // up to 256 weight rows x 64 bf16 = 32 KB
constexpr int kProHead = 128 * 64 * 2;    // one head's weight rows of a K step: 16 KB
constexpr int kProThreads = 256;
constexpr uint16_t kProBoth = 0x3;        // both CTAs of the cluster
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

// Work items of a CTA pair, per 256 token rows: the head pairs (2p, 2p + 1), then (n_heads odd) the lone last
// head.  Head index hkv is the key head.  This CTA's rows are row0 .. row0 + 127; accumulator columns
// 128 u .. 128 u + 127 hold head h0 + u.
struct ProItem {
  int row0, h0, n_heads;
};

__host__ __device__ __forceinline__ int pro_items_per_256(int hkv) {
  const int n_heads = hkv + 1;
  return n_heads / 2 + (n_heads & 1);
}
__host__ __device__ __forceinline__ int pro_items(int total_q, int hkv) {
  return ((total_q + 255) / 256) * pro_items_per_256(hkv);
}

__device__ __forceinline__ ProItem pro_item(const PrologueParams& p, int j, int rank) {
  const int n_heads = p.hkv + 1, n_pairs = n_heads / 2, per = pro_items_per_256(p.hkv);
  const int sub = j % per;
  ProItem it;
  const bool lone = sub >= n_pairs;
  it.row0 = (j / per) * 256 + 128 * rank;
  it.h0 = lone ? n_heads - 1 : 2 * sub;
  it.n_heads = lone ? 1 : 2;
  return it;
}

// Loads weight rows [r0, r0 + n) (n = 64 or 128) of head h for K block kb into dst, multicast to both CTAs.
// The key head's map has 64-row boxes, the query heads' 128-row boxes (each K step of a query head is one box).
__device__ __forceinline__ void load_weights(const PrologueParams& p, const CUtensorMap* tm_wq,
                                             const CUtensorMap* tm_wk, uint8_t* dst, uint64_t* bar, int h, int kb,
                                             int r0, int n) {
  if (h < p.hkv) {  // n == 128: only the key head is ever split (the lone head of an even hkv)
    tma_load_2d_multicast(dst, tm_wq, bar, kb * 64, h * 128 + r0, kProBoth);
  } else {
    for (int q = 0; q < n; q += 64) tma_load_2d_multicast(dst + q * 128, tm_wk, bar, kb * 64, r0 + q, kProBoth);
  }
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kProThreads, 1)
    index_prologue_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wq,
                          const __grid_constant__ CUtensorMap tm_wk, PrologueParams p) {
  extern __shared__ uint8_t smem_raw[];
  WsHeader* hdr = p.hdr;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_buf = base;                                   // kProStages x 16 KB
  uint8_t* b_buf = base + kProStages * kProATile;          // kProStages x 32 KB
  ProSmem& sm = *reinterpret_cast<ProSmem*>(base + kProStages * (kProATile + kProBTile));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int n_items = pro_items(p.total_q, p.hkv);
  const int kblocks = p.d_model / 64;
  // both CTAs of a pair see the same flag (the planning kernel before set it), so both skip or both run
  const bool run = !(hdr->status & kFlagBadSeqlens);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kProStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 2);  // both CTAs' MMA warps release a stage
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
  cluster_sync();  // the peer's barriers are initialised before anything is multicast to them
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (!run) {
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int j = cluster; j < n_items && ok; j += n_clusters) {
        const ProItem w = pro_item(p, j, rank);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int st = it % kProStages;
          // the slot is free once both CTAs' MMAs have read its previous fill
          if (it >= kProStages && !mbar_wait(&sm.empty[st], ((it / kProStages) - 1) & 1, abort_flag)) {
            report_timeout(abort_flag, hdr, 701);
            ok = false;
            break;
          }
          // this CTA's X rows (rows past the end read as zeros and count their bytes), and the item's weight
          // rows of this K step, half from each CTA
          mbar_arrive_expect_tx(&sm.full[st], kProATile + w.n_heads * kProHead);
          tma_load_2d(a_buf + st * kProATile, &tm_x, &sm.full[st], kb * 64, w.row0);
          uint8_t* b = b_buf + st * kProBTile;
          if (w.n_heads == 2)
            load_weights(p, &tm_wq, &tm_wk, b + rank * kProHead, &sm.full[st], w.h0 + rank, kb, 0, 128);
          else
            load_weights(p, &tm_wq, &tm_wk, b + rank * (kProHead / 2), &sm.full[st], w.h0, kb, 64 * rank, 64);
        }
      }
      // let every copy into this CTA land before it can exit
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
      for (int j = cluster; j < n_items && ok; j += n_clusters, ++a_iter) {
        const ProItem w = pro_item(p, j, rank);
        const uint32_t idesc = idesc_bf16(128, 128 * w.n_heads, false);
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
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + ab * 256, sdesc_sw128(aa + kk * 32, 16, 1024), sdesc_sw128(ba + kk * 32, 16, 1024),
                      idesc, (acc || kk > 0) ? 1u : 0u);
          umma_commit_multicast(&sm.empty[st], kProBoth);
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
    for (int j = cluster; j < n_items; j += n_clusters, ++a_iter) {
      const ProItem w = pro_item(p, j, rank);
      const int ab = a_iter & 1;
      if (!mbar_wait_warp(&sm.acc_full[ab], (a_iter >> 1) & 1, abort_flag)) {
        report_timeout(abort_flag, hdr, 721);
        break;
      }
      tc_fence_after();
      for (int hh = 0; hh < w.n_heads; ++hh) {  // accumulator slot: head h0 + hh of this CTA's rows
        const int i = w.row0 + r;
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
          const int h = w.h0 + hh;
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
  // neither CTA leaves while the other may still multicast into it or arrive on its barriers
  cluster_sync();
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
  // persistent CTA pairs: as many as can be resident at once (a GPC with an odd number of free SMs leaves one
  // idle), at most one per item
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (sms / 2)));
  cfg.blockDim = dim3(kProThreads);
  cfg.dynamicSmemBytes = kProSmemBytes;
  cfg.stream = stream;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, index_prologue_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const long long n = items < clusters ? items : clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * n));
  e = cudaLaunchKernelEx(&cfg, index_prologue_kernel, tx, twq, twk, p);
  note_launches(1);
  return e;
}

}  // namespace msa
