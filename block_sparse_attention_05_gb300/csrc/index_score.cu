// index_score.cu -- Index Branch scoring on the tensor cores.
//
// "MiniMax Sparse Attention: let each query pick its own blocks", section
// "The mechanism, precisely" (first bullet) and Figure 1: token scores
// Q_idx . K_idx^T, max-pooled over 128-token key blocks, then top-k blocks
// with the query's own (local) block always kept.
//
// Work item: a tile of 128 rows of Q_idx viewed as [T * Hkv, d_idx]; with
// Hkv = 4 that is 32 consecutive queries x 4 groups, so one K_idx tile (the
// shared index-key head) serves every group at once.  The CTA walks the key
// blocks 0..L_max of the tile in pairs; each pair is one 128 x 256 x d_idx
// tcgen05 MMA (bf16 in, fp32 accumulate in TMEM, two 256-column
// accumulators): N = 256 halves the shared-memory operand traffic per FLOP
// of a 128-key MMA, which is what limits a 128 x 128 MMA from shared memory.
// The epilogue warps reduce each accumulator row (one TMEM lane per thread) to
// the two blocks' pooled scores with the causal limit of that row.  In the
// fused mode the epilogue keeps a running top-(k-1) of the non-local blocks
// per row in registers and writes the final selection; otherwise it writes
// pooled scores.
//
// Warp roles (256 threads): warp 0 = TMA producer and work claiming, warp 1 =
// MMA issuer, warp 2 = TMEM allocator, warp 3 idle, warps 4..7 = epilogue.
// Work items are claimed dynamically (atomic counter) from a list sorted by
// descending cost, so the persistent grid balances itself.
//
// fp8 index inputs (E4M3 codes, d_idx 128): kind::f8f6f4 MMAs over 16 KB Q_idx
// tiles and 32 KB pair tiles (a 6-stage ring), and 384 threads: warps 4..7 and
// 8..11 are two epilogue groups, one per block of a pair, with registers moved
// to them from warps 0..3 (setmaxnreg); a block's pooled score is its maximum
// code dot product times its K_idx scale and the row's Q_idx scale.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

// Tiles: 128 rows x 128 bf16 columns (two 64-column halves of 128-byte rows),
// or x 128 E4M3 codes (one 128-byte row) for an fp8 index; the K_idx ring holds
// pairs of key blocks, as many as fit the same 192 KB.  The fp8 MMAs take half
// the time of the bf16 ones, so the fp8 kernel has two epilogue warpgroups,
// one per block of a pair, each keeping its own top-k list per row; at the end
// of a work item the second hands its lists to the first through shared
// memory (kMergeBytes) to be merged.
template <bool FP8>
struct IdxCfg {
  static constexpr int kStagesK = FP8 ? 6 : 3;
  static constexpr int kQTile = FP8 ? 128 * 128 : 128 * 128 * 2;
  static constexpr int kKPair = 2 * kQTile;
  static constexpr int kEpiGroups = FP8 ? 2 : 1;
  static constexpr int kThreads = 128 + 128 * kEpiGroups;
  static constexpr int kMergeBytes = FP8 ? 128 * 15 * 8 : 0;  // 128 rows x up to 15 keys
  // fp8: registers per thread after the reallocation (warps 0-3: TMA, MMA and TMEM allocation; the two
  // epilogue warpgroups load a whole block's 128 accumulator columns at once)
  static constexpr int kCtlRegs = 96, kEpiRegs = 200;
  static constexpr int kRegsNeeded = 128 * kCtlRegs + 128 * kEpiGroups * kEpiRegs;
};
constexpr int kIdxMaxStagesK = 6;

struct IdxSmem {
  uint64_t q_full, q_empty;
  uint64_t k_full[kIdxMaxStagesK], k_empty[kIdxMaxStagesK];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t work_full[2], work_empty[2];
  uint64_t mma_done;
  uint64_t merge_full, merge_empty;  // fp8: the second epilogue group's lists written / read
  int work[2];
  uint32_t tmem_base;
  int abort_flag;
};

template <bool FP8>
constexpr size_t idx_smem_bytes() {
  return 1024 /*align slack*/ + IdxCfg<FP8>::kQTile + IdxCfg<FP8>::kStagesK * IdxCfg<FP8>::kKPair +
         sizeof(IdxSmem) + IdxCfg<FP8>::kMergeBytes;
}
static_assert(idx_smem_bytes<true>() <= 232448 && idx_smem_bytes<false>() <= 232448, "shared memory per CTA");

__device__ __forceinline__ void tile_geometry(const SeqInfo& si, int t0, int qt, int& nq, int& lmax) {
  nq = min(qt, si.q_len - t0);
  const int last_pos = si.kv_len - si.q_len + t0 + nq - 1;
  lmax = last_pos >> 7;
}

}  // namespace

// FP8: Q_idx and K_idx are E4M3 codes (kind::f8f6f4 MMAs, K = 32 codes per
// instruction) with one scale per Q_idx row and one per key block; a block's
// pooled score is its maximum code dot product times the two scales (positive,
// so scaling the maximum is the maximum of the scaled scores).
template <int CAP, bool FUSED, bool FP8>
__global__ void __launch_bounds__(IdxCfg<FP8>::kThreads, 1)
    index_score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       IndexParams p) {
  constexpr int kIdxStagesK = IdxCfg<FP8>::kStagesK, kQTile = IdxCfg<FP8>::kQTile, kKPair = IdxCfg<FP8>::kKPair;
  constexpr int kEpi = IdxCfg<FP8>::kEpiGroups;
  extern __shared__ uint8_t smem_raw[];
  WsHeader* hdr = p.hdr;
  if (hdr->status & kFlagBadSeqlens) return;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_buf = base;                      // one 128-row tile
  uint8_t* k_buf = base + kQTile;             // kIdxStagesK pairs of key blocks
  IdxSmem& sm = *reinterpret_cast<IdxSmem*>(base + kQTile + kIdxStagesK * kKPair);
  // fp8: merge buffer, key j of row r at [j * 128 + r]
  uint64_t* merge_keys = reinterpret_cast<uint64_t*>(base + kQTile + kIdxStagesK * kKPair + sizeof(IdxSmem));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = static_cast<int>(hdr->n_qtiles);
  const int kchunks = FP8 ? 1 : p.d_idx >> 6;      // 128-byte chunks per row
  const int ksteps = p.d_idx >> (FP8 ? 5 : 4);     // UMMA K = 32 bytes per step
  const uint32_t row_tx = p.d_idx * (FP8 ? 1u : 2u);  // bytes of one row

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.acc_full[i], 1);
      mbar_init(&sm.acc_empty[i], 128 * kEpi);
      mbar_init(&sm.work_full[i], 1);
      mbar_init(&sm.work_empty[i], 1 + 4 * kEpi);  // the MMA warp and every epilogue warp
    }
    mbar_init(&sm.merge_full, 128);
    mbar_init(&sm.merge_empty, 128);
    for (int i = 0; i < kIdxStagesK; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
    }
    mbar_init(&sm.mma_done, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
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

  // fp8: the control warpgroup gives registers to the two epilogue warpgroups (each warpgroup reallocates at
  // the top of its own branch; the launcher checked that the launch allocation covers the counts)
  if (warp < 4) {
  if constexpr (FP8) regs_release<IdxCfg<FP8>::kCtlRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t q_iter = 0, k_iter = 0;
      for (uint32_t w = 0;; ++w) {
        const int slot = w & 1;
        if (w >= 2 && !mbar_wait(&sm.work_empty[slot], ((w >> 1) - 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 101);
          break;
        }
        const int u = static_cast<int>(atomicAdd(&hdr->counter[0], 1u));
        const int item = (u < n_tiles && !*abort_flag) ? u : -1;
        sm.work[slot] = item;
        mbar_arrive(&sm.work_full[slot]);
        if (item < 0) break;
        const int2 tile = p.tiles[item];
        const SeqInfo si = p.seq[tile.x];
        int nq, lmax;
        tile_geometry(si, tile.y, p.qt, nq, lmax);
        const int row0 = (si.q_start + tile.y) * p.hkv;
        if (q_iter >= 1 && !mbar_wait(&sm.q_empty, (q_iter - 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 102);
          break;
        }
        mbar_arrive_expect_tx(&sm.q_full, 128u * row_tx);
        for (int c = 0; c < kchunks; ++c) tma_load_2d(q_buf + c * 16384, &tm_q, &sm.q_full, c * 64, row0);
        ++q_iter;
        bool ok = true;
        for (int bp = 0; 2 * bp <= lmax; ++bp) {
          const int ks = k_iter % kIdxStagesK;
          if (k_iter >= kIdxStagesK &&
              !mbar_wait(&sm.k_empty[ks], ((k_iter / kIdxStagesK) - 1) & 1, abort_flag)) {
            report_timeout(abort_flag, hdr, 103);
            ok = false;
            break;
          }
          // keys 256 bp .. 256 bp + 255 of the sequence (past its end: zero fill
          // or the next sequence's keys, both masked by the causal limit)
          mbar_arrive_expect_tx(&sm.k_full[ks], 256u * row_tx);
          for (int c = 0; c < kchunks; ++c)
            tma_load_2d(k_buf + ks * kKPair + c * 32768, &tm_k, &sm.k_full[ks], c * 64, si.k_start + bp * 256);
          ++k_iter;
        }
        if (!ok) break;
      }
      // Let every issued copy land before the CTA can exit (matters only
      // after an abort; in a normal run the MMA warp consumed them all).
      if (q_iter > 0) mbar_wait(&sm.q_full, (q_iter - 1) & 1, nullptr);
      for (int s = 0; s < kIdxStagesK; ++s)
        if (k_iter > static_cast<uint32_t>(s)) {
          const uint32_t last = ((k_iter - 1 - s) / kIdxStagesK) * kIdxStagesK + s;
          mbar_wait(&sm.k_full[s], (last / kIdxStagesK) & 1, nullptr);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = FP8 ? idesc_e4m3(128, 256) : idesc_bf16(128, 256, false);
      uint32_t q_iter = 0, k_iter = 0, a_iter = 0;
      for (uint32_t w = 0;; ++w) {
        const int slot = w & 1;
        if (!mbar_wait(&sm.work_full[slot], (w >> 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 111);
          break;
        }
        const int item = sm.work[slot];
        mbar_arrive(&sm.work_empty[slot]);
        if (item < 0) break;
        const int2 tile = p.tiles[item];
        const SeqInfo si = p.seq[tile.x];
        int nq, lmax;
        tile_geometry(si, tile.y, p.qt, nq, lmax);
        if (!mbar_wait(&sm.q_full, q_iter & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 112);
          break;
        }
        const uint32_t qa = smem_u32(q_buf);
        bool ok = true;
        for (int bp = 0; 2 * bp <= lmax; ++bp) {
          const int ks = k_iter % kIdxStagesK;
          const int ab = a_iter & 1;
          if (!mbar_wait(&sm.k_full[ks], (k_iter / kIdxStagesK) & 1, abort_flag) ||
              (a_iter >= 2 && !mbar_wait(&sm.acc_empty[ab], ((a_iter >> 1) - 1) & 1, abort_flag))) {
            report_timeout(abort_flag, hdr, 113);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ka = smem_u32(k_buf + ks * kKPair);
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint32_t qoff = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * 32768 + (kk & 3) * 32;
            if constexpr (FP8)
              umma_e4m3(tmem + ab * 256, sdesc_sw128(qa + qoff, 16, 1024), sdesc_sw128(ka + koff, 16, 1024), idesc,
                        kk > 0 ? 1u : 0u);
            else
              umma_bf16(tmem + ab * 256, sdesc_sw128(qa + qoff, 16, 1024), sdesc_sw128(ka + koff, 16, 1024), idesc,
                        kk > 0 ? 1u : 0u);
          }
          umma_commit(&sm.k_empty[ks]);
          umma_commit(&sm.acc_full[ab]);
          ++k_iter;
          ++a_iter;
        }
        if (!ok) break;
        umma_commit(&sm.q_empty);
        ++q_iter;
      }
      // all MMAs retired before TMEM can be released
      umma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, nullptr);
    }
  }
  } else {
    // ------------------------------------------------------------ epilogue
    if constexpr (FP8) regs_claim<IdxCfg<FP8>::kEpiRegs>();
    const int row = (warp & 3) * 32 + lane;  // TMEM lane == tile row
    const int eg = (warp - 4) >> 2;           // epilogue group: block eg of each pair (fp8), both blocks (bf16)
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    uint32_t a_iter = 0, n_items = 0;
    for (uint32_t w = 0;; ++w) {
      const int slot = w & 1;
      if (!mbar_wait_warp(&sm.work_full[slot], (w >> 1) & 1, abort_flag)) {
        report_timeout(abort_flag, hdr, 121);
        break;
      }
      const int item = sm.work[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.work_empty[slot]);
      if (item < 0) break;
      const int2 tile = p.tiles[item];
      const SeqInfo si = p.seq[tile.x];
      int nq, lmax;
      tile_geometry(si, tile.y, p.qt, nq, lmax);
      const int tq = row / p.hkv;               // query offset inside the tile
      const bool valid = tq < nq;
      const int t = tile.y + tq;
      const int pos = si.kv_len - si.q_len + t;
      const int local = pos >> 7;
      const int64_t grow = static_cast<int64_t>(si.q_start + tile.y) * p.hkv + row;  // global Q_idx row
      float q_sc = 1.f;
      int blk0 = 0;
      if constexpr (FP8) {
        q_sc = valid ? p.q_scale[grow] : 1.f;
        blk0 = p.blk_off[tile.x];
      }
      TopkList<CAP> list;
      list.clear();
      bool ok = true;
      for (int bp = 0; 2 * bp <= lmax; ++bp) {
        const int ab = a_iter & 1;
        float sc = 1.f;  // fp8: the combined scale of this group's block (a block past the tile's last: unused)
        if constexpr (FP8) {
          if (2 * bp + eg <= lmax) sc = q_sc * p.k_scale[blk0 + 2 * bp + eg];
        }
        if (!mbar_wait_warp(&sm.acc_full[ab], (a_iter >> 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 122);
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2 / kEpi; ++hh) {  // block 2 bp + h: accumulator columns 128 h .. 128 h + 127
          const int h = kEpi == 2 ? eg : hh;
          const int b = 2 * bp + h;
          if constexpr (kEpi == 1) {
            uint32_t r[4][32];
            float cmax[4];  // the load's own maximum of each 32-column chunk
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_max_32cols(lane_addr + ab * 256 + h * 128 + c * 32, r[c], cmax[c]);
            tmem_ld_wait_max4(cmax);
            if (hh == 1) {
              tc_fence_before();
              mbar_arrive(&sm.acc_empty[ab]);
            }
            if (valid && b <= local) {
              const int lim = (b == local) ? (pos & 127) : 127;
              float m0 = cmax[0], m1 = cmax[1], m2 = cmax[2], m3 = cmax[3];
              if (lim < 127) {  // the query's own block: only keys up to its position
                m0 = m1 = m2 = m3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                  m0 = fmaxf(m0, c <= lim ? __uint_as_float(r[0][c]) : -INFINITY);
                  m1 = fmaxf(m1, c + 32 <= lim ? __uint_as_float(r[1][c]) : -INFINITY);
                  m2 = fmaxf(m2, c + 64 <= lim ? __uint_as_float(r[2][c]) : -INFINITY);
                  m3 = fmaxf(m3, c + 96 <= lim ? __uint_as_float(r[3][c]) : -INFINITY);
                }
              }
              const float m = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
              if constexpr (FUSED) {
                if (b < local) list.insert(topk_key(m, b));
              } else {
                p.pooled[grow * p.pooled_stride + b] = m;
              }
            }
          } else {
            // this group's block, all 128 columns in flight at once
            const bool take = valid && b <= local;
            uint32_t r[4][32];
            float cmax[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_max_32cols(lane_addr + ab * 256 + h * 128 + c * 32, r[c], cmax[c]);
            tmem_ld_wait_max4(cmax);
            tc_fence_before();
            mbar_arrive(&sm.acc_empty[ab]);
            float m0 = cmax[0], m1 = cmax[1], m2 = cmax[2], m3 = cmax[3];
            const int lim = (b == local) ? (pos & 127) : 127;
            if (take && lim < 127) {  // the query's own block: only keys up to its position
              m0 = m1 = m2 = m3 = -INFINITY;
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                m0 = fmaxf(m0, c <= lim ? __uint_as_float(r[0][c]) : -INFINITY);
                m1 = fmaxf(m1, c + 32 <= lim ? __uint_as_float(r[1][c]) : -INFINITY);
                m2 = fmaxf(m2, c + 64 <= lim ? __uint_as_float(r[2][c]) : -INFINITY);
                m3 = fmaxf(m3, c + 96 <= lim ? __uint_as_float(r[3][c]) : -INFINITY);
              }
            }
            float m = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
            if (take) {
              m *= sc;
              if constexpr (FUSED) {
                if (b < local) list.insert(topk_key(m, b));
              } else {
                p.pooled[grow * p.pooled_stride + b] = m;
              }
            }
          }
        }
        ++a_iter;
      }
      if (!ok) break;
      if constexpr (FUSED) {
        if constexpr (kEpi == 2) {
          // the second group's lists go to the first through shared memory (bounded waits on both sides)
          static_assert(CAP <= 15, "merge buffer holds 15 keys per row");
          if (eg == 1) {
            if (n_items > 0 && !mbar_wait_warp(&sm.merge_empty, (n_items - 1) & 1, abort_flag)) {
              report_timeout(abort_flag, hdr, 123);
              break;
            }
#pragma unroll
            for (int j = 0; j < CAP; ++j) merge_keys[j * 128 + row] = list.k[j];
            mbar_arrive(&sm.merge_full);
          } else {
            if (!mbar_wait_warp(&sm.merge_full, n_items & 1, abort_flag)) {
              report_timeout(abort_flag, hdr, 124);
              break;
            }
#pragma unroll
            for (int j = 0; j < CAP; ++j) list.insert(merge_keys[j * 128 + row]);
            mbar_arrive(&sm.merge_empty);
          }
        }
        if (valid && eg == 0) {
          int chosen[CAP];
#pragma unroll
          for (int j = 0; j < CAP; ++j)
            chosen[j] = (j < p.topk - 1 && list.k[j] != 0ull) ? topk_key_block(list.k[j]) : -1;
          write_selection<CAP>(p.idx + grow * p.topk, p.topk, chosen, local);
        }
      }
      ++n_items;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t index_score_smem_bytes(bool fp8) { return fp8 ? idx_smem_bytes<true>() : idx_smem_bytes<false>(); }

template <int CAP, bool FUSED, bool FP8>
static cudaError_t launch_index(const CUtensorMap& tq, const CUtensorMap& tk, const IndexParams& p, int grid,
                                cudaStream_t stream) {
  auto* fn = index_score_kernel<CAP, FUSED, FP8>;
  constexpr size_t smem = idx_smem_bytes<FP8>();
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if constexpr (FP8) {
    // the register reallocation's increases must fit in the launch allocation, or they would never complete
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < IdxCfg<FP8>::kCtlRegs || fa.numRegs * IdxCfg<FP8>::kThreads < IdxCfg<FP8>::kRegsNeeded)
      return cudaErrorInvalidConfiguration;
  }
  fn<<<grid, IdxCfg<FP8>::kThreads, smem, stream>>>(tq, tk, p);
  note_launches(1);
  return cudaGetLastError();
}

template <bool FP8>
static cudaError_t launch_index_dtype(const CUtensorMap& tq, const CUtensorMap& tk, const IndexParams& p,
                                     bool fused, int grid, cudaStream_t stream) {
  if (!fused) return launch_index<1, false, FP8>(tq, tk, p, grid, stream);
  if (p.topk <= 4) return launch_index<3, true, FP8>(tq, tk, p, grid, stream);
  if (p.topk <= 8) return launch_index<7, true, FP8>(tq, tk, p, grid, stream);
  return launch_index<15, true, FP8>(tq, tk, p, grid, stream);
}

cudaError_t launch_index_score(const CUtensorMap& tq, const CUtensorMap& tk, const IndexParams& p, bool fused,
                               bool fp8, int grid, cudaStream_t stream) {
  return fp8 ? launch_index_dtype<true>(tq, tk, p, fused, grid, stream)
             : launch_index_dtype<false>(tq, tk, p, fused, grid, stream);
}

}  // namespace msa
