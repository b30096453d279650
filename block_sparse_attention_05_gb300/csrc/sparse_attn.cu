// sparse_attn.cu -- Main Branch for prefill: exact softmax attention over each
// query's selected key blocks, KV-outer on the tensor cores.
//
// "MiniMax Sparse Attention: let each query pick its own blocks", section "The
// mechanism, precisely" (second bullet): exact attention over only the
// selected blocks; every head of a group reuses the group's block set, so the
// key/value reads stay block-contiguous.  The atlas record of the report
// describes the kernel family this follows: KV-outer, queries that selected
// the same block gathered and concatenated into one tensor-core tile, partial
// results with their own LSE combined in a second phase.
//
// Work item ("chunk", from the schedule): one key block (sequence s, block b,
// group g) and up to qpc queries that selected it.  The block's K and V
// (128 tokens x 128 dims each) are loaded once by TMA; the queries are taken
// qpt at a time (qpt x G heads = 128 rows; G = 16 gives 8 queries per tile),
// their Q rows gathered by TMA.  Per tile:
//   S = Q K^T                 tcgen05, 128 x 128 x 128, fp32 in TMEM
//   P = exp2(S*c - max)       softmax warpgroup, one TMEM lane (row) per thread,
//                             causal limit per row (only the local block is cut);
//                             P is split into bf16 hi + lo parts written back
//                             over S in TMEM
//   O = P_hi V + P_lo V       tcgen05 with A read from TMEM, V MN-major in smem
//   partial O / l and LSE     written per (query, group, slot, head)
// The tile covers exactly one key block, so no running rescale is needed.
//
// Warp roles (384 threads): warp 0 = TMA producer and chunk claiming, warp 1 =
// MMA issuer, warp 2 = TMEM allocator, warp 3 idle, warps 4..7 and 8..11 = two
// softmax/epilogue warpgroups taking alternate tiles (each owns an S and an O
// accumulator in TMEM: 2 x (128 + 128) = 512 columns).  Q tiles live in a
// 3-stage ring, freed as soon as QK^T retires; K/V are double-buffered across
// chunks.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kQStages = 3;
constexpr int kWorkSlots = 4;
constexpr int kQTileBytes = 128 * 128 * 2;   // 32 KB
constexpr int kKVBytes = 2 * kQTileBytes;     // K + V of one block, 64 KB
constexpr int kAttnThreads = 384;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnSmem {
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], s_free[2], p_full[2], o_full[2], o_free[2];
  uint64_t work_full[kWorkSlots], work_empty[kWorkSlots];
  uint64_t mma_done;
  int work[kWorkSlots];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kAttnSmemBytes = 1024 + 2 * kKVBytes + kQStages * kQTileBytes + sizeof(AttnSmem);

struct ChunkInfo {
  int g, b, s, begin, count, ntile;
  int krow;
};

__device__ __forceinline__ ChunkInfo decode_chunk(const AttnParams& p, int item) {
  const int4 c = p.chunks[item];
  ChunkInfo ci;
  const long long bk = c.x;
  ci.g = static_cast<int>(bk % p.hkv);
  const int gb = static_cast<int>((bk / p.hkv) % p.total_blocks);
  ci.s = find_seq(p.blk_off, p.num_seqs, gb);
  ci.b = gb - p.blk_off[ci.s];
  ci.begin = c.y;
  ci.count = c.z;
  ci.ntile = (c.z + p.qpt - 1) / p.qpt;
  ci.krow = p.seq[ci.s].k_start + ci.b * kBlock;
  return ci;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace

__global__ void __launch_bounds__(kAttnThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  WsHeader* hdr = p.hdr;
  if (hdr->status & kFlagBadSeqlens) return;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv_buf = base;                       // 2 x (K 32 KB | V 32 KB)
  uint8_t* q_buf = base + 2 * kKVBytes;         // kQStages x 32 KB
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(base + 2 * kKVBytes + kQStages * kQTileBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_chunks = static_cast<int>(hdr->n_chunks);
  const int G = p.group;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.kv_full[i], 1);
      mbar_init(&sm.kv_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_free[i], 1);
      mbar_init(&sm.p_full[i], 128);
      mbar_init(&sm.o_full[i], 1);
      mbar_init(&sm.o_free[i], 128);
    }
    for (int i = 0; i < kWorkSlots; ++i) {
      mbar_init(&sm.work_full[i], 1);
      mbar_init(&sm.work_empty[i], 9);  // MMA thread + 8 softmax warps
    }
    mbar_init(&sm.mma_done, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t q_iter = 0, kv_iter = 0;
      for (uint32_t w = 0;; ++w) {
        const int slot = w % kWorkSlots;
        if (w >= kWorkSlots &&
            !mbar_wait(&sm.work_empty[slot], ((w / kWorkSlots) - 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 201);
          break;
        }
        const int u = static_cast<int>(atomicAdd(&hdr->counter[1], 1u));
        const int item = (u < n_chunks && !*abort_flag) ? u : -1;
        sm.work[slot] = item;
        mbar_arrive(&sm.work_full[slot]);
        if (item < 0) break;
        const ChunkInfo ci = decode_chunk(p, item);
        const int kvb = kv_iter & 1;
        if (kv_iter >= 2 && !mbar_wait(&sm.kv_empty[kvb], ((kv_iter >> 1) - 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 202);
          break;
        }
        uint8_t* kvp = kv_buf + kvb * kKVBytes;
        mbar_arrive_expect_tx(&sm.kv_full[kvb], kKVBytes);
        tma_load_3d(kvp, &tm_k, &sm.kv_full[kvb], 0, ci.g, ci.krow);
        tma_load_3d(kvp + 16384, &tm_k, &sm.kv_full[kvb], 64, ci.g, ci.krow);
        tma_load_3d(kvp + 32768, &tm_v, &sm.kv_full[kvb], 0, ci.g, ci.krow);
        tma_load_3d(kvp + 49152, &tm_v, &sm.kv_full[kvb], 64, ci.g, ci.krow);
        ++kv_iter;
        bool ok = true;
        for (int tt = 0; tt < ci.ntile; ++tt) {
          const int qs = q_iter % kQStages;
          if (q_iter >= kQStages &&
              !mbar_wait(&sm.q_empty[qs], ((q_iter / kQStages) - 1) & 1, abort_flag)) {
            report_timeout(abort_flag, hdr, 203);
            ok = false;
            break;
          }
          uint8_t* qp = q_buf + qs * kQTileBytes;
          mbar_arrive_expect_tx(&sm.q_full[qs], kQTileBytes);
          for (int ql = 0; ql < p.qpt; ++ql) {
            int e = ci.begin + tt * p.qpt + ql;
            if (e >= ci.begin + ci.count) e = ci.begin;  // pad the last tile with a real row
            const int qi = p.entries[e] >> 5;
            tma_load_3d(qp + ql * G * 128, &tm_q, &sm.q_full[qs], 0, ci.g * G, qi);
            tma_load_3d(qp + 16384 + ql * G * 128, &tm_q, &sm.q_full[qs], 64, ci.g * G, qi);
          }
          ++q_iter;
        }
        if (!ok) break;
      }
      for (int s = 0; s < kQStages; ++s)
        if (q_iter > static_cast<uint32_t>(s)) {
          const uint32_t last = ((q_iter - 1 - s) / kQStages) * kQStages + s;
          mbar_wait(&sm.q_full[s], (last / kQStages) & 1, nullptr);
        }
      for (int s = 0; s < 2; ++s)
        if (kv_iter > static_cast<uint32_t>(s)) {
          const uint32_t last = ((kv_iter - 1 - s) / 2) * 2 + s;
          mbar_wait(&sm.kv_full[s], (last >> 1) & 1, nullptr);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16(128, 128, false);
      const uint32_t idesc_pv = idesc_bf16(128, 128, true);
      uint32_t w_iter = 0, kv_iter = 0;
      uint32_t t = 0;                 // global tile counter (== Q stage use counter)
      // the chunk being walked
      int have_chunk = 0, tt = 0, ntile = 0, cur_kvb = 0;
      // the previous tile, waiting for its PV
      bool prev_valid = false;
      uint32_t prev_t = 0;
      int prev_kvb = 0;
      bool prev_last = false;
      bool done = false;
      while (true) {
        // ---- next tile
        bool next_valid = false;
        int next_kvb = 0;
        bool next_last = false;
        bool new_chunk = false;
        if (!done) {
          if (!have_chunk || tt >= ntile) {
            const int slot = w_iter % kWorkSlots;
            if (!mbar_wait(&sm.work_full[slot], (w_iter / kWorkSlots) & 1, abort_flag)) {
              report_timeout(abort_flag, hdr, 211);
              break;
            }
            const int item = sm.work[slot];
            mbar_arrive(&sm.work_empty[slot]);
            ++w_iter;
            if (item < 0) {
              done = true;
            } else {
              const ChunkInfo ci = decode_chunk(p, item);
              have_chunk = 1;
              tt = 0;
              ntile = ci.ntile;
              cur_kvb = kv_iter & 1;
              new_chunk = true;
            }
          }
          if (!done) {
            next_valid = true;
            next_kvb = cur_kvb;
            next_last = (tt == ntile - 1);
          }
        }
        if (next_valid) {
          const int qs = t % kQStages;
          const int w = t & 1;
          const uint32_t n = t >> 1;
          if (new_chunk) {
            if (!mbar_wait(&sm.kv_full[next_kvb], (kv_iter >> 1) & 1, abort_flag)) {
              report_timeout(abort_flag, hdr, 212);
              break;
            }
            ++kv_iter;
          }
          if (!mbar_wait(&sm.q_full[qs], (t / kQStages) & 1, abort_flag) ||
              (n >= 1 && !mbar_wait(&sm.s_free[w], (n - 1) & 1, abort_flag))) {
            report_timeout(abort_flag, hdr, 213);
            break;
          }
          tc_fence_after();
          const uint32_t qa = smem_u32(q_buf + qs * kQTileBytes);
          const uint32_t ka = smem_u32(kv_buf + next_kvb * kKVBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_bf16(tmem + w * 256, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), idesc_qk,
                      kk > 0 ? 1u : 0u);
          }
          umma_commit(&sm.s_full[w]);
          umma_commit(&sm.q_empty[qs]);  // the Q stage is free once QK^T has retired
          ++tt;
        }
        if (prev_valid) {
          const int w = prev_t & 1;
          const uint32_t n = prev_t >> 1;
          if (!mbar_wait(&sm.p_full[w], n & 1, abort_flag) ||
              (n >= 1 && !mbar_wait(&sm.o_free[w], (n - 1) & 1, abort_flag))) {
            report_timeout(abort_flag, hdr, 214);
            break;
          }
          tc_fence_after();
          // P sits in the S columns of TMEM as bf16 pairs: high parts in columns
          // 0..63, low parts (p - bf16(p)) in 64..127; O = P_hi V + P_lo V.
          const uint32_t pa = tmem + w * 256;
          const uint32_t va = smem_u32(kv_buf + prev_kvb * kKVBytes + 32768);
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16_ts(tmem + w * 256 + 128, pa + part * 64 + kk * 8, sdesc_sw128(va + kk * 2048, 16384, 1024),
                           idesc_pv, (part | kk) ? 1u : 0u);
          umma_commit(&sm.o_full[w]);
          umma_commit(&sm.s_free[w]);  // S/P columns reusable once PV has retired
          if (prev_last) umma_commit(&sm.kv_empty[prev_kvb]);
        }
        if (!next_valid) break;
        prev_valid = true;
        prev_t = t;
        prev_kvb = next_kvb;
        prev_last = next_last;
        ++t;
      }
      umma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int wg = (warp - 4) >> 2;                 // 0 or 1: which tiles, which TMEM half
    const int r = (warp & 3) * 32 + lane;           // TMEM lane == tile row
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + wg * 256;
    const int q_local = r / G, hh = r % G;
    uint32_t t = 0, w_iter = 0;
    bool ok = true;
    while (ok) {
      const int slot = w_iter % kWorkSlots;
      if (!mbar_wait_warp(&sm.work_full[slot], (w_iter / kWorkSlots) & 1, abort_flag)) {
        report_timeout(abort_flag, hdr, 221);
        break;
      }
      const int item = sm.work[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.work_empty[slot]);
      ++w_iter;
      if (item < 0) break;
      const ChunkInfo ci = decode_chunk(p, item);
      for (int tt = 0; tt < ci.ntile; ++tt, ++t) {
        if ((t & 1) != static_cast<uint32_t>(wg)) continue;
        const uint32_t n = t >> 1;
        const int e = ci.begin + tt * p.qpt + q_local;
        const bool valid = e < ci.begin + ci.count;
        int qi = 0, slot_id = 0, lim = -1;
        if (valid) {
          const int ent = p.entries[e];
          qi = ent >> 5;
          slot_id = ent & 31;
          const SeqInfo si = p.seq[ci.s];
          const int pos = si.kv_len - si.q_len + (qi - si.q_start);
          lim = pos - ci.b * kBlock;               // keys 0..lim of this block are visible
        }
        if (!mbar_wait_warp(&sm.s_full[wg], n & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 222);
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32cols(lane_addr + c * 32, sr[c]);
        tmem_ld_wait();

        // softmax over the visible keys of this block (base-2, scale folded in)
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = (c * 32 + j <= lim) ? __uint_as_float(sr[c][j]) * p.scale_log2 : -INFINITY;
            sr[c][j] = __float_as_uint(x);
            mx = fmaxf(mx, x);
          }
        const float mref = (mx == -INFINITY) ? 0.f : mx;
        float l = 0.f;
        // P = hi + lo, both bf16, written over the S columns: hi pairs to columns
        // 0..63, lo pairs to 64..127 (two bf16 per 32-bit column, key 2c in the
        // low half).  Splitting keeps P at ~16 significant bits for the PV product.
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a = exp2f(__uint_as_float(sr[c][2 * j]) - mref);
            const float b = exp2f(__uint_as_float(sr[c][2 * j + 1]) - mref);
            l += a + b;
            const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
            hi[j] = *reinterpret_cast<const uint32_t*>(&h);
            lo[j] = pack_bf16(a - __low2float(h), b - __high2float(h));
          }
          tmem_st_16cols(lane_addr + c * 16, hi);
          tmem_st_16cols(lane_addr + 64 + c * 16, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full[wg]);

        if (!mbar_wait_warp(&sm.o_full[wg], n & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 223);
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        __nv_bfloat16* orow =
            p.part.o + ((static_cast<int64_t>(qi) * p.hkv + ci.g) * p.topk + slot_id) * G * kHeadDim +
            static_cast<int64_t>(hh) * kHeadDim;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t orr[32];
          tmem_ld_32cols(lane_addr + 128 + c * 32, orr);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(orr[j + 0]) * inv_l, __uint_as_float(orr[j + 1]) * inv_l);
              v.y = pack_bf16(__uint_as_float(orr[j + 2]) * inv_l, __uint_as_float(orr[j + 3]) * inv_l);
              v.z = pack_bf16(__uint_as_float(orr[j + 4]) * inv_l, __uint_as_float(orr[j + 5]) * inv_l);
              v.w = pack_bf16(__uint_as_float(orr[j + 6]) * inv_l, __uint_as_float(orr[j + 7]) * inv_l);
              *reinterpret_cast<uint4*>(orow + c * 32 + j) = v;
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&sm.o_free[wg]);
        if (valid) {
          p.part.lse[((static_cast<int64_t>(qi) * p.hkv + ci.g) * p.topk + slot_id) * G + hh] =
              (mx == -INFINITY) ? -INFINITY : (mx + log2f(l)) * kLn2;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t sparse_attn_smem_bytes() { return kAttnSmemBytes; }

cudaError_t launch_sparse_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const AttnParams& p, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kAttnSmemBytes));
  if (e != cudaSuccess) return e;
  sparse_attn_kernel<<<grid, kAttnThreads, kAttnSmemBytes, stream>>>(tq, tk, tv, p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
