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
//                             over S in TMEM (each 32-key chunk over its own
//                             columns: 16 hi, then 16 lo)
//   O = P_hi V + P_lo V       tcgen05 with A read from TMEM, V MN-major in smem
//   partial O / l and LSE     written per (query, group, slot, head)
// The tile covers exactly one key block, so no running rescale is needed.
//
// Warp roles (512 threads): warp 0 = TMA producer and chunk claiming, warps 1
// and 3 = one MMA issuer per softmax warpgroup, warp 2 = TMEM allocator,
// warps 4..7 and 8..11 = two
// softmax warpgroups taking alternate tiles (each owns an S/P and an O
// accumulator in TMEM: 2 x (128 + 128) = 512 columns), warps 12..15 = the
// epilogue warpgroup (O read-back, normalisation, partial stores) for every
// tile.  The softmax warpgroups hand each row's max and sum to the epilogue
// through a 4-slot shared buffer.  Q tiles live in a 2-stage ring, freed as
// soon as QK^T retires; K/V are double-buffered across chunks.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kQStages = 2;
constexpr int kWorkSlots = 4;
constexpr int kStatSlots = 4;
constexpr int kQTileBytes = 128 * 128 * 2;   // 32 KB
constexpr int kKVBytes = 2 * kQTileBytes;     // K + V of one block, 64 KB
constexpr int kAttnThreads = 512;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnSmem {
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], s_free[2], p_full[2], o_full[2], o_free[2];
  uint64_t stat_full[kStatSlots];
  uint64_t work_full[kWorkSlots], work_empty[kWorkSlots];
  uint64_t mma_done[2];
  float2 stat[kStatSlots][128];  // per tile slot and row: (max in scaled log2 units, sum of P)
  int work[kWorkSlots];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kAttnSmemBytes = 1024 + 2 * kKVBytes + kQStages * kQTileBytes + sizeof(AttnSmem);

struct ChunkInfo {
  int g, b, s, begin, count, ntile, krow;
};

__device__ __forceinline__ ChunkInfo decode_chunk(const AttnParams& p, int item) {
  const int4 c = p.chunks[item];
  ChunkInfo ci;
  ci.begin = c.x;
  ci.count = c.y;
  ci.g = c.z & 0xFF;
  ci.b = c.z >> 8;
  ci.s = c.w;
  ci.ntile = (c.y + p.qpt - 1) / p.qpt;
  ci.krow = p.seq[ci.s].k_start + ci.b * kBlock;
  return ci;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x on the special-function unit (approximate, flushes subnormals; 2^-inf = 0).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The row of a tile: which query and slot it holds (or none, for padding rows).
struct RowInfo {
  bool valid;
  int qi, slot, lim;
};

__device__ __forceinline__ RowInfo row_info(const AttnParams& p, const ChunkInfo& ci, int tt, int q_local) {
  RowInfo ri{false, 0, 0, -1};
  const int e = ci.begin + tt * p.qpt + q_local;
  if (e < ci.begin + ci.count) {
    const int ent = p.entries[e];
    ri.valid = true;
    ri.qi = ent >> 5;
    ri.slot = ent & 31;
    const SeqInfo si = p.seq[ci.s];
    const int pos = si.kv_len - si.q_len + (ri.qi - si.q_start);
    ri.lim = pos - ci.b * kBlock;  // keys 0..lim of this block are visible
  }
  return ri;
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
      mbar_init(&sm.kv_empty[i], 2);  // one arrival per MMA issuer
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_free[i], 1);
      mbar_init(&sm.p_full[i], 128);
      mbar_init(&sm.o_full[i], 1);
      mbar_init(&sm.o_free[i], 128);
    }
    for (int i = 0; i < kStatSlots; ++i) mbar_init(&sm.stat_full[i], 128);
    for (int i = 0; i < kWorkSlots; ++i) {
      mbar_init(&sm.work_full[i], 1);
      mbar_init(&sm.work_empty[i], 14);  // 2 MMA threads + 8 softmax warps + 4 epilogue warps
    }
    mbar_init(&sm.mma_done[0], 1);
    mbar_init(&sm.mma_done[1], 1);
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
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per softmax warpgroup: warp 1 drives the even tiles,
    // warp 3 the odd ones, so a wait for one warpgroup never stalls the other.
    // Tile t uses Q stage t % 2 == its warpgroup, so each stage has one consumer.
    if (lane == 0) {
      const int wg = (warp == 1) ? 0 : 1;
      const uint32_t idesc_qk = idesc_bf16(128, 128, false);
      const uint32_t idesc_pv = idesc_bf16(128, 128, true);
      const uint32_t s_col = tmem + wg * 256, o_col = tmem + wg * 256 + 128;
      uint32_t w_iter = 0, kv_iter = 0, t = 0;
      bool ok = true;
      while (ok) {
        const int slot = w_iter % kWorkSlots;
        if (!mbar_wait(&sm.work_full[slot], (w_iter / kWorkSlots) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 211);
          break;
        }
        const int item = sm.work[slot];
        mbar_arrive(&sm.work_empty[slot]);
        ++w_iter;
        if (item < 0) break;
        const ChunkInfo ci = decode_chunk(p, item);
        const int kvb = kv_iter & 1;
        // every issuer waits for every chunk's K/V, used or not, so that it can
        // never arrive on kv_empty for a later use of this buffer too early
        if (!mbar_wait(&sm.kv_full[kvb], (kv_iter >> 1) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 212);
          break;
        }
        ++kv_iter;
        // this issuer's tiles of the chunk: t0 + tt with (t0 + tt) & 1 == wg
        const int first = ((t & 1) == static_cast<uint32_t>(wg)) ? 0 : 1;
        const int mine = (ci.ntile > first) ? (ci.ntile - first + 1) / 2 : 0;
        const uint32_t ka = smem_u32(kv_buf + kvb * kKVBytes);
        const uint32_t va = ka + 32768;
        for (int m = 0; m < mine; ++m) {
          const uint32_t tm = t + first + 2 * m;
          const uint32_t n = tm >> 1;
          // ---- S = Q K^T
          if (!mbar_wait(&sm.q_full[wg], n & 1, abort_flag) ||
              (n >= 1 && !mbar_wait(&sm.s_free[wg], (n - 1) & 1, abort_flag))) {
            report_timeout(abort_flag, hdr, 213);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qa = smem_u32(q_buf + wg * kQTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_bf16(s_col, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), idesc_qk,
                      kk > 0 ? 1u : 0u);
          }
          umma_commit(&sm.s_full[wg]);
          umma_commit(&sm.q_empty[wg]);  // the Q stage is free once QK^T has retired
          // ---- O = P_hi V + P_lo V
          if (!mbar_wait(&sm.p_full[wg], n & 1, abort_flag) ||
              (n >= 1 && !mbar_wait(&sm.o_free[wg], (n - 1) & 1, abort_flag))) {
            report_timeout(abort_flag, hdr, 214);
            ok = false;
            break;
          }
          tc_fence_after();
          // P sits in the S columns of TMEM as bf16 pairs, per 32 keys: the high
          // parts (16 columns), then the low parts (p - bf16(p), 16 columns).
          // K-step kk covers keys 16kk..16kk+15.
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16_ts(o_col, s_col + (kk >> 1) * 32 + part * 16 + (kk & 1) * 8,
                           sdesc_sw128(va + kk * 2048, 16384, 1024), idesc_pv, (part | kk) ? 1u : 0u);
          umma_commit(&sm.o_full[wg]);
          umma_commit(&sm.s_free[wg]);  // S/P columns reusable once PV has retired
          if (m == mine - 1) umma_commit(&sm.kv_empty[kvb]);
        }
        if (!ok) break;
        if (mine == 0) mbar_arrive(&sm.kv_empty[kvb]);
        t += ci.ntile;
      }
      umma_commit(&sm.mma_done[wg]);
      mbar_wait(&sm.mma_done[wg], 0, nullptr);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax
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
        const RowInfo ri = row_info(p, ci, tt, q_local);
        if (!mbar_wait_warp(&sm.s_full[wg], n & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 222);
          ok = false;
          break;
        }
        tc_fence_after();
        // pass 1: row max over the visible keys (raw scores)
        float mx = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld_32cols(lane_addr + c * 32, v);
          tmem_ld_wait();
          if (ri.lim >= 127) {
#pragma unroll
            for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(v[j]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) mx = fmaxf(mx, (c * 32 + j <= ri.lim) ? __uint_as_float(v[j]) : -INFINITY);
          }
        }
        const float ms = (mx == -INFINITY) ? 0.f : mx * p.scale_log2;  // max in scaled log2 units
        // pass 2: P = 2^(s*c - ms), its sum, and the bf16 hi + lo split written over S
        float l = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld_32cols(lane_addr + c * 32, v);
          tmem_ld_wait();
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int k0 = c * 32 + 2 * j;
            float a = exp2_approx(fmaf(__uint_as_float(v[2 * j]), p.scale_log2, -ms));
            float b = exp2_approx(fmaf(__uint_as_float(v[2 * j + 1]), p.scale_log2, -ms));
            if (k0 > ri.lim) a = 0.f;
            if (k0 + 1 > ri.lim) b = 0.f;
            l += a + b;
            const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
            hi[j] = *reinterpret_cast<const uint32_t*>(&h);
            lo[j] = pack_bf16(a - __low2float(h), b - __high2float(h));
          }
          // keys 32c..32c+31 of this row: hi pairs to columns 32c..32c+15, lo pairs
          // to 32c+16..32c+31 -- only columns this pass has already read
          tmem_st_16cols(lane_addr + c * 32, hi);
          tmem_st_16cols(lane_addr + c * 32 + 16, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full[wg]);
        sm.stat[t % kStatSlots][r] = make_float2(mx == -INFINITY ? -INFINITY : ms, l);
        mbar_arrive(&sm.stat_full[t % kStatSlots]);
        if (ri.valid)
          p.part.lse[((static_cast<int64_t>(ri.qi) * p.hkv + ci.g) * p.topk + ri.slot) * G + hh] =
              (mx == -INFINITY) ? -INFINITY : (ms + log2f(l)) * kLn2;
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogue
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int q_local = r / G, hh = r % G;
    uint32_t t = 0, w_iter = 0;
    bool ok = true;
    while (ok) {
      const int slot = w_iter % kWorkSlots;
      if (!mbar_wait_warp(&sm.work_full[slot], (w_iter / kWorkSlots) & 1, abort_flag)) {
        report_timeout(abort_flag, hdr, 231);
        break;
      }
      const int item = sm.work[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.work_empty[slot]);
      ++w_iter;
      if (item < 0) break;
      const ChunkInfo ci = decode_chunk(p, item);
      for (int tt = 0; tt < ci.ntile; ++tt, ++t) {
        const int w = t & 1;
        const RowInfo ri = row_info(p, ci, tt, q_local);
        if (!mbar_wait_warp(&sm.o_full[w], (t >> 1) & 1, abort_flag) ||
            !mbar_wait_warp(&sm.stat_full[t % kStatSlots], (t / kStatSlots) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 232);
          ok = false;
          break;
        }
        tc_fence_after();
        const float2 st = sm.stat[t % kStatSlots][r];
        const float inv_l = (st.y > 0.f) ? 1.f / st.y : 0.f;
        __nv_bfloat16* orow =
            p.part.o + ((static_cast<int64_t>(ri.qi) * p.hkv + ci.g) * p.topk + ri.slot) * G * kHeadDim +
            static_cast<int64_t>(hh) * kHeadDim;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld_32cols(lane_addr + w * 256 + 128 + c * 32, o);
          tmem_ld_wait();
          if (ri.valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(o[j + 0]) * inv_l, __uint_as_float(o[j + 1]) * inv_l);
              v.y = pack_bf16(__uint_as_float(o[j + 2]) * inv_l, __uint_as_float(o[j + 3]) * inv_l);
              v.z = pack_bf16(__uint_as_float(o[j + 4]) * inv_l, __uint_as_float(o[j + 5]) * inv_l);
              v.w = pack_bf16(__uint_as_float(o[j + 6]) * inv_l, __uint_as_float(o[j + 7]) * inv_l);
              *reinterpret_cast<uint4*>(orow + c * 32 + j) = v;
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&sm.o_free[w]);
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
