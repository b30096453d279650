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
//   S = Q K^T                 tcgen05 (bf16), 128 x 128 x 128, fp32 in TMEM
//   P = exp2(S*c - m)         softmax warpgroup, one TMEM lane (row) per thread,
//                             causal limit per row (only the local block is cut);
//                             one pass over S; P written back over S in TMEM
//                             as fp16, m a per-row reference (below)
//   U = P V16                 tcgen05 (fp16) with A read from TMEM, V16 = the
//                             fp16 copy of V, MN-major in smem
//   U / l, LSE, log weight    written per (query, group, slot, head), U / l in
//                             fp16 (below 2^14 in V16 units); the log weight
//                             W = LSE + e ln 2 undoes V's 2^-e scale
// fp8 K/V (E4M3 codes with one scale per key block and KV head) run on exact
// 16-bit copies of the codes: the tile's K scale multiplies its logits and the
// log of its V scale is added to the log weight.
// The tile covers exactly one key block, so no running rescale of U is needed.
//
// Warp roles (512 threads): warp 0 = producer (chunk claiming, K and Q
// gathers, L2 prefetches), warps 1 and 3 = one MMA issuer per softmax
// warpgroup, warp 2 = TMEM allocator, then V loader, warps 4..7 and 8..11 =
// two softmax warpgroups taking alternate tiles (each owns an S/P and a U
// accumulator in TMEM: 2 x (128 + 128) = 512 columns), warps 12..15 = the
// epilogue warpgroup (U read-back, normalisation, partial stores) for every
// tile, which gets each row's sum of P through a 4-slot shared buffer.  Q
// tiles live in a 4-stage ring (two stages per MMA issuer), each freed as soon
// as its QK^T retires.  K and V have one buffer each with their own barriers:
// the next chunk's K is loaded once the current chunk's last QK^T retires and
// its V once the last PV does, which chunks of about 16 tiles hide.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kQStages = 4;     // tile t uses stage t % 4: stages 0, 2 feed issuer 0, stages 1, 3 issuer 1
constexpr int kWorkSlots = 4;
constexpr int kStatSlots = 4;
constexpr int kQPrefetch = 4;  // Q rows are prefetched into L2 this many tiles ahead of their gather
constexpr int kQTileBytes = 128 * 128 * 2;   // 32 KB
constexpr int kKVTileBytes = kQTileBytes;     // K or V of one block, 32 KB
constexpr int kAttnThreads = 512;
constexpr float kLn2 = 0.6931471805599453f;

struct ChunkInfo {
  int g, b, s, begin, count, ntile, krow;
};

// Per tile and row, softmax -> epilogue: the sum of P and where the row goes
// (0 for a padding row).
struct RowStat {
  float l;
  int pad;
  unsigned long long orow;
};

constexpr int kMaxChunkEntries = 16 * kTilesPerChunk;  // qpt <= 16 queries per tile

struct AttnSmem {
  uint8_t stage[4][32 * 64];     // epilogue: per warp, 32 rows x 32 bf16 (one quarter of the row)
  int ent[2][kMaxChunkEntries];  // producer: entries of the current and the next chunk
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t k_full, k_empty, v_full, v_empty;
  uint64_t s_full[2], s_free[2], p_full[2], o_full[2], o_free[2];
  uint64_t stat_full[kStatSlots];
  uint64_t work_full[kWorkSlots], work_empty[kWorkSlots];
  uint64_t mma_done[2];
  RowStat stat[kStatSlots][128];
  ChunkInfo work_ci[kWorkSlots];  // the published chunks, decoded by the producer
  int work[kWorkSlots];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kAttnSmemBytes = 1024 + 2 * kKVTileBytes + kQStages * kQTileBytes + sizeof(AttnSmem);


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

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
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
    ri.qi = ent >> kSlotBits;
    ri.slot = ent & kSlotMask;
    const SeqInfo si = p.seq[ci.s];
    const int pos = si.kv_len - si.q_len + (ri.qi - si.q_start);
    ri.lim = pos - ci.b * kBlock;  // keys 0..lim of this block are visible
  }
  return ri;
}

// Multiplies this lane's first n8 groups of 8 P columns (fp16 pairs) by f, an
// exact power of two.  Warp-collective (tcgen05 loads and stores); rare, so
// kept out of line to leave the softmax loop its registers.
__device__ __noinline__ void rescale_p(uint32_t lane_addr, int n8, float f) {
  const __half2 f2 = __float2half2_rn(f);
  tmem_st_wait();
  for (int cc = 0; cc < n8; ++cc) {
    uint32_t w8[8];
    tmem_ld_8cols(lane_addr + cc * 8, w8);
    tmem_ld_wait_regs8(w8);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&w8[j]), f2);
      w8[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    tmem_st_8cols(lane_addr + cc * 8, w8);
  }
}

}  // namespace

__global__ void __launch_bounds__(kAttnThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  WsHeader* hdr = p.hdr;
  if (hdr->status & kFlagBadSeqlens) return;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* k_buf = base;                        // K of the current chunk, 32 KB
  uint8_t* v_buf = base + kKVTileBytes;         // V (fp16 copy) of the current chunk, 32 KB
  uint8_t* q_buf = base + 2 * kKVTileBytes;     // kQStages x 32 KB
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(base + 2 * kKVTileBytes + kQStages * kQTileBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_chunks = static_cast<int>(hdr->n_chunks);
  const int G = p.group;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
    }
    mbar_init(&sm.k_full, 1);
    mbar_init(&sm.k_empty, 2);  // one arrival per MMA issuer
    mbar_init(&sm.v_full, 1);
    mbar_init(&sm.v_empty, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_free[i], 1);
      mbar_init(&sm.p_full[i], 128);
      mbar_init(&sm.o_full[i], 1);
      mbar_init(&sm.o_free[i], 128);
    }
    for (int i = 0; i < kStatSlots; ++i) mbar_init(&sm.stat_full[i], 128);
    for (int i = 0; i < kWorkSlots; ++i) {
      mbar_init(&sm.work_full[i], 1);
      mbar_init(&sm.work_empty[i], 15);  // 2 MMA threads + V loader + 8 softmax + 4 epilogue warps
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
  const float v_shift = static_cast<float>(v_scale_shift(hdr->vmax_bits));  // V copy = V * 2^-v_shift

  if (warp == 0) {
    // ------------------------------------------------------------ producer warp
    // Claims chunks one ahead of the one it feeds: while chunk w's K/V and Q
    // tiles are loaded into shared memory, chunk w+1's entries already sit in
    // shared memory and its K and V are on their way into L2.  Along with the
    // Q gather of each tile, the Q rows of the tile kQPrefetch places later
    // (in this chunk or the next) are prefetched into L2, so that the gathers
    // find their rows there; spread this way, the prefetches never queue up
    // in front of a gather.
    uint32_t q_iter = 0, kv_iter = 0;
    auto claim = [&]() -> int {
      int u = -1;
      if (lane == 0) {
        u = static_cast<int>(atomicAdd(&hdr->counter[1], 1u));
        if (u >= n_chunks || *abort_flag) u = -1;
      }
      return __shfl_sync(0xFFFFFFFFu, u, 0);
    };
    auto stage_chunk = [&](int item, int buf) {
      if (item < 0) return;
      const ChunkInfo ci = decode_chunk(p, item);
      for (int e = lane; e < ci.count; e += 32) sm.ent[buf][e] = p.entries[ci.begin + e];
      if (lane < 4) tma_prefetch_3d((lane & 2) ? &tm_v : &tm_k, (lane & 1) * 64, ci.g, ci.krow);
      __syncwarp();
    };
    // L2 prefetch of the Q rows of tile tt of a staged chunk (one lane per
    // query): a query's G heads of group g are G * 256 contiguous bytes of Q.
    auto prefetch_q = [&](const ChunkInfo& c, int buf, int tt) {
      const int e = tt * p.qpt + lane;
      if (lane < p.qpt && e < c.count) {
        const int qi = sm.ent[buf][e] >> kSlotBits;
        bulk_prefetch_l2(p.q + (static_cast<int64_t>(qi) * p.hkv + c.g) * G * kHeadDim, G * kHeadDim * 2);
      }
    };
    int cur = claim();
    stage_chunk(cur, 0);
    if (cur >= 0) {
      const ChunkInfo c0 = decode_chunk(p, cur);
      for (int tt = 0; tt < kQPrefetch && tt < c0.ntile; ++tt) prefetch_q(c0, 0, tt);
    }
    for (uint32_t w = 0;; ++w) {
      const int item = cur;
      const int buf = w & 1;
      int nxt = -1;
      ChunkInfo nci{};
      if (item >= 0) {
        nxt = claim();
        stage_chunk(nxt, buf ^ 1);  // chunk w-1's loads are all issued: its entries are free
        if (nxt >= 0) nci = decode_chunk(p, nxt);
      }
      const int slot = w % kWorkSlots;
      if (w >= kWorkSlots && !mbar_wait_warp(&sm.work_empty[slot], ((w / kWorkSlots) - 1) & 1, abort_flag)) {
        if (lane == 0) report_timeout(abort_flag, hdr, 201);
        break;
      }
      ChunkInfo ci{};
      if (item >= 0) ci = decode_chunk(p, item);
      if (lane == 0) {
        sm.work[slot] = item;
        sm.work_ci[slot] = ci;
        mbar_arrive(&sm.work_full[slot]);
      }
      if (item < 0) break;
      // K of this chunk, once every QK^T of the previous chunk has retired
      // (V is loaded by warp 2 once every PV of the previous chunk has).
      if (kv_iter >= 1 && !mbar_wait_warp(&sm.k_empty, (kv_iter - 1) & 1, abort_flag)) {
        if (lane == 0) report_timeout(abort_flag, hdr, 202);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&sm.k_full, kKVTileBytes);
        tma_load_3d(k_buf, &tm_k, &sm.k_full, 0, ci.g, ci.krow);
        tma_load_3d(k_buf + 16384, &tm_k, &sm.k_full, 64, ci.g, ci.krow);
      }
      ++kv_iter;
      bool ok = true;
      for (int tt = 0; tt < ci.ntile; ++tt) {
        const int qs = q_iter % kQStages;
        if (q_iter >= kQStages && !mbar_wait_warp(&sm.q_empty[qs], ((q_iter / kQStages) - 1) & 1, abort_flag)) {
          if (lane == 0) report_timeout(abort_flag, hdr, 203);
          ok = false;
          break;
        }
        {
          const int ahead = tt + kQPrefetch;
          if (ahead < ci.ntile) prefetch_q(ci, buf, ahead);
          else if (nxt >= 0 && ahead - ci.ntile < nci.ntile) prefetch_q(nci, buf ^ 1, ahead - ci.ntile);
        }
        // The gather: one TMA box per query brings its G heads of group g
        // (G * 256 contiguous bytes of Q) in the layout the MMA reads: 8-row
        // groups 2 KB apart, each holding the rows' first 64 dims (1 KB,
        // 128-byte swizzle) and then their last 64.
        if (lane == 0) mbar_arrive_expect_tx(&sm.q_full[qs], kQTileBytes);
        __syncwarp();
        if (lane < p.qpt) {  // one lane per query of the tile
          int e = tt * p.qpt + lane;
          if (e >= ci.count) e = 0;  // pad the last tile with a real row
          const int qg = (sm.ent[buf][e] >> kSlotBits) * p.hkv + ci.g;
          tma_load_5d(q_buf + qs * kQTileBytes + lane * G * 256, &tm_q, &sm.q_full[qs], qg);
        }
        ++q_iter;
      }
      if (!ok) break;
      cur = nxt;
    }
    if (lane == 0) {
      for (int s = 0; s < kQStages; ++s)
        if (q_iter > static_cast<uint32_t>(s)) {
          const uint32_t last = ((q_iter - 1 - s) / kQStages) * kQStages + s;
          mbar_wait(&sm.q_full[s], (last / kQStages) & 1, nullptr);
        }
      if (kv_iter > 0) mbar_wait(&sm.k_full, (kv_iter - 1) & 1, nullptr);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ V loader
    // (after allocating TMEM) loads each chunk's V once every PV of the
    // previous chunk has retired, so that a chunk change stalls neither the
    // Q gathers nor the first QK^T of the next chunk.
    uint32_t w_iter = 0, v_iter = 0;
    for (;;) {
      const int slot = w_iter % kWorkSlots;
      if (!mbar_wait_warp(&sm.work_full[slot], (w_iter / kWorkSlots) & 1, abort_flag)) {
        if (lane == 0) report_timeout(abort_flag, hdr, 241);
        break;
      }
      const int item = sm.work[slot];
      const ChunkInfo ci = sm.work_ci[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.work_empty[slot]);
      ++w_iter;
      if (item < 0) break;
      if (v_iter >= 1 && !mbar_wait_warp(&sm.v_empty, (v_iter - 1) & 1, abort_flag)) {
        if (lane == 0) report_timeout(abort_flag, hdr, 242);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&sm.v_full, kKVTileBytes);
        tma_load_3d(v_buf, &tm_v, &sm.v_full, 0, ci.g, ci.krow);
        tma_load_3d(v_buf + 16384, &tm_v, &sm.v_full, 64, ci.g, ci.krow);
      }
      ++v_iter;
    }
    if (lane == 0 && v_iter > 0) mbar_wait(&sm.v_full, (v_iter - 1) & 1, nullptr);
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per softmax warpgroup: warp 1 drives the even tiles,
    // warp 3 the odd ones, so a wait for one warpgroup never stalls the other.
    // Tile t uses Q stage t % 4, so stages 0 and 2 belong to warp 1 and
    // stages 1 and 3 to warp 3: each stage has one consumer.
    if (lane == 0) {
      const int wg = (warp == 1) ? 0 : 1;
      const uint32_t idesc_qk = idesc_bf16(128, 128, false);
      const uint32_t idesc_pv = idesc_f16(128, 128, true);
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
        const ChunkInfo ci = sm.work_ci[slot];
        mbar_arrive(&sm.work_empty[slot]);
        ++w_iter;
        if (item < 0) break;
        // every issuer waits for every chunk's K and V, used or not, so that it
        // never arrives on k_empty / v_empty for a later fill too early
        const uint32_t kv_par = kv_iter & 1;
        if (!mbar_wait(&sm.k_full, kv_par, abort_flag)) {
          report_timeout(abort_flag, hdr, 212);
          break;
        }
        ++kv_iter;
        // this issuer's tiles of the chunk: t0 + tt with (t0 + tt) & 1 == wg
        const int first = ((t & 1) == static_cast<uint32_t>(wg)) ? 0 : 1;
        const int mine = (ci.ntile > first) ? (ci.ntile - first + 1) / 2 : 0;
        const uint32_t ka = smem_u32(k_buf);
        const uint32_t va = smem_u32(v_buf);
        for (int m = 0; m < mine; ++m) {
          const uint32_t tm = t + first + 2 * m;
          const uint32_t n = tm >> 1;
          // ---- S = Q K^T
          const int qs = tm & (kQStages - 1);
          if (!mbar_wait(&sm.q_full[qs], (tm / kQStages) & 1, abort_flag) ||
              (n >= 1 && !mbar_wait(&sm.s_free[wg], (n - 1) & 1, abort_flag))) {
            report_timeout(abort_flag, hdr, 213);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qa = smem_u32(q_buf + qs * kQTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;  // K: 64-dim halves 16 KB apart
            const uint32_t qoff = (kk >> 2) * 1024 + (kk & 3) * 32;   // Q: halves interleaved per row group
            umma_bf16(s_col, sdesc_sw128(qa + qoff, 16, 2048), sdesc_sw128(ka + koff, 16, 1024), idesc_qk,
                      kk > 0 ? 1u : 0u);
          }
          umma_commit(&sm.s_full[wg]);
          umma_commit(&sm.q_empty[qs]);  // the Q stage is free once QK^T has retired
          if (m == mine - 1) umma_commit(&sm.k_empty);
          if (m == 0 && !mbar_wait(&sm.v_full, kv_par, abort_flag)) {
            report_timeout(abort_flag, hdr, 215);
            ok = false;
            break;
          }
          // ---- U = P V (fp16)
          if (!mbar_wait(&sm.p_full[wg], n & 1, abort_flag) ||
              (n >= 1 && !mbar_wait(&sm.o_free[wg], (n - 1) & 1, abort_flag))) {
            report_timeout(abort_flag, hdr, 214);
            ok = false;
            break;
          }
          tc_fence_after();
          // P sits in the S columns of TMEM as fp16 pairs: K-step kk (keys
          // 16kk..16kk+15) in columns 8kk..8kk+7.
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16_ts(o_col, s_col + kk * 8, sdesc_sw128(va + kk * 2048, 16384, 1024), idesc_pv, kk ? 1u : 0u);
          umma_commit(&sm.o_full[wg]);
          umma_commit(&sm.s_free[wg]);  // S/P columns reusable once PV has retired
          if (m == mine - 1) umma_commit(&sm.v_empty);
        }
        if (!ok) break;
        if (mine == 0) {
          mbar_arrive(&sm.k_empty);
          if (!mbar_wait(&sm.v_full, kv_par, abort_flag)) {
            report_timeout(abort_flag, hdr, 216);
            break;
          }
          mbar_arrive(&sm.v_empty);
        }
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
      const ChunkInfo ci = sm.work_ci[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.work_empty[slot]);
      ++w_iter;
      if (item < 0) break;
      // the tile's logit scale and the log of V's scale: fp8 K/V carry one scale per (key block, KV head),
      // a bf16 V copy the power of two 2^v_shift
      float sc_log2 = p.scale_log2, lnv = v_shift * kLn2;
      if (p.k_scale) {
        const long long srow = (static_cast<long long>(p.blk_off[ci.s]) + ci.b) * p.hkv + ci.g;
        sc_log2 *= p.k_scale[srow];
        lnv = logf(p.v_scale[srow]);
      }
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
        // One pass over S, 32 keys at a time, each step's load issued one step
        // ahead.  The exponent reference m starts at the max of the first
        // step's visible keys; a later step whose max exceeds it by more than
        // 2^15 first rescales the P already stored by an exact power of two and
        // raises m (rare), so every P lies in [0, 2^15] and fits fp16.  P goes
        // back over the step's own S columns as fp16 pairs: keys 32c..32c+31
        // -> columns 16c..16c+15 (keys 16k..16k+15 in columns 8k..8k+7, one
        // PV K-step each).  With l = sum_k P_k the epilogue stores U / l,
        // U = sum_k P_k v_k over V scaled by 2^-e: the block's normalised output
        // times 2^-e, so its LSE is (m + log2 l) ln 2 and its log weight that
        // LSE + e ln 2.
        const int lim = ri.valid ? ri.lim : kBlock - 1;  // padding rows: computed, never stored
        const bool warp_full = __all_sync(0xFFFFFFFFu, lim >= kBlock - 1);
        float2 l2 = make_float2(0.f, 0.f);
        float m_ref = 0.f;
        {
          uint32_t va[32], vb[32];
          // score j of step c, -inf past the row's causal limit on the masked path
          auto sval = [&](const uint32_t (&v)[32], int c, bool masked, int j) {
            return (!masked || c * 32 + j <= lim) ? __uint_as_float(v[j]) : -INFINITY;
          };
          // cmax: the load's own maximum of the step's 32 scores (used when no key is masked)
          auto process = [&](const uint32_t (&v)[32], int c, bool masked, float cmax) {
            float cm = cmax;
            if (masked) {
              float t8[11];
#pragma unroll
              for (int j = 0; j < 10; ++j)
                t8[j] = fmax3(sval(v, c, masked, 3 * j), sval(v, c, masked, 3 * j + 1), sval(v, c, masked, 3 * j + 2));
              t8[10] = fmaxf(sval(v, c, masked, 30), sval(v, c, masked, 31));
              cm = fmaxf(fmax3(fmax3(t8[0], t8[1], t8[2]), fmax3(t8[3], t8[4], t8[5]), fmax3(t8[6], t8[7], t8[8])),
                         fmaxf(t8[9], t8[10]));
            }
            if (c == 0) m_ref = (cm == -INFINITY) ? 0.f : cm * sc_log2;
            // The rescale uses warp-collective TMEM loads and stores, so the
            // whole warp enters it when any of its rows needs it; the other rows
            // scale by exactly 1.
            const bool need = cm != -INFINITY && cm * sc_log2 - m_ref > 15.f;
            if (__any_sync(0xFFFFFFFFu, need)) {
              const float kexp = need ? ceilf(cm * sc_log2 - m_ref) : 0.f;
              const float f = exp2f(-kexp);
              rescale_p(lane_addr, 2 * c, f);
              l2.x *= f;
              l2.y *= f;
              m_ref += kexp;
            }
            const float2 sc = make_float2(sc_log2, sc_log2), nm = make_float2(-m_ref, -m_ref);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t pk[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int k = 16 * h + 2 * j;
                const float2 z = ffma2(make_float2(sval(v, c, masked, k), sval(v, c, masked, k + 1)), sc, nm);
                const float2 x = make_float2(exp2_approx(z.x), exp2_approx(z.y));
                l2 = fadd2(l2, x);
                const __half2 hx = __floats2half2_rn(x.x, x.y);
                pk[j] = *reinterpret_cast<const uint32_t*>(&hx);
              }
              tmem_st_8cols(lane_addr + c * 16 + h * 8, pk);
            }
          };
          float ma, mb;
          tmem_ld_max_32cols(lane_addr, va, ma);
          tmem_ld_wait_regs_max(va, ma);
          if (warp_full) {
            tmem_ld_max_32cols(lane_addr + 32, vb, mb);
            process(va, 0, false, ma);
            tmem_ld_wait_regs_max(vb, mb);
            tmem_ld_max_32cols(lane_addr + 64, va, ma);
            process(vb, 1, false, mb);
            tmem_ld_wait_regs_max(va, ma);
            tmem_ld_max_32cols(lane_addr + 96, vb, mb);
            process(va, 2, false, ma);
            tmem_ld_wait_regs_max(vb, mb);
            process(vb, 3, false, mb);
          } else {
            tmem_ld_32cols(lane_addr + 32, vb);
            process(va, 0, true, 0.f);
            tmem_ld_wait_regs(vb);
            tmem_ld_32cols(lane_addr + 64, va);
            process(vb, 1, true, 0.f);
            tmem_ld_wait_regs(va);
            tmem_ld_32cols(lane_addr + 96, vb);
            process(va, 2, true, 0.f);
            tmem_ld_wait_regs(vb);
            process(vb, 3, true, 0.f);
          }
        }
        const float l = l2.x + l2.y;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full[wg]);
        {
          RowStat rs;
          rs.l = l;
          rs.pad = 0;
          rs.orow = ri.valid ? reinterpret_cast<unsigned long long>(
                                   p.part.o +
                                   ((static_cast<int64_t>(ri.qi) * p.hkv + ci.g) * p.topk + ri.slot) * G * kHeadDim +
                                   static_cast<int64_t>(hh) * kHeadDim)
                             : 0ull;
          sm.stat[t % kStatSlots][r] = rs;
        }
        mbar_arrive(&sm.stat_full[t % kStatSlots]);
        if (ri.valid) {
          const int64_t at = ((static_cast<int64_t>(ri.qi) * p.hkv + ci.g) * p.topk + ri.slot) * G + hh;
          const bool empty = lim < 0;
          const float lse2 = m_ref + log2f(l);
          p.part.lse[at] = empty ? -INFINITY : lse2 * kLn2;
          p.part.ow[at] = empty ? -INFINITY : lse2 * kLn2 + lnv;
        }
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogue
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    uint8_t* stg = sm.stage[warp & 3];
    uint32_t t = 0, w_iter = 0;
    bool ok = true;
    while (ok) {
      const int slot = w_iter % kWorkSlots;
      if (!mbar_wait_warp(&sm.work_full[slot], (w_iter / kWorkSlots) & 1, abort_flag)) {
        report_timeout(abort_flag, hdr, 231);
        break;
      }
      const int item = sm.work[slot];
      const ChunkInfo ci = sm.work_ci[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.work_empty[slot]);
      ++w_iter;
      if (item < 0) break;
      for (int tt = 0; tt < ci.ntile; ++tt, ++t) {
        const int w = t & 1;
        if (!mbar_wait_warp(&sm.o_full[w], (t >> 1) & 1, abort_flag) ||
            !mbar_wait_warp(&sm.stat_full[t % kStatSlots], (t / kStatSlots) & 1, abort_flag)) {
          report_timeout(abort_flag, hdr, 232);
          ok = false;
          break;
        }
        tc_fence_after();
        const RowStat rs = sm.stat[t % kStatSlots][r];
        const float inv_l = (rs.l > 0.f) ? 1.f / rs.l : 0.f;
        // Each lane owns one row (one TMEM lane); the rows of one query are
        // contiguous in the partial buffer.  A quarter of the row (32 values)
        // at a time goes through this warp's staging area (16-byte chunks
        // XOR-swizzled by row pair, so neither side has bank conflicts) and
        // leaves as 32-byte stores, two lanes per row, that fill whole 64-byte
        // runs of 16 rows (half the store instructions of 16-byte stores:
        // 10.38 -> 10.05 ms at 128K).
        const unsigned long long orow = rs.orow;
        unsigned long long rowp[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) rowp[k] = __shfl_sync(0xFFFFFFFFu, orow, 16 * k + (lane >> 1));
        const int ck = (lane & 1) * 2;  // the first of the two 16-byte chunks this lane stores
        auto emit = [&](const uint32_t (&o)[32], int quarter) {
          uint4 pk[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float2 il = make_float2(inv_l, inv_l);
            float2 z;
            z = fmul2(make_float2(__uint_as_float(o[8 * c + 0]), __uint_as_float(o[8 * c + 1])), il);
            pk[c].x = pack_f16(z.x, z.y);
            z = fmul2(make_float2(__uint_as_float(o[8 * c + 2]), __uint_as_float(o[8 * c + 3])), il);
            pk[c].y = pack_f16(z.x, z.y);
            z = fmul2(make_float2(__uint_as_float(o[8 * c + 4]), __uint_as_float(o[8 * c + 5])), il);
            pk[c].z = pack_f16(z.x, z.y);
            z = fmul2(make_float2(__uint_as_float(o[8 * c + 6]), __uint_as_float(o[8 * c + 7])), il);
            pk[c].w = pack_f16(z.x, z.y);
            *reinterpret_cast<uint4*>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = pk[c];
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int R = 16 * k + (lane >> 1);
            const uint4 v0 = *reinterpret_cast<const uint4*>(stg + R * 64 + ((ck ^ ((R >> 1) & 3)) << 4));
            const uint4 v1 = *reinterpret_cast<const uint4*>(stg + R * 64 + (((ck + 1) ^ ((R >> 1) & 3)) << 4));
            if (rowp[k]) st_global_32b(reinterpret_cast<uint16_t*>(rowp[k]) + quarter * 32 + ck * 8, v0, v1);
          }
          __syncwarp();
        };
        uint32_t va[32], vb[32];
        const uint32_t o_addr = lane_addr + w * 256 + 128;
        tmem_ld_32cols(o_addr, va);
        tmem_ld_wait_regs(va);
        tmem_ld_32cols(o_addr + 32, vb);
        emit(va, 0);
        tmem_ld_wait_regs(vb);
        tmem_ld_32cols(o_addr + 64, va);
        emit(vb, 1);
        tmem_ld_wait_regs(va);
        tmem_ld_32cols(o_addr + 96, vb);
        emit(va, 2);
        tmem_ld_wait_regs(vb);
        tc_fence_before();
        mbar_arrive(&sm.o_free[w]);  // every read of this U accumulator is done
        emit(vb, 3);
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
