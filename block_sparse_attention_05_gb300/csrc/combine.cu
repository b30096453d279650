// combine.cu -- second phase of the two-phase softmax: merge the per-block
// partial results of each (query, head) with their log-sum-exp weights.
//
// The Main Branch computes, for every selected block (one "slot"), a partial
// output normalised within the block, O_s, and its log-sum-exp L_s.  Exact
// softmax attention over the union of the blocks is then
//     L = log sum_s exp(L_s),   O = sum_s exp(L_s - L) O_s .
// The stored partial is U_s = O_s exp(L_s - W_s) with its own log weight W_s
// (W_s = L_s when it is stored normalised), so the merge is
//     O = sum_s exp(W_s - L) U_s .
// (The atlas record of the report lists a two-phase combine with per-partial
// LSE buffers and no atomics; this kernel is that second phase.)
//
// One warp per two heads of a query (same group, G >= 8): each half-warp
// owns a head, its lanes 8 of the 128 output columns and, for the slot
// loads, one slot each (slots hl, hl + 16, ... when k > 16).  Every load -- the slots' block indices, LSEs, log
// weights and all k partial rows -- is issued before any is used, so a row
// costs one memory round trip; the sequence lookup that decides which slots
// are valid runs alongside.  Slots whose block index is -1 or past the
// query's causal end hold no partial (their memory is never written, so its
// contents are only ever selected away, never multiplied) and are skipped,
// matching the scheduler.
//
// The kernel is a grid-stride loop (two CTAs per SM), and each warp first
// prefetches into L2 the partial rows of the item it takes next.  A warp's
// loads are bounded by its registers (16 slots x 16 bytes per lane); the
// prefetches hold none, so the HBM stream keeps running while the warps
// combine rows that are already in L2.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kCombineWarps = 8;

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

struct PairRef {
  int i, h, g, hh;
  int64_t sel_base;
};

__device__ __forceinline__ PairRef pair_ref(const CombineParams& p, int64_t pair, int half) {
  PairRef r;
  r.i = static_cast<int>(pair / (p.hq >> 1));
  r.h = static_cast<int>(pair % (p.hq >> 1)) * 2 + half;
  r.g = r.h / p.group;
  r.hh = r.h % p.group;
  r.sel_base = (static_cast<int64_t>(r.i) * p.hkv + r.g) * p.topk;
  return r;
}

// NG groups of 16 slots (topk <= 16 NG): lane hl of a half-warp holds slots hl, hl + 16, ... for the
// log-sum-exp, and the partial rows are loaded and accumulated 16 slots at a time.
// F16: the partial rows are fp16 (prefill), else bf16 (decode).
template <int NG, bool F16>
__global__ void __launch_bounds__(32 * kCombineWarps, 2) combine_kernel(CombineParams p) {
  griddep_wait();  // the partials come from the Main Branch kernel
  if (p.hdr->status & kFlagBadSeqlens) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const int64_t n_pairs = static_cast<int64_t>(p.total_q) * (p.hq >> 1);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCombineWarps;
  const int64_t slot_stride = static_cast<int64_t>(p.group) * kHeadDim;
  for (int64_t pair = static_cast<int64_t>(blockIdx.x) * kCombineWarps + warp; pair < n_pairs; pair += stride) {
    // the next item's rows: lane (half, hl) covers slots hl + 16 j of head 2 * pair + half, 256 bytes = 2 lines
    if (pair + stride < n_pairs) {
      const PairRef nx = pair_ref(p, pair + stride, half);
#pragma unroll
      for (int j = 0; j < NG; ++j)
        if (hl + 16 * j < p.topk) {
          const uint16_t* row = p.part.o + ((nx.sel_base + hl + 16 * j) * p.group + nx.hh) * kHeadDim;
          prefetch_l2(row);
          prefetch_l2(row + 64);
        }
    }
    const PairRef r = pair_ref(p, pair, half);
    const int i = r.i, h = r.h, hh = r.hh;
    const int64_t sel_base = r.sel_base;

    int b[NG];
    float l_s[NG], w_s[NG];
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const int sl = hl + 16 * j;
      b[j] = -1;
      l_s[j] = -INFINITY;
      w_s[j] = -INFINITY;
      if (sl < p.topk) {
        b[j] = p.idx[sel_base + sl];
        l_s[j] = p.part.lse[(sel_base + sl) * p.group + hh];
        w_s[j] = p.part.ow[(sel_base + sl) * p.group + hh];
      }
    }
    const uint16_t* base = p.part.o + (sel_base * p.group + hh) * kHeadDim + hl * 8;
    uint4 raw[16];
#pragma unroll
    for (int sl = 0; sl < 16; ++sl)
      raw[sl] = (sl < p.topk) ? __ldcs(reinterpret_cast<const uint4*>(base + sl * slot_stride))
                              : make_uint4(0, 0, 0, 0);

    const int s = p.one_query_per_seq ? i : find_seq(p.cu_q, p.num_seqs, i);
    const SeqInfo si = p.seq[s];
    const int local = (si.kv_len - si.q_len + (i - si.q_start)) >> 7;
    bool valid[NG];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      valid[j] = hl + 16 * j < p.topk && b[j] >= 0 && b[j] <= local;
      if (!valid[j]) l_s[j] = -INFINITY;
      m = fmaxf(m, l_s[j]);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NG; ++j) sum += valid[j] ? expf(l_s[j] - m) : 0.f;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    const float L = m + logf(sum);
    float w[NG];
#pragma unroll
    for (int j = 0; j < NG; ++j) w[j] = valid[j] ? expf(w_s[j] - L) : 0.f;

    // acc[j] holds columns 2j, 2j + 1: one packed fma per 16-bit pair (the same single rounding per
    // element as two scalar fmas); a bf16 widens to fp32 by moving its bits to the high half, an fp16 pair
    // by conversion
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      if (j > 0) {  // the next 16 slots' rows (the first 16 were issued before the weights)
#pragma unroll
        for (int sl = 0; sl < 16; ++sl)
          raw[sl] = (16 * j + sl < p.topk)
                        ? __ldcs(reinterpret_cast<const uint4*>(base + (16 * j + sl) * slot_stride))
                        : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int sl = 0; sl < 16; ++sl) {
        const float ws = __shfl_sync(0xFFFFFFFFu, w[j], (lane & 16) | sl);
        if (16 * j + sl < p.topk && ws != 0.f) {
          const uint32_t v[4] = {raw[sl].x, raw[sl].y, raw[sl].z, raw[sl].w};
          const float2 w2 = make_float2(ws, ws);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float2 x;
            if constexpr (F16) x = __half22float2(*reinterpret_cast<const __half2*>(&v[c]));
            else x = make_float2(__uint_as_float(v[c] << 16), __uint_as_float(v[c] & 0xFFFF0000u));
            acc[c] = ffma2(w2, x, acc[c]);
          }
        }
      }
    }
    const bool empty = (m == -INFINITY);
    uint4 out;
    uint32_t* ow = &out.x;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const __nv_bfloat162 t = __floats2bfloat162_rn(acc[c].x, acc[c].y);
      ow[c] = *reinterpret_cast<const uint32_t*>(&t);
    }
    const int64_t orow = static_cast<int64_t>(i) * p.hq + h;
    *reinterpret_cast<uint4*>(p.o + orow * kHeadDim + hl * 8) = out;
    if (hl == 0) p.lse[orow] = empty ? -INFINITY : L;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, bool f16_partials, cudaStream_t stream) {
  const int64_t pairs = static_cast<int64_t>(p.total_q) * (p.hq >> 1);  // hq is a multiple of 8
  if (pairs == 0) return cudaSuccess;
  int64_t grid = (pairs + kCombineWarps - 1) / kCombineWarps;
  if (grid > 2LL * p.sms) grid = 2LL * p.sms;
  const unsigned g = static_cast<unsigned>(grid);
  const int ng = (p.topk + 15) / 16;
  auto* fn = f16_partials ? (ng <= 1 ? combine_kernel<1, true> : ng == 2 ? combine_kernel<2, true>
                             : ng == 3 ? combine_kernel<3, true> : combine_kernel<4, true>)
                         : (ng <= 1 ? combine_kernel<1, false> : ng == 2 ? combine_kernel<2, false>
                             : ng == 3 ? combine_kernel<3, false> : combine_kernel<4, false>);
  const cudaError_t e = launch_pdl(fn, dim3(g), dim3(32 * kCombineWarps), 0, stream, p);
  note_launches(1);
  return e;
}

}  // namespace msa
