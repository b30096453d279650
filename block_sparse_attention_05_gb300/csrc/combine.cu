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
// One warp per (query, head): lanes own 4 of the 128 output columns and loop
// over the slots; the slot weights come from a warp reduction over the LSEs.
// Slots whose block index is -1 or past the query's causal end hold no partial
// and are skipped, matching the scheduler.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kCombineWarps = 8;
constexpr int kMaxTopk = 16;

__global__ void __launch_bounds__(32 * kCombineWarps) combine_kernel(CombineParams p) {
  if (p.hdr->status & kFlagBadSeqlens) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kCombineWarps + warp;  // (query, head)
  if (row >= static_cast<int64_t>(p.total_q) * p.hq) return;
  const int i = static_cast<int>(row / p.hq);
  const int h = static_cast<int>(row % p.hq);
  const int g = h / p.group, hh = h % p.group;
  const int s = find_seq(p.cu_q, p.num_seqs, i);
  const SeqInfo si = p.seq[s];
  const int local = (si.kv_len - si.q_len + (i - si.q_start)) >> 7;
  const int64_t sel_base = (static_cast<int64_t>(i) * p.hkv + g) * p.topk;

  float l_s = -INFINITY, w_s = -INFINITY;
  if (lane < p.topk) {
    const int b = p.idx[sel_base + lane];
    if (b >= 0 && b <= local) {
      l_s = p.part.lse[(sel_base + lane) * p.group + hh];
      w_s = p.part.ow[(sel_base + lane) * p.group + hh];
    }
  }
  float m = l_s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  float sum = (l_s == -INFINITY) ? 0.f : expf(l_s - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  const float L = m + logf(sum);
  const float w = (l_s == -INFINITY) ? 0.f : expf(w_s - L);

  // issue every slot's load before using any (memory-level parallelism)
  const __nv_bfloat16* base = p.part.o + (sel_base * p.group + hh) * kHeadDim + lane * 4;
  const int64_t slot_stride = static_cast<int64_t>(p.group) * kHeadDim;
  uint2 raw[kMaxTopk];
  float wsl[kMaxTopk];
#pragma unroll
  for (int sl = 0; sl < kMaxTopk; ++sl) {
    wsl[sl] = __shfl_sync(0xFFFFFFFFu, w, sl);
    raw[sl] = make_uint2(0u, 0u);
    if (sl < p.topk && wsl[sl] != 0.f) raw[sl] = __ldcs(reinterpret_cast<const uint2*>(base + sl * slot_stride));
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int sl = 0; sl < kMaxTopk; ++sl) {
    const float ws = wsl[sl];
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw[sl].x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw[sl].y);
    acc[0] = fmaf(ws, __low2float(a), acc[0]);
    acc[1] = fmaf(ws, __high2float(a), acc[1]);
    acc[2] = fmaf(ws, __low2float(b), acc[2]);
    acc[3] = fmaf(ws, __high2float(b), acc[3]);
  }
  const bool empty = (m == -INFINITY);
  __nv_bfloat162 o01 = __floats2bfloat162_rn(acc[0], acc[1]);
  __nv_bfloat162 o23 = __floats2bfloat162_rn(acc[2], acc[3]);
  uint2 out;
  out.x = *reinterpret_cast<uint32_t*>(&o01);
  out.y = *reinterpret_cast<uint32_t*>(&o23);
  *reinterpret_cast<uint2*>(p.o + row * kHeadDim + lane * 4) = out;
  if (lane == 0) p.lse[row] = empty ? -INFINITY : L;
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.total_q) * p.hq;
  if (rows == 0) return cudaSuccess;
  const int64_t grid = (rows + kCombineWarps - 1) / kCombineWarps;
  combine_kernel<<<static_cast<unsigned>(grid), 32 * kCombineWarps, 0, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
