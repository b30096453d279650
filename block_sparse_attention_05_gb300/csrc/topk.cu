// topk.cu -- top-k block selection over pooled rows, local block forced in.
//
// "MiniMax Sparse Attention: let each query pick its own blocks", section "The
// mechanism, precisely": keep the top-k blocks, the block the query sits in is
// always kept.  The selection needs no exponential: it compares pooled scores
// only (the atlas record lists an exp-free TopK for the small-k regime built
// from per-thread register lists merged with shuffles; this kernel follows the
// same idea on GB300: per-lane sorted register lists of 64-bit keys, then a
// warp merge by repeated shuffle-max, then a merge across warps).
//
// One CTA of W warps per row.  Warp w scans a contiguous slice of the row, each
// lane keeping the CAP best (score, block) keys of its strided subset; k-1
// rounds of warp max extract the warp's best k-1; warp 0 merges the W lists.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kTopkMaxWarps = 8;

template <int CAP>
__global__ void __launch_bounds__(32 * kTopkMaxWarps) topk_pooled_kernel(TopkParams p) {
  __shared__ uint64_t cand[kTopkMaxWarps][CAP];
  if (p.hdr->status & kFlagBadSeqlens) return;
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!index_ok(p.hdr, row, static_cast<long long>(p.total_q) * p.hkv, 502)) return;
  const int nwarps = blockDim.x >> 5;
  const int i = row / p.hkv;
  const int s = find_seq(p.cu_q, p.num_seqs, i);
  const SeqInfo si = p.seq[s];
  const int pos = si.kv_len - si.q_len + (i - si.q_start);
  const int nb = (pos >> 7) + 1;
  const int local = nb - 1;
  const int want = min(p.topk - 1, nb - 1);
  const float* pr = p.pooled + static_cast<int64_t>(row) * p.pooled_stride;

  // this warp's slice of the non-local blocks [0, local)
  const int per = (local + nwarps - 1) / nwarps;
  const int lo = warp * per, hi = min(local, lo + per);
  TopkList<CAP> lst;
  lst.clear();
  // eight loads in flight per lane before any insertion (one memory round
  // trip per eight values instead of one per value)
  for (int b0 = lo + lane; b0 < hi; b0 += 8 * 32) {
    float v[8];
    unsigned ok = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int b = b0 + 32 * j;
      const bool use = b < hi && index_ok(p.hdr, b, p.max_nb, 501);
      v[j] = use ? pr[b] : 0.f;
      ok |= use ? (1u << j) : 0u;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (ok & (1u << j)) lst.insert(topk_key(v[j], b0 + 32 * j));
  }
#pragma unroll
  for (int r = 0; r < CAP; ++r) {
    if (r < want) {
      const uint64_t best = warp_max_u64(lst.k[0]);
      if (best != 0ull && lst.k[0] == best) lst.pop();
      if (lane == 0) cand[warp][r] = best;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  TopkList<CAP> fin;
  fin.clear();
  for (int j = lane; j < nwarps * want; j += 32) fin.insert(cand[j / want][j % want]);
  int chosen[CAP];
#pragma unroll
  for (int r = 0; r < CAP; ++r) {
    chosen[r] = -1;
    if (r < want) {
      const uint64_t best = warp_max_u64(fin.k[0]);
      if (best != 0ull && fin.k[0] == best) fin.pop();
      if (best != 0ull) chosen[r] = topk_key_block(best);
    }
  }
  if (lane == 0 && index_ok(p.hdr, local, p.max_nb, 503))
    write_selection<CAP>(p.idx + static_cast<int64_t>(row) * p.topk, p.topk, chosen, local);
}

}  // namespace

cudaError_t launch_topk_pooled(const TopkParams& p, int max_nb, cudaStream_t stream) {
  const int rows = p.total_q * p.hkv;
  if (rows == 0) return cudaSuccess;
  int warps = max_nb / 256;
  warps = warps < 1 ? 1 : (warps > kTopkMaxWarps ? kTopkMaxWarps : warps);
  const dim3 grid(rows), block(32 * warps);
  if (p.topk <= 4) topk_pooled_kernel<3><<<grid, block, 0, stream>>>(p);
  else if (p.topk <= 8) topk_pooled_kernel<7><<<grid, block, 0, stream>>>(p);
  else topk_pooled_kernel<15><<<grid, block, 0, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
