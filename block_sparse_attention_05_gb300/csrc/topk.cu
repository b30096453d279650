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
// That needs registers for k-1 keys per lane, so it serves k <= 16; larger k
// (up to 64) take topk_radix_kernel below: a radix selection of the (k-1)-th
// best key, eight bits of the 64-bit key per pass over the row, then every
// key at or above it, written in block order by a compaction scan.
//
// Long rows in small batches (decode: a few rows of thousands of blocks) take
// topk_threshold_kernel: 1024 threads per row, each reducing its strided share
// of the row to one maximum; a bitonic sort of those maxima (in registers:
// shuffles within a warp, shared memory across warps) gives the want-th
// largest, T.  At least want keys reach T (the want threads whose maxima do)
// and at most want x (keys per thread) do, so the keys >= T are a small
// candidate set holding the answer; each candidate's rank among them is
// counted directly, and the want best are written in block order.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kTopkMaxWarps = 8;

template <int CAP>
__global__ void __launch_bounds__(32 * kTopkMaxWarps) topk_pooled_kernel(TopkParams p) {
  __shared__ uint64_t cand[kTopkMaxWarps][CAP];
  griddep_wait();  // the pooled rows come from the kernel before
  if (p.hdr->status & kFlagBadSeqlens) return;
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!index_ok(p.hdr, row, static_cast<long long>(p.total_q) * p.hkv, 502)) return;
  const int nwarps = blockDim.x >> 5;
  const int i = row / p.hkv;
  const int s = p.one_query_per_seq ? i : find_seq(p.cu_q, p.num_seqs, i);
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

constexpr int kRadixThreads = 256;

// Selection of one row by radix select.  The candidates are the non-local
// causal blocks b < local; want = min(k - 1, local) of them are kept.  Keys
// are distinct (they embed the block index), so the want-th largest key T is
// unique and the kept set is exactly {b : key(b) >= T}.  Each pass takes the
// next 8 bits of T: a histogram of that byte over the keys that agree with T
// on the bytes already fixed, then the byte whose bin holds the rank still
// wanted.  When that bin holds exactly the rank still wanted, every key in it
// is kept and the remaining bytes need not be fixed.
__global__ void __launch_bounds__(kRadixThreads) topk_radix_kernel(TopkParams p) {
  __shared__ uint32_t hist[256];
  __shared__ int s_digit, s_rem, s_exact;
  __shared__ int s_warp_tot[kRadixThreads / 32];
  griddep_wait();  // the pooled rows come from the kernel before
  if (p.hdr->status & kFlagBadSeqlens) return;
  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!index_ok(p.hdr, row, static_cast<long long>(p.total_q) * p.hkv, 511)) return;
  const int i = row / p.hkv;
  const int s = p.one_query_per_seq ? i : find_seq(p.cu_q, p.num_seqs, i);
  const SeqInfo si = p.seq[s];
  const int pos = si.kv_len - si.q_len + (i - si.q_start);
  const int local = pos >> 7;  // also the number of non-local causal blocks
  const int want = min(p.topk - 1, local);
  if (!index_ok(p.hdr, local, p.max_nb, 512)) return;
  const float* pr = p.pooled + static_cast<int64_t>(row) * p.pooled_stride;

  uint64_t prefix = 0, mask = 0;
  if (want > 0 && want < local) {
    int remaining = want;
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int h = tid; h < 256; h += kRadixThreads) hist[h] = 0u;
      __syncthreads();
      for (int b = tid; b < local; b += kRadixThreads) {
        const uint64_t key = topk_key(pr[b], b);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l holds bins 255 - 8l .. 248 - 8l (descending); counts above each lane by a shuffle scan
        uint32_t c[8];
        uint32_t tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[255 - 8 * lane - j];
          tot += c[j];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t above = incl - tot;  // keys in bins above this lane's
        const bool here = above < static_cast<uint32_t>(remaining) && incl >= static_cast<uint32_t>(remaining);
        if (here) {
          uint32_t cum = above;
          int j = 0;
          while (cum + c[j] < static_cast<uint32_t>(remaining)) cum += c[j++];
          s_digit = 255 - 8 * lane - j;
          s_rem = remaining - static_cast<int>(cum);
          s_exact = (c[j] == static_cast<uint32_t>(remaining) - cum) ? 1 : 0;
        }
      }
      __syncthreads();
      const int d = s_digit;
      remaining = s_rem;
      const bool exact = s_exact != 0;
      __syncthreads();  // every thread has read the decision before the next pass clears the histogram
      prefix |= static_cast<uint64_t>(d) << shift;
      mask |= static_cast<uint64_t>(0xFFu) << shift;
      if (exact) break;
    }
  }

  // kept blocks, written in ascending order: thread t owns the contiguous blocks [t * per, (t + 1) * per)
  const int per = (local + kRadixThreads - 1) / kRadixThreads;
  const int lo = tid * per, hi = min(local, lo + per);
  auto kept = [&](int b) {
    if (want == 0) return false;
    return (topk_key(pr[b], b) & mask) >= prefix;
  };
  int cnt = 0;
  for (int b = lo; b < hi; ++b) cnt += kept(b) ? 1 : 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp_tot[warp] = incl;
  __syncthreads();
  int base = incl - cnt;
  for (int w = 0; w < warp; ++w) base += s_warp_tot[w];
  int32_t* out = p.idx + static_cast<int64_t>(row) * p.topk;
  for (int b = lo; b < hi; ++b)
    if (kept(b)) {
      if (index_ok(p.hdr, base, p.topk - 1, 513)) out[base] = b;
      ++base;
    }
  if (tid == 0) {
    out[want] = local;
    for (int j = want + 1; j < p.topk; ++j) out[j] = -1;
  }
}

constexpr int kThrThreads = 1024;
constexpr int kThrMaxPerThread = 32;  // rows of up to 32 x 1024 blocks
constexpr int kThrCandMax = 63 * kThrMaxPerThread;
constexpr int kThrReg = 8;

__global__ void __launch_bounds__(kThrThreads) topk_threshold_kernel(TopkParams p) {
  __shared__ uint64_t xch[2][kThrThreads];  // bitonic exchanges between warps (double-buffered)
  __shared__ uint64_t kth;
  __shared__ uint64_t cand[kThrCandMax];
  __shared__ int chosen[64];
  __shared__ int n_cand;
  griddep_wait();  // the pooled rows come from the kernel before
  if (p.hdr->status & kFlagBadSeqlens) return;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  if (!index_ok(p.hdr, row, static_cast<long long>(p.total_q) * p.hkv, 521)) return;
  const int i = row / p.hkv;
  const int s = p.one_query_per_seq ? i : find_seq(p.cu_q, p.num_seqs, i);
  const SeqInfo si = p.seq[s];
  const int pos = si.kv_len - si.q_len + (i - si.q_start);
  const int local = pos >> 7;  // also the number of non-local causal blocks
  const int want = min(p.topk - 1, local);
  if (!index_ok(p.hdr, local, p.max_nb, 522) || local > kThrThreads * kThrMaxPerThread) return;
  const float* pr = p.pooled + static_cast<int64_t>(row) * p.pooled_stride;
  int32_t* out = p.idx + static_cast<int64_t>(row) * p.topk;
  if (want > 0) {
    // the first kThrReg keys of the thread's share stay in registers (all loads in flight at once); rows
    // longer than kThrReg x 1024 blocks read the rest twice
    float v[kThrReg];
#pragma unroll
    for (int r = 0; r < kThrReg; ++r) {
      const int b = tid + r * kThrThreads;
      v[r] = b < local ? pr[b] : 0.f;
    }
    uint64_t mx = 0ull;
#pragma unroll
    for (int r = 0; r < kThrReg; ++r) {
      const int b = tid + r * kThrThreads;
      const uint64_t key = b < local ? topk_key(v[r], b) : 0ull;
      mx = key > mx ? key : mx;
    }
    for (int b = tid + kThrReg * kThrThreads; b < local; b += kThrThreads) {
      const uint64_t key = topk_key(pr[b], b);
      mx = key > mx ? key : mx;
    }
    if (tid == 0) n_cand = 0;
    // bitonic sort of the maxima, descending, one key per thread in a register: partners closer than
    // a warp exchange by shuffle, farther ones through shared memory
    int xb = 0;
    for (int k = 2; k <= kThrThreads; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        uint64_t y;
        if (j < 32) {
          y = __shfl_xor_sync(0xFFFFFFFFu, mx, j);
        } else {
          xch[xb][tid] = mx;
          __syncthreads();
          y = xch[xb][tid ^ j];
          xb ^= 1;
        }
        // the lower index of a pair keeps the larger key in a descending run ((tid & k) == 0)
        const bool keep_max = ((tid & j) == 0) == ((tid & k) == 0);
        mx = keep_max ? (y > mx ? y : mx) : (y < mx ? y : mx);
      }
    }
    // want <= min(local, 63) threads hold a key, so T > 0 is a real key
    if (tid == want - 1) kth = mx;
    __syncthreads();
    const uint64_t T = kth;
    // at most want x kThrMaxPerThread keys reach T; the guard only makes that explicit
    auto keep = [&](uint64_t key) {
      if (key >= T) {
        const int c = atomicAdd(&n_cand, 1);
        if (c < kThrCandMax) cand[c] = key;
      }
    };
#pragma unroll
    for (int r = 0; r < kThrReg; ++r) {
      const int b = tid + r * kThrThreads;
      if (b < local) keep(topk_key(v[r], b));
    }
    for (int b = tid + kThrReg * kThrThreads; b < local; b += kThrThreads) keep(topk_key(pr[b], b));
    __syncthreads();
    const int nc = min(n_cand, kThrCandMax);
    // rank of each candidate among the candidates (keys are distinct); the want best are kept
    for (int c = tid; c < nc; c += kThrThreads) {
      const uint64_t key = cand[c];
      int rank = 0;
      for (int j = 0; j < nc; ++j) rank += cand[j] > key ? 1 : 0;
      if (rank < want) chosen[rank] = topk_key_block(key);
    }
    __syncthreads();
    // in block order: the position of a kept block is the number of kept blocks below it
    if (tid < want) {
      const int b = chosen[tid];
      int at = 0;
      for (int j = 0; j < want; ++j) at += chosen[j] < b ? 1 : 0;
      out[at] = b;
    }
  }
  if (tid == 0) {
    out[want] = local;
    for (int j = want + 1; j < p.topk; ++j) out[j] = -1;
  }
}

}  // namespace

template <int CAP>
static cudaError_t launch_topk_cap(const TopkParams& p, int max_nb, cudaStream_t stream) {
  const int rows = p.total_q * p.hkv;
  int warps = max_nb / 256;
  warps = warps < 1 ? 1 : (warps > kTopkMaxWarps ? kTopkMaxWarps : warps);
  const cudaError_t e = launch_pdl(topk_pooled_kernel<CAP>, dim3(rows), dim3(32 * warps), 0, stream, p);
  note_launches(1);
  return e;
}

cudaError_t launch_topk_pooled(const TopkParams& p, int max_nb, cudaStream_t stream) {
  const int rows = p.total_q * p.hkv;
  if (rows == 0) return cudaSuccess;
  // a few long rows (decode batches): one 1024-thread CTA per row
  if (max_nb >= 2048 && max_nb <= kThrThreads * kThrMaxPerThread && rows <= 1024) {
    cudaError_t e = launch_pdl(topk_threshold_kernel, dim3(rows), dim3(kThrThreads), 0, stream, p);
    note_launches(1);
    return e;
  }
  if (p.topk > 16) {
    cudaError_t e = launch_pdl(topk_radix_kernel, dim3(rows), dim3(kRadixThreads), 0, stream, p);
    note_launches(1);
    return e;
  }
  if (p.topk <= 4) return launch_topk_cap<3>(p, max_nb, stream);
  if (p.topk <= 8) return launch_topk_cap<7>(p, max_nb, stream);
  return launch_topk_cap<15>(p, max_nb, stream);
}

}  // namespace msa
