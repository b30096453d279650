// plan.cu -- per-call planning on the device: validate cu_seqlens against the
// host-side sizes, derive per-sequence facts, and build the work list of the
// index-scoring kernel sorted by descending cost (a counting sort over the
// number of key blocks each tile scans).  Also a device-wide exclusive scan.
// Nothing here is read back by the host.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

// Exclusive scan across a CTA (blockDim.x a multiple of 32, <= 1024).
// sh must hold 32 ints.  *total receives the CTA-wide sum.
__device__ int block_excl_scan(int v, int* sh, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? sh[warp - 1] : 0);
  *total = sh[nw - 1];
  __syncthreads();
  return excl;
}

__device__ __forceinline__ int tile_cost(const SeqInfo& si, int t0, int qt) {
  const int nq = min(qt, si.q_len - t0);
  const int last_pos = si.kv_len - si.q_len + t0 + nq - 1;
  return (last_pos >> 7) + 1;
}

__global__ void __launch_bounds__(1024) plan_kernel(PlanParams p) {
  __shared__ int sh[32];
  __shared__ int s_bad;
  griddep_wait();  // the kernel before may still read this workspace's header
  // a call starts from a clear workspace header (status flags, work counters)
  static_assert(sizeof(WsHeader) % 4 == 0, "header cleared as 32-bit words");
  for (int w = threadIdx.x; w < static_cast<int>(sizeof(WsHeader) / 4); w += blockDim.x)
    reinterpret_cast<uint32_t*>(p.hdr)[w] = 0u;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();

  for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
    const int q0 = p.cu_q[s], q1 = p.cu_q[s + 1], k0 = p.cu_k[s], k1 = p.cu_k[s + 1];
    const int ql = q1 - q0, kl = k1 - k0;
    bool bad = ql < 0 || kl < ql || ql > p.max_q || kl > p.max_k || q0 < 0 || k0 < 0 || q1 > p.total_q ||
               k1 > p.total_k;
    if (s == 0 && (q0 != 0 || k0 != 0)) bad = true;
    if (s == p.num_seqs - 1 && (q1 != p.total_q || k1 != p.total_k)) bad = true;
    if (bad) atomicOr(&s_bad, 1);
    SeqInfo si;
    si.q_start = q0;
    si.q_len = ql;
    si.k_start = k0;
    si.kv_len = kl;
    p.seq[s] = si;
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      atomicOr(&p.hdr->status, kFlagBadSeqlens);
      p.hdr->n_qtiles = 0;
    }
    return;
  }

  // exclusive prefixes over sequences: key blocks, index tiles
  int carry_b = 0, carry_t = 0;
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int s = base + threadIdx.x;
    int nb = 0, nt = 0;
    if (s < p.num_seqs) {
      const SeqInfo si = p.seq[s];
      nb = (si.kv_len + kBlock - 1) / kBlock;
      nt = p.qt > 0 ? (si.q_len + p.qt - 1) / p.qt : 0;
    }
    int tot_b, tot_t;
    const int eb = block_excl_scan(nb, sh, &tot_b);
    const int et = block_excl_scan(nt, sh, &tot_t);
    if (s < p.num_seqs) {
      p.blk_off[s] = carry_b + eb;
      p.tile_base[s] = carry_t + et;
    }
    carry_b += tot_b;
    carry_t += tot_t;
  }
  if (threadIdx.x == 0) {
    p.blk_off[p.num_seqs] = carry_b;
    p.tile_base[p.num_seqs] = carry_t;
  }
  if (p.qt == 0) {
    if (threadIdx.x == 0) p.hdr->n_qtiles = 0;
    return;
  }
  const int n_tiles = carry_t;
  for (int c = threadIdx.x; c < p.max_nb + 2; c += blockDim.x) {
    p.hist[c] = 0;
    p.cursor[c] = 0;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < n_tiles; j += blockDim.x) {
    const int s = find_seq(p.tile_base, p.num_seqs, j);
    const int t0 = (j - p.tile_base[s]) * p.qt;
    atomicAdd(&p.hist[tile_cost(p.seq[s], t0, p.qt)], 1);
  }
  __syncthreads();
  // start[c] = number of tiles with cost > c  (descending order), kept in cursor[]
  int carry = 0;
  for (int base = 0; base < p.max_nb; base += blockDim.x) {
    const int r = base + threadIdx.x;
    const int c = p.max_nb - r;  // cost, descending
    const int h = (r < p.max_nb) ? p.hist[c] : 0;
    int tot;
    const int e = block_excl_scan(h, sh, &tot);
    if (r < p.max_nb) p.cursor[c] = carry + e;
    carry += tot;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < n_tiles; j += blockDim.x) {
    const int s = find_seq(p.tile_base, p.num_seqs, j);
    const int t0 = (j - p.tile_base[s]) * p.qt;
    const int pos = atomicAdd(&p.cursor[tile_cost(p.seq[s], t0, p.qt)], 1);
    p.tiles[pos] = make_int2(s, t0);
  }
  if (threadIdx.x == 0) p.hdr->n_qtiles = static_cast<uint32_t>(n_tiles);
}

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;
constexpr int kScanTile = kScanThreads * kScanItems;

__global__ void __launch_bounds__(kScanThreads) scan_reduce_kernel(const int32_t* in, int n, int32_t* part,
                                                                    const WsHeader* hdr) {
  __shared__ int sh[32];
  if (hdr->status & kFlagBadSeqlens) return;
  const int base = blockIdx.x * kScanTile + threadIdx.x * kScanItems;
  int s = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i)
    if (base + i < n) s += in[base + i];
  int tot;
  block_excl_scan(s, sh, &tot);
  if (threadIdx.x == 0) part[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kScanThreads) scan_parts_kernel(int32_t* part, int nparts, const WsHeader* hdr) {
  __shared__ int sh[32];
  if (hdr->status & kFlagBadSeqlens) return;
  int carry = 0;
  for (int base = 0; base < nparts; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int v = i < nparts ? part[i] : 0;
    int tot;
    const int e = block_excl_scan(v, sh, &tot);
    if (i < nparts) part[i] = carry + e;
    carry += tot;
  }
  if (threadIdx.x == 0) part[nparts] = carry;
}

__global__ void __launch_bounds__(kScanThreads) scan_down_kernel(const int32_t* in, int32_t* out, int n,
                                                                  const int32_t* part, int nparts,
                                                                  uint32_t* total_dst, const WsHeader* hdr) {
  __shared__ int sh[32];
  if (hdr->status & kFlagBadSeqlens) return;
  const int base = blockIdx.x * kScanTile + threadIdx.x * kScanItems;
  int v[kScanItems];
  int s = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    v[i] = (base + i < n) ? in[base + i] : 0;
    s += v[i];
  }
  int tot;
  int e = block_excl_scan(s, sh, &tot) + part[blockIdx.x];
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    if (base + i < n) out[base + i] = e;
    e += v[i];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    out[n] = part[nparts];
    if (total_dst) *total_dst = static_cast<uint32_t>(part[nparts]);
  }
}

}  // namespace

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
  const cudaError_t e = launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, stream, p);
  note_launches(1);
  return e;
}

int scan_tmp_ints(int n) { return (n + kScanTile - 1) / kScanTile + 1; }

cudaError_t launch_exclusive_scan(const int32_t* in, int32_t* out, int n, int32_t* tmp, uint32_t* total_dst,
                                  const WsHeader* hdr, cudaStream_t stream) {
  const int nparts = (n + kScanTile - 1) / kScanTile;
  if (nparts > 0) scan_reduce_kernel<<<nparts, kScanThreads, 0, stream>>>(in, n, tmp, hdr);
  scan_parts_kernel<<<1, kScanThreads, 0, stream>>>(tmp, nparts, hdr);
  scan_down_kernel<<<nparts > 0 ? nparts : 1, kScanThreads, 0, stream>>>(in, out, n, tmp, nparts, total_dst,
                                                                         hdr);
  note_launches(nparts > 0 ? 3 : 2);
  return cudaGetLastError();
}

}  // namespace msa
