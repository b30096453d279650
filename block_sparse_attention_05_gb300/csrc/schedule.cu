// schedule.cu -- inverts the block selection for the KV-outer Main Branch.
//
// For every incidence (query i, group g, slot) whose selected block b is
// valid, the incidence goes to bucket (window(i), g, key block (s, b)).  A
// counting sort (count, exclusive scan, scatter) gathers each bucket's queries
// contiguously, and every bucket is cut into chunks of at most `qpc` queries
// -- a block that many queries selected becomes several chunks, so no work item
// is much larger than another.  Buckets are ordered window-major, then by
// group: the chunks of one window and one group run together, so that group's
// Q rows of the window and its K/V stay hot in L2 while every key block they
// selected is visited.  Each chunk descriptor carries (begin, count,
// g | b << 8, s) so the attention kernel needs no lookup.
// (The atlas record of the report lists KV-outer sparse attention with query
// gathering, pre-scheduled tile chunking for hot KV blocks and dynamic load
// balancing; these kernels build that schedule on the device, with nothing
// read back by the host.)
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

__device__ __forceinline__ bool incidence(const ScheduleParams& p, int64_t e, int& i, int& slot, long long& bucket) {
  const int b = p.idx[e];
  if (b < 0) return false;
  const int per_q = p.hkv * p.topk;
  i = static_cast<int>(e / per_q);
  const int g = static_cast<int>((e / p.topk) % p.hkv);
  slot = static_cast<int>(e % p.topk);
  const int s = find_seq(p.cu_q, p.num_seqs, i);
  const SeqInfo si = p.seq[s];
  const int pos = si.kv_len - si.q_len + (i - si.q_start);
  if (b > (pos >> 7)) return false;  // not a causal block of this query: ignored
  const long long w = i / p.window;
  bucket = (w * p.hkv + g) * p.total_blocks + p.blk_off[s] + b;
  return true;
}

__global__ void sched_count_kernel(ScheduleParams p) {
  if (p.hdr->status & kFlagBadSeqlens) return;
  const int64_t n = static_cast<int64_t>(p.total_q) * p.hkv * p.topk;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int i, slot;
    long long bucket;
    if (incidence(p, e, i, slot, bucket)) atomicAdd(&p.count[bucket], 1);
  }
}

__global__ void sched_nchunk_kernel(ScheduleParams p) {
  if (p.hdr->status & kFlagBadSeqlens) return;
  for (long long bk = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; bk < p.n_buckets;
       bk += static_cast<long long>(gridDim.x) * blockDim.x)
    p.nchunk[bk] = (p.count[bk] + p.qpc - 1) / p.qpc;
}

__global__ void sched_fill_kernel(ScheduleParams p) {
  if (p.hdr->status & kFlagBadSeqlens) return;
  const int64_t n = static_cast<int64_t>(p.total_q) * p.hkv * p.topk;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int i, slot;
    long long bucket;
    if (incidence(p, e, i, slot, bucket)) {
      const int at = p.bucket_start[bucket] + atomicAdd(&p.cursor[bucket], 1);
      p.entries[at] = (i << 5) | slot;
    }
  }
}

__global__ void sched_chunks_kernel(ScheduleParams p) {
  if (p.hdr->status & kFlagBadSeqlens) return;
  for (long long bk = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; bk < p.n_buckets;
       bk += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int cnt = p.count[bk];
    if (cnt == 0) continue;
    const int begin = p.bucket_start[bk];
    const int c0 = p.chunk_start[bk];
    const int g = static_cast<int>((bk / p.total_blocks) % p.hkv);
    const int gb = static_cast<int>(bk % p.total_blocks);
    const int s = find_seq(p.blk_off, p.num_seqs, gb);
    const int b = gb - p.blk_off[s];
    for (int c = 0; c * p.qpc < cnt; ++c)
      p.chunks[c0 + c] = make_int4(begin + c * p.qpc, min(p.qpc, cnt - c * p.qpc), g | (b << 8), s);
  }
}

int grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > 65535LL * 16) g = 65535LL * 16;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_schedule(const ScheduleParams& p, cudaStream_t stream) {
  const long long n_inc = static_cast<long long>(p.total_q) * p.hkv * p.topk;
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.count, 0, sizeof(int32_t) * p.n_buckets, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.cursor, 0, sizeof(int32_t) * p.n_buckets, stream)) != cudaSuccess) return e;
  note_launches(2);
  sched_count_kernel<<<grid_for(n_inc, 256), 256, 0, stream>>>(p);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = launch_exclusive_scan(p.count, p.bucket_start, static_cast<int>(p.n_buckets), p.scan_tmp, &p.hdr->n_entries,
                            p.hdr, stream);
  if (e != cudaSuccess) return e;
  sched_nchunk_kernel<<<grid_for(p.n_buckets, 256), 256, 0, stream>>>(p);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = launch_exclusive_scan(p.nchunk, p.chunk_start, static_cast<int>(p.n_buckets), p.scan_tmp, &p.hdr->n_chunks,
                            p.hdr, stream);
  if (e != cudaSuccess) return e;
  sched_fill_kernel<<<grid_for(n_inc, 256), 256, 0, stream>>>(p);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  sched_chunks_kernel<<<grid_for(p.n_buckets, 256), 256, 0, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
