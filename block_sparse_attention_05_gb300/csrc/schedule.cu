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

// Count and fill aggregate per CTA before touching the global counters: a CTA
// takes kSchedQueries consecutive queries (all their groups and slots), counts
// its incidences per bucket in a shared-memory hash table, and only then adds
// each bucket's total to (count) or reserves a range of (cursor) in global
// memory -- one global atomic per distinct bucket instead of one per incidence.
// The hot buckets (the local block, which every query of a block selects, and
// blocks many queries agree on) are exactly the contended ones.  An incidence
// whose bucket finds no table slot within kHashProbes probes falls back to a
// global atomic; the probe sequence of a key is fixed and a slot, once taken,
// keeps its key, so a key either has a slot for every incidence of the CTA or
// for none, and the two passes of the fill agree.
constexpr int kSchedThreads = 256;
constexpr int kSchedQueries = 128;  // divides the 4096-query window
constexpr int kHashBits = 12;
constexpr int kHashSlots = 1 << kHashBits;
constexpr int kHashProbes = 64;

struct BucketTable {
  int key[kHashSlots];  // bucket, or -1 when free
  int val[kHashSlots];
};

__device__ __forceinline__ void table_clear(BucketTable& t) {
  for (int h = threadIdx.x; h < kHashSlots; h += blockDim.x) {
    t.key[h] = -1;
    t.val[h] = 0;
  }
}

__device__ __forceinline__ uint32_t table_home(int key) {
  return (static_cast<uint32_t>(key) * 2654435761u) >> (32 - kHashBits);
}

// Slot of `key`, claiming a free one on the way; -1 when all probed slots hold other keys.
__device__ __forceinline__ int table_insert(BucketTable& t, int key) {
  uint32_t h = table_home(key);
  for (int n = 0; n < kHashProbes; ++n, h = (h + 1) & (kHashSlots - 1)) {
    const int old = atomicCAS(&t.key[h], -1, key);
    if (old == -1 || old == key) return static_cast<int>(h);
  }
  return -1;
}

// Slot of `key` after the inserts are done (no slot changes any more); -1 when it has none.
__device__ __forceinline__ int table_find(const BucketTable& t, int key) {
  uint32_t h = table_home(key);
  for (int n = 0; n < kHashProbes; ++n, h = (h + 1) & (kHashSlots - 1)) {
    const int k = t.key[h];
    if (k == key) return static_cast<int>(h);
    if (k == -1) return -1;
  }
  return -1;
}

// The CTA's queries, resolved once: query i's incidence (g, slot) selecting
// block b lands in bucket base[i] + g * total_blocks + b, and counts only when
// 0 <= b <= lim[i] (a causal block of the query).
struct CtaQueries {
  int base[kSchedQueries];  // (window * hkv) * total_blocks + blk_off[seq]
  int lim[kSchedQueries];   // the query's local block
  int i0, nq;
};

__device__ __forceinline__ void load_queries(const ScheduleParams& p, CtaQueries& cq) {
  const int i0 = blockIdx.x * kSchedQueries;
  const int nq = min(kSchedQueries, p.total_q - i0);
  if (threadIdx.x == 0) {
    cq.i0 = i0;
    cq.nq = nq;
  }
  for (int q = threadIdx.x; q < nq; q += blockDim.x) {
    const int i = i0 + q;
    const int s = find_seq(p.cu_q, p.num_seqs, i);
    const SeqInfo si = p.seq[s];
    const int pos = si.kv_len - si.q_len + (i - si.q_start);
    cq.base[q] = (i / p.window) * p.hkv * p.total_blocks + p.blk_off[s];
    cq.lim[q] = pos >> 7;
  }
}

// Visits the CTA's incidences in kSchedBatch-deep batches of independent loads
// (coalesced over the flat [query, group, slot] order of idx), calling
// f(bucket, query, slot) for each counted one.
constexpr int kSchedBatch = 8;

template <typename F>
__device__ __forceinline__ void for_each_incidence(const ScheduleParams& p, const CtaQueries& cq, F&& f) {
  const int per_q = p.hkv * p.topk;
  const int n = cq.nq * per_q;
  const int32_t* idx = p.idx + static_cast<int64_t>(cq.i0) * per_q;
  for (int l0 = threadIdx.x; l0 < n; l0 += kSchedThreads * kSchedBatch) {
    int bv[kSchedBatch];
#pragma unroll
    for (int u = 0; u < kSchedBatch; ++u) {
      const int l = l0 + u * kSchedThreads;
      bv[u] = l < n ? __ldg(idx + l) : -1;
    }
#pragma unroll
    for (int u = 0; u < kSchedBatch; ++u) {
      const int l = l0 + u * kSchedThreads;
      const int q = l / per_q;
      const int r = l - q * per_q;
      const int g = r / p.topk;
      const int slot = r - g * p.topk;
      if (bv[u] < 0 || bv[u] > cq.lim[q]) continue;  // empty slot, or not a causal block: ignored
      f(cq.base[q] + g * p.total_blocks + bv[u], cq.i0 + q, slot);
    }
  }
}

__global__ void __launch_bounds__(kSchedThreads) sched_count_kernel(ScheduleParams p) {
  __shared__ BucketTable t;
  __shared__ CtaQueries cq;
  if (p.hdr->status & kFlagBadSeqlens) return;
  table_clear(t);
  load_queries(p, cq);
  __syncthreads();
  for_each_incidence(p, cq, [&](int bucket, int, int) {
    const int h = table_insert(t, bucket);
    if (h >= 0)
      atomicAdd(&t.val[h], 1);
    else
      atomicAdd(&p.count[bucket], 1);
  });
  __syncthreads();
  for (int h = threadIdx.x; h < kHashSlots; h += kSchedThreads)
    if (t.key[h] >= 0) atomicAdd(&p.count[t.key[h]], t.val[h]);
}

__global__ void sched_nchunk_kernel(ScheduleParams p) {
  if (p.hdr->status & kFlagBadSeqlens) return;
  for (long long bk = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; bk < p.n_buckets;
       bk += static_cast<long long>(gridDim.x) * blockDim.x)
    p.nchunk[bk] = (p.count[bk] + p.qpc - 1) / p.qpc;
}

__global__ void __launch_bounds__(kSchedThreads) sched_fill_kernel(ScheduleParams p) {
  __shared__ BucketTable t;
  __shared__ CtaQueries cq;
  if (p.hdr->status & kFlagBadSeqlens) return;
  table_clear(t);
  load_queries(p, cq);
  __syncthreads();
  for_each_incidence(p, cq, [&](int bucket, int, int) {
    const int h = table_insert(t, bucket);
    if (h >= 0) atomicAdd(&t.val[h], 1);
  });
  __syncthreads();
  // reserve each bucket's range once; the slot then holds the CTA's next entry position
  for (int h = threadIdx.x; h < kHashSlots; h += kSchedThreads) {
    const int key = t.key[h];
    if (key >= 0) t.val[h] = p.bucket_start[key] + atomicAdd(&p.cursor[key], t.val[h]);
  }
  __syncthreads();
  for_each_incidence(p, cq, [&](int bucket, int i, int slot) {
    const int h = table_find(t, bucket);
    const int at = h >= 0 ? atomicAdd(&t.val[h], 1) : p.bucket_start[bucket] + atomicAdd(&p.cursor[bucket], 1);
    p.entries[at] = (i << kSlotBits) | slot;
  });
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
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.count, 0, sizeof(int32_t) * p.n_buckets, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.cursor, 0, sizeof(int32_t) * p.n_buckets, stream)) != cudaSuccess) return e;
  note_launches(2);
  // one CTA per kSchedQueries queries (at least one, so the launch list is the same for every size)
  const int cta_grid = p.total_q > 0 ? (p.total_q + kSchedQueries - 1) / kSchedQueries : 1;
  sched_count_kernel<<<cta_grid, kSchedThreads, 0, stream>>>(p);
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
  sched_fill_kernel<<<cta_grid, kSchedThreads, 0, stream>>>(p);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  sched_chunks_kernel<<<grid_for(p.n_buckets, 256), 256, 0, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
