// common.cuh -- device primitives shared by the sm_103a kernels: bounded
// mbarrier waits, TMA tile loads, tcgen05 (UMMA) issue / commit / TMEM loads,
// shared-memory matrix descriptors, and the top-k key order.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

// ----------------------------------------------------------------------------
// Workspace header: first 256 bytes of every workspace.
// ----------------------------------------------------------------------------
enum : uint32_t { kFlagTimeout = 1u, kFlagBadSeqlens = 2u, kFlagBadIndex = 4u };

// Compile with -DMSA_CHECKED=1 to make the kernels verify their computed
// indices before each global or shared access they are not certain of; a
// failed check records (site, index, bound) in the workspace header, raises
// kFlagBadIndex and skips the access.
#ifndef MSA_CHECKED
#define MSA_CHECKED 0
#endif

struct WsHeader {
  uint32_t status;          // MSA_DEVICE_* bits
  uint32_t n_qtiles;        // index-scoring work items
  uint32_t n_chunks;        // sparse-attention work items
  uint32_t n_entries;       // (query, group, slot) incidences
  uint32_t counter[8];      // persistent-kernel claim counters
  uint32_t timeout_site;    // where a wait gave up (debug)
  uint32_t bad_site;        // first failed index check: site
  long long bad_index, bad_bound;
  uint32_t vmax_bits;       // fp32 bits of max |V| (prefill Main Branch, fp16 copy of V)
};

// The prefill Main Branch multiplies P by an fp16 copy of V scaled by 2^-e,
// where e is the smallest shift that brings max |V| below 2^14 (e = 0 for any
// V already in that range, and for a V holding inf or NaN, which then
// propagates as it would unscaled).  From the fp32 bits of max |V|.
__host__ __device__ __forceinline__ int v_scale_shift(uint32_t vmax_bits) {
  if (vmax_bits >= 0x7F800000u) return 0;
  const int E = static_cast<int>(vmax_bits >> 23) - 127;  // max |V| < 2^(E+1)
  return E > 13 ? E - 13 : 0;
}

// Per-sequence facts derived once from cu_seqlens.
struct SeqInfo {
  int32_t q_start, q_len, k_start, kv_len;
};

constexpr int kBlock = 128;       // key block size (tokens)
constexpr int kHeadDim = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with the programmatic
// stream serialization attribute may be set up while the previous kernel on
// the stream drains; griddep_wait() returns once that kernel has completed and
// its writes are visible (immediately when the kernel was launched without the
// attribute).  Every such kernel calls it before touching memory the previous
// kernel writes or reads.  No kernel here triggers its dependents early: on the
// decode chain an early trigger (dependent CTAs resident while the index scan
// streams) measured 0.375 ms per decode_1m step against 0.343 without it and
// 0.352 without programmatic launches at all.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) when *abort becomes nonzero or after kWaitLimitNs; the
// caller then records the failure and leaves its loop.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  // The clock is read only every 64 failed tries (the first read starts the
  // limit): a read of the global timer takes long enough to delay noticing
  // the phase completion if it sat between every few tries.
  uint64_t t0 = 0;
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 63) {
      if (abort_flag && *abort_flag) return false;
      const uint64_t now = global_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kWaitLimitNs) return false;
    }
  }
}

// Warp-wide wait.  try_wait may release the lanes of a warp at different
// times, so a plain per-lane spin can leave the warp diverged; the code after
// a wait executes warp-collective .sync.aligned instructions (ldmatrix,
// mma.sync, tcgen05.ld/st) that need every lane converged.  __all_sync
// reconverges the warp and makes the outcome uniform.  Every lane must call it.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xFFFFFFFFu, ok) != 0;
}

// Records a failed wait: sets the CTA abort flag and the workspace status.
__device__ __forceinline__ void report_timeout(volatile int* abort_flag, WsHeader* hdr, uint32_t site) {
  *abort_flag = 1;
  atomicOr(&hdr->status, kFlagTimeout);
  atomicExch(&hdr->timeout_site, site);
}

// First row of key block b of sequence s: packed (k_start + 128 b) or, with a
// block table, its page times 128.  A page outside the cache is recorded in
// the status (always, not only in checked builds) and mapped to a row past
// the end of the cache, which a TMA load reads as zeros instead of faulting.
__device__ __forceinline__ int key_block_row(const int32_t* block_table, int bt_stride, long long n_pages,
                                             int k_start, int s, int b, WsHeader* hdr) {
  if (!block_table) return k_start + b * 128;
  const int page = block_table[static_cast<long long>(s) * bt_stride + b];
  if (page < 0 || page >= n_pages) {
    if (atomicCAS(&hdr->bad_site, 0u, 601u) == 0u) {
      hdr->bad_index = page;
      hdr->bad_bound = n_pages;
    }
    atomicOr(&hdr->status, kFlagBadIndex);
    return static_cast<int>(n_pages) * 128;
  }
  return page * 128;
}

// True when 0 <= i < n; otherwise (in checked builds) records the failure.
__device__ __forceinline__ bool index_ok(WsHeader* hdr, long long i, long long n, uint32_t site) {
#if MSA_CHECKED
  if (i < 0 || i >= n) {
    if (atomicCAS(&hdr->bad_site, 0u, site) == 0u) {
      hdr->bad_index = i;
      hdr->bad_bound = n;
    }
    atomicOr(&hdr->status, kFlagBadIndex);
    return false;
  }
#else
  (void)hdr; (void)i; (void)n; (void)site;
#endif
  return true;
}

// ----------------------------------------------------------------------------
// TMA (tiled bulk tensor copies global -> shared, completion on an mbarrier)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// tma_load_2d into the same shared-memory offset of every CTA of the cluster
// in cta_mask, each CTA's barrier at `bar`'s offset receiving its bytes.
__device__ __forceinline__ void tma_load_2d_multicast(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                                      int c1, uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "h"(cta_mask)
      : "memory");
}

// Thread-block clusters: this CTA's rank, and a barrier over every thread of the cluster (release / acquire).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Brings `bytes` contiguous bytes into L2 (16-byte aligned, a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}
// 5D box at coordinates (0, 0, 0, 0, c4).
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %3, %3, %3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(0), "r"(c4)
      : "memory");
}
// Brings a tensor-map box into L2 (no shared memory, no completion signal).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// One 32-byte global store (dst 32-byte aligned): lo to bytes 0..15, hi to 16..31.
__device__ __forceinline__ void st_global_32b(void* dst, const uint4& lo, const uint4& hi) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(lo.x), "r"(lo.y),
               "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
               : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA issue, commit, TMEM -> register loads
// ----------------------------------------------------------------------------
// Whole warp.  Writes the allocated TMEM base address to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T with kind::f8f6f4, both operands E4M3 (K =
// 32 codes, 32 bytes, per instruction), fp32 accumulate.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same with A read from tensor memory (columns a_tmem.., one row per lane, two
// 16-bit elements per 32-bit column along K).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// umma_commit arriving on `bar`'s offset in every CTA of the cluster in cta_mask.
__device__ __forceinline__ void umma_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               ::"r"(smem_u32(bar)), "h"(cta_mask)
               : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its TMEM
// lane (lane = (warp % 4) * 32 + laneid, encoded in taddr bits 31..16).
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// As tmem_ld_32cols, and `mx` receives the maximum of the 32 values (the load's
// own reduction, tcgen05.ld.red).  Valid after a wait that names it.
__device__ __forceinline__ void tmem_ld_max_32cols(uint32_t taddr, uint32_t (&r)[32], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(mx)
      : "r"(taddr));
}
// Waits for this thread's TMEM loads; the four maxima count as written here.
__device__ __forceinline__ void tmem_ld_wait_max4(float (&mx)[4]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+f"(mx[0]), "+f"(mx[1]), "+f"(mx[2]), "+f"(mx[3])::"memory");
}

// Waits for this thread's TMEM loads and marks r as written by the wait, so the
// compiler cannot read or move r between the load and this point.  This lets a
// load be issued ahead of the computation on an earlier chunk.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
        "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
        "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
        "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// As tmem_ld_wait_regs, for a load made by tmem_ld_max_32cols: its maximum
// counts as written here too.
__device__ __forceinline__ void tmem_ld_wait_regs_max(uint32_t (&r)[32], float& mx) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
        "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
        "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
        "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+f"(mx)
      :
      : "memory");
}

// Warpgroup register reallocation: every thread of the warpgroup executes it.
// The increases of a CTA draw on the registers its warps were launched with
// (threads x the kernel's register count), so a launcher checks the sum of the
// warpgroups' new counts against that before launching.
template <int N>
__device__ __forceinline__ void regs_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_claim() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Marks r and mx as written here, with no instruction: placed after a wait for
// a second load still in r, it keeps the compiler from reading r before it.
__device__ __forceinline__ void tmem_regs_written(uint32_t (&r)[32], float& mx) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+f"(mx)
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld_8cols(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait_regs8(uint32_t (&r)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}

// Packed pairs of fp32 (one instruction each on sm_100 and later).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// Three-input max (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Each thread of the warp writes 8 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_st_8cols(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format) for a tile stored in the
// 128-byte swizzled layout that TMA writes with CU_TENSOR_MAP_SWIZZLE_128B:
// rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte offset).
// For K-major operands the leading byte offset is unused; for MN-major
// operands it is the distance between 64-element column chunks.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M x N tile.
// b_mn_major: B stored with N contiguous (else K contiguous).  A is K-major.
// Same as idesc_bf16 with A and B both fp16.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4)                                  // D format: f32 (A, B format 0: f16)
         | ((b_mn_major ? 1u : 0u) << 16)           // B major
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4)                                  // D format: f32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | ((b_mn_major ? 1u : 0u) << 16)           // B major
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Instruction descriptor, kind::f8f6f4: E4M3 A and B (format code 0 for both),
// fp32 D, both K-major, M x N tile.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4)                                  // D format: f32 (A, B format 0: E4M3)
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// ----------------------------------------------------------------------------
// Top-k key order: larger key = better block.  Score descending first, then
// block index ascending.  +0 and -0 map to the same key (they compare equal).
// Key 0 is "empty" (below every real key).
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint64_t topk_key(float score, int block) {
  float s = (score == 0.0f) ? 0.0f : score;
  uint32_t u = __float_as_uint(s);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(block));
}
__device__ __forceinline__ int topk_key_block(uint64_t key) {
  return static_cast<int>(~static_cast<uint32_t>(key & 0xFFFFFFFFu));
}

// Sorted (descending) register list of the CAP best keys seen so far.
// Keys must be distinct (they embed the block index), so the order is total.
template <int CAP>
struct TopkList {
  uint64_t k[CAP];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int j = 0; j < CAP; ++j) k[j] = 0ull;
  }
  __device__ __forceinline__ void insert(uint64_t x) {
    if (x > k[CAP - 1]) {
      k[CAP - 1] = x;
#pragma unroll
      for (int j = CAP - 1; j > 0; --j) {
        const uint64_t a = k[j - 1], b = k[j];
        const bool sw = b > a;
        k[j - 1] = sw ? b : a;
        k[j] = sw ? a : b;
      }
    }
  }
  // Removes the head (the best key).
  __device__ __forceinline__ void pop() {
#pragma unroll
    for (int j = 0; j + 1 < CAP; ++j) k[j] = k[j + 1];
    k[CAP - 1] = 0ull;
  }
};

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t y = __shfl_xor_sync(0xFFFFFFFFu, x, off);
    x = y > x ? y : x;
  }
  return x;
}

// Writes the ascending selection {chosen blocks} U {local}, -1 padded, to
// out[0..k).  chosen[] holds up to CAP block indices (-1 = none), all < local.
template <int CAP>
__device__ __forceinline__ void write_selection(int32_t* out, int k, const int (&chosen)[CAP], int local) {
  int v[CAP + 1];
#pragma unroll
  for (int j = 0; j < CAP; ++j) v[j] = chosen[j] < 0 ? 0x7FFFFFFF : chosen[j];
  v[CAP] = local;
  // odd-even transposition sort, ascending
#pragma unroll
  for (int pass = 0; pass < CAP + 1; ++pass) {
#pragma unroll
    for (int j = (pass & 1); j + 1 < CAP + 1; j += 2) {
      const int a = v[j], b = v[j + 1];
      v[j] = a < b ? a : b;
      v[j + 1] = a < b ? b : a;
    }
  }
#pragma unroll
  for (int j = 0; j < CAP + 1; ++j)
    if (j < k) out[j] = (v[j] == 0x7FFFFFFF) ? -1 : v[j];
}

// Largest s in [0, num_seqs) with cu[s] <= row (the sequence owning `row`;
// empty sequences are skipped because they share their prefix value).
__device__ __forceinline__ int find_seq(const int32_t* cu, int num_seqs, int row) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace msa
