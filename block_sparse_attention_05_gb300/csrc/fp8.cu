// fp8.cu -- fp8 (E4M3) K/V: quantization, and the widening copies the prefill
// Main Branch reads.
//
// The atlas record of the report states that the kernels handle fp8 as well
// (provenance of section 4.2) without giving a format.  This library reads it
// as OCP E4M3 codes with one fp32 scale per (key block of 128 tokens of a
// sequence, KV head), for K and V separately: scale = amax / 448 over the
// block's rows of that head (1 when amax = 0), code = round-to-nearest-even of
// x / scale (fp32 division), saturated to +-448; value = code * scale.  Scales
// are stored [n_key_blocks, num_kv_heads], key block b of sequence s at row
// (key blocks of the sequences before s) + b.  One scale per block and head
// makes the scale a single number per Main Branch tile.
//
// quantize_kv_fp8_kernel: one CTA per (key block, KV head): max |x| of the
// block's K (and V) rows of that head, then the codes.  HBM-bound: 2 bytes read
// and 1 written per element.
// quantize_index_fp8_kernel: the same codes for the index inputs (an option
// beside the bf16 index, since a quantized index selects other blocks): K_idx
// with one scale per key block of a sequence (the index-key head is shared),
// Q_idx with one scale per (query row, group).
// kv8_widen_kernel: the prefill Main Branch multiplies on the tensor cores in
// bf16 (QK^T) and fp16 (PV), so it reads 16-bit copies of the fp8 codes (K as
// bf16, V as fp16); both conversions are exact (an E4M3 value has 4
// significant bits and an exponent within both formats' normal ranges), and the
// scales are applied per tile (to the logits and to the partial's log weight).
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ uint32_t bf16_abs_bits(uint32_t w) { return w & 0x7FFFu; }

// max |x| over the 16 KB (128 rows x 128 dims) of one head's block, as fp32 bits
__device__ __forceinline__ float block_absmax(const __nv_bfloat16* x, int hkv, int rows, uint32_t* red) {
  uint32_t m = 0;
  for (int c = threadIdx.x; c < rows * 16; c += kQuantThreads) {  // 16-byte chunks: 16 per row
    const int r = c >> 4, col = (c & 15) * 8;
    const uint4 v = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(r) * hkv * kHeadDim + col);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = max(m, max(bf16_abs_bits(w[j]), bf16_abs_bits(w[j] >> 16)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  uint32_t t = 0;
  for (int w = 0; w < kQuantThreads / 32; ++w) t = max(t, red[w]);
  __syncthreads();
  return __uint_as_float(t << 16);  // bf16 bits -> fp32 (|x|; no NaN on finite inputs)
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

__device__ __forceinline__ void quantize_block(const __nv_bfloat16* x, uint8_t* out, int hkv, int rows, float s) {
  for (int c = threadIdx.x; c < rows * 16; c += kQuantThreads) {
    const int r = c >> 4, col = (c & 15) * 8;
    const int64_t at = static_cast<int64_t>(r) * hkv * kHeadDim + col;
    const uint4 v = *reinterpret_cast<const uint4*>(x + at);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __fdiv_rn(__uint_as_float(w[j] << 16), s);
      f[2 * j + 1] = __fdiv_rn(__uint_as_float(w[j] & 0xFFFF0000u), s);
    }
    uint2 q;
    q.x = e4m3x4(f[0], f[1], f[2], f[3]);
    q.y = e4m3x4(f[4], f[5], f[6], f[7]);
    *reinterpret_cast<uint2*>(out + at) = q;
  }
}

__global__ void __launch_bounds__(kQuantThreads) quantize_kv_fp8_kernel(QuantParams p) {
  __shared__ uint32_t red[kQuantThreads / 32];
  if (p.hdr->status & kFlagBadSeqlens) return;
  const int gb = blockIdx.x / p.hkv, g = blockIdx.x % p.hkv;
  if (gb >= p.blk_off[p.num_seqs]) return;  // past the last key block (the grid is an upper bound)
  const int s = find_seq(p.blk_off, p.num_seqs, gb);
  const int b = gb - p.blk_off[s];
  const SeqInfo si = p.seq[s];
  const int rows = min(kBlock, si.kv_len - b * kBlock);
  const int64_t at = (static_cast<int64_t>(si.k_start) + b * kBlock) * p.hkv * kHeadDim + g * kHeadDim;
  const float ak = block_absmax(p.k + at, p.hkv, rows, red);
  const float av = block_absmax(p.v + at, p.hkv, rows, red);
  const float sk = ak > 0.f ? __fdiv_rn(ak, 448.0f) : 1.0f;
  const float sv = av > 0.f ? __fdiv_rn(av, 448.0f) : 1.0f;
  if (threadIdx.x == 0) {
    p.k_scale[static_cast<int64_t>(gb) * p.hkv + g] = sk;
    p.v_scale[static_cast<int64_t>(gb) * p.hkv + g] = sv;
  }
  quantize_block(p.k + at, p.k8 + at, p.hkv, rows, sk);
  quantize_block(p.v + at, p.v8 + at, p.hkv, rows, sv);
}

// Index inputs (d_idx 128): CTAs 0 .. key_ctas - 1 take one key block of K_idx
// each (the K/V block routines above with one head), the others eight Q_idx
// rows each, one warp per (query row, group) with four values per lane.  Same
// rounding as K/V: scale = amax / 448 (1 when 0), code = RNE(x / scale),
// saturated.
__global__ void __launch_bounds__(kQuantThreads) quantize_index_fp8_kernel(IndexQuantParams p) {
  __shared__ uint32_t red[kQuantThreads / 32];
  if (p.hdr->status & kFlagBadSeqlens) return;
  if (blockIdx.x < p.key_ctas) {
    const int gb = blockIdx.x;
    if (!p.k_idx || gb >= p.blk_off[p.num_seqs]) return;  // CTA-uniform, before block_absmax's barriers
    const int s = find_seq(p.blk_off, p.num_seqs, gb);
    const int b = gb - p.blk_off[s];
    const SeqInfo si = p.seq[s];
    const int rows = min(kBlock, si.kv_len - b * kBlock);
    const int64_t at = (static_cast<int64_t>(si.k_start) + b * kBlock) * kHeadDim;
    const float a = block_absmax(p.k_idx + at, 1, rows, red);
    const float sc = a > 0.f ? __fdiv_rn(a, 448.0f) : 1.0f;
    if (threadIdx.x == 0) p.k_scale[gb] = sc;
    quantize_block(p.k_idx + at, p.k8 + at, 1, rows, sc);
    return;
  }
  if (!p.q_idx) return;
  const long long r =
      (static_cast<long long>(blockIdx.x) - p.key_ctas) * (kQuantThreads / 32) + (threadIdx.x >> 5);
  if (r >= static_cast<long long>(p.total_q) * p.hkv) return;
  const int lane = threadIdx.x & 31;
  const uint2 v = *reinterpret_cast<const uint2*>(p.q_idx + r * kHeadDim + lane * 4);
  uint32_t m = max(max(bf16_abs_bits(v.x), bf16_abs_bits(v.x >> 16)), max(bf16_abs_bits(v.y), bf16_abs_bits(v.y >> 16)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  const float a = __uint_as_float(m << 16);
  const float sc = a > 0.f ? __fdiv_rn(a, 448.0f) : 1.0f;
  const float f0 = __fdiv_rn(__uint_as_float(v.x << 16), sc), f1 = __fdiv_rn(__uint_as_float(v.x & 0xFFFF0000u), sc);
  const float f2 = __fdiv_rn(__uint_as_float(v.y << 16), sc), f3 = __fdiv_rn(__uint_as_float(v.y & 0xFFFF0000u), sc);
  *reinterpret_cast<uint32_t*>(p.q8 + r * kHeadDim + lane * 4) = e4m3x4(f0, f1, f2, f3);
  if (lane == 0) p.q_scale[r] = sc;
}

__global__ void __launch_bounds__(256) kv8_widen_kernel(const uint4* __restrict__ k8, const uint4* __restrict__ v8,
                                                        uint4* __restrict__ k16, uint4* __restrict__ v16,
                                                        long long n16, const WsHeader* hdr) {
  if (hdr->status & kFlagBadSeqlens) return;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 kc = __ldcs(k8 + i), vc = __ldcs(v8 + i);
    const uint32_t kw[4] = {kc.x, kc.y, kc.z, kc.w}, vw[4] = {vc.x, vc.y, vc.z, vc.w};
    uint32_t ko[8], vo[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __nv_fp8x2_storage_t kp = static_cast<__nv_fp8x2_storage_t>((kw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
      const __nv_fp8x2_storage_t vp = static_cast<__nv_fp8x2_storage_t>((vw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
      const __half2_raw kh = __nv_cvt_fp8x2_to_halfraw2(kp, __NV_E4M3);
      const __half2_raw vh = __nv_cvt_fp8x2_to_halfraw2(vp, __NV_E4M3);
      const __half2 k2 = *reinterpret_cast<const __half2*>(&kh);
      const __nv_bfloat162 kb = __floats2bfloat162_rn(__low2float(k2), __high2float(k2));  // exact
      ko[j] = *reinterpret_cast<const uint32_t*>(&kb);
      vo[j] = static_cast<uint32_t>(vh.x) | (static_cast<uint32_t>(vh.y) << 16);
    }
    k16[2 * i] = make_uint4(ko[0], ko[1], ko[2], ko[3]);
    k16[2 * i + 1] = make_uint4(ko[4], ko[5], ko[6], ko[7]);
    v16[2 * i] = make_uint4(vo[0], vo[1], vo[2], vo[3]);
    v16[2 * i + 1] = make_uint4(vo[4], vo[5], vo[6], vo[7]);
  }
}

}  // namespace

cudaError_t launch_quantize_kv_fp8(const QuantParams& p, long long max_blocks, cudaStream_t stream) {
  const long long grid = max_blocks * p.hkv;
  if (grid <= 0) return cudaSuccess;
  quantize_kv_fp8_kernel<<<static_cast<unsigned>(grid), kQuantThreads, 0, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_quantize_index_fp8(const IndexQuantParams& p, cudaStream_t stream) {
  const long long q_ctas =
      p.q_idx ? (static_cast<long long>(p.total_q) * p.hkv + kQuantThreads / 32 - 1) / (kQuantThreads / 32) : 0;
  const long long grid = p.key_ctas + q_ctas;
  if (grid <= 0) return cudaSuccess;
  quantize_index_fp8_kernel<<<static_cast<unsigned>(grid), kQuantThreads, 0, stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_kv8_widen(const uint8_t* k8, const uint8_t* v8, __nv_bfloat16* k16, __half* v16,
                             long long n_elems, const WsHeader* hdr, int sms, cudaStream_t stream) {
  const long long n16 = n_elems / 16;  // rows of 128 codes: a multiple of 16
  if (n16 == 0) return cudaSuccess;
  const long long want = (n16 + 255) / 256, cap = static_cast<long long>(sms) * 8;
  kv8_widen_kernel<<<static_cast<unsigned>(want < cap ? want : cap), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(k8), reinterpret_cast<const uint4*>(v8), reinterpret_cast<uint4*>(k16),
      reinterpret_cast<uint4*>(v16), n16, hdr);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
