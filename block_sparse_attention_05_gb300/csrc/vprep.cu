// vprep.cu -- fp16 copy of V for the prefill Main Branch.
//
// "MiniMax Sparse Attention: let each query pick its own blocks", section "The
// mechanism, precisely" (second bullet): the Main Branch is exact softmax
// attention over the selected blocks, O = softmax(S) V.  The prefill kernel
// keeps P in fp16 on the tensor cores (eleven significant bits, where bf16 has
// eight), and one tcgen05 MMA takes both operands in the same type, so V is
// multiplied in fp16 too.  Every bf16 value whose magnitude lies in fp16's
// normal range converts exactly; to keep large V in range the copy is scaled
// by 2^-e (v_scale_shift), an exact power of two that the partial's log
// weight takes back out.
//
// Two grid-stride passes over V (HBM-bound, 2 bytes read per element each,
// 2 written by the second): max |V| by integer atomicMax on the fp32 bits
// (non-negative floats order like their bit patterns), then the copy.
#include "common.cuh"
#include "kernels.h"

namespace msa {

namespace {

constexpr int kPrepThreads = 256;

__global__ void __launch_bounds__(kPrepThreads) v_absmax_kernel(const uint4* __restrict__ v, long long n16,
                                                                 WsHeader* hdr) {
  uint32_t m = 0;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 x = __ldcs(v + i);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0 && m) atomicMax(&hdr->vmax_bits, m << 16);  // bf16 bits -> fp32 bits
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float sigma) {
  const float a = __uint_as_float(w << 16) * sigma;
  const float b = __uint_as_float(w & 0xFFFF0000u) * sigma;
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kPrepThreads) v_to_f16_kernel(const uint4* __restrict__ v, uint4* __restrict__ v16,
                                                                 long long n16, const WsHeader* hdr) {
  const int e = v_scale_shift(hdr->vmax_bits);
  const float sigma = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, e <= 114
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 x = __ldcs(v + i);
    uint4 y;
    y.x = bf16x2_to_f16x2(x.x, sigma);
    y.y = bf16x2_to_f16x2(x.y, sigma);
    y.z = bf16x2_to_f16x2(x.z, sigma);
    y.w = bf16x2_to_f16x2(x.w, sigma);
    v16[i] = y;
  }
}

}  // namespace

cudaError_t launch_v_prep(const __nv_bfloat16* v, __half* v16, long long n_elems, WsHeader* hdr, int sms,
                          cudaStream_t stream) {
  const long long n16 = n_elems / 8;  // rows of 128 elements: always a multiple of 8
  if (n16 == 0) return cudaSuccess;
  long long want = (n16 + kPrepThreads - 1) / kPrepThreads;
  const long long cap = static_cast<long long>(sms) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  v_absmax_kernel<<<grid, kPrepThreads, 0, stream>>>(reinterpret_cast<const uint4*>(v), n16, hdr);
  v_to_f16_kernel<<<grid, kPrepThreads, 0, stream>>>(reinterpret_cast<const uint4*>(v), reinterpret_cast<uint4*>(v16),
                                                      n16, hdr);
  note_launches(2);
  return cudaGetLastError();
}

}  // namespace msa
