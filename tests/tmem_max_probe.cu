// Checks the TMEM load with a max reduction that the index max-pool and the
// softmax rely on: one warp writes 32 known fp32 values per TMEM lane (32
// columns), reads them back with tcgen05.ld.red ... .max.f32, and the host
// compares the returned values and each lane's reduction with its own maximum.
// One CTA of one warp, 32 TMEM columns, every access in bounds.
#include <cstdio>
#include <cstdint>
#include <cmath>
#include <cuda_runtime.h>
__global__ void probe(const float* in, float* red_out, float* val_out) {
  __shared__ uint32_t tbase;
  const int lane = threadIdx.x;
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(&tbase))) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t taddr = tbase;  // lane 0..31 of the warp, column 0
  uint32_t w[32];
  for (int c = 0; c < 32; ++c) w[c] = __float_as_uint(in[lane * 32 + c]);
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
               "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
               ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
               "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]),
               "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
               "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31]) : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  uint32_t r[32];
  float red;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=f"(red)
      : "r"(taddr) : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+f"(red) :: "memory");
  red_out[lane] = red;
  for (int c = 0; c < 32; ++c) val_out[lane * 32 + c] = __uint_as_float(r[c]);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(taddr) : "memory");
}
int main() {
  const int n = 32 * 32;
  float h_in[n], h_red[32], h_val[n];
  unsigned s = 12345u;
  for (int i = 0; i < n; ++i) { s = s * 1664525u + 1013904223u; h_in[i] = ((int)(s >> 8) % 20001 - 10000) * 0.37f; }
  h_in[3 * 32 + 7] = -0.0f; h_in[5 * 32 + 0] = 1e30f; h_in[9 * 32 + 31] = -1e30f;
  for (int c = 0; c < 32; ++c) h_in[11 * 32 + c] = -5.0f - c;  // all negative row
  float *d_in, *d_red, *d_val;
  cudaMalloc(&d_in, n * 4); cudaMalloc(&d_red, 32 * 4); cudaMalloc(&d_val, n * 4);
  cudaMemcpy(d_in, h_in, n * 4, cudaMemcpyHostToDevice);
  probe<<<1, 32>>>(d_in, d_red, d_val);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) { printf("error %s\n", cudaGetErrorString(e)); return 1; }
  cudaMemcpy(h_red, d_red, 32 * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(h_val, d_val, n * 4, cudaMemcpyDeviceToHost);
  int bad_val = 0, bad_red = 0;
  for (int l = 0; l < 32; ++l) {
    float m = -INFINITY;
    for (int c = 0; c < 32; ++c) { m = fmaxf(m, h_in[l * 32 + c]); if (h_val[l * 32 + c] != h_in[l * 32 + c]) ++bad_val; }
    if (h_red[l] != m) { ++bad_red; if (bad_red < 4) printf("lane %d: red %g expected %g\n", l, h_red[l], m); }
  }
  printf("values mismatched %d of %d, reductions mismatched %d of 32\n", bad_val, n, bad_red);
  return (bad_val || bad_red) ? 2 : 0;
}
