// Instruction-rate probe for the GB300 (sm_103a): lane-operations per clock per
// SM of the instructions the emulated FP8 GEMM's inner loop is built from.  Each
// of 1024 threads per CTA (one CTA per SM) runs NCH independent chains of one
// operation for ITERS iterations; the CTA's clock64 span gives the rate.
// Prints one line per operation: "<name> <lane-ops per clock per SM>".
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#define ITERS 4096
#define NCH 8

__device__ __forceinline__ float mul_rz(float a, float b) {
  float r;
  asm volatile("mul.rz.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float mul_rn(float a, float b) {
  float r;
  asm volatile("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float add_rn(float a, float b) {
  float r;
  asm volatile("add.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

template <int MODE>
__global__ void probe(unsigned long long* cycles, unsigned* sink, float f0, float fk, unsigned u0) {
  const unsigned long long t0 = clock64();
  unsigned u[NCH];
  float f[NCH];
  for (int i = 0; i < NCH; ++i) {
    u[i] = u0 + i * 977u + threadIdx.x;
    f[i] = f0 * (float)(i + 1 + (threadIdx.x & 7));
  }
  const unsigned ku = u0 ^ 0x1234u;
#pragma unroll 1
  for (int it = 0; it < ITERS; ++it) {
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      if (MODE == 0) f[i] = mul_rz(f[i], fk);                        // FMUL.RZ, subnormal results
      if (MODE == 1) f[i] = mul_rn(f[i], fk);                        // FMUL, normal results
      if (MODE == 2) f[i] = add_rn(f[i], fk);                        // FADD of subnormals
      if (MODE == 3) u[i] = __viaddmax_s16x2(u[i], ku, ku);          // DPX 16x2 add + max
      if (MODE == 4) u[i] = u[i] * ku + 7u;                          // IMAD
      if (MODE == 5) u[i] = __byte_perm(u[i], ku, 0x3276);           // PRMT
    }
  }
  unsigned acc = 0;
  for (int i = 0; i < NCH; ++i) acc ^= u[i] ^ __float_as_uint(f[i]);
  const unsigned long long t1 = clock64();
  if (acc == 0xdeadbeefu) sink[threadIdx.x] = acc;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int MODE>
static int run(const char* name, float f0, float fk, int nsm) {
  unsigned long long* d_cyc = nullptr;
  unsigned* d_sink = nullptr;
  if (cudaMalloc(&d_cyc, nsm * sizeof(unsigned long long)) != cudaSuccess) return 1;
  if (cudaMalloc(&d_sink, 1024 * sizeof(unsigned)) != cudaSuccess) return 1;
  probe<MODE><<<nsm, 1024>>>(d_cyc, d_sink, f0, fk, 3u);   // warm-up
  probe<MODE><<<nsm, 1024>>>(d_cyc, d_sink, f0, fk, 3u);
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  unsigned long long h[1024];
  cudaMemcpy(h, d_cyc, nsm * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  unsigned long long mx = 0;
  for (int i = 0; i < nsm; ++i) mx = h[i] > mx ? h[i] : mx;
  printf("%s %.1f\n", name, 1024.0 * ITERS * NCH / (double)mx);
  cudaFree(d_cyc);
  cudaFree(d_sink);
  return 0;
}

int main() {
  int nsm = 0;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  if (nsm <= 0 || nsm > 1024) return 1;
  int rc = 0;
  // x * (1 - 2^-24) rounded toward zero stays subnormal for the whole run
  rc |= run<0>("fmul_rz_subnormal", 1e-41f, 0.99999994f, nsm);
  rc |= run<1>("fmul_rn_normal", 1.0f, 1.0000001f, nsm);
  rc |= run<2>("fadd_subnormal", 1e-42f, 1e-42f, nsm);
  rc |= run<3>("viaddmax_s16x2", 1.0f, 1.0f, nsm);
  rc |= run<4>("imad", 1.0f, 1.0f, nsm);
  rc |= run<5>("prmt", 1.0f, 1.0f, nsm);
  return rc;
}
