// Instruction-rate probe for the GB300 (sm_103a): lane-operations per clock per
// SM of the instructions the emulated FP8 GEMM's inner loop is built from.  Each
// of 1024 threads per CTA (one CTA per SM) runs NCH independent chains of one
// operation for ITERS iterations; the CTA's clock64 span gives the rate.
// Prints one line per operation: "<name> <lane-ops per clock per SM>", then the
// packed-vs-scalar mismatch counts "<name> <count>".
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
// packed fp32 pairs (f32x2), as the GEMM's pass 2 issues them
typedef unsigned long long u64;
__device__ __forceinline__ u64 mul_rz2(u64 a, u64 b) {
  u64 r;
  asm volatile("mul.rz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ u64 mul_rn2(u64 a, u64 b) {
  u64 r;
  asm volatile("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ u64 add_rn2(u64 a, u64 b) {
  u64 r;
  asm volatile("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ u64 pk(float lo, float hi) {
  return ((u64)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}

template <int MODE>
__global__ void probe(unsigned long long* cycles, unsigned* sink, float f0, float fk, unsigned u0) {
  const unsigned long long t0 = clock64();
  unsigned u[NCH];
  float f[NCH];
  u64 v[NCH];
  for (int i = 0; i < NCH; ++i) {
    u[i] = u0 + i * 977u + threadIdx.x;
    f[i] = f0 * (float)(i + 1 + (threadIdx.x & 7));
    v[i] = pk(f[i], f[i] * 1.5f);
  }
  const unsigned ku = u0 ^ 0x1234u;
  const u64 k2 = pk(fk, fk);
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
      if (MODE == 6) v[i] = mul_rz2(v[i], k2);                       // packed FMUL.RZ, subnormal
      if (MODE == 7) v[i] = mul_rn2(v[i], k2);                       // packed FMUL
      if (MODE == 8) v[i] = add_rn2(v[i], k2);                       // packed FADD of subnormals
    }
  }
  unsigned acc = 0;
  for (int i = 0; i < NCH; ++i) acc ^= u[i] ^ __float_as_uint(f[i]) ^ (unsigned)v[i] ^ (unsigned)(v[i] >> 32);
  const unsigned long long t1 = clock64();
  if (acc == 0xdeadbeefu) sink[threadIdx.x] = acc;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// lane-operations per clock: packed modes do two per lane and instruction
template <int MODE>
static int run(const char* name, float f0, float fk, int nsm) {
  const double ops = MODE >= 6 ? 2.0 : 1.0;
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
  printf("%s %.1f\n", name, ops * 1024.0 * ITERS * NCH / (double)mx);
  cudaFree(d_cyc);
  cudaFree(d_sink);
  return 0;
}

// Packed against scalar on random pairs: count of lanes whose bits differ (NaN
// results compare as NaN, whatever their payload), for mul.rn, mul.rz and add.rn.
__global__ void agree(const unsigned* x, const unsigned* y, int n, unsigned* bad) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a0 = __uint_as_float(x[2 * i]), a1 = __uint_as_float(x[2 * i + 1]);
  const float b0 = __uint_as_float(y[2 * i]), b1 = __uint_as_float(y[2 * i + 1]);
  const u64 A = pk(a0, a1), B = pk(b0, b1);
  const u64 r[3] = {mul_rn2(A, B), mul_rz2(A, B), add_rn2(A, B)};
  const float s0[3] = {mul_rn(a0, b0), mul_rz(a0, b0), add_rn(a0, b0)};
  const float s1[3] = {mul_rn(a1, b1), mul_rz(a1, b1), add_rn(a1, b1)};
  for (int m = 0; m < 3; ++m) {
    const unsigned got[2] = {(unsigned)r[m], (unsigned)(r[m] >> 32)};
    const unsigned want[2] = {__float_as_uint(s0[m]), __float_as_uint(s1[m])};
    for (int h = 0; h < 2; ++h) {
      const bool nan_w = (want[h] & 0x7FFFFFFFu) > 0x7F800000u;
      const bool ok = nan_w ? (got[h] & 0x7FFFFFFFu) > 0x7F800000u : got[h] == want[h];
      if (!ok) atomicAdd(&bad[m], 1u);
    }
  }
}

static unsigned rng_state = 12345u;
static unsigned rnd() {   // xorshift32
  rng_state ^= rng_state << 13;
  rng_state ^= rng_state >> 17;
  rng_state ^= rng_state << 5;
  return rng_state;
}

static int agreement(int n) {
  unsigned* hx = new unsigned[2 * (size_t)n];
  unsigned* hy = new unsigned[2 * (size_t)n];
  for (int i = 0; i < 2 * n; ++i) {
    if (i % 4 == 0) {      // any bit pattern
      hx[i] = rnd();
      hy[i] = rnd();
    } else {               // small times mid-range operands: products near and below 2^-126
      hx[i] = (rnd() & 0x807FFFFFu) | ((rnd() % 40u) << 23);
      hy[i] = (rnd() & 0x807FFFFFu) | ((60u + rnd() % 80u) << 23);
    }
  }
  unsigned *dx = nullptr, *dy = nullptr, *dbad = nullptr;
  int rc = 1;
  if (cudaMalloc(&dx, 8 * (size_t)n) == cudaSuccess && cudaMalloc(&dy, 8 * (size_t)n) == cudaSuccess &&
      cudaMalloc(&dbad, 3 * sizeof(unsigned)) == cudaSuccess) {
    cudaMemcpy(dx, hx, 8 * (size_t)n, cudaMemcpyHostToDevice);
    cudaMemcpy(dy, hy, 8 * (size_t)n, cudaMemcpyHostToDevice);
    cudaMemset(dbad, 0, 3 * sizeof(unsigned));
    agree<<<(n + 255) / 256, 256>>>(dx, dy, n, dbad);
    unsigned hb[3] = {0, 0, 0};
    if (cudaDeviceSynchronize() == cudaSuccess &&
        cudaMemcpy(hb, dbad, sizeof hb, cudaMemcpyDeviceToHost) == cudaSuccess) {
      printf("f32x2_mismatch_mul_rn %u\nf32x2_mismatch_mul_rz %u\nf32x2_mismatch_add_rn %u\n",
             hb[0], hb[1], hb[2]);
      rc = 0;
    }
  }
  cudaFree(dx);
  cudaFree(dy);
  cudaFree(dbad);
  delete[] hx;
  delete[] hy;
  return rc;
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
  rc |= run<6>("f32x2_fmul_rz_subnormal", 1e-41f, 0.99999994f, nsm);
  rc |= run<7>("f32x2_fmul_rn_normal", 1.0f, 1.0000001f, nsm);
  rc |= run<8>("f32x2_fadd_subnormal", 1e-42f, 1e-42f, nsm);
  rc |= agreement(1 << 22);
  return rc;
}
