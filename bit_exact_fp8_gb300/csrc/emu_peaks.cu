// emu_peaks.cu -- libemupeaks: instruction-rate microbenchmark of the GB300 (sm_103a)
// pipes that the emulated FP8 GEMM issues on.  bench.py reads these rates as the
// denominators of its roofline (measured, not nominal), and the test suite checks
// that the packed f32x2 arithmetic rounds every half exactly as the scalar
// instruction does, which the GEMM's pass 2 relies on.
//
// Rates: one CTA of 1024 threads per SM; every thread runs NCH independent chains
// of one operation for ITERS iterations; the slowest CTA's clock64 span gives
// lane-operations per clock per SM (a packed f32x2 instruction counts as two).
// Nothing here waits on anything: every kernel is a fixed number of arithmetic
// iterations.
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#include "emu_peaks.h"

namespace {

constexpr int ITERS = 4096;
constexpr int NCH = 8;
constexpr int THREADS = 1024;

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
__device__ __forceinline__ unsigned lop3_xor3(unsigned a, unsigned b, unsigned c) {
  unsigned r;
  asm volatile("lop3.b32 %0, %1, %2, %3, 0x96;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ unsigned iadd3(unsigned a, unsigned b, unsigned c) {
  unsigned r;
  asm volatile("add.u32 %0, %1, %2;\n\tadd.u32 %0, %0, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ u64 pk(float lo, float hi) {
  return ((u64)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}

// The measured operations.  MIX: the GEMM's arithmetic mix per MAC, 1.5 packed
// FP32 instructions (exact product, truncating multiply, exact add) and 0.5 DPX
// add-max: per iteration six packed chains and two DPX chains, i.e. four MACs.
// The modes above take their second and third operands from kernel arguments (the
// same for every thread); the _vector modes take every operand from registers that
// differ per thread, as the GEMM's operands do.  MIX_VEC: four outputs' exact
// product, truncating multiply and add (each product fed by another output's sum)
// and four DPX add-max of per-thread labels, i.e. eight MACs per iteration.
enum Mode {
  FMUL_RZ_SUB, FMUL_RN, FADD_SUB, F2_FMUL_RZ_SUB, F2_FMUL_RN, F2_FADD_SUB,
  DPX_VIADDMAX, IMAD, IADD3, LOP3, PRMT, IMAD_IADD3, MIX, DPX_VEC, F2_FMUL_RZ_VEC, MIX_VEC,
  MIX_TILE, NUM_MODES
};
const char* const kNames[NUM_MODES] = {
    "fmul_rz_subnormal", "fmul_rn_normal", "fadd_subnormal",
    "f32x2_fmul_rz_subnormal", "f32x2_fmul_rn_normal", "f32x2_fadd_subnormal",
    "dpx_viaddmax_s16x2", "imad", "iadd3", "lop3", "prmt", "imad_iadd3_mixed",
    "emulation_mix_macs", "dpx_viaddmax_s16x2_vector", "f32x2_fmul_rz_subnormal_vector",
    "emulation_mix_vector_macs", "emulation_tile_macs"};

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
probe(unsigned long long* cycles, unsigned* sink, float f0, float fk, unsigned u0) {
  const unsigned long long t0 = clock64();
  unsigned u[NCH];
  float f[NCH];
  u64 v[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    u[i] = u0 + i * 977u + threadIdx.x;
    f[i] = f0 * (float)(i + 1 + (threadIdx.x & 7));
    v[i] = pk(f[i], f[i] * 1.5f);
  }
  const unsigned ku = u0 ^ 0x1234u, kv = u0 * 3u + 1u;
  const u64 k2 = pk(fk, fk);
  unsigned wu[NCH], wv[NCH];             // per-thread operands of the _vector modes
  u64 w2[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    wu[i] = ku + (unsigned)(threadIdx.x * 7 + i);
    wv[i] = kv ^ (unsigned)(threadIdx.x * 13 + i);
    w2[i] = pk(fk * (1.0f + 0.125f * (float)((threadIdx.x + i) & 3)), fk);
  }
#pragma unroll 1
  for (int it = 0; it < ITERS; ++it) {
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      if (MODE == FMUL_RZ_SUB) f[i] = mul_rz(f[i], fk);
      if (MODE == FMUL_RN) f[i] = mul_rn(f[i], fk);
      if (MODE == FADD_SUB) f[i] = add_rn(f[i], fk);
      if (MODE == F2_FMUL_RZ_SUB) v[i] = mul_rz2(v[i], k2);
      if (MODE == F2_FMUL_RN) v[i] = mul_rn2(v[i], k2);
      if (MODE == F2_FADD_SUB) v[i] = add_rn2(v[i], k2);
      if (MODE == DPX_VIADDMAX) u[i] = __viaddmax_s16x2(u[i], ku, kv);
      if (MODE == IMAD) u[i] = u[i] * ku + kv;
      if (MODE == IADD3) u[i] = iadd3(u[i], ku, kv);
      if (MODE == LOP3) u[i] = lop3_xor3(u[i], ku, kv);
      if (MODE == PRMT) u[i] = __byte_perm(u[i], ku, 0x3276);
      if (MODE == IMAD_IADD3) u[i] = (i & 1) ? iadd3(u[i], ku, kv) : u[i] * ku + kv;
      if (MODE == MIX) {
        if (i < 6) v[i] = (i % 3 == 0) ? mul_rn2(v[i], k2) : (i % 3 == 1) ? mul_rz2(v[i], k2)
                                                                         : add_rn2(v[i], k2);
        else u[i] = __viaddmax_s16x2(u[i], ku, kv);
      }
      if (MODE == DPX_VEC) u[i] = __viaddmax_s16x2(wu[i], wv[i], u[i]);
      if (MODE == F2_FMUL_RZ_VEC) v[i] = mul_rz2(v[i], w2[i]);
      if (MODE == MIX_VEC) {
        if (i < 4) {
          const u64 x = mul_rn2(v[(i + 1) & 3], w2[i]);
          v[i] = add_rn2(v[i], mul_rz2(x, w2[i + 4]));
        } else {
          u[i] = __viaddmax_s16x2(wu[i], wv[i], u[i]);
        }
      }
    }
  }
  unsigned acc = 0;
#pragma unroll
  for (int i = 0; i < NCH; ++i)
    acc ^= u[i] ^ __float_as_uint(f[i]) ^ (unsigned)v[i] ^ (unsigned)(v[i] >> 32);
  const unsigned long long t1 = clock64();
  if (acc == 0xdeadbeefu) sink[threadIdx.x] = acc;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// The GEMM's inner loop on a 4 x 4 thread tile: per k-pair the thread loads its
// four A and four B value pairs and label pairs from a decoded stage in shared
// memory (the 128 x 64 tile's layout), then per output one exact product,
// truncating multiply and add (packed f32x2 on the k-pair) and one DPX add-max.  No
// decode, no per-block scale or normalisation, no barrier: the ceiling of the
// kernel's arithmetic and operand traffic.  512 threads per SM, the GEMM's budget of
// 128 registers; 32 MACs per thread and k-pair.
constexpr int TILE_THREADS = 512;
constexpr int TILE_ITERS = 2048;
__global__ void __launch_bounds__(TILE_THREADS, 1)
probe_tile(unsigned long long* cycles, unsigned* sink, float f0, float fk, unsigned u0) {
  __shared__ __align__(16) u64 sA[16][128];
  __shared__ __align__(16) u64 sB[16][64];
  __shared__ __align__(16) unsigned sAl[16][128];
  __shared__ __align__(16) unsigned sBl[16][64];
  for (int x = threadIdx.x; x < 16 * 128; x += TILE_THREADS) {
    const int kp = x / 128, r = x % 128;
    sA[kp][r] = pk(f0 * (float)(1 + (x & 7)), f0 * (float)(2 + (x & 3)));
    sAl[kp][r] = u0 + (unsigned)x * 0x00010001u;
    if (r < 64) {
      sB[kp][r] = pk(fk * (float)(1 + (x & 3)), fk);
      sBl[kp][r] = u0 ^ ((unsigned)x * 0x00030003u);
    }
  }
  __syncthreads();
  const unsigned long long t0 = clock64();
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  u64 pa[4][4], sc2[4][4];
  unsigned e2[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      pa[i][j] = pk(f0, f0 * 0.5f);
      sc2[i][j] = pk(fk * (float)(1 + ((i + j + threadIdx.x) & 3)), fk);
      e2[i][j] = 0x80008000u;
    }
#pragma unroll 4
  for (int it = 0; it < TILE_ITERS; ++it) {
    const int kp = it & 15;
    u64 a2[4], b2[4];
    unsigned la[4], lb[4];
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
      const ulonglong2 va = *reinterpret_cast<const ulonglong2*>(&sA[kp][ty * 4 + i]);
      a2[i] = va.x; a2[i + 1] = va.y;
      const ulonglong2 vb = *reinterpret_cast<const ulonglong2*>(&sB[kp][tx * 2 + i * 16]);
      b2[i] = vb.x; b2[i + 1] = vb.y;
    }
    const uint4 qa = *reinterpret_cast<const uint4*>(&sAl[kp][ty * 4]);
    const uint4 qb = *reinterpret_cast<const uint4*>(&sBl[kp][tx * 4]);
    la[0] = qa.x; la[1] = qa.y; la[2] = qa.z; la[3] = qa.w;
    lb[0] = qb.x; lb[1] = qb.y; lb[2] = qb.z; lb[3] = qb.w;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pa[i][j] = add_rn2(pa[i][j], mul_rz2(mul_rn2(a2[i], b2[j]), sc2[i][j]));
        e2[i][j] = __viaddmax_s16x2(la[i], lb[j], e2[i][j]);
      }
  }
  unsigned acc = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc ^= e2[i][j] ^ (unsigned)pa[i][j] ^ (unsigned)(pa[i][j] >> 32);
  const unsigned long long t1 = clock64();
  if (acc == 0xdeadbeefu) sink[threadIdx.x] = acc;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

int run_tile(int nsm, unsigned long long* d_cyc, unsigned* d_sink, double* rate) {
  probe_tile<<<nsm, TILE_THREADS>>>(d_cyc, d_sink, 1e-41f, 0.99999994f, 3u);   // warm-up
  probe_tile<<<nsm, TILE_THREADS>>>(d_cyc, d_sink, 1e-41f, 0.99999994f, 3u);
  if (cudaDeviceSynchronize() != cudaSuccess) return -4;
  unsigned long long h[1024];
  if (cudaMemcpy(h, d_cyc, nsm * sizeof(unsigned long long), cudaMemcpyDeviceToHost) != cudaSuccess)
    return -4;
  unsigned long long mx = 1;
  for (int i = 0; i < nsm; ++i) mx = h[i] > mx ? h[i] : mx;
  *rate = 32.0 * (double)TILE_THREADS * TILE_ITERS / (double)mx;
  return 0;
}

// operations one iteration of one chain counts for, per mode
double ops_per_chain_iter(int mode) {
  switch (mode) {
    case F2_FMUL_RZ_SUB: case F2_FMUL_RN: case F2_FADD_SUB: return 2.0;
    case F2_FMUL_RZ_VEC: return 2.0;
    case MIX: return 4.0 / NCH;            // four MACs per iteration over all chains
    case MIX_VEC: return 8.0 / NCH;        // eight MACs per iteration over all chains
    default: return 1.0;
  }
}

template <int MODE>
int run_mode(int nsm, unsigned long long* d_cyc, unsigned* d_sink, float f0, float fk, double* rate) {
  probe<MODE><<<nsm, THREADS>>>(d_cyc, d_sink, f0, fk, 3u);   // warm-up
  probe<MODE><<<nsm, THREADS>>>(d_cyc, d_sink, f0, fk, 3u);
  if (cudaDeviceSynchronize() != cudaSuccess) return -4;
  unsigned long long h[1024];
  if (cudaMemcpy(h, d_cyc, nsm * sizeof(unsigned long long), cudaMemcpyDeviceToHost) != cudaSuccess)
    return -4;
  unsigned long long mx = 1;
  for (int i = 0; i < nsm; ++i) mx = h[i] > mx ? h[i] : mx;
  *rate = ops_per_chain_iter(MODE) * (double)THREADS * ITERS * NCH / (double)mx;
  return 0;
}

// Packed against scalar on random pairs: lanes whose bits differ (NaN results
// compare as NaN, whatever their payload), for mul.rn, mul.rz and add.rn.
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

unsigned xorshift32(unsigned& s) {
  s ^= s << 13;
  s ^= s >> 17;
  s ^= s << 5;
  return s;
}

}  // namespace

extern "C" {

int emu_peaks_count(void) { return NUM_MODES; }

const char* emu_peaks_name(int i) { return (i >= 0 && i < NUM_MODES) ? kNames[i] : ""; }

// rates[i]: lane-operations per clock per SM of mode i on the current device
// (emulation_mix_macs: MACs of the GEMM's arithmetic mix per clock per SM).
// Returns 0, or -4 on a CUDA error.  Synchronous; allocates and frees two small
// buffers.
int emu_peaks_measure(double* rates) {
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      nsm <= 0 || nsm > 1024)
    return -4;
  unsigned long long* d_cyc = nullptr;
  unsigned* d_sink = nullptr;
  if (cudaMalloc(&d_cyc, nsm * sizeof(unsigned long long)) != cudaSuccess) return -4;
  if (cudaMalloc(&d_sink, THREADS * sizeof(unsigned)) != cudaSuccess) {
    cudaFree(d_cyc);
    return -4;
  }
  int rc = 0;
  // x * (1 - 2^-24) rounded toward zero stays subnormal for the whole run;
  // 4096 additions of 1e-42 stay below 2^-126
  rc |= run_mode<FMUL_RZ_SUB>(nsm, d_cyc, d_sink, 1e-41f, 0.99999994f, &rates[FMUL_RZ_SUB]);
  rc |= run_mode<FMUL_RN>(nsm, d_cyc, d_sink, 1.0f, 1.0000001f, &rates[FMUL_RN]);
  rc |= run_mode<FADD_SUB>(nsm, d_cyc, d_sink, 1e-42f, 1e-42f, &rates[FADD_SUB]);
  rc |= run_mode<F2_FMUL_RZ_SUB>(nsm, d_cyc, d_sink, 1e-41f, 0.99999994f, &rates[F2_FMUL_RZ_SUB]);
  rc |= run_mode<F2_FMUL_RN>(nsm, d_cyc, d_sink, 1.0f, 1.0000001f, &rates[F2_FMUL_RN]);
  rc |= run_mode<F2_FADD_SUB>(nsm, d_cyc, d_sink, 1e-42f, 1e-42f, &rates[F2_FADD_SUB]);
  rc |= run_mode<DPX_VIADDMAX>(nsm, d_cyc, d_sink, 1.0f, 1.0f, &rates[DPX_VIADDMAX]);
  rc |= run_mode<IMAD>(nsm, d_cyc, d_sink, 1.0f, 1.0f, &rates[IMAD]);
  rc |= run_mode<IADD3>(nsm, d_cyc, d_sink, 1.0f, 1.0f, &rates[IADD3]);
  rc |= run_mode<LOP3>(nsm, d_cyc, d_sink, 1.0f, 1.0f, &rates[LOP3]);
  rc |= run_mode<PRMT>(nsm, d_cyc, d_sink, 1.0f, 1.0f, &rates[PRMT]);
  rc |= run_mode<IMAD_IADD3>(nsm, d_cyc, d_sink, 1.0f, 1.0f, &rates[IMAD_IADD3]);
  rc |= run_mode<MIX>(nsm, d_cyc, d_sink, 1e-41f, 0.99999994f, &rates[MIX]);
  rc |= run_mode<DPX_VEC>(nsm, d_cyc, d_sink, 1.0f, 1.0f, &rates[DPX_VEC]);
  rc |= run_mode<F2_FMUL_RZ_VEC>(nsm, d_cyc, d_sink, 1e-41f, 0.99999994f, &rates[F2_FMUL_RZ_VEC]);
  rc |= run_mode<MIX_VEC>(nsm, d_cyc, d_sink, 1e-41f, 0.99999994f, &rates[MIX_VEC]);
  rc |= run_tile(nsm, d_cyc, d_sink, &rates[MIX_TILE]);
  cudaFree(d_cyc);
  cudaFree(d_sink);
  return rc ? -4 : 0;
}

// bad[0..2]: halves of n random pairs where mul.rn / mul.rz / add.rn .f32x2 differ
// from the scalar instruction (subnormal results included).  Returns 0 or -4.
int emu_peaks_f32x2_agreement(int n, unsigned* bad) {
  if (n <= 0 || !bad) return -1;
  unsigned* hx = new unsigned[2 * (size_t)n];
  unsigned* hy = new unsigned[2 * (size_t)n];
  unsigned s = 12345u;
  for (int i = 0; i < 2 * n; ++i) {
    if (i % 4 == 0) {      // any bit pattern
      hx[i] = xorshift32(s);
      hy[i] = xorshift32(s);
    } else {               // small times mid-range operands: products near and below 2^-126
      hx[i] = (xorshift32(s) & 0x807FFFFFu) | ((xorshift32(s) % 40u) << 23);
      hy[i] = (xorshift32(s) & 0x807FFFFFu) | ((60u + xorshift32(s) % 80u) << 23);
    }
  }
  unsigned *dx = nullptr, *dy = nullptr, *dbad = nullptr;
  int rc = -4;
  if (cudaMalloc(&dx, 8 * (size_t)n) == cudaSuccess && cudaMalloc(&dy, 8 * (size_t)n) == cudaSuccess &&
      cudaMalloc(&dbad, 3 * sizeof(unsigned)) == cudaSuccess &&
      cudaMemcpy(dx, hx, 8 * (size_t)n, cudaMemcpyHostToDevice) == cudaSuccess &&
      cudaMemcpy(dy, hy, 8 * (size_t)n, cudaMemcpyHostToDevice) == cudaSuccess &&
      cudaMemset(dbad, 0, 3 * sizeof(unsigned)) == cudaSuccess) {
    agree<<<(n + 255) / 256, 256>>>(dx, dy, n, dbad);
    if (cudaDeviceSynchronize() == cudaSuccess &&
        cudaMemcpy(bad, dbad, 3 * sizeof(unsigned), cudaMemcpyDeviceToHost) == cudaSuccess)
      rc = 0;
  }
  cudaFree(dx);
  cudaFree(dy);
  cudaFree(dbad);
  delete[] hx;
  delete[] hy;
  return rc;
}

}  // extern "C"
