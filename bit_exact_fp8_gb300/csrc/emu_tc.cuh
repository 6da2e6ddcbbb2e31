// emu_tc.cuh -- 5th-generation tensor cores (tcgen05, sm_100+ "a" targets) as a source
// of exact products, and the per-device self-test that gates their use.
//
// The emulation needs, for every output (m, n) and k, the exact product a'_mk * b'_nk
// of the pre-scaled operand values (at most four significant bits each, in
// [2^-62, 2^-30] and [2^-63, 2^-31]).  A tcgen05.mma of kind::f16 (bf16 operands, fp32
// accumulator, D = A * B with the input D disabled) computes, per output element, a
// sum of 16 products.  Given a B operand in which every column has exactly one
// nonzero k, each element of D is a single product plus zeros: at most eight
// significant bits, inside the fp32 normal range, so no rounding, alignment or
// truncation inside the tensor core can act on it -- provided the unit computes the
// products of bf16 inputs exactly and adds exact zeros without change.  That is what
// the self-test below checks on the device, over every pair of finite codes of the
// two FP8 formats, before anything relies on it.  (Only bf16 inputs are used: the
// FP8 kinds of the MMA are never used.)  An Inf or NaN operand would meet the zeros
// of the expanded B (Inf * 0 = NaN), so blocks holding such codes do not take this
// path.
//
// Operand layout in shared memory: K-major, no swizzle.  Core matrices of 8 rows x 16
// bytes (8 bf16 along K); within one, row r at byte 16 r.  Element (row, k) of a
// rows x 16 tile sits at ((row / 8) * 2 + k / 8) * 128 + (row % 8) * 16 + (k % 8) * 2:
// the two K-adjacent core matrices are 128 bytes apart (the descriptor's leading
// dimension byte offset) and the 8-row groups 256 bytes apart (its stride byte
// offset).
#pragma once
#include <cstdint>

namespace emu {

// shared-memory matrix descriptor (sm_100 format): start address, leading and stride
// byte offsets (all >> 4), version 1, no swizzle
__device__ __forceinline__ uint64_t tc_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major, N and M
__device__ __forceinline__ uint32_t tc_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] = A * B (the accumulator's previous contents ignored)
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, 0, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc)
      : "memory");
}
// the mbarrier completes once the MMAs this thread issued before are done
__device__ __forceinline__ void tc_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
               : "memory");
}
// 32 consecutive columns of this warp's 32 TMEM lanes, one lane per thread
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// the same wait, with the registers of a 16-column load tied to it: their uses cannot
// move above it, while other arithmetic may overlap a load still in flight
__device__ __forceinline__ void tc_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// byte offset of element (row, k) in a K-major, unswizzled rows x 16 bf16 tile
__device__ __forceinline__ uint32_t tc_kmajor_off(int row, int k) {
  return (uint32_t)(((row >> 3) * 2 + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

constexpr int kTcM = 128, kTcN = 256, kTcK = 16;
constexpr int kTcSmem = kTcM * kTcK * 2 + kTcN * kTcK * 2 + 64;   // A, B, barrier and TMEM slot

// The gate.  One CTA of 128 threads per call (fmt 0: E4M3FN, 1: E5M2).  Row m of A
// holds the code m + 128 r (`round` r = 0, 1) at every k, column n of the expanded B
// the code n at k = n % 16 and zeros elsewhere, so output (m, n) is the product of
// those two codes and over the two rounds every pair of codes meets once.  A NaN or
// Inf code is replaced by 1.0.  Each output's bits are compared with the fp32
// product of the two pre-scaled values (a zero product matches either zero: the
// emulation never lets a zero term's sign reach a result); mismatches are counted
// into *bad.  status[0] = 1 if the completion wait gave up.
__global__ void __launch_bounds__(128, 1)
emu_tc_selftest_kernel(int fmt_a, int fmt_b, int round, unsigned* bad, int* status) {
  extern __shared__ __align__(1024) unsigned char tsm[];
  unsigned char* sA = tsm;                             // 128 x 16 bf16
  unsigned char* sB = tsm + kTcM * kTcK * 2;           // 256 x 16 bf16 (the expanded B)
  const uint32_t bar = smem_u32(tsm + kTcM * kTcK * 2 + kTcN * kTcK * 2);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(tsm + kTcM * kTcK * 2 + kTcN * kTcK * 2 + 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t one_a = fmt_a == 1 ? 0x3Cu : 0x38u;
  const uint32_t one_b = fmt_b == 1 ? 0x3Cu : 0x38u;
  auto finite = [](uint32_t code, int fmt) {
    const uint32_t mag = code & 0x7Fu;
    return fmt == 1 ? mag < 0x7Cu : mag != 0x7Fu;
  };
  auto code_a = [&](int m, int) {
    const uint32_t c = (uint32_t)(m + 128 * round) & 255u;
    return finite(c, fmt_a) ? c : one_a;
  };
  auto code_b = [&](int n) {
    const uint32_t c = (uint32_t)n & 255u;
    return finite(c, fmt_b) ? c : one_b;
  };
  auto bf16_of = [](uint32_t entry) { return (uint16_t)(entry >> 16); };   // value bits 31..20
  // A: row m, k -> value of code_a(m, k); B: column n holds its value at k = n % 16 only
  for (int k = 0; k < kTcK; ++k)
    *reinterpret_cast<uint16_t*>(sA + tc_kmajor_off(tid, k)) = bf16_of(lut_entry(code_a(tid, k), fmt_a, kPreA));
  for (int n = tid; n < kTcN; n += 128)
    for (int k = 0; k < kTcK; ++k)
      *reinterpret_cast<uint16_t*>(sB + tc_kmajor_off(n, k)) =
          k == (n & 15) ? bf16_of(lut_entry(code_b(n), fmt_b, kPreB)) : (uint16_t)0;
  fence_proxy_async();                                  // operands visible to the tensor core
  if (tid == 0) {
    mbar_init(bar, 1u);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    tc_alloc(smem_u32(tslot), (uint32_t)kTcN);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    tc_mma_bf16(tmem, tc_smem_desc(smem_u32(sA), 128u, 256u), tc_smem_desc(smem_u32(sB), 128u, 256u),
                tc_idesc_bf16(kTcM, kTcN));
    tc_commit(bar);
  }
  bool done = mbar_wait_bounded(bar, 0u, kWaitPolls);
  if (!done) done = mbar_wait_bounded(bar, 0u, kWaitPolls);    // once more before giving up
  done = __syncthreads_and(done);                       // the TMEM loads below are warp-wide
  tc_fence_after();
  unsigned nbad = 0;
  if (done) {
    const int m = 32 * warp + lane;                      // this thread's TMEM lane = row m
#pragma unroll 1
    for (int c0 = 0; c0 < kTcN; c0 += 32) {
      uint32_t r[32];
      tc_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, r);
      tc_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int n = c0 + i;
        const float va = __uint_as_float(lut_entry(code_a(m, n & 15), fmt_a, kPreA) & 0xFFF00000u);
        const float vb = __uint_as_float(lut_entry(code_b(n), fmt_b, kPreB) & 0xFFF00000u);
        const uint32_t want = __float_as_uint(fmul_rn(va, vb));
        if (r[i] != want && !(((r[i] | want) & 0x7FFFFFFFu) == 0u)) ++nbad;
      }
    }
  } else if (tid == 0) {
    status[0] = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, (uint32_t)kTcN);
  if (nbad) atomicAdd(bad, nbad);
}

}  // namespace emu

namespace emu {

// 16 consecutive columns of this warp's 32 TMEM lanes
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// ---------------------------------------------------------------------------
// The W tile with tensor-core products (fast chains, 32-product blocks, E4M3FN A).
// 128 x 64 outputs per CTA, one CTA per SM, 640 threads:
//   * warps 16-18 decode each K-stage: A into two bf16 tiles of 128 x 16 (K-major,
//     one per 16-k slice), B's values into eight "expanded" 256 x 16 tiles -- tile
//     (s, q) has column n = 16 jl + kk holding b(16 q + jl, 16 s + kk) at k = kk and
//     zeros elsewhere, so the MMA of A slice s with it gives, in TMEM column n of lane
//     m, the single product a(m, 16 s + kk) * b(16 q + jl, 16 s + kk) -- plus the
//     label pairs row by row and every 16-code chunk's label maximum (as in the
//     sparse W kernel).  The zeros are written once; a stage rewrites only the 2048
//     values.
//   * warp 19 allocates all 512 TMEM columns and issues the eight MMAs of a block
//     (kind::f16, bf16 inputs, fp32 accumulator, 128 x 256 x 16) into two 256-column
//     buffers in turn, each as soon as the consumers have read the buffer's previous
//     group; tcgen05.commit completes the buffer's TFULL barrier.
//   * warps 0-15 hold one TMEM lane (row) and 16 outputs each (columns 16 q + 4 w' +
//     t, w' = warp / 4, t < 4); per block they take E as in the sparse W kernel, then
//     read each group's products with tcgen05.ld (one output's 16 k per load) and run
//     the truncating multiply and the add: two packed FP32 instructions per output
//     and k-pair instead of three, and no shared-memory operand loads.
// An E4M3FN A has no Inf; a NaN code in A meets the expanded zeros and turns every
// product of its row and slice into NaN, where the emulated result is NaN anyway; an
// Inf or NaN in B meets only its own product.  So the products are right for every
// input.  Every wait is bounded; warp 19 releases the TMEM after the consumers'
// last read (or after a wait gave up) before it exits.
template <int LREP_>
struct WtShape {
  using TS = TileShape<4, 4, 32, 16, 32, 1, LREP_>;
  static constexpr int BM = 128, BN = 64, BK = 32;
  static constexpr int NC = 512, NP = 128, NDEC = 96, NTH = NC + NP;
  static constexpr int OUT = BM * BN;
  static constexpr int KPR = BK / 2, LROW = KPR + 4;
  static constexpr int A_TILE = BM * 16 * 2;                        // one 16-k slice
  static constexpr int B_TILE = 256 * 16 * 2;
  static constexpr int A_OFF = TS::NS * TS::RAW_STAGE;              // 2 stages x 2 slices
  static constexpr int B_OFF = A_OFF + 2 * 2 * A_TILE;              // 8 expanded tiles
  static constexpr int LBUF = ((BM + BN) * LROW + 2 * (BM + BN)) * 4;   // label rows, chunk maxima
  static constexpr int L_OFF = B_OFF + 8 * B_TILE;
  static constexpr int LUT_OFF = L_OFF + 2 * LBUF;
  static constexpr int BAR_OFF = LUT_OFF + 2 * 256 * LREP_ * 4;
  // barriers: raw ring, FULL[2], EMPTY[2], TFULL[2], TEMPTY[2], BDONE, DONE; TMEM slot
  static constexpr int NBAR = TS::NS + 10;
  static constexpr int LIST_OFF = (BAR_OFF + NBAR * 8 + 8 + 127) / 128 * 128;
  static constexpr int LIST_BYTES = 32 * 16 * 2;
  static constexpr int RES_OFF = LIST_OFF + (NC / 32) * LIST_BYTES;
  static constexpr int CST_OFF = RES_OFF + (NC / 32) * LIST_BYTES;
  static constexpr int SMEM_BYTES = CST_OFF + OUT * 4 + TS::RAW_ALIGN;
  static_assert(TS::BM == BM && TS::BN == BN && TS::BK == BK && TS::SWZ, "the W geometry");
  static_assert(A_OFF % 1024 == 0 && L_OFF % 16 == 0 && (LBUF % 16) == 0, "aligned regions");
};

template <int LREP>
__global__ void __launch_bounds__(WtShape<LREP>::NTH, 1)
emu_wst_kernel(const GemmParams p, const __grid_constant__ CUtensorMap tmA,
               const __grid_constant__ CUtensorMap tmB) {
  using WS = WtShape<LREP>;
  using TS = typename WS::TS;
  constexpr int BM = WS::BM, BN = WS::BN, BK = WS::BK, NS = TS::NS;
  constexpr int NC = WS::NC, LROW = WS::LROW, NDEC = WS::NDEC;
  constexpr int A_CHUNKS = BM * BK / 16, B_CHUNKS = BN * BK / 16;
  constexpr int PER_DEC = (A_CHUNKS + B_CHUNKS) / NDEC;
  static_assert((A_CHUNKS + B_CHUNKS) % NDEC == 0, "whole chunk rounds");

  extern __shared__ __align__(128) unsigned char smem_dyn[];
  unsigned char* const smem =
      smem_dyn + ((TS::RAW_ALIGN - (smem_u32(smem_dyn) & (TS::RAW_ALIGN - 1))) & (TS::RAW_ALIGN - 1));
  uint32_t* lutA = reinterpret_cast<uint32_t*>(smem + WS::LUT_OFF);
  uint32_t* lutB = lutA + 256 * LREP;
  const uint32_t bar0 = smem_u32(smem + WS::BAR_OFF);
  const uint32_t full0 = bar0 + 8u * NS, empty0 = full0 + 16u, tfull0 = empty0 + 16u;
  const uint32_t tempty0 = tfull0 + 16u, bdone = tempty0 + 16u, done_bar = bdone + 8u;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + WS::BAR_OFF + WS::NBAR * 8);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t m0 = ((int64_t)blockIdx.y + p.m_tile0) * BM;
  const int64_t n0 = (int64_t)blockIdx.x * BN;
  const int s = blockIdx.z;
  fill_luts<LREP, WS::NTH>(lutA, reinterpret_cast<uint32_t*>(smem), p.fmt_a, p.fmt_b, tid);

  const int K = (int)p.K;
  const int kt = p.S == 1 ? BK : p.ktile;
  const int T = (K + kt - 1) / kt;
  int t_begin, t_end, t_stride;
  if (p.S == 1) { t_begin = 0; t_end = T; t_stride = 1; }
  else if (p.scheme == 0) {
    const int q = (T + p.S - 1) / p.S;
    t_begin = s * q; t_end = t_begin + q < T ? t_begin + q : T; t_stride = 1;
  } else { t_begin = s; t_end = T; t_stride = p.S; }
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + t_stride - 1) / t_stride : 0;
  const int spt = kt / BK;
  int n_stages = n_tiles * spt;
  if (n_tiles > 0) {
    const int t_last = t_begin + (n_tiles - 1) * t_stride;
    const int len_last = K - t_last * kt < kt ? K - t_last * kt : kt;
    n_stages -= spt - (len_last + BK - 1) / BK;
  }

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(bar0 + 8u * i, 1u);
    for (int i = 0; i < 2; ++i) {
      mbar_init(full0 + 8u * i, WS::NDEC / 32);   // one arrival per decoder warp
      mbar_init(empty0 + 8u * i, NC / 32);        // one per consumer warp
      mbar_init(tfull0 + 8u * i, 1u);             // the MMA commit
      mbar_init(tempty0 + 8u * i, NC / 32);
    }
    mbar_init(bdone, 1u);                         // a block's MMAs done (commit)
    mbar_init(done_bar, NC / 32);                 // the consumers' last TMEM read done
    fence_mbar_init();
  }
  // the expanded tiles' fixed zeros (the MMAs read them through the async proxy)
  for (int i = tid; i < 8 * WS::B_TILE / 16; i += WS::NTH)
    reinterpret_cast<uint4*>(smem + WS::B_OFF)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async();
  if (warp == 19) {
    tc_alloc(smem_u32(tslot), 512u);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();                                // tables, barriers, zeros, TMEM ready
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp >= 16 && warp < 19) {
    // ---- decoders
    const int pt = tid - NC;
    auto stage_k = [&](int st) -> int {
      if (spt == 1) return (t_begin + st * t_stride) * kt;
      return (t_begin + (st / spt) * t_stride) * kt + (st % spt) * BK;
    };
    int issued = 0;
    auto issue = [&](int st) {
      issued = st + 1;
      const int slot = st % NS;
      const uint32_t bar = bar0 + 8u * slot;
      const uint32_t dst = smem_u32(smem + slot * TS::RAW_STAGE);
      const int k = stage_k(st);
      mbar_arrive_expect_tx(bar, (uint32_t)(TS::RAW_A + TS::RAW_B));
      tma_load_2d(dst, &tmA, k, (int)m0, bar);
      tma_load_2d(dst + TS::RAW_A, &tmB, k, (int)n0, bar);
    };
    auto raw_wait = [&](int st) {
      return mbar_wait_bounded(bar0 + 8u * (uint32_t)(st % NS), (uint32_t)((st / NS) & 1), kWaitPolls);
    };
    if (pt == 0) {
      fence_proxy_async();
      for (int st = 0; st < NS && st < n_stages; ++st) issue(st);
    }
    const uint32_t* lA = lutA + lane % LREP;
    const uint32_t* lB = lutB + lane % LREP;
    for (int st = 0; st < n_stages; ++st) {
      const int sb = st & 1;
      // the raw stage has landed; the consumers are done with stage st - 2 (this
      // buffer's labels); the MMAs of block st - 1 are done (the expanded tiles)
      bool ok = raw_wait(st);
      if (st >= 2)
        ok = mbar_wait_bounded(empty0 + 8u * (uint32_t)sb, (uint32_t)(((st - 2) >> 1) & 1), kWaitPolls) && ok;
      if (st >= 1) ok = mbar_wait_bounded(bdone, (uint32_t)((st - 1) & 1), kWaitPolls) && ok;
      if (ok) {
        const unsigned char* raw = smem + (st % NS) * TS::RAW_STAGE;
        const uint32_t raw_u32 = smem_u32(raw);
        unsigned char* aT = smem + WS::A_OFF + sb * 2 * WS::A_TILE;
        unsigned char* bT = smem + WS::B_OFF;
        uint32_t* sL = reinterpret_cast<uint32_t*>(smem + WS::L_OFF + sb * WS::LBUF);
        int* sMx = reinterpret_cast<int*>(sL + (BM + BN) * LROW);
#pragma unroll 1
        for (int r = 0; r < PER_DEC; ++r) {
          const int c = pt + r * NDEC;
          const bool isA = c < A_CHUNKS;
          const int cb = isA ? c : c - A_CHUNKS;
          const int rows = isA ? BM : BN;
          const int row = cb % rows, h = cb / rows;
          const int off_row = isA ? row * BK : TS::RAW_A + row * BK;
          const int hs = h ^ (int)(((raw_u32 + (uint32_t)off_row) >> 7) & 1u);
          const uint4 q4 = *reinterpret_cast<const uint4*>(raw + off_row + hs * 16);
          const uint32_t w[4] = {q4.x, q4.y, q4.z, q4.w};
          const uint32_t* lt = isA ? lA : lB;
          uint32_t e[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) e[j] = lt[__byte_perm(w[j >> 2], 0u, 0x4440u | (j & 3)) * LREP];
          uint32_t lp[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) lp[i] = __byte_perm(e[2 * i], e[2 * i + 1], 0x5410);
          const int lr = isA ? row : BM + row;
          uint32_t* lrow = sL + lr * LROW + h * 8;
          *reinterpret_cast<uint4*>(lrow) = make_uint4(lp[0], lp[1], lp[2], lp[3]);
          *reinterpret_cast<uint4*>(lrow + 4) = make_uint4(lp[4], lp[5], lp[6], lp[7]);
          uint32_t mx = __vmaxs2(__vmaxs2(__vmaxs2(lp[0], lp[1]), __vmaxs2(lp[2], lp[3])),
                                 __vmaxs2(__vmaxs2(lp[4], lp[5]), __vmaxs2(lp[6], lp[7])));
          mx = __vmaxs2(mx, __byte_perm(mx, 0u, 0x1032));
          sMx[h * (BM + BN) + lr] = (int)mx >> 16;
          if (isA) {            // two 8-code rows of the slice's core matrices
            unsigned char* at = aT + h * WS::A_TILE;
            *reinterpret_cast<uint4*>(at + tc_kmajor_off(row, 0)) =
                make_uint4(__byte_perm(e[0], e[1], 0x7632), __byte_perm(e[2], e[3], 0x7632),
                           __byte_perm(e[4], e[5], 0x7632), __byte_perm(e[6], e[7], 0x7632));
            *reinterpret_cast<uint4*>(at + tc_kmajor_off(row, 8)) =
                make_uint4(__byte_perm(e[8], e[9], 0x7632), __byte_perm(e[10], e[11], 0x7632),
                           __byte_perm(e[12], e[13], 0x7632), __byte_perm(e[14], e[15], 0x7632));
          } else {              // column row = 16 q + jl: tile (h, q), column 16 jl + kk at k = kk
            unsigned char* bt = bT + (h * 4 + row / 16) * WS::B_TILE;
            const int jl = row % 16;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              *reinterpret_cast<uint16_t*>(bt + tc_kmajor_off(16 * jl + kk, kk)) = (uint16_t)(e[kk] >> 16);
          }
        }
      }
      fence_proxy_async();                       // the tiles, for the tensor core
      if (named_sync_or(1, WS::NP, !ok)) {       // decoded (with warp 19), or someone gave up
        atomicExch(&g_emu_device_status, kStatusWaitTimeout);
        if (pt == 0)
          for (int x = st; x < issued; ++x) (void)raw_wait(x);
        return;
      }
      if (pt == 0 && st + NS < n_stages) {
        fence_proxy_async();
        issue(st + NS);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(full0 + 8u * (uint32_t)sb);
    }
    return;
  }

  if (warp == 19) {
    // ---- the MMA issuer; it also owns the TMEM
    const uint32_t idesc = tc_idesc_bf16(128, 256);
    bool err = false;
    int groups = 0;
    for (int st = 0; st < n_stages; ++st) {
      if (named_sync_or(1, WS::NP, err)) { err = true; break; }     // stage st decoded
      tc_fence_after();
      const uint32_t aT = smem_u32(smem + WS::A_OFF + (st & 1) * 2 * WS::A_TILE);
      const uint32_t bT = smem_u32(smem + WS::B_OFF);
#pragma unroll 1
      for (int g = 0; g < 8 && !err; ++g) {
        const int gg = 8 * st + g, buf = gg & 1;
        if (gg >= 2) {        // the consumers have read this buffer's previous group
          const bool ok = mbar_wait_bounded(tempty0 + 8u * (uint32_t)buf, (uint32_t)(((gg - 2) >> 1) & 1),
                                            kWaitPolls);
          if (!__all_sync(0xFFFFFFFFu, ok)) { err = true; break; }
        }
        tc_fence_after();
        if (lane == 0) {
          // group g: quarter g / 2 of the outputs' columns, k-slice g % 2
          const int sl = g & 1, qt = g >> 1;
          tc_mma_bf16(tmem + (uint32_t)(buf * 256), tc_smem_desc(aT + (uint32_t)(sl * WS::A_TILE), 128u, 256u),
                      tc_smem_desc(bT + (uint32_t)((4 * sl + qt) * WS::B_TILE), 128u, 256u), idesc);
          tc_commit(tfull0 + 8u * (uint32_t)buf);
          if (g == 7) tc_commit(bdone);
        }
        __syncwarp();
        groups = gg + 1;
      }
    }
    if (err) atomicExch(&g_emu_device_status, kStatusWaitTimeout);
    // the TMEM goes back once the MMAs issued are done and the consumers have read
    if (groups > 0)
      (void)mbar_wait_bounded(tfull0 + 8u * (uint32_t)((groups - 1) & 1), (uint32_t)(((groups - 1) >> 1) & 1),
                              kWaitPolls);
    (void)mbar_wait_bounded(done_bar, 0u, kWaitPolls);
    tc_fence_after();
    tc_dealloc(tmem, 512u);
    return;
  }

  // ---- consumers: warp w holds TMEM lanes 32 (w % 4) .. (the rows) and the columns
  // 16 q + 4 (w / 4) + t, q, t < 4 (output o = 4 q + t)
  const int sub = warp & 3, wq = warp >> 2;
  const int ml = 32 * sub + lane;
  float4* const cst = reinterpret_cast<float4*>(smem + WS::CST_OFF) + tid;   // quarter q: + q * NC
  uint16_t* const list = reinterpret_cast<uint16_t*>(smem + WS::LIST_OFF + warp * WS::LIST_BYTES);
  uint16_t* const ep_res = reinterpret_cast<uint16_t*>(smem + WS::RES_OFF + warp * WS::LIST_BYTES);
  const uint32_t tlane = tmem + ((uint32_t)(32 * sub) << 16);
#pragma unroll
  for (int q = 0; q < 4; ++q) cst[q * NC] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  bool failed = false;
  for (int st = 0; st < n_stages && !failed; ++st) {
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(full0 + 8u * (uint32_t)(st & 1), (uint32_t)((st >> 1) & 1),
                                                    kWaitPolls))) {
      failed = true;
      break;
    }
    const uint32_t* sL = reinterpret_cast<const uint32_t*>(smem + WS::L_OFF + (st & 1) * WS::LBUF);
    const int* sMx = reinterpret_cast<const int*>(sL + (BM + BN) * LROW);
    float cv[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 c4 = cst[q * NC];
      cv[4 * q] = c4.x; cv[4 * q + 1] = c4.y; cv[4 * q + 2] = c4.z; cv[4 * q + 3] = c4.w;
    }
    // the bound U = row maximum + column maximum of the block's labels against e(c),
    // two outputs per word in 16-bit halves
    const int ra = max(sMx[ml], sMx[(BM + BN) + ml]);
    const uint32_t rap = __byte_perm((uint32_t)ra, 0u, 0x1010);
    uint32_t need = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int4 x0 = *reinterpret_cast<const int4*>(sMx + BM + 16 * q + 4 * wq);
      const int4 x1 = *reinterpret_cast<const int4*>(sMx + (BM + BN) + BM + 16 * q + 4 * wq);
      const int rb[4] = {max(x0.x, x1.x), max(x0.y, x1.y), max(x0.z, x1.z), max(x0.w, x1.w)};
#pragma unroll
      for (int tp = 0; tp < 2; ++tp) {
        const int o = 4 * q + 2 * tp;
        const uint32_t c16 = __byte_perm(__float_as_uint(cv[o]), __float_as_uint(cv[o + 1]), 0x7632) & 0x7F807F80u;
        const uint32_t rbp = __byte_perm((uint32_t)rb[2 * tp], (uint32_t)rb[2 * tp + 1], 0x5410);
        const uint32_t gt = __vcmpgts2(__vadd2(rap, rbp), c16);
        need |= ((gt & 1u) | ((gt >> 15) & 2u)) << o;
      }
    }
    // the warp's list of outputs that need E_p; one listed output per lane and round
    const int cnt = __popc(need);
    int before = 0, total = 0;
#pragma unroll
    for (int bit = 0; bit < 5; ++bit) {
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, (cnt >> bit) & 1);
      before += __popc(bal & ((1u << lane) - 1u)) << bit;
      total += __popc(bal) << bit;
    }
    uint4* const own = reinterpret_cast<uint4*>(ep_res + lane * 16);
    own[0] = make_uint4(0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u);
    own[1] = own[0];
    for (uint32_t m = need; m; m &= m - 1) list[before++] = (uint16_t)(lane * 16 + __ffs(m) - 1);
    __syncwarp();
    for (int it = lane; it < total; it += 32) {
      const int item = list[it], o = item & 15;
      const uint32_t* la = sL + (32 * sub + (item >> 4)) * LROW;
      const uint32_t* lb = sL + (BM + 16 * (o >> 2) + 4 * wq + (o & 3)) * LROW;
      uint32_t e[4] = {0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u};
#pragma unroll
      for (int k = 0; k < WS::KPR; k += 4) {
        const uint4 a4 = *reinterpret_cast<const uint4*>(la + k);
        const uint4 b4 = *reinterpret_cast<const uint4*>(lb + k);
        e[0] = __viaddmax_s16x2(a4.x, b4.x, e[0]);
        e[1] = __viaddmax_s16x2(a4.y, b4.y, e[1]);
        e[2] = __viaddmax_s16x2(a4.z, b4.z, e[2]);
        e[3] = __viaddmax_s16x2(a4.w, b4.w, e[3]);
      }
      uint32_t x = __vmaxs2(__vmaxs2(e[0], e[1]), __vmaxs2(e[2], e[3]));
      x = __vmaxs2(x, __byte_perm(x, 0u, 0x1032));
      ep_res[item] = (uint16_t)(x >> 16);
    }
    __syncwarp();
    // per quarter q of this thread's outputs (o = 4 q + t): scales from E = max(E_p, e(c))
    // clamped, then the two groups (k-slices) of the quarter's products from the tensor
    // cores, then the normalisation: four accumulators live at a time
#pragma unroll
    for (int q = 0; q < 4 && !failed; ++q) {
      const float4 c4 = cst[q * NC];
      const float cv4[4] = {c4.x, c4.y, c4.z, c4.w};
      const uint2 rq = *reinterpret_cast<const uint2*>(ep_res + lane * 16 + 4 * q);
      const uint32_t rw2[2] = {rq.x, rq.y};
      uint32_t scb[4];
      f32x2_t pa[4];
#pragma unroll
      for (int tp = 0; tp < 2; ++tp) {
        const uint32_t c16 = __byte_perm(__float_as_uint(cv4[2 * tp]), __float_as_uint(cv4[2 * tp + 1]), 0x7632) &
                             0x7F807F80u;
        const uint32_t e16 = __vmins2(__vmaxs2(rw2[tp], c16), 0x3A803A80u);
        scb[2 * tp] = kScaleBase - (e16 << 16);
        scb[2 * tp + 1] = kScaleBase - (e16 & 0xFFFF0000u);
        pa[2 * tp] = pack2(fmul_rz(cv4[2 * tp], __uint_as_float(scb[2 * tp])), 0.0f);
        pa[2 * tp + 1] = pack2(fmul_rz(cv4[2 * tp + 1], __uint_as_float(scb[2 * tp + 1])), 0.0f);
      }
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
        const int gg = 8 * st + 2 * q + sl, buf = gg & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(tfull0 + 8u * (uint32_t)buf, (uint32_t)((gg >> 1) & 1),
                                                        kWaitPolls))) {
          failed = true;
          break;
        }
        tc_fence_after();
        // one load per output (its 16 k), the next output's load in flight while this
        // one's products are truncated and added (two chains per output)
        const uint32_t tcol = tlane + (uint32_t)(buf * 256 + 4 * wq * 16);
        uint32_t r0[16], r1[16];
        tc_ld16(tcol, r0);
        tc_wait_ld16(r0);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          uint32_t(&cur)[16] = (t & 1) ? r1 : r0;
          uint32_t(&nxt)[16] = (t & 1) ? r0 : r1;
          if (t < 3) tc_ld16(tcol + (uint32_t)(16 * (t + 1)), nxt);
          const float scf = __uint_as_float(scb[t]);
          const f32x2_t s2 = pack2(scf, scf);
          f32x2_t pb = pack2(0.0f, 0.0f);
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            pa[t] = fadd2_rn(pa[t], fmul2_rz(pack2(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), s2));
            pb = fadd2_rn(pb, fmul2_rz(pack2(__uint_as_float(cur[2 * i + 2]), __uint_as_float(cur[2 * i + 3])), s2));
          }
          pa[t] = fadd2_rn(pa[t], pb);
          if (t < 3) tc_wait_ld16(nxt);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8u * (uint32_t)buf);
      }
      if (failed) break;
      // normalise: c' = S * 2^(E-13) * 2^-93, truncated to 14 significant bits
      float cn[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float inv = __uint_as_float(kInvBase - scb[t]);
        cn[t] = __uint_as_float(__float_as_uint(fmul_rn(sum_halves(pa[t]), inv)) & kKeep14);
      }
      cst[q * NC] = make_float4(cn[0], cn[1], cn[2], cn[3]);
    }
    if (failed) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8u * (uint32_t)(st & 1));
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(done_bar);
  if (failed) {
    atomicExch(&g_emu_device_status, kStatusWaitTimeout);
    return;
  }

  float res[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 c4 = cst[q * NC];
    res[4 * q] = fmul_rn(c4.x, kTwo93);
    res[4 * q + 1] = fmul_rn(c4.y, kTwo93);
    res[4 * q + 2] = fmul_rn(c4.z, kTwo93);
    res[4 * q + 3] = fmul_rn(c4.w, kTwo93);
  }
  const int64_t m = m0 + ml;
  if (m >= p.M) return;
  if (p.S > 1) {
    float* dst = p.partial + (int64_t)s * p.M * p.N + m * p.N;
#pragma unroll
    for (int o = 0; o < 16; ++o) {
      const int64_t n = n0 + 16 * (o >> 2) + 4 * wq + (o & 3);
      if (n < p.N) dst[n] = res[o];
    }
    return;
  }
  const float alpha = fmul_rn(__ldg(p.scale_a), __ldg(p.scale_b));
  const OutStore store(p);
#pragma unroll
  for (int o = 0; o < 16; ++o) {
    const int64_t n = n0 + 16 * (o >> 2) + 4 * wq + (o & 3);
    if (n < p.N) store(p, m * p.N + n, fma_plus0(res[o], alpha));
  }
}

}  // namespace emu
