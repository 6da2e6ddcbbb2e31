/*
 * emu_fp8.h -- C ABI of libemufp8, the GB300 (sm_103a) emulated FP8 scaled GEMM.
 *
 * The library computes out = (A @ B) * scale_a * scale_b for FP8 operands bit for
 * bit as a reference tensor-core platform computes torch._scaled_mm ("User guide",
 * section 1 "What mmaemu does, in one paragraph", and section 3 "A first GEMM",
 * of the mmaemu v0.1 documentation):
 *
 *   - each operand code is decoded to an exact significand and exponent; a
 *     subnormal keeps the exponent emin ("Validation evidence", table "Claims and
 *     their recordings", first row);
 *   - the exact products of a K-block of the preset's width, with the incoming
 *     fp32 accumulator c, are aligned to the block's largest exponent (zero
 *     products left out), each term truncated toward zero to F fraction bits, and
 *     the block sum truncated to F+1 significant bits; a zero result is +0
 *     (same table, rows 1-2; table "Scope", rows "Ada instruction model" and
 *     "Hopper preset"; the H100 PCIe probe table, first row);
 *   - fast accumulation chains the blocks over K; slow accumulation restarts the
 *     chain every R elements and adds the chunk results in K order in fp32
 *     (H100 PCIe probe table, second row; "Scope", row "Slow accumulation");
 *   - an explicit split-K factor S cuts K into contiguous runs of k-tiles
 *     (hopper) or deals k-tiles round-robin (ada); the partials are added in fp32,
 *     serially, or pairwise for ada ("Claims and their recordings", split rows;
 *     H100 PCIe probe table, split row);
 *   - the epilogue is alpha = RN32(scale_a * scale_b), y = fma(acc, alpha, +0),
 *     bf16/fp16 rounded from y; a NaN code in row m of A or column n of B makes
 *     output (m, n) the canonical NaN ("Limitations of mmaemu v0.1", section
 *     "Corrections of earlier statements").
 *
 * Every entry point is host-callable and asynchronous: arguments are checked on
 * the host before any launch, and then every kernel is enqueued on the caller's
 * stream.  No entry point synchronises with the device or allocates memory.
 */
#ifndef EMU_FP8_H
#define EMU_FP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  0 is success; every error is negative and leaves nothing enqueued
   (EMU_ECUDA: a launch failed; kernels before it may have been enqueued). */
#define EMU_OK 0
#define EMU_EINVAL (-1)        /* null pointer, bad enum, negative size, workspace too small */
#define EMU_EREJECT (-2)       /* a call torch 2.7.1 / cuBLAS rejects ("Limitations of mmaemu
                                  v0.1", table "Features outside v0.1": e5m2 x e5m2, K or N not a
                                  multiple of 16, storage not 16-byte aligned)                  */
#define EMU_EUNSUPPORTED (-3)  /* outside the modelled scope: scale_result with a non-FP8
                                  output, split_S above 64, a preset the kernels do not
                                  implement (bias and row-wise scales have no argument here:
                                  the Python layer raises for them)                            */
#define EMU_ECUDA (-4)         /* a CUDA launch error (cudaGetLastError)                        */

/* FP8 operand formats (OCP): E4M3FN (bias 7, no Inf, S.1111.111 = NaN) and E5M2
   (bias 15, exponent 31 = Inf/NaN). */
typedef enum { EMU_E4M3FN = 0, EMU_E5M2 = 1 } emu_fp8_t;

/* Output dtypes: fp32 (the epilogue's y), bf16 or fp16 rounded to nearest even from y,
   or FP8 (E4M3FN, E5M2): y times scale_result (a separate fp32 multiply, when given)
   rounded to nearest even and saturated to the format's largest finite value; NaN is
   0x7F ("Validation evidence", table "Claims and their recordings", fp8-output row). */
typedef enum {
  EMU_OUT_F32 = 0, EMU_OUT_BF16 = 1, EMU_OUT_F16 = 2, EMU_OUT_E4M3FN = 3, EMU_OUT_E5M2 = 4
} emu_out_t;

/* Instruction/platform preset ("Validation evidence", H100 PCIe probe table and
   "Claims and their recordings").  The kernels implement block_width 16 or 32,
   frac_bits 13, restart a multiple of 32 (of block_width for 16), c_in_alignment 1,
   ktile 64 or 128; other values return EMU_EUNSUPPORTED. */
typedef struct {
  int32_t block_width;     /* B: products per block: 32 (hopper), 16 (ada)              */
  int32_t frac_bits;       /* F: retained fraction bits: 13                             */
  int32_t restart;         /* R: slow-accumulation chunk length: 128                    */
  int32_t c_in_alignment;  /* 1: the accumulator takes part in the block's alignment    */
  int32_t split_scheme;    /* 0: contiguous runs of k-tiles (hopper), 1: round-robin    */
  int32_t ktile;           /* k-tile width of the split rule: 128 (hopper), 64 (ada)    */
  int32_t combine;         /* 0: serial p0 + p1 + ...; 1: pairwise tree (ada)           */
} emu_preset_t;

/* Fill *out with a named preset: "hopper" (H100 PCIe) or "ada" (RTX 4060).
   Returns EMU_OK, or EMU_EINVAL for a null pointer or an unknown name. */
int emu_preset_get(const char* name, emu_preset_t* out);

/* Bytes of device workspace emu_scaled_mm needs for these sizes: S * M * N * 4
   rounded up to 256 for split_S > 1 (the fp32 split partials), 0 for split_S == 1
   or an empty output.  Returns 0 for invalid sizes, and SIZE_MAX when the product
   does not fit in size_t (no workspace can then be large enough). */
size_t emu_workspace_bytes(int64_t M, int64_t N, int32_t split_S);

/*
 * out[M,N] = emulated (A @ B) * scale_a * scale_b.
 *
 *   A          device, [M,K] row-major FP8 codes (lda = K), format fmt_a
 *   B          device, [K,N] column-major FP8 codes: B[k,n] at byte n*K + k (the w.t()
 *              of a row-major [N,K] weight), format fmt_b
 *   scale_a/b  device pointers to one fp32 each (tensor-wise scales; they multiply)
 *   out        device, [M,N] row-major, element type out_dtype
 *   fast_accum 1: fast accumulation (one chain per split); 0: slow (restart every R)
 *   split_S    >= 1: explicit split-K factor; the partials go through the workspace
 *   preset     host pointer, see emu_preset_t
 *   workspace  device scratch of at least emu_workspace_bytes(M, N, split_S) bytes
 *              (may be NULL when that is 0); its contents on entry do not matter
 *   stream     a cudaStream_t (NULL: the legacy default stream)
 *
 * Ownership: all buffers belong to the caller; the call keeps no pointer after it
 * returns.  Alignment: A, B and out must be 16-byte aligned (EMU_EREJECT otherwise).
 * Sizes: M, N, K >= 0, K and N multiples of 16 (EMU_EREJECT otherwise), K < 2^31.
 * M == 0 or N == 0 enqueues nothing; K == 0 gives +0 outputs (NaN if alpha is NaN).
 * E5M2 x E5M2 is rejected (EMU_EREJECT).  E5M2 Inf codes follow IEEE on the
 * products (Inf*0 -> NaN, +Inf and -Inf -> NaN, otherwise +-Inf).
 * Results do not depend on the previous contents of out or of the workspace.
 * The call may be captured in a CUDA graph (stream capture): its launches, with
 * the operand tensor maps encoded at capture, replay on whatever the same buffers
 * hold then, so the buffers must stay where they were at capture.
 */
int emu_scaled_mm(const uint8_t* A, emu_fp8_t fmt_a,
                  const uint8_t* B, emu_fp8_t fmt_b,
                  int64_t M, int64_t N, int64_t K,
                  const float* scale_a, const float* scale_b,
                  void* out, emu_out_t out_dtype,
                  int32_t fast_accum, int32_t split_S,
                  const emu_preset_t* preset,
                  void* workspace, size_t workspace_bytes,
                  void* stream);

/*
 * emu_scaled_mm with torch._scaled_mm's scale_result: a device pointer to one fp32
 * that multiplies y, as a separate fp32 multiply, before the FP8 output conversion
 * ("Validation evidence", table "Claims and their recordings": "scale_result is a
 * separate fp32 multiply before saturation to the format's maximum").  NULL means
 * none; a non-NULL scale_result with a non-FP8 output returns EMU_EUNSUPPORTED, and
 * e4m3 x e4m3 -> e5m2 returns EMU_EREJECT (cuBLASLt refuses it).  emu_scaled_mm is
 * this call with scale_result = NULL.
 */
int emu_scaled_mm_ex(const uint8_t* A, emu_fp8_t fmt_a,
                     const uint8_t* B, emu_fp8_t fmt_b,
                     int64_t M, int64_t N, int64_t K,
                     const float* scale_a, const float* scale_b,
                     const float* scale_result,
                     void* out, emu_out_t out_dtype,
                     int32_t fast_accum, int32_t split_S,
                     const emu_preset_t* preset,
                     void* workspace, size_t workspace_bytes,
                     void* stream);

/*
 * emu_scaled_mm_noalloc: emu_scaled_mm for callers that cannot allocate device
 * memory. (This entry point is an addition of this library; the documentation
 * pages have no counterpart.)
 *
 * emu_scaled_mm itself allocates nothing, but with split_S > 1 it needs a
 * caller-owned workspace for the fp32 split partials.  Some callers have no way
 * to get one: a plugin or custom-op interface that hands the library only the
 * input and output buffers, code whose memory is fixed at start-up and that must
 * not call cudaMalloc (or a caching allocator) later, or a host framework that
 * owns every allocation on the device.  This entry point keeps the partials in a
 * file-scope static device array of EMU_NOALLOC_SCRATCH_BYTES bytes instead, so
 * the caller passes only inputs and outputs.  It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *
 * Arguments, layouts, ownership and status codes are those of emu_scaled_mm,
 * without the workspace.  Limit: split_S * M * N * 4 bytes (rounded up to 256)
 * must fit in EMU_NOALLOC_SCRATCH_BYTES (4 MiB: split_S * M * N <= 1,048,576);
 * larger calls return EMU_EUNSUPPORTED before any launch.
 *
 * The array exists once per GPU that loads the library and is held until the
 * process exits.  The first call on a device, with that device current, looks up
 * the array's device address (cudaGetSymbolAddress) and caches it: make that first
 * call before any CUDA stream capture.  Every call on a device shares the one
 * array and leaves its partials there; each call writes every partial before it
 * reads it, so nothing needs clearing.  Calls whose kernels overlap on the GPU
 * (on different streams, or from different host threads, without ordering
 * between them) race on the array and may return wrong results: order them on
 * one stream or serialise them.
 */
#define EMU_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

int emu_scaled_mm_noalloc(const uint8_t* A, emu_fp8_t fmt_a,
                          const uint8_t* B, emu_fp8_t fmt_b,
                          int64_t M, int64_t N, int64_t K,
                          const float* scale_a, const float* scale_b,
                          void* out, emu_out_t out_dtype,
                          int32_t fast_accum, int32_t split_S,
                          const emu_preset_t* preset,
                          void* stream);

/*
 * emu_scaled_mm_host: the same GEMM with the operands and the result in HOST memory,
 * the copies overlapped with the compute.  (An addition of this library; the pages
 * have no counterpart: they describe the arithmetic, not the data movement.)
 *
 * N is cut into `chunks` column slabs (widths multiples of 16; chunks <= 0 picks
 * one slab per 64 MiB of B; never more than 16 slabs, nor more than N / 16).  One stream copies the scales, A and then B
 * slab by slab into the device staging buffer; each slab's GEMM starts on one of
 * four compute streams as soon as its B slab has landed, so slab c + 1 uploads
 * while slab c computes; a third stream copies each finished slab of the result
 * back into its columns of out_host (a strided 2-D copy).  Every output depends
 * only on its row of A and column of B, so the bits equal those of one
 * emu_scaled_mm_ex call on the whole problem.
 *
 *   A_host, B_host  host, layouts as in emu_scaled_mm (B: [N,K] bytes, n-major)
 *   scale_a/b       the fp32 scales by value
 *   scale_result    host pointer to one fp32 (FP8 outputs), or NULL
 *   out_host        host, [M,N] row-major, element type out_dtype
 *   staging         device buffer of at least emu_host_staging_bytes(M, N, K,
 *                   split_S, out_dtype) bytes, 256-byte aligned; scratch only
 *   chunks          number of column slabs (<= 0: one per 64 MiB of B)
 *   stream          the caller's stream: the work starts after what the stream
 *                   holds at the call, and the stream waits for the last copy back
 *
 * Asynchronous: the call returns once everything is enqueued; out_host holds the
 * result when `stream` has completed, and the host buffers must stay valid and
 * unchanged until then.  Pinned host memory (cudaHostAlloc / pin_memory) lets the
 * copies overlap the compute; pageable memory works, without the overlap.  Calls
 * issued on different caller streams with different staging buffers overlap one
 * call's uploads with another's GEMM.  The
 * call keeps no pointer after the stream completes.  Status codes and argument
 * checks are those of emu_scaled_mm_ex; EMU_EINVAL also for a short or misaligned
 * staging buffer; EMU_ECUDA when a copy or a stream operation fails.  When a step
 * fails after others were enqueued, the caller's stream is still ordered after
 * them, so the buffers may be released once it completes (out_host then holds no
 * valid result).  Calls from several host threads are serialised while they enqueue.
 */
size_t emu_host_staging_bytes(int64_t M, int64_t N, int64_t K, int32_t split_S,
                              emu_out_t out_dtype);

int emu_scaled_mm_host(const uint8_t* A_host, emu_fp8_t fmt_a,
                       const uint8_t* B_host, emu_fp8_t fmt_b,
                       int64_t M, int64_t N, int64_t K,
                       float scale_a, float scale_b, const float* scale_result,
                       void* out_host, emu_out_t out_dtype,
                       int32_t fast_accum, int32_t split_S,
                       const emu_preset_t* preset,
                       void* staging, size_t staging_bytes,
                       int32_t chunks, void* stream);

/*
 * Device status of the library on the current device: *status = 0, or 1 when a
 * kernel's wait for its TMA loads gave up (each wait polls a bounded number of
 * times instead of hanging; the CTA then returns early and the outputs of that
 * call are not valid).  Synchronous: it waits for the device.  reset != 0 clears
 * the status afterwards.  Returns EMU_OK or EMU_EINVAL/EMU_ECUDA.
 */
int emu_device_status(int32_t* status, int32_t reset);

/*
 * The CTA tile the GEMM entry points launch for this problem (the format pair and
 * the output dtype do not enter the choice), by its name: "M40", "M32", "M64",
 * "S", "K8", "K4", "K8H", "K4H", "C2", "C4", "C1", "C1L" or "W", or "none" when M,
 * N or K is 0.  The choice is
 * this library's cost model of the GB300 (an estimate per tile of issue and
 * latency time, fitted to measurements), not a behaviour of the pages' platforms;
 * every tile gives the same bits.  sm_count > 0 stands in for the device's SM
 * count, so the call needs no device; 0 asks the current device (152 when none is
 * visible).  EMU_FP8_TILE=<name> forces a tile, as for the GEMM calls.  name
 * receives the NUL-terminated name (name_len bytes at most; 4 suffice).  Returns
 * EMU_OK, or the status the GEMM entry points return for the same sizes, split and
 * preset, or EMU_EINVAL for a null or short buffer or a negative sm_count.
 */
int emu_tile_for(int64_t M, int64_t N, int64_t K, int32_t fast_accum, int32_t split_S,
                 const emu_preset_t* preset, int32_t sm_count, char* name, size_t name_len);

/*
 * Self-test of the bounded wait: enqueues a one-CTA kernel whose barrier can never
 * complete, so its wait gives up after a short limit and sets the device status
 * to 1 (read it with emu_device_status).  It exercises the failure path without a
 * fault or a hang; the pages have no counterpart.
 */
int emu_selftest_wait_timeout(void* stream);

/*
 * Self-test of the tensor cores as a source of exact products: on the current
 * device, tcgen05.mma of bf16 operands (fp32 accumulator) with a B operand whose
 * every column has one nonzero k, so that each output is one product of two
 * pre-scaled FP8 values; over the four format pairs, every pair of finite codes meets
 * once.  *mismatches (caller-owned) = outputs whose bits differ from the exact fp32
 * product (0: the tensor cores return exact products; a zero product may carry
 * either sign), or 0xFFFFFFFF if a completion wait gave up.  Synchronous; allocates
 * and frees two words of device memory.  Returns EMU_OK, EMU_EINVAL (null pointer) or
 * EMU_ECUDA.  ("User guide" section 6 and "Limitations of mmaemu v0.1": the pages'
 * tensor-core kernels rely on properties of the tensor cores; this is the check of
 * the one property a product path needs.)  The W tile takes its products from the
 * tensor cores only when the environment has EMU_FP8_TC=1 and this test, run once
 * per device on first use, finds no mismatch; otherwise it computes them itself.
 */
int emu_tc_selftest(uint32_t* mismatches);

/* Message of the last error returned on the calling host thread ("" if none). */
const char* emu_last_error(void);

/* ABI version of this header: 1. */
int emu_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EMU_FP8_H */
