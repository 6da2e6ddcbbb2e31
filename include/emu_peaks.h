/*
 * emu_peaks.h -- C ABI of libemupeaks, the instruction-rate microbenchmark of the
 * GB300 (sm_103a) pipes that libemufp8's GEMM kernels issue on.  It is measurement
 * infrastructure, not part of the GEMM: the documentation pages have no counterpart.
 * bench.py divides its achieved rates by these measured rates (times the SM count
 * and the maximum SM clock) to report roofline fractions against measured, not
 * nominal, peaks; the test suite uses the agreement check, on which the GEMM's
 * packed pass 2 rests.
 *
 * Every call is synchronous on the current device, allocates and frees its own
 * small device buffers, and runs kernels of a fixed number of arithmetic
 * iterations (nothing waits on anything).
 */
#ifndef EMU_PEAKS_H
#define EMU_PEAKS_H

#ifdef __cplusplus
extern "C" {
#endif

/* Number of measured operations. */
int emu_peaks_count(void);

/* Name of operation i ("" when out of range): fmul_rz_subnormal, fmul_rn_normal,
   fadd_subnormal, their f32x2_ forms, dpx_viaddmax_s16x2, imad, iadd3, lop3, prmt,
   imad_iadd3_mixed, emulation_mix_macs, dpx_viaddmax_s16x2_vector,
   f32x2_fmul_rz_subnormal_vector, emulation_mix_vector_macs, emulation_tile_macs. */
const char* emu_peaks_name(int i);

/* rates[i] (emu_peaks_count() doubles, caller-owned host memory): lane-operations per
   clock per SM of operation i, from one CTA of 1024 threads per SM each running 8
   independent chains (a packed f32x2 instruction counts two operations);
   emulation_mix_macs: MACs per clock per SM of the GEMM's per-MAC arithmetic, 1.5
   packed f32x2 instructions and 0.5 DPX add-max.  The operations without _vector
   take their second and third operands from kernel arguments, the same in every
   thread; the _vector ones take all operands from per-thread registers, as the GEMM
   does (emulation_mix_vector_macs: the same mix so fed); emulation_tile_macs: MACs
   per clock per SM of the GEMM's inner loop on a 4 x 4 thread tile from registers
   (512 threads per SM).  Returns 0, or -4 on a CUDA error. */
int emu_peaks_measure(double* rates);

/* bad[0..2] (3 caller-owned unsigned ints): halves of n random operand pairs on which
   mul.rn.f32x2, mul.rz.f32x2 and add.rn.f32x2 differ bit for bit from the scalar
   instruction (NaN results compare as NaN), subnormal results included.  Returns 0,
   -1 for n <= 0 or a null bad, -4 on a CUDA error. */
int emu_peaks_f32x2_agreement(int n, unsigned* bad);

#ifdef __cplusplus
}
#endif

#endif /* EMU_PEAKS_H */
