/*
 * arf_oracle.h: CPU oracle for the all-reduce fusion epilogue.
 *
 * TEST INFRASTRUCTURE, not part of the library. Only the test suite, the
 * package's smoke check and the benchmark's CPU-baseline leg load it. It
 * shares no code, header, table or helper with the CUDA library; the two
 * agree only on the meaning of the arguments below.
 *
 * Enum values (plain ints, so this header stands alone):
 *   pattern 0 = kAllReduce, 1 = kARResidualRMSNorm
 *   dtype   0 = bf16,       1 = fp16
 * All [M,H] buffers are contiguous row-major host arrays of 16-bit codes.
 */
#ifndef ARF_ORACLE_H
#define ARF_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Decode a 16-bit code of `dtype` to the exact binary32 value. */
float arf_oracle_widen(int dtype, uint16_t bits);

/* Round a binary32 / binary64 value to the nearest `dtype` value,
 * ties to even; NaN stays a quiet NaN, overflow gives +-inf. */
uint16_t arf_oracle_narrow_f32(int dtype, float v);
uint16_t arf_oracle_narrow_f64(int dtype, double v);

/* Array forms of the three converters above (n elements). */
void arf_oracle_widen_n(int dtype, const uint16_t* in, float* out, int64_t n);
void arf_oracle_narrow_f32_n(int dtype, const float* in, uint16_t* out, int64_t n);
void arf_oracle_narrow_f64_n(int dtype, const double* in, uint16_t* out, int64_t n);

/* Inverse RMS of one stored row x[0..H-1] (codes of `dtype`), in binary64:
 * 1 / sqrt(sum(x^2) / H + eps). Also returns sum(x^2) through ss_out
 * when it is not NULL. */
double arf_oracle_inv_rms(int dtype, const uint16_t* x, int64_t H, float eps,
                          double* ss_out);

/* The epilogue with general layouts: every [M,H] tensor has its own row
 * stride (in elements, >= H), and the partials may be binary32 (pdtype 2)
 * instead of the I/O dtype (pdtype == dtype). binary32 partials enter the
 * binary32 rank-order sum as they are. Same return convention as below. */
int arf_oracle_run_general(int pattern, int W, const void* const* partials, int pdtype, int64_t ld_partials,
                           const void* residual, int64_t ld_residual, const void* gamma, float eps,
                           void* out, int64_t ld_out, void* residual_out, int64_t ld_residual_out,
                           int64_t M, int64_t H, int dtype);

/* The epilogue on host buffers.
 *   partials: host array of W host pointers, each to an [M,H] tensor.
 *   kAllReduce writes out only; residual, gamma, residual_out may be NULL.
 *   kARResidualRMSNorm writes residual_out and out.
 * Returns 0 on success, 1 on an invalid argument (nothing written). */
int arf_oracle_run(int pattern, int W, const void* const* partials,
                   const void* residual, const void* gamma, float eps,
                   void* out, void* residual_out, int64_t M, int64_t H,
                   int dtype);

#ifdef __cplusplus
}
#endif

#endif /* ARF_ORACLE_H */
