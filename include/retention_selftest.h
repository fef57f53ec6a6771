/*
 * retention_selftest.h -- tensor-core self-test of libretention.so.
 *
 * No counterpart on the pages: this checks the sm_103a tensor-core
 * building blocks (shared-memory operand layouts, TMEM operands and the
 * accumulator's lane layout) that the retention kernels rely on.
 */
#ifndef RETENTION_SELFTEST_H
#define RETENTION_SELFTEST_H

#include "retention.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One CTA computes D = A * B^T with a chain of tcgen05 MMAs (bf16 inputs,
 * fp32 accumulation).  A: [M][K] bf16, B: [N][K] bf16 (device, row-major).
 * a_mode: 0 = A in shared memory K-major, 1 = MN-major, 2 = A in TMEM.
 * b_mode: 0 = K-major, 1 = MN-major.  M in {64,128}, N in 32..256 (multiple
 * of 32), K in {64,128}.  a_lbo/a_sbo/b_lbo/b_sbo: byte strides used in the
 * MN-major descriptors.  D: [128][N] fp32 device buffer receiving all 128
 * TMEM lanes of the accumulator.  status: device word, set non-zero if the
 * MMA completion wait ran out.  Returns a ret_status value.
 */
int retention_tc_probe(int a_mode, int b_mode, int M, int N, int K, int a_lbo, int a_sbo,
                       int b_lbo, int b_sbo, const void *A, const void *B, float *D,
                       unsigned *status, ret_stream_t stream);

/*
 * The accumulator-scaling operand of tcgen05.mma (PTX ISA, tcgen05.mma
 * "scale-input-d": D = A * B + D * 2^-n).  One CTA computes D = A * B^T
 * (A, B: [128][64] bf16 device, K-major in shared memory), then runs the
 * same MMA chain again with the first MMA given scale n (0..15), so that
 * D' = A B^T (1 + 2^-n).  D: [128][128] fp32 device.  Returns a ret_status.
 */
int retention_tc_probe_scale_d(int n, const void *A, const void *B, float *D,
                               unsigned *status, ret_stream_t stream);

/*
 * The CTA-pair MMA (PTX ISA, tcgen05.mma with .cta_group::2): the two CTAs
 * of a cluster compute D = A * B^T for 256 rows, CTA r holding rows
 * 128 r .. 128 r + 127 of A and columns N/2 r .. N/2 (r + 1) - 1 of B in
 * its shared memory (K-major, 128-byte swizzled) and receiving its 128 rows
 * of D in its TMEM; the even CTA issues the MMAs.  A: [256][K], B: [N][K]
 * bf16 device; D: [256][N] fp32 device; tbase_out: two device words, the
 * TMEM address each CTA's allocation returned.  N in {128, 256}, K in
 * {64, 128}.  status as above.  Returns a ret_status value.
 */
int retention_tc_probe_pair(int N, int K, const void *A, const void *B, float *D,
                            unsigned *tbase_out, unsigned *status, ret_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif
