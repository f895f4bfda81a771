/*
 * oracle.h -- plain, slow CPU reference of the gradient-averaging hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this code.  It shares nothing
 * with the CUDA library (no header, helper, table or constant generator):
 * every function below is written straight from the pages it cites.
 *
 * Sources (cited by page title and section):
 *  [H]  "Horovod: Fast and Easy Distributed Deep Learning in TensorFlow"
 *       (explainer page), section "The Ring-Allreduce Algorithm" and
 *       section "Tensor Fusion: Why Small Tensors Break Ring-Allreduce".
 *  [R]  "Collective Communication: Ring All-Reduce" tutorial, section 4
 *       (step-by-step schedule), section 5 (data volume), section 7
 *       (ring simulator).
 *  [T]  "THC: Accelerating Distributed Deep Learning Using Tensor
 *       Homomorphic Compression", section 2 (NMSE definition), section 4
 *       (stochastic quantization, uniform SQ, Uniform THC / Algorithm 1).
 *  [S]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *       1, 2, 3", SC'11 -- definition of the Philox4x32 generator.
 *  [ST] Sanders, Speck, Traff, "Two-tree algorithms for full bandwidth
 *       broadcast, reduction and scan", Parallel Computing 35 (2009) --
 *       the two complementary binary trees read into the tutorial's
 *       double-binary-tree all-reduce ([R], "Design Alternatives &
 *       Collective Comparison Matrix: Ring vs. Tree vs. NVLS").
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math), so
 * every float expression is evaluated as written, one IEEE rounding per op.
 */
#ifndef GAR_ORACLE_H
#define GAR_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes and reduction ops used by the oracle's own interface */
#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_SUM 0
#define ORACLE_AVG 1

/* ---------------- Philox4x32 [S] ---------------- */
void oracle_philox4x32(const uint32_t ctr[4], const uint32_t key[2], int rounds,
                       uint32_t out[4]);

/* ---------------- ring all-reduce [H], [R] ---------------- */
/* chunk length used for a buffer of n elements split over p workers */
int64_t oracle_ring_chunk_len(int64_t n, int p);

/* Literal schedule: p-1 scatter-reduce steps then (if phases == 2) p-1
 * all-gather steps, run in place on p fp32 host buffers.  sent_elems[w]
 * receives the number of elements worker w put on the wire; *steps the
 * number of synchronous ring steps executed.  Returns 0 or -1 (bad args). */
int oracle_ring_schedule_f32(float *const *bufs, int p, int64_t n, int op, int phases,
                             int64_t *sent_elems, int *steps);

/* Closed form of the same schedule: every element's ring-order fp32 fold,
 * written to out[n] (all workers receive this value). */
int oracle_ring_fold_f32(const float *const *x, int p, int64_t n, int op, float *out);
/* the same, only for the element indices idx[k], k < count */
int oracle_ring_fold_f32_at(const float *const *x, int p, int64_t n, int op,
                            const int64_t *idx, int64_t count, float *out);

/* bf16 variants: inputs are bf16 bit patterns, partial sums are fp32, the
 * averaged value is rounded to bf16 (nearest-even) on output.
 * out_f32 (may be NULL) receives the fp32 value before that rounding. */
float oracle_bf16_to_f32(uint16_t h);
uint16_t oracle_f32_to_bf16(float f);
void oracle_f32_to_bf16_n(const float *in, int64_t n, uint16_t *out);
int oracle_ring_fold_bf16(const uint16_t *const *x, int p, int64_t n, int op, uint16_t *out,
                          float *out_f32);
int oracle_ring_fold_bf16_at(const uint16_t *const *x, int p, int64_t n, int op,
                             const int64_t *idx, int64_t count, uint16_t *out);
int oracle_ring_schedule_bf16(uint16_t *const *bufs, int p, int64_t n, int op,
                              int64_t *sent_elems, int *steps);
/* Sampled forms for buffers too large to copy to the host: vals[w * count + k]
 * is worker w's value at element e[k] of its n-element buffer. */
int oracle_ring_fold_f32_samples(const float *vals, int p, int64_t n, int op, const int64_t *e,
                                 int64_t count, float *out);
int oracle_ring_fold_bf16_samples(const uint16_t *vals, int p, int64_t n, int op,
                                  const int64_t *e, int64_t count, uint16_t *out);

/* Bidirectional dual ring ([R] section 11, exercise 1 and its worked
 * solution): the buffer is cut into 2p sub-chunks; sub-chunks 0..p-1 go
 * round the clockwise ring, p..2p-1 round the counter-clockwise ring, both
 * in the same 2(p-1) steps.  Literal schedule (fp32, in place) and its
 * closed form. */
int64_t oracle_bidir_subchunk_len(int64_t n, int p);
int oracle_bidir_schedule_f32(float *const *bufs, int p, int64_t n, int op, int64_t *sent_elems,
                              int *steps);
int oracle_bidir_fold_f32(const float *const *x, int p, int64_t n, int op, float *out);
/* sampled form: vals[w * count + k] = worker w's value at element e[k] */
int oracle_bidir_fold_f32_samples(const float *vals, int p, int64_t n, int op, const int64_t *e,
                                  int64_t count, float *out);

/* Double binary tree ([R] "Design Alternatives & Collective Comparison
 * Matrix"; construction [ST]).  Tree 1: the in-order binary tree on labels
 * 1..p (a run's root is its label with the most trailing zero bits), label l
 * on rank l - 1; tree 2: the same shape, label l on rank p - l (p even) or
 * (l - 2) mod p (p odd).  Elements [0, ceil(n/2)) go over tree 1, the rest
 * over tree 2; a node's partial sum is (own + left child's) + right child's
 * in fp32; the root's sum (/ p for AVG) is broadcast.
 * oracle_dbtree_build fills parent/left/right[rank] (-1: none) for tree 0 or
 * 1 and returns the root rank (-1: bad arguments). */
int oracle_dbtree_build(int p, int tree, int32_t *parent, int32_t *left, int32_t *right);
int64_t oracle_dbtree_half(int64_t n);
/* literal schedule (fp32, in place): reduce up both trees, then broadcast */
int oracle_dbtree_schedule_f32(float *const *bufs, int p, int64_t n, int op, int64_t *sent_elems,
                               int *steps);
/* closed forms; bf16 inputs are widened, summed in fp32, rounded once */
int oracle_dbtree_fold_f32(const float *const *x, int p, int64_t n, int op, float *out);
int oracle_dbtree_fold_bf16(const uint16_t *const *x, int p, int64_t n, int op, uint16_t *out);
/* sampled forms: vals[w * count + k] = worker w's value at element e[k] */
int oracle_dbtree_fold_f32_samples(const float *vals, int p, int64_t n, int op, const int64_t *e,
                                   int64_t count, float *out);
int oracle_dbtree_fold_bf16_samples(const uint16_t *vals, int p, int64_t n, int op, const int64_t *e,
                                    int64_t count, uint16_t *out);

/* ---------------- Tensor Fusion [H] ---------------- */
/* Next-fit plan.  dtype[i] is ORACLE_F32 or ORACLE_BF16.  Outputs per tensor:
 * seg_buffer[i], seg_offset[i] (elements from the buffer start); per buffer:
 * buf_numel[b] (elements, from 0 to the end of the last tensor).  buf_numel
 * must have room for count entries.  Returns the number of buffers or -1. */
int oracle_fusion_plan(const int64_t *numel, const int32_t *dtype, int count,
                       int64_t capacity_bytes, int align_bytes, int32_t *seg_buffer,
                       int64_t *seg_offset, int64_t *buf_numel);
/* Copy the tensors of `buffer` into fusion_buf; every other byte of
 * fusion_buf[0, buf_numel) is set to zero. */
int oracle_fusion_pack(const void *const *src, const int32_t *seg_buffer,
                       const int64_t *seg_offset, const int64_t *numel, int count, int buffer,
                       void *fusion_buf, int64_t buf_numel, int elem_bytes);
int oracle_fusion_unpack(const void *fusion_buf, const int32_t *seg_buffer,
                         const int64_t *seg_offset, const int64_t *numel, int count, int buffer,
                         void *const *dst, int elem_bytes);

/* ---------------- uniform THC [T] ---------------- */
void oracle_thc_range(const float *const *x, int p, int64_t n, float *m, float *M);
/* fp32 position t = (x - m) * (L / (M - m)) clamped to [0, L] */
float oracle_thc_position(float x, float m, float M, int b);
/* index of one coordinate of worker `worker` at element index e */
uint32_t oracle_thc_index(float x, float m, float M, int b, uint64_t seed, int worker,
                          int64_t e);
int oracle_thc_encode(const float *x, int64_t n, float m, float M, int b, uint64_t seed,
                      int worker, uint32_t *packed);
int oracle_thc_unpack(const uint32_t *packed, int64_t n, int b, uint8_t *idx);
int oracle_thc_aggregate(const uint32_t *const *packed, int p, int64_t n, int b,
                         uint16_t *sums);
int oracle_thc_decode(const uint16_t *sums, int64_t n, float m, float M, int b, int p,
                      double *avg);
/* Sampled THC round: vals[w * count + k] is worker w's value at element e[k];
 * idx[w * count + k] (may be NULL) receives its index, avg[k] the decoded
 * average of element e[k]. */
int oracle_thc_allreduce_samples(const float *vals, int p, const int64_t *e, int64_t count, int b,
                                 uint64_t seed, float m, float M, uint8_t *idx, double *avg);
/* Straggler dropping ([T] section 8, stragglers): only the workers whose bit
 * is set in `arrived` are encoded (each with its own worker id) and summed;
 * the decode divides by their number.  packed may be NULL; entries of
 * workers that did not arrive are not written. */
int oracle_thc_allreduce_masked(const float *const *x, int p, uint64_t arrived, int64_t n, int b,
                                uint64_t seed, float m, float M, double *avg, uint32_t *const *packed);
/* encode every worker, aggregate, decode; packed may be NULL */
int oracle_thc_allreduce(const float *const *x, int p, int64_t n, int b, uint64_t seed,
                         float m, float M, double *avg, uint32_t *const *packed);

/* ---------------- non-uniform THC [T] section 5, Algorithm 2 ---------------- */
/* table[0..L], L = 2^b - 1: strictly increasing integers, table[0] = 0,
 * table[L] = g.  Returns 0 if valid, -1 otherwise. */
int oracle_nuhc_check_table(const uint16_t *table, int b, int g);
/* fp32 position on the granularity-g grid: clamp((x - m) * (g / (M - m)), 0, g) */
float oracle_nuhc_position(float x, float m, float M, int g);
uint32_t oracle_nuhc_index(float x, float m, float M, int b, int g, const uint16_t *table,
                           uint64_t seed, int worker, int64_t e);
int oracle_nuhc_encode(const float *x, int64_t n, float m, float M, int b, int g,
                       const uint16_t *table, uint64_t seed, int worker, uint32_t *packed);
/* the PS: sums[e] = sum over workers of table[index] */
/* oracle_nuhc_encode of elements e0 .. e0 + n - 1 of a longer vector (x[k] =
 * element e0 + k; e0 a multiple of 32 / b): the whole vector's words
 * e0 / (32 / b) onwards. */
int oracle_nuhc_encode_at(const float *x, int64_t n, int64_t e0, float m, float M, int b, int g,
                          const uint16_t *table, uint64_t seed, int worker, uint32_t *packed);
int oracle_nuhc_aggregate(const uint32_t *const *packed, int p, int64_t n, int b,
                          const uint16_t *table, uint16_t *sums);
int oracle_nuhc_decode(const uint16_t *sums, int64_t n, float m, float M, int g, int p,
                       double *avg);

/* ---------------- RHT pre/post-processing [T] section 5 ---------------- */
/* Rademacher diagonal D: d_i = -1 when bit (i mod 128) of the 128-bit
 * Philox4x32-10 block with counter (i/128 low, i/128 high, 0xFFFFFFFF, 0)
 * and key (seed low, seed high) is set (word (i/32) mod 4, bit i mod 32),
 * else +1.  The worker slot 0xFFFFFFFF keeps this stream apart from the
 * quantization draws; every worker uses the same D (same seed). */
int oracle_rht_signs(int64_t n, uint64_t seed, int8_t *d);
/* y = (1/sqrt(n)) H D x (inverse = 0) or x = (1/sqrt(n)) D H y (inverse = 1),
 * n a power of two, H the Sylvester-Hadamard matrix, in fp64. */
int oracle_rht(const double *in, int64_t n, uint64_t seed, int inverse, double *out);
/* Norm-based range: l = max_w ||x_w||_2, M = (t_p / sqrt(n)) l, m = -M (fp64). */
void oracle_rht_norm_range(const double *const *x, int p, int64_t n, double t_p, double *m,
                           double *M);

/* ---------------- NMSE [T] ---------------- */
/* Error feedback ([T] section 5): x = grad + e before the rotation, and
 * e = x - x_hat after it (x_hat: the worker's own quantized vector, decoded
 * and rotated back).  fp32, one rounding per element. */
void oracle_ef_apply(const float *grad, const float *e, float *x, int64_t n);
void oracle_ef_update(float *e, const float *x, const float *x_hat, int64_t n);

double oracle_nmse(const float *x, const float *x_hat, int64_t n);
double oracle_nmse_f64(const double *x, const double *x_hat, int64_t n);

/* ---------------- wire-vector checksum ---------------- */
/* Silent-data-corruption check of the packed indices, for failure
 * detection (the pages fix no checksum): s1 = sum w_i and
 * s2 = sum (i + 1) w_i over the n 32-bit words, both mod 2^32; returns
 * (s2 << 32) | s1.  s1 changes with any flipped bit; a swap of words i and j
 * changes s2 by (j - i)(w_i - w_j) mod 2^32, so only swaps where that product
 * is 0 mod 2^32 go unseen. */
uint64_t oracle_checksum(const uint32_t *w, int64_t n);

#ifdef __cplusplus
}
#endif
#endif
