/*
 * gar.h -- C ABI of the GB300 gradient-averaging library (libgar.so).
 *
 * The library averages the gradients of P data-parallel workers whose
 * buffers all live in one GPU's HBM.  Three parts, each a hand-written
 * sm_103a CUDA kernel family behind the calls below:
 *
 *   1. Tensor Fusion   -- many small gradient tensors packed into large
 *                         fusion buffers and scattered back afterwards.
 *   2. Ring all-reduce -- the reduce-scatter + all-gather chunk schedule,
 *                         computed as one pass that reproduces, bit for bit,
 *                         the fp32 sum order of the 2(P-1)-step ring.
 *   3. Uniform THC     -- shared range, Philox-driven stochastic quantization
 *                         to b-bit indices, integer summation of the indices
 *                         without decompression, one decode to the average.
 *
 * Sources (cited by page title and section):
 *   [H] "Horovod: Fast and Easy Distributed Deep Learning in TensorFlow"
 *       (explainer page): "The Ring-Allreduce Algorithm"; "Tensor Fusion:
 *       Why Small Tensors Break Ring-Allreduce" (steps 1-6).
 *   [R] "Collective Communication: Ring All-Reduce" tutorial: section 4
 *       (schedule), section 5 (per-worker volume 2(P-1)/P of the buffer),
 *       section 7 (ring simulator).
 *   [T] "THC: Accelerating Distributed Deep Learning Using Tensor
 *       Homomorphic Compression": section 2 (NMSE), section 4 (stochastic
 *       quantization, uniform SQ on a global range, Uniform THC /
 *       Algorithm 1), section 5 (index vectors summed at the PS).
 *   [S] Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3"
 *       (SC'11): Philox4x32-10.
 *   [ST] Sanders, Speck, Traff, "Two-tree algorithms for full bandwidth
 *       broadcast, reduction and scan" (Parallel Computing, 2009): the two
 *       complementary trees of the double-binary-tree all-reduce that [R]
 *       compares with the ring ("Design Alternatives & Collective
 *       Comparison Matrix: Ring vs. Tree vs. NVLS").
 *
 * Conventions shared by every call
 *   - Ownership: the caller owns every buffer.  "device" pointers are CUDA
 *     device (or managed) memory; "host" arrays (pointer tables, plans) are
 *     read during the call only and may be freed when it returns.  No call
 *     allocates device memory.
 *   - Asynchrony: device work is enqueued on `stream` (a cudaStream_t; NULL
 *     is the legacy default stream) and the call returns without waiting.
 *     The status covers argument checks and the launch itself.
 *   - Errors: every call returns GAR_OK (0) or a negative gar_status; nothing
 *     exits, traps or prints.  gar_last_error() returns a message for the
 *     last failing call on the calling thread.
 *   - Limits: 1 <= P <= GAR_MAX_WORKERS; sizes are element counts (int64).
 *   - Alignment: device buffers with 16-byte aligned base addresses take
 *     the vectorised paths; other addresses are accepted and take scalar
 *     paths (same results).  Element alignment (4 B for fp32 and uint32,
 *     2 B for bf16 and uint16) is required: GAR_EALIGN otherwise.
 */
#ifndef GAR_H
#define GAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *gar_stream_t;

typedef enum {
    GAR_OK = 0,
    GAR_EINVAL = -1,    /* null pointer, bad size, P, b, op, buffer id ...      */
    GAR_EDTYPE = -2,    /* unknown dtype, or mixed dtypes where one is required */
    GAR_EALIGN = -3,    /* pointer not aligned to its element size              */
    GAR_EOVERFLOW = -4, /* P * (2^b - 1) exceeds the 16-bit index sum           */
    GAR_ECUDA = -5      /* the CUDA runtime reported an error at launch         */
} gar_status;

typedef enum { GAR_F32 = 0, GAR_BF16 = 1 } gar_dtype;

/* Bits of the device status word (gar_sync_status). */
typedef enum {
    GAR_STATUS_NONFINITE = 1 /* a THC range pass saw a NaN or an infinite input */
} gar_device_status;
typedef enum { GAR_SUM = 0, GAR_AVG = 1 } gar_op;

#define GAR_MAX_WORKERS 64

/* One tensor's place in a fusion plan. */
typedef struct {
    int32_t buffer;   /* fusion buffer id, 0-based                    */
    int32_t reserved; /* 0                                            */
    int64_t offset;   /* first element of the tensor inside the buffer */
    int64_t numel;    /* number of elements                           */
} gar_seg;

/* Library version (major * 10000 + minor * 100 + patch). */
int gar_version(void);

/* Message for the last non-OK status returned on this thread ("" if none).
 * The string stays valid until the next failing call on the thread. */
const char *gar_last_error(void);

/* Number of CUDA kernels this library has launched in this process (all
 * threads, all devices), for accounting; never reset. */
uint64_t gar_launch_count(void);

/* ===================================================================== */
/* Tensor Fusion [H] "Tensor Fusion", steps 1-6                          */
/* ===================================================================== */

/* gar_fusion_plan -- host only, no device work.
 * Plans the fusion of `count` tensors taken in list (= ready) order
 * (step 1): a tensor joins the open buffer if it has that buffer's dtype
 * and fits in the room left, its start rounded up to `align_bytes`;
 * otherwise the open buffer is closed and the tensor opens the next one
 * (next-fit).  A tensor larger than the capacity gets a buffer to itself.
 * Step 2's buffer size is `capacity_bytes` (64 MB default in Horovod).
 *   numel[count], dtype[count]  host, per tensor (gar_dtype)
 *   capacity_bytes              > 0
 *   align_bytes                 > 0, a multiple of every used element size
 *                               (16 lets every tensor start on a 16-B line)
 *   segs[count]                 host, out: the tensor's buffer and offset
 *   n_buffers                   host, out: number of buffers
 *   buf_numel[count]            host, out: elements of each buffer, from 0
 *                               to the end of its last tensor (only the first
 *                               *n_buffers entries are written)
 * Errors: GAR_EINVAL (null, count < 0, numel < 0, bad capacity/alignment),
 *         GAR_EDTYPE (unknown dtype). */
int gar_fusion_plan(const int64_t *numel, const int32_t *dtype, int32_t count,
                    int64_t capacity_bytes, int32_t align_bytes, gar_seg *segs,
                    int32_t *n_buffers, int64_t *buf_numel);

/* gar_fusion_pack -- step 3: copy the tensors that the plan puts in `buffer`
 * into `fusion_buf` at their offsets; the alignment gaps between them are
 * zero-filled.  One worker's tensors per call.
 *   src[count]    host array of device pointers (entries of tensors in other
 *                 buffers are ignored and may be NULL)
 *   segs, dtype   the plan and the per-tensor dtypes given to the plan
 *   fusion_buf    device, buf_numel elements of the buffer's dtype
 * Errors: GAR_EINVAL (bad buffer id, a segment outside buf_numel, null
 *         pointer), GAR_EDTYPE (dtypes differ within the buffer),
 *         GAR_EALIGN, GAR_ECUDA. */
int gar_fusion_pack(const void *const *src, const gar_seg *segs, const int32_t *dtype,
                    int32_t count, int32_t buffer, void *fusion_buf, int64_t buf_numel,
                    gar_stream_t stream);

/* gar_fusion_unpack -- step 5: copy each tensor of `buffer` from `fusion_buf`
 * back to dst[i] (host array of device pointers).  Errors as for pack. */
int gar_fusion_unpack(const void *fusion_buf, const gar_seg *segs, const int32_t *dtype,
                      int32_t count, int32_t buffer, void *const *dst, gar_stream_t stream);

/* gar_fusion_pack_all -- step 3 for every worker and every fusion buffer in
 * one pass (the same bytes as P * n_buffers gar_fusion_pack calls, in a
 * handful of launches).  Optionally also THC's preliminary round ([T] section
 * 4, Algorithm 1): d_mM[2b], d_mM[2b+1] = min and max over all workers'
 * fusion buffer b, its zero padding included -- the same values
 * gar_thc_range gives on the packed buffers -- computed while copying.
 *   src[P * count]          host array: src[w * count + i] = worker w's tensor i
 *   segs, dtype, count      the plan and per-tensor dtypes
 *   fusion_bufs[P * n_buffers]  host array: fusion_bufs[w * n_buffers + b] =
 *                           worker w's buffer b (device, buf_numel[b] elements)
 *   d_mM                    device, 2 * n_buffers floats, or NULL (no range);
 *                           fp32 plans only
 * Only buffers that at least one of the `count` tensors belongs to are
 * written (their range entries too), so a slice of a plan (e.g. one buffer's
 * tensors) packs just those buffers.
 * Errors: GAR_EINVAL, GAR_EDTYPE (mixed dtypes in a buffer, or a range asked
 *         of bf16 tensors), GAR_EALIGN, GAR_ECUDA. */
int gar_fusion_pack_all(const void *const *src, int32_t P, const gar_seg *segs, const int32_t *dtype,
                        int32_t count, void *const *fusion_bufs, const int64_t *buf_numel,
                        int32_t n_buffers, float *d_mM, gar_stream_t stream);

/* gar_fused_allreduce -- steps 3-5 in one pass: for every fusion buffer of
 * the plan, the ring all-reduce (as gar_ring_allreduce_sim, over the
 * buffer's buf_numel elements with its chunking) is applied, reading the
 * workers' tensors directly and writing each worker's result tensors
 * directly; the fusion buffers themselves are never materialised.  Results
 * are bit-identical to pack -> ring all-reduce -> unpack.
 *   src[P * count]  host array: src[w * count + i] = worker w's tensor i
 *   dst[P * count]  host array, same layout; dst may equal src (in place)
 *   segs, dtype     plan and per-tensor dtypes; buf_numel[n_buffers]
 *   op              GAR_SUM or GAR_AVG
 * Errors: GAR_EINVAL, GAR_EDTYPE, GAR_EALIGN, GAR_ECUDA. */
int gar_fused_allreduce(const void *const *src, void *const *dst, int32_t P,
                        const gar_seg *segs, const int32_t *dtype, int32_t count,
                        const int64_t *buf_numel, int32_t n_buffers, int32_t op,
                        gar_stream_t stream);

/* gar_fused_allreduce_range -- gar_fused_allreduce that also computes THC's
 * preliminary round for the plan's buffers ([T] section 4, Algorithm 1) from
 * the same reads: d_mM[2b], d_mM[2b+1] = min and max over the workers' inputs
 * of fusion buffer b, the packed buffer's zero padding included -- the values
 * gar_fusion_pack_all with a range gives for the same arguments.  Meant with
 * dst != src, so that the original gradients stay available to THC.  Only
 * buffers that at least one of the tensors belongs to get range entries.
 *   d_mM  device, 2 * n_buffers floats; fp32 plans only
 * Errors: as gar_fused_allreduce; GAR_EDTYPE for bf16 tensors. */
int gar_fused_allreduce_range(const void *const *src, void *const *dst, int32_t P, const gar_seg *segs,
                              const int32_t *dtype, int32_t count, const int64_t *buf_numel,
                              int32_t n_buffers, int32_t op, float *d_mM, gar_stream_t stream);

/* gar_checksum -- *d_out (device, one uint64) = (s2 << 32) | s1 with
 * s1 = sum w_i and s2 = sum (i + 1) w_i over the n 32-bit words d_words
 * (device, 4-byte aligned), both mod 2^32: a check against silent data
 * corruption of THC's wire vectors (a worker's packed indices as sent and
 * as the parameter server receives them).  A flipped bit changes s1; a swap
 * of words i and j changes s2 unless (j - i)(w_i - w_j) = 0 mod 2^32 (e.g.
 * words 2^16 apart whose values differ by a multiple of 2^16).  The value
 * does not depend on the order of the device's partial sums.  n = 0 gives 0.
 * Errors: GAR_EINVAL (n < 0, NULL), GAR_EALIGN, GAR_ECUDA. */
int gar_checksum(const uint32_t *d_words, int64_t n, uint64_t *d_out, gar_stream_t stream);

/* gar_sync_status -- waits for `stream`, then *status (host) = the device
 * status word of the current device: bits that kernels set for conditions
 * they find on the device.  GAR_STATUS_NONFINITE: a THC range pass
 * (gar_thc_range, gar_fusion_pack_all or gar_fused_allreduce_range with a
 * range) saw a NaN or an infinite input; the range skips NaN and takes
 * infinities in, so the quantization of such a round is meaningless.  The
 * word is set to 0 when clear != 0.  Kernels queued on other streams may set
 * bits at any time.  No kernel of this library waits on a flag or a peer, so
 * there is no timeout condition to report.
 * Errors: GAR_EINVAL (status NULL), GAR_ECUDA. */
int gar_sync_status(gar_stream_t stream, uint32_t *status, int32_t clear);

/* ===================================================================== */
/* Ring all-reduce [H] "The Ring-Allreduce Algorithm", [R] sections 4, 5, 7 */
/* ===================================================================== */

/* gar_ring_allreduce_sim -- the ring all-reduce of P worker buffers held in
 * one GPU's memory, in place: afterwards every bufs[w] holds the result.
 * The buffer is cut into P chunks of ceil(N / P) elements (the trailing
 * chunks short or empty when P does not divide N).  Chunk c starts on worker
 * c and gains one worker per scatter-reduce hop, so every element of chunk c
 * becomes the fp32 fold x_c + x_{c+1} + ... + x_{c+P-1} (indices mod P),
 * left to right; the all-gather hands that value to every worker.  GAR_AVG
 * then divides by P (fp32, round to nearest even).  bf16 buffers are widened
 * exactly, folded in fp32 and rounded to bf16 (nearest even) once, at the
 * end.  The result equals the literal 2(P-1)-step schedule bit for bit.
 *   bufs[P]  host array of device pointers, each N elements of `dtype`
 * Errors: GAR_EINVAL, GAR_EDTYPE, GAR_EALIGN, GAR_ECUDA. */
int gar_ring_allreduce_sim(void *const *bufs, int32_t P, int64_t N, int32_t dtype, int32_t op,
                           gar_stream_t stream);

/* gar_ring_allreduce_sim_out -- the same result written to n_out separate
 * device buffers out[n_out] (1 = reduce to one output, P = one per worker);
 * the inputs bufs[P] are only read.  Outputs must not overlap the inputs. */
int gar_ring_allreduce_sim_out(const void *const *bufs, int32_t P, int64_t N, int32_t dtype,
                               int32_t op, void *const *out, int32_t n_out,
                               gar_stream_t stream);

/* gar_ring_allreduce_bidir -- the bidirectional dual ring ([R] section 11,
 * exercise 1): the buffer is cut into 2P sub-chunks of ceil(N / 2P)
 * elements; sub-chunks 0..P-1 travel the clockwise ring exactly as in
 * gar_ring_allreduce_sim (sub-chunk c folds x_c + x_{c+1} + ...), sub-chunks
 * P..2P-1 travel the counter-clockwise ring (sub-chunk P + c folds
 * x_c + x_{c-1} + ..., indices mod P), in the same 2(P-1) steps.  In place,
 * fp32 or bf16, GAR_SUM or GAR_AVG as gar_ring_allreduce_sim.
 * Errors: GAR_EINVAL, GAR_EDTYPE, GAR_EALIGN, GAR_ECUDA. */
int gar_ring_allreduce_bidir(void *const *bufs, int32_t P, int64_t N, int32_t dtype, int32_t op,
                             gar_stream_t stream);

/* gar_ring_allreduce_steps -- the literal schedule, one launch per ring
 * step: P-1 scatter-reduce steps (worker i adds worker i-1's chunk
 * (i-s-1) mod P into its own), P-1 all-gather steps (worker i overwrites its
 * chunk (i-s) mod P with worker i-1's), then, for GAR_AVG, one element-wise
 * division by P.  In place, fp32 only (a bf16 schedule would round the
 * partial sums held in the buffers).  A checking path, not a fast one.
 *   steps       host, out (may be NULL): ring steps executed, 2(P-1)
 *   sent_elems  host, out (may be NULL): [P] elements each worker sent
 * Errors: GAR_EINVAL, GAR_EDTYPE (bf16), GAR_EALIGN, GAR_ECUDA. */
int gar_ring_allreduce_steps(void *const *bufs, int32_t P, int64_t N, int32_t op,
                             int32_t *steps, int64_t *sent_elems, gar_stream_t stream);

/* gar_dbtree_allreduce -- the double-binary-tree all-reduce ([R] "Design
 * Alternatives & Collective Comparison Matrix"; trees of [ST]) as a fold
 * order, in place: afterwards every bufs[w] holds the result.  Both trees
 * have the shape of the in-order binary tree on the labels 1..P (a run of
 * labels is rooted at its label with the most trailing zero bits).  Elements
 * [0, ceil(N/2)) are reduced over tree 1, label l on rank l - 1; the rest
 * over tree 2, label l on rank P - l (P even) or (l - 2) mod P (P odd).  A
 * node's partial sum is its own value plus its left child's partial sum,
 * then plus its right child's, in fp32; the root's sum (divided by P for
 * GAR_AVG, round to nearest even) is what every rank receives.  bf16
 * buffers are widened exactly, folded in fp32 and rounded to bf16 once.
 *   bufs[P]  host array of distinct device pointers, N elements of `dtype`
 * Errors: GAR_EINVAL, GAR_EDTYPE, GAR_EALIGN, GAR_ECUDA. */
int gar_dbtree_allreduce(void *const *bufs, int32_t P, int64_t N, int32_t dtype, int32_t op,
                         gar_stream_t stream);

/* gar_dbtree_parents -- host only: parent[w] = the parent rank of rank w in
 * tree 0 or 1 of gar_dbtree_allreduce, -1 for the root.
 *   parent  host, out: P entries
 * Errors: GAR_EINVAL. */
int gar_dbtree_parents(int32_t P, int32_t tree, int32_t *parent);

/* ===================================================================== */
/* Uniform THC [T] section 4 (Algorithm 1) and section 5                 */
/* ===================================================================== */
/* Encoding of one coordinate x of worker `worker` at element index e, with
 * L = 2^b - 1 and the shared range [m, M] (all in fp32, one rounding each):
 *     t = clamp((x - m) * (L / (M - m)), 0, L)       (t = 0 when M == m)
 *     j = floor(t),  f = t - j
 *     r = word (e mod 4) of Philox4x32-10 [S] with key (seed low 32 bits,
 *         seed high 32 bits) and counter (e/4 low, e/4 high, worker, 0)
 *     u = (r mod 2^23) / 2^23
 *     index = j + (u < f ? 1 : 0)
 * so the index rounds up with probability f (to within 2^-23) and the
 * quantized value m + index (M - m) / L is unbiased.  Indices are packed
 * least-significant-bits first: element e in word e / (32/b) at bit
 * (e mod (32/b)) * b; the last word is zero-padded.  b in {1, 2, 4, 8}. */

/* Number of uint32 words that hold N packed b-bit indices (0 if b is bad). */
int64_t gar_thc_words(int64_t N, int32_t b);

/* gar_thc_range -- the preliminary round: d_mM[0] = min, d_mM[1] = max over
 * all P * N entries (NaN entries are skipped; N = 0 gives +inf, -inf).
 *   x[P]  host array of device fp32 pointers;  d_mM  device, 2 floats.
 * Errors: GAR_EINVAL, GAR_EALIGN, GAR_ECUDA. */
int gar_thc_range(const float *const *x, int32_t P, int64_t N, float *d_mM,
                  gar_stream_t stream);

/* gar_thc_encode -- one worker's quantization to packed b-bit indices.
 *   x       device, N fp32;  d_mM  device [m, M] (e.g. from gar_thc_range)
 *   packed  device, gar_thc_words(N, b) uint32 words, fully written
 * Errors: GAR_EINVAL, GAR_EALIGN, GAR_ECUDA. */
int gar_thc_encode(const float *x, int64_t N, const float *d_mM, int32_t b, uint64_t seed,
                   int32_t worker, uint32_t *packed, gar_stream_t stream);

/* gar_thc_aggregate -- the PS step: sums[e] = sum over workers of their
 * index e, as exact integers, without decoding anything.
 *   packed[P]  host array of device pointers (gar_thc_words(N, b) words each)
 *   sums       device, N uint16
 * Errors: GAR_EINVAL, GAR_EOVERFLOW (P * (2^b - 1) > 65535), GAR_EALIGN,
 *         GAR_ECUDA. */
int gar_thc_aggregate(const uint32_t *const *packed, int32_t P, int64_t N, int32_t b,
                      uint16_t *sums, gar_stream_t stream);

/* gar_thc_decode -- each worker's last step: the index sum divided by the
 * number of workers, mapped back onto the grid:
 *     avg[e] = fma(sums[e], ((M - m) / L) / P, m)      (fp32, one rounding
 * per operation; within 1e-6 max(|m|, |M|) of the exact value).
 *   sums  device, N uint16;  d_mM  device [m, M];  avg  device, N fp32
 * Errors: GAR_EINVAL, GAR_EALIGN, GAR_ECUDA. */
int gar_thc_decode(const uint16_t *sums, int64_t N, const float *d_mM, int32_t b, int32_t P,
                   float *avg, gar_stream_t stream);

/* gar_thc_allreduce_fused -- encode (every worker), aggregate and decode in
 * one pass over the P inputs: avg equals gar_thc_decode(gar_thc_aggregate(
 * gar_thc_encode(x[w]) for w < P)) bit for bit.  If packed is non-NULL,
 * packed[w] (device, gar_thc_words(N, b) words) also receives worker w's
 * packed indices, the vector THC puts on the wire.
 * Errors: GAR_EINVAL, GAR_EOVERFLOW, GAR_EALIGN, GAR_ECUDA. */
int gar_thc_allreduce_fused(const float *const *x, int32_t P, int64_t N, int32_t b,
                            uint64_t seed, const float *d_mM, float *avg,
                            uint32_t *const *packed, gar_stream_t stream);

/* gar_thc_allreduce_fused_masked -- straggler dropping ([T] section 8,
 * stragglers: the PS waits only for the workers that arrived).  Only the
 * workers whose bit is set in `arrived` (bit w = worker w, w < P) are
 * encoded, each under its own worker id, and summed; the decode divides by
 * their number.  x[w] and packed[w] of the other workers are not read or
 * written (they may be NULL).  With every bit set this is
 * gar_thc_allreduce_fused bit for bit; it also equals gar_thc_encode of the
 * arrived workers -> gar_thc_aggregate over their vectors -> gar_thc_decode
 * with their number.  Errors: as gar_thc_allreduce_fused, and GAR_EINVAL when
 * no worker arrived. */
int gar_thc_allreduce_fused_masked(const float *const *x, int32_t P, uint64_t arrived, int64_t N,
                                   int32_t b, uint64_t seed, const float *d_mM, float *avg,
                                   uint32_t *const *packed, gar_stream_t stream);

/* gar_thc_allreduce_fused_plan -- uniform THC of every fusion buffer of a
 * plan ([H] "Tensor Fusion" feeding [T] Algorithm 1), read straight from the
 * workers' tensors and written straight to the output tensors: for each
 * buffer b the result is bit-identical to gar_fusion_pack_all ->
 * gar_thc_allreduce_fused over buffer b (worker ids 0..P-1, the packed
 * buffer's element index keying the Philox draws, zero padding encoded as
 * zeros) -> gar_fusion_unpack of the average.
 *   src[P * count]   host array: src[w * count + i] = worker w's tensor i
 *   segs, dtype      the plan; every tensor fp32; buf_numel[n_buffers]
 *   d_mM             device, [n_buffers][2]: each buffer's shared [m, M]
 *                    (from gar_fusion_pack_all or gar_fused_allreduce_range)
 *   out[count]       host array: device output tensor of each tensor (the
 *                    average every worker decodes)
 *   packed           NULL, or host array [P * n_buffers]: packed[w *
 *                    n_buffers + b] receives worker w's indices of buffer b
 *                    (gar_thc_words(buf_numel[b], b) words)
 * Only buffers that at least one of the tensors belongs to are processed.
 * Errors: GAR_EINVAL (bad b/P/plan, NULL, more than min(128, 2048 / P)
 * tensors meeting one packed word -- for b <= 2 one 8-element part of a
 * word), GAR_EDTYPE (bf16), GAR_EOVERFLOW,
 * GAR_EALIGN, GAR_ECUDA. */
int gar_thc_allreduce_fused_plan(const float *const *src, int32_t P, const gar_seg *segs,
                                 const int32_t *dtype, int32_t count, const int64_t *buf_numel,
                                 int32_t n_buffers, int32_t b, uint64_t seed, const float *d_mM,
                                 float *const *out, uint32_t *const *packed, gar_stream_t stream);

/* Bytes of device workspace gar_thc_allreduce_fused_plan_nmse needs for a
 * plan with these buffers and `count` tensors at b bits (0 for bad b or
 * counts).  An upper bound: one pair of doubles per CTA the call can run. */
size_t gar_thc_plan_nmse_workspace_bytes(const int64_t *buf_numel, int32_t n_buffers, int32_t count,
                                         int32_t b);

/* gar_thc_allreduce_fused_plan_nmse -- gar_thc_allreduce_fused_plan (same
 * outputs and wire vectors, bit for bit) that also takes, in the same pass,
 * the two sums of NMSE ([T] section 2) of the decoded average against a
 * reference -- the exact average, e.g. the ring all-reduce's output:
 *   d_pair[0] = sum (ref - avg)^2,  d_pair[1] = sum ref^2
 * over every element of the call's tensors (alignment gaps excluded), so
 * that no second pass over the averages is needed.  Terms in fp32, summed
 * pairwise over a word and over a thread's words and across a warp in fp32,
 * then across warps and CTAs in fp64 in a fixed order: deterministic, within
 * 2e-6 relative of all-fp64 sums.  gar_nmse_combine of the pairs of several
 * calls (e.g. one per fusion buffer) gives the NMSE over all of them.
 *   ref[count]     host array: device reference tensor of each tensor (fp32,
 *                  the tensor's numel, 4-byte aligned)
 *   d_pair         device, two doubles, 8-byte aligned
 *   d_workspace    device, at least gar_thc_plan_nmse_workspace_bytes(...)
 *                  bytes, 8-byte aligned, caller-owned, not shared with a
 *                  concurrent call
 * Other arguments and errors as gar_thc_allreduce_fused_plan; GAR_EINVAL
 * also for a NULL ref, d_pair or workspace, or a workspace too small. */
int gar_thc_allreduce_fused_plan_nmse(const float *const *src, int32_t P, const gar_seg *segs,
                                      const int32_t *dtype, int32_t count, const int64_t *buf_numel,
                                      int32_t n_buffers, int32_t b, uint64_t seed, const float *d_mM,
                                      float *const *out, uint32_t *const *packed,
                                      const float *const *ref, double *d_pair, void *d_workspace,
                                      size_t workspace_bytes, gar_stream_t stream);

/* ===================================================================== */
/* Non-uniform THC [T] section 5, Algorithm 2                            */
/* ===================================================================== */
/* With granularity g (2^b - 1 <= g <= 16383) the grid is m + k (M - m)/g,
 * k = 0..g, but a worker may only send the 2^b points whose k is a value of
 * the lookup table T (host array of 2^b uint16, strictly increasing,
 * T[0] = 0, T[2^b - 1] = g; the pages give no optimal tables, so T is the
 * caller's).  Encoding in fp32, one rounding per operation:
 *     t = clamp((x - m) * (g / (M - m)), 0, g)        (t = 0 when M == m)
 *     z = the largest z <= 2^b - 2 with T[z] <= t
 *     index = z + 1 if u < (t - T[z]) / (T[z + 1] - T[z]) exactly, else z
 *             (u: the Philox draw of uniform THC; decided as
 *              u (T[z + 1] - T[z]) < t - T[z], whose sides are exact)
 * Packing as for uniform THC.  The PS looks every index up in T and sums the
 * table values; each worker decodes avg = fma(S, ((M - m)/g)/P, m).  With
 * g = 2^b - 1 and T the identity this is exactly uniform THC. */

/* gar_nuhc_encode -- one worker's indices (see gar_thc_encode for layout).
 * Errors: GAR_EINVAL (bad b, g or table, NULL), GAR_EALIGN, GAR_ECUDA. */
int gar_nuhc_encode(const float *x, int64_t N, const float *d_mM, int32_t b, int32_t g,
                    const uint16_t *table, uint64_t seed, int32_t worker, uint32_t *packed,
                    gar_stream_t stream);

/* gar_nuhc_aggregate -- sums[e] = sum over workers of T[index] (uint16).
 * g is taken as T[2^b - 1].  Errors: GAR_EINVAL, GAR_EOVERFLOW (P * g >
 * 65535), GAR_EALIGN (sums must be 4-byte aligned), GAR_ECUDA. */
int gar_nuhc_aggregate(const uint32_t *const *packed, int32_t P, int64_t N, int32_t b,
                       const uint16_t *table, uint16_t *sums, gar_stream_t stream);

/* gar_nuhc_decode -- avg[e] = fma(sums[e], ((M - m)/g)/P, m) in fp32.
 * Errors: GAR_EINVAL, GAR_EALIGN, GAR_ECUDA. */
int gar_nuhc_decode(const uint16_t *sums, int64_t N, const float *d_mM, int32_t g, int32_t P,
                    float *avg, gar_stream_t stream);

/* gar_nuhc_allreduce_fused -- encode every worker, look up, sum and decode in
 * one pass; equal bit for bit to decode(aggregate(encode)).  packed may be
 * NULL.  Errors: GAR_EINVAL, GAR_EOVERFLOW, GAR_EALIGN, GAR_ECUDA. */
int gar_nuhc_allreduce_fused(const float *const *x, int32_t P, int64_t N, int32_t b, int32_t g,
                             const uint16_t *table, uint64_t seed, const float *d_mM, float *avg,
                             uint32_t *const *packed, gar_stream_t stream);

/* gar_nuhc_allreduce_fused_masked -- straggler dropping ([T] section 8,
 * stragglers: the PS waits only for the workers that arrived) with
 * non-uniform THC ([T] section 5, Algorithm 2).  Only the workers whose bit
 * is set in `arrived` (bit w = worker w, w < P) are encoded, each under its
 * own worker id, and their table values summed; the decode divides by their
 * number.  x[w] and packed[w] of the other workers are not read or written
 * (they may be NULL).  With every bit set this is gar_nuhc_allreduce_fused
 * bit for bit; it also equals gar_nuhc_encode of the arrived workers (their
 * own ids) -> gar_nuhc_aggregate over their vectors -> gar_nuhc_decode with
 * their number.  Errors: as gar_nuhc_allreduce_fused (GAR_EOVERFLOW when the
 * number arrived times g exceeds 65535), and GAR_EINVAL when no worker
 * arrived. */
int gar_nuhc_allreduce_fused_masked(const float *const *x, int32_t P, uint64_t arrived, int64_t N, int32_t b,
                                    int32_t g, const uint16_t *table, uint64_t seed, const float *d_mM, float *avg,
                                    uint32_t *const *packed, gar_stream_t stream);

/* ===================================================================== */
/* Pre- and post-processing [T] section 5 (RHT, truncation, error feedback) */
/* ===================================================================== */
/* Before non-uniform THC each worker adds its error-feedback vector to its
 * gradient (x = grad + e), rotates it with the randomized Hadamard transform
 * and quantizes against the range [-M, M] set from the largest worker norm
 * (values outside are clamped: the truncation).  After the decode each
 * worker applies the inverse rotation to the average estimate and updates
 * e.  Every worker draws the same D (same seed).  Vectors whose length is
 * not a power of two are zero-padded to one by the caller. */

/* gar_rht -- out = (1/sqrt(n)) H D in (inverse = 0) or
 * out = (1/sqrt(n)) D H in (inverse = 1), H the n x n Sylvester-Hadamard
 * matrix, D = diag(d), d_i = -1 when bit (i mod 128) of the Philox4x32-10
 * block with key (seed low, seed high) and counter (i/128 low, i/128 high,
 * 0xFFFFFFFF, 0) is set (word (i/32) mod 4, bit i mod 32), else +1.
 * in, out: device, n fp32, 16-byte aligned, caller-owned; out == in runs in
 * place, any other overlap is rejected.  n: a power of two, 1 <= n <= 2^31.
 * fp32 butterflies (a + b, a - b), the 1/sqrt(n) factor (rounded to fp32)
 * applied once at the end: each output is within about
 * (log2 n + 2) 2^-24 ||in|| of the exact value.  Kernels: n < 4096 one CTA;
 * else one 4096-element tile pass plus ceil((log2 n - 12) / 8) strided
 * passes, each one read and one write of the vector.
 * Errors: GAR_EINVAL (n not a power of two or above 2^31, NULL, bad inverse,
 * partial overlap), GAR_EALIGN, GAR_ECUDA. */
int gar_rht(const float *in, float *out, int64_t n, uint64_t seed, int32_t inverse,
            gar_stream_t stream);

/* Bytes of device workspace gar_rht_norm_range needs (0 for bad P or n). */
size_t gar_rht_norm_range_workspace_bytes(int32_t P, int64_t n);

/* gar_rht_norm_range -- the range of the rotated vectors without rotating
 * them first (the rotation keeps norms): l = max over workers of ||x_w||_2,
 * d_mM[0] = -M, d_mM[1] = M with M = (t_p / sqrt(n)) l, rounded to fp32.
 * x: host array of P device pointers to n fp32 each (4-byte aligned).
 * t_p > 0: the truncation threshold for a p fraction outside,
 * Phi^-1(1 - p/2).  d_mM: device, two floats.  Squares are formed in fp32
 * (four summed pairwise) and accumulated in fp64 in a fixed order
 * (deterministic; relative error below 1e-6).  d_workspace: device, 8-byte
 * aligned, caller-owned, not shared with a concurrent call.
 * Errors: GAR_EINVAL (P outside [1, 64], n < 1, NULL, t_p not positive,
 * workspace too small), GAR_EALIGN, GAR_ECUDA. */
int gar_rht_norm_range(const float *const *x, int32_t P, int64_t n, double t_p, float *d_mM,
                       void *d_workspace, size_t workspace_bytes, gar_stream_t stream);

/* gar_ef_apply -- x = grad + e, elementwise fp32 (one rounding).
 * gar_ef_update -- e = x - x_hat, elementwise fp32, where x_hat is the value
 * this worker's x came back as (its own quantized vector, decoded and
 * inverse-rotated).  Device pointers, n fp32 each, 4-byte aligned; the
 * output may be one of the inputs exactly, any other overlap is rejected;
 * n = 0 is a no-op.  Errors: GAR_EINVAL, GAR_EALIGN, GAR_ECUDA. */
int gar_ef_apply(const float *grad, const float *e, float *x, int64_t n, gar_stream_t stream);
int gar_ef_update(float *e, const float *x, const float *x_hat, int64_t n, gar_stream_t stream);

/* The same worker steps fused into the transform's own passes ([T] section
 * 5: error feedback, the randomized Hadamard transform, the norm-based
 * range, and the update of e from the worker's own quantized vector), so
 * that x = grad + e, the decoded own vector and x_hat are never written to
 * memory.  Results are bit for bit those of the separate calls named below. */

/* Tiles (4096 elements; 1 when n < 4096) of a transform of n elements: the
 * per-tile sums of squares gar_rht_ef_forward writes.  0 for a bad n. */
int64_t gar_rht_tiles(int64_t n);

/* gar_rht_ef_forward -- y = (1/sqrt(n)) H D (grad + e): bit for bit
 * gar_ef_apply(grad, e, x) then gar_rht(x, y, n, seed, 0), reading grad and
 * e once and writing y.  d_sumsq (device, gar_rht_tiles(n) doubles, 8-byte
 * aligned, or NULL): the sums of squares of x = grad + e per tile (fp32
 * squares summed pairwise, fp64 per tile), for gar_rht_norm_range_from_sums.
 * grad, e, y: device, n fp32, 16-byte aligned; y must not overlap grad or e.
 * n: a power of two, 1 <= n <= 2^31.
 * Errors: GAR_EINVAL (n, NULL, overlap), GAR_EALIGN, GAR_ECUDA. */
int gar_rht_ef_forward(const float *grad, const float *e, float *y, int64_t n, uint64_t seed,
                       double *d_sumsq, gar_stream_t stream);

/* gar_rht_norm_range_from_sums -- the norm-based range of gar_rht_norm_range
 * from the P workers' per-tile sums of squares (d_sumsq[w]: device,
 * gar_rht_tiles(n) doubles each, as gar_rht_ef_forward wrote them): each
 * worker's tiles added in a fixed order in fp64, the largest sum l^2 taken,
 * d_mM = (-M, M) with M = (t_p / sqrt(n)) l rounded to fp32.  Within 1e-6
 * relative of the exact value (the sums are ordered differently from
 * gar_rht_norm_range's, so the two may differ in the last bit).
 * Errors: GAR_EINVAL (P outside [1, 64], n, NULL, t_p not positive),
 * GAR_EALIGN, GAR_ECUDA. */
int gar_rht_norm_range_from_sums(const double *const *d_sumsq, int32_t P, int64_t n, double t_p,
                                 float *d_mM, gar_stream_t stream);

/* gar_rht_ef_update -- the worker's error-feedback update from its own wire
 * vector: e = (grad + e) - x_hat, x_hat = (1/sqrt(n)) D H y_hat, where
 * y_hat[i] = fma(S_i, (M - m) / steps, m) is the worker's own index i
 * decoded on the grid (S_i = table[idx_i] for non-uniform THC, idx_i for
 * uniform THC with table = NULL and steps = 2^b - 1).  Bit for bit
 * gar_nuhc_aggregate / gar_thc_aggregate of [packed] alone, then the decode
 * with P = 1, gar_rht(inverse), and gar_ef_update(e, gar_ef_apply(grad, e),
 * x_hat).  packed: device, the worker's gar_thc_words(n, b) words (4-byte
 * aligned); table: host, 2^b entries from 0 to steps, strictly increasing,
 * or NULL; d_mM: device [m, M]; grad, e: device, n fp32 (e read and
 * rewritten in place); tmp: device scratch of n fp32 for the transform's
 * intermediate passes (caller-owned, not shared with a concurrent call; its
 * contents after the call are undefined: where it is 128-byte aligned its
 * cache lines are dropped from L2 unwritten once read); grad, e, tmp
 * 16-byte aligned and pairwise disjoint.
 * Errors: GAR_EINVAL (n, b, steps, table, NULL, overlap), GAR_EALIGN,
 * GAR_ECUDA. */
int gar_rht_ef_update(const uint32_t *packed, int32_t b, int32_t steps, const uint16_t *table,
                      const float *d_mM, const float *grad, float *e, float *tmp, int64_t n, uint64_t seed,
                      gar_stream_t stream);

/* ===================================================================== */
/* NMSE [T] section 2: ||x - x_hat||^2 / ||x||^2                          */
/* ===================================================================== */

/* Bytes of device workspace gar_nmse needs for N elements. */
size_t gar_nmse_workspace_bytes(int64_t N);

/* gar_nmse -- *d_out (device, one double) = sum (x - x_hat)^2 / sum x^2,
 * NaN when sum x^2 = 0.  Per-element terms are formed in fp32 and summed in
 * fp64 in a fixed order (deterministic on a given GPU model: the order
 * follows the grid, one wave of the device's SMs; within 2e-6 relative of
 * an all-fp64 sum).  x, x_hat: device, N fp32.  d_workspace: device, at least
 * gar_nmse_workspace_bytes(N) bytes, 8-byte aligned, caller-owned, not
 * shared with a concurrent call.
 * Errors: GAR_EINVAL (null, N < 0, workspace too small), GAR_EALIGN,
 *         GAR_ECUDA. */
int gar_nmse(const float *x, const float *x_hat, int64_t N, double *d_out, void *d_workspace,
             size_t workspace_bytes, gar_stream_t stream);

/* gar_nmse_sums -- the two sums of NMSE ([T] section 2) over one range, not
 * divided: d_pair[0] = sum (x - x_hat)^2, d_pair[1] = sum x^2, with the
 * per-element terms and summation order of gar_nmse (gar_nmse_combine of this
 * one pair gives gar_nmse's result bit for bit).  NMSE over a vector held in
 * several ranges -- the fusion buffers of a plan, averaged one after another,
 * or the slices of a vector split across devices -- is gar_nmse_combine of
 * their pairs.  x, x_hat: device, N fp32 (4-byte aligned).  d_pair: device,
 * two doubles (8-byte aligned).  d_workspace: as for gar_nmse, not shared with
 * a concurrent call.
 * Errors: GAR_EINVAL (null, N < 0, workspace too small), GAR_EALIGN,
 *         GAR_ECUDA. */
int gar_nmse_sums(const float *x, const float *x_hat, int64_t N, double *d_pair, void *d_workspace,
                  size_t workspace_bytes, gar_stream_t stream);

/* gar_nmse_combine -- *d_out = (sum of d_pairs[2i]) / (sum of d_pairs[2i+1])
 * over i < n, each sum added in index order in fp64; NaN when the second sum
 * is 0.  d_pairs: device, n pairs from gar_nmse_sums (8-byte aligned).
 * Errors: GAR_EINVAL (n < 1, null), GAR_EALIGN, GAR_ECUDA. */
int gar_nmse_combine(const double *d_pairs, int32_t n, double *d_out, gar_stream_t stream);

/* gar_nmse_noalloc -- no counterpart in the pages: a library convenience.
 * The same NMSE as gar_nmse (same kernels, same summation order, same result)
 * for callers that cannot provide a workspace because they may not allocate
 * device memory themselves -- for instance a plug-in running inside a host
 * framework whose allocator owns all of the device's memory, or a
 * latency-critical path that must not pay cudaMalloc's implicit device-wide
 * synchronisation.  The caller still passes x, x_hat (device, N fp32) and
 * d_out (device, one double).  The call allocates nothing: the per-block
 * partial sums go to a fixed 16 KiB array inside the library (1024 pairs of
 * doubles; every GPU that loads the library holds it until the process
 * exits).  Every N >= 0 fits, because the reduction never uses more than 1024
 * blocks; a size needing more partial sums than the array holds would be
 * rejected with GAR_EINVAL.  The first call on a device looks up that array's
 * device address (cudaGetSymbolAddress) with the device current; make that
 * first call before any stream capture.  The address is kept for the life of
 * the process: after cudaDeviceReset() on a device the library's image is
 * loaded anew and the kept address is stale, so do not call this entry point
 * on that device again.  All calls on a device share the
 * array and it keeps the last call's contents (nothing in it needs to start
 * at zero); calls that overlap on the GPU, e.g. on two streams, race.
 * Errors: GAR_EINVAL (null, N < 0), GAR_EALIGN, GAR_ECUDA. */
int gar_nmse_noalloc(const float *x, const float *x_hat, int64_t N, double *d_out,
                     gar_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GAR_H */
