// thc_fused.cuh -- the fused THC kernels (encode every worker -> integer
// sum -> decode in one pass), over packed buffers and over a Tensor Fusion
// plan, and the index decision they share with the separate kernels of
// thc.cu ([T] section 4, Uniform THC / Algorithm 1; [H] "Tensor Fusion").
//
// The fused kernels are compiled once for any worker count (kP = 0) and once
// each for P = 4, 8, 16 and 64 (kP = P: the worker loop unrolled, its
// pointers and worker ids at fixed parameter offsets), each fixed count in a
// translation unit of its own (thc_p<P>.cu) so that the library builds in
// parallel.  Results do not depend on kP.
#pragma once

#include <cstdint>
#include <type_traits>

#include "common.cuh"

namespace gar {
namespace thc {

constexpr int kThreads = 256;

// The fused kernels' unit of work: E elements whose b-bit indices fill one
// store -- a whole 32-bit wire word for b >= 4 (E = 32 / b), 16 bits for
// b = 2 and 8 bits for b = 1 (E = 8, the registers of a b = 4 word).  The
// wire vectors keep their layout: unit u is bits [j E b, (j + 1) E b) of
// word u / (32 / (E b)), j = u mod (32 / (E b)), written as its own 8-, 16-
// or 32-bit slice (little endian); adjacent threads write the slices of one
// word.
template <int B>
constexpr int unit_elems() {
    return B >= 4 ? 32 / B : 8;
}
template <int B>
using UnitT = std::conditional_t<(B >= 4), uint32_t, std::conditional_t<(B == 2), uint16_t, uint8_t>>;
inline int unit_elems_of(int b) { return b >= 4 ? 32 / b : 8; }
// Units of the wire words of N elements (the last word's spare units too).
inline int64_t thc_units(int64_t words, int b) { return words * (32 / (unit_elems_of(b) * b)); }

// Resident CTAs per SM the fused kernels are compiled for (caps registers at
// 65536 / (256 * n)).
constexpr int kFusedMinBlocks = 4;
template <int B>
constexpr int fused_min_blocks() {
    return kFusedMinBlocks;
}

__device__ __forceinline__ float range_scale(float m, float M, float L) {
    return (M == m) ? 0.0f : __fdiv_rn(L, __fsub_rn(M, m));
}

// The index decision.  The grid position t = clamp((x - m) sc, 0, L) rounds
// up to j + 1 iff u < f (j = min(floor t, L - 1), f = t - j, u the 23-bit
// uniform), i.e. the index is ceil(t - u): for t < L, t - u = j + (f - u)
// with f - u in (-1, 1), whose ceiling is j + [u < f]; for t = L it is L.
// With 1 + u read as the float whose mantissa is the 23 random bits, two
// additions rounded up give it without any int <-> float conversion:
//   z = t - (1 + u), rounded up: ceil(z) = ceil(t - u) - 1, since rounding up
//       never passes an integer (every integer below 2^24 is a float);
//   z + 1.5 * 2^23, rounded up, lies in [2^23, 2^24), where the floats are
//       the integers, so it equals 1.5 * 2^23 + ceil(z) exactly.
// Its bit pattern is bits(1.5 * 2^23) + ceil(t - u) - 1: the index plus
// kIndexBias.  Callers sum and pack the biased values and remove the bias
// once per sum or word.
constexpr uint32_t kIndexBias = 0x4B3FFFFFu;  // bits(1.5 * 2^23) - 1
constexpr float kCeilMagic = 12582912.0f;     // 1.5 * 2^23

__device__ __forceinline__ uint32_t index_biased(float x, float m, float sc, float L, uint32_t r) {
    float t = __fmul_rn(__fsub_rn(x, m), sc);
    t = fminf(fmaxf(t, 0.0f), L);
    const float one_u = __uint_as_float((r & 0x007FFFFFu) | 0x3F800000u);
    return __float_as_uint(__fadd_ru(__fsub_ru(t, one_u), kCeilMagic));
}

// The same decision for two elements at once: the fp32 adds, subtracts and
// multiplies go through the packed f32x2 instructions (two IEEE binary32
// operations per instruction, each lane rounded exactly as the scalar
// operation, subnormals kept), halving their issue slots; min / max stay
// scalar.  Bit for bit equal to two index_biased calls.
__device__ __forceinline__ uint64_t pack_f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 unpack_f2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t sub_rn_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul_rn_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add_rm_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rm.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub_rp_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rp.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add_rp_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rp.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ void index_biased2(float x0, float x1, uint64_t m2, uint64_t sc2, float L, uint32_t r0,
                                              uint32_t r1, uint32_t &a0, uint32_t &a1) {
    float2 t = unpack_f2(mul_rn_f2(sub_rn_f2(pack_f2(x0, x1), m2), sc2));
    t.x = fminf(fmaxf(t.x, 0.0f), L);
    t.y = fminf(fmaxf(t.y, 0.0f), L);
    const uint64_t one_u = pack_f2(__uint_as_float((r0 & 0x007FFFFFu) | 0x3F800000u),
                                   __uint_as_float((r1 & 0x007FFFFFu) | 0x3F800000u));
    const float2 c = unpack_f2(add_rp_f2(sub_rp_f2(pack_f2(t.x, t.y), one_u), pack_f2(kCeilMagic, kCeilMagic)));
    a0 = __float_as_uint(c.x);
    a1 = __float_as_uint(c.y);
}

__device__ __forceinline__ uint4 philox_block(int64_t q, int worker, const PhiloxKeys &k) {
    return philox10(make_uint4(static_cast<uint32_t>(q), static_cast<uint32_t>(static_cast<uint64_t>(q) >> 32),
                               static_cast<uint32_t>(worker), 0u),
                    k);
}

// Sum over the 32/B fields of a packed word of (kIndexBias << field shift),
// mod 2^32: packing the biased indices with plain shifted adds and removing
// this once leaves the exact word (the fields never overlap).
template <int B, int E = 32 / B>
__host__ __device__ constexpr uint32_t pack_bias() {
    uint32_t s = 0;
    for (int i = 0; i < E; ++i) s += kIndexBias << (i * B);
    return s;
}

__device__ __forceinline__ uint32_t pick(const uint4 &r, int i) {
    return i == 0 ? r.x : (i == 1 ? r.y : (i == 2 ? r.z : r.w));
}

__device__ __forceinline__ float decode_step(const float *mM, float L, float fp, float &m) {
    m = mM[0];
    const float delta = __fdiv_rn(__fsub_rn(mM[1], m), L);
    return __fdiv_rn(delta, fp);
}
// S < 2^23: the float with mantissa S, minus 2^23, is S exactly
__device__ __forceinline__ float small_to_float(uint32_t s) {
    return __fsub_rn(__uint_as_float(0x4B000000u | s), 8388608.0f);
}


// ------------------------------------------------------------------ fused
struct FusedParams {
    PhiloxKeys keys;
    const float *x[GAR_MAX_WORKERS];    // the P contributing workers, slot by slot
    uint32_t *packed[GAR_MAX_WORKERS];  // all NULL when the wire vectors are not wanted
    int32_t wid[GAR_MAX_WORKERS];       // worker id of each slot (keys its Philox stream)
    const float *mM;
    float *avg;
    int64_t N;
    int64_t nunits;  // units of work: the wire words' units (see unit_elems)
    int32_t P;    // contributing workers (the decode divides by this)
    int32_t vec;  // inputs and avg 16-byte aligned
    float L;
    float fp;
};

// Constants of one launch: range, quantization scale, decode step.
struct Coder {
    float m, sc, k, km;
    uint64_t m2, sc2;  // (m, m) and (sc, sc) as f32x2 operands
    uint32_t bias;     // P * kIndexBias (mod 2^32): removed once from each index sum
};

__device__ __forceinline__ Coder make_coder_at(const float *mM, float L, float fp, int P) {
    Coder c;
    c.m = mM[0];
    c.sc = range_scale(c.m, mM[1], L);
    c.k = decode_step(mM, L, fp, c.km);
    c.bias = static_cast<uint32_t>(P) * kIndexBias;
    c.m2 = pack_f2(c.m, c.m);
    c.sc2 = pack_f2(c.sc, c.sc);
    return c;
}
template <class Prm>
__device__ __forceinline__ Coder make_coder(const Prm &p) {
    return make_coder_at(p.mM, p.L, p.fp, p.P);
}

// One worker's contribution to a unit of E = 4G elements: Philox draws,
// indices added to the running sums s, the packed slice stored if wanted.
template <int B, bool kPacked, int G, class Prm>
__device__ __forceinline__ void fused_one_worker(const float4 (&v)[G], uint32_t (&s)[4 * G], int64_t e0, int64_t w,
                                                 int wk, uint32_t *pk, const Prm &p, const Coder &c) {
    uint32_t word = 0;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 r = philox_block((e0 >> 2) + g, p.wid[wk], p.keys);
        uint32_t a0, a1, a2, a3;
        index_biased2(v[g].x, v[g].y, c.m2, c.sc2, p.L, r.x, r.y, a0, a1);
        index_biased2(v[g].z, v[g].w, c.m2, c.sc2, p.L, r.z, r.w, a2, a3);
        s[4 * g] += a0;
        s[4 * g + 1] += a1;
        s[4 * g + 2] += a2;
        s[4 * g + 3] += a3;
        if (kPacked)
            word += (a0 << (4 * g * B)) + (a1 << ((4 * g + 1) * B)) + (a2 << ((4 * g + 2) * B)) +
                    (a3 << ((4 * g + 3) * B));
    }
    if (kPacked)
        __stcs(reinterpret_cast<UnitT<B> *>(pk) + w, static_cast<UnitT<B>>(word - pack_bias<B, 4 * G>()));
}

template <int G>
__device__ __forceinline__ void load_group(float4 (&v)[G], const float *x) {
#pragma unroll
    for (int g = 0; g < G; ++g) v[g] = __ldcs(reinterpret_cast<const float4 *>(x) + g);
}

// Unit w (elements w*E .. w*E + E - 1) with every operand 16-byte aligned:
// worker slot wk's E inputs start at xs[wk] + xoff, the E averages go to avg.
// Two register buffers, the worker loop unrolled by two: one worker's loads
// are in flight while the other is quantized, with no copies.
// How far the worker loop (two workers an iteration) is unrolled: fully for
// a fixed count of up to 16 workers, partly for 64.
template <int B, int kP>
constexpr int fused_unroll() {
    if (kP == 0) return 1;
    return kP <= 16 ? 64 : 8;
}

// A thread's running sums for NMSE ([T] section 2) of the decoded average
// against a reference: sum (ref - avg)^2 and sum ref^2, fp32.
struct NmseAcc {
    float num = 0.0f, den = 0.0f;
};

// sum (r - a)^2 and sum r^2 over four lanes, pairwise
__device__ __forceinline__ void nmse_terms4(const float4 &r, const float4 &a, float &num, float &den) {
    const float d0 = __fsub_rn(r.x, a.x), d1 = __fsub_rn(r.y, a.y), d2 = __fsub_rn(r.z, a.z), d3 = __fsub_rn(r.w, a.w);
    num = __fadd_rn(__fadd_rn(__fmul_rn(d0, d0), __fmul_rn(d1, d1)), __fadd_rn(__fmul_rn(d2, d2), __fmul_rn(d3, d3)));
    den = __fadd_rn(__fadd_rn(__fmul_rn(r.x, r.x), __fmul_rn(r.y, r.y)), __fadd_rn(__fmul_rn(r.z, r.z), __fmul_rn(r.w, r.w)));
}

// kP > 0: the worker count is kP, known at compile time (the worker loop is
// unrolled, its pointers and worker ids taken at fixed parameter offsets);
// kP = 0: p.P.  kNmse: also add the word's NMSE terms against ref (the
// reference values of the same E elements) to acc.
template <int B, bool kPacked, int kP = 0, bool kNmse = false, class Prm>
__device__ __forceinline__ void fused_word_vec(const Prm &p, const Coder &c, const float *const *xs, int64_t xoff,
                                               uint32_t *const *pks, float *avg, int64_t w,
                                               const float *ref = nullptr, NmseAcc *acc = nullptr) {
    constexpr int E = unit_elems<B>();
    constexpr int G = E / 4;  // float4 groups (and Philox blocks) per unit
    const int P = kP > 0 ? kP : p.P;
    const int64_t e0 = w * E;
    uint32_t s[E];
#pragma unroll
    for (int i = 0; i < E; ++i) s[i] = 0;
    float4 va[G], vb[G];
    load_group(va, xs[0] + xoff);
    float4 rv[kNmse ? G : 1];  // the reference values, in flight while the last workers are quantized
#pragma unroll(fused_unroll<B, kP>())
    for (int wk = 0; wk < P; wk += 2) {
        const bool has1 = wk + 1 < P;
        if constexpr (kNmse) {
            if (wk + 2 >= P) load_group(rv, ref);
        }
        if (has1) load_group(vb, xs[wk + 1] + xoff);
        fused_one_worker<B, kPacked>(va, s, e0, w, wk, kPacked ? pks[wk] : nullptr, p, c);
        if (wk + 2 < P) load_group(va, xs[wk + 2] + xoff);
        if (has1) fused_one_worker<B, kPacked>(vb, s, e0, w, wk + 1, kPacked ? pks[wk + 1] : nullptr, p, c);
    }
    float4 *dst = reinterpret_cast<float4 *>(avg);
    float num = 0.0f, den = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float4 a = make_float4(__fmaf_rn(small_to_float(s[4 * g] - c.bias), c.k, c.km),
                                     __fmaf_rn(small_to_float(s[4 * g + 1] - c.bias), c.k, c.km),
                                     __fmaf_rn(small_to_float(s[4 * g + 2] - c.bias), c.k, c.km),
                                     __fmaf_rn(small_to_float(s[4 * g + 3] - c.bias), c.k, c.km));
        __stcs(dst + g, a);
        if constexpr (kNmse) {
            float n4, d4;
            nmse_terms4(rv[g], a, n4, d4);
            num = g == 0 ? n4 : __fadd_rn(num, n4);
            den = g == 0 ? d4 : __fadd_rn(den, d4);
        }
    }
    if constexpr (kNmse) {
        acc->num = __fadd_rn(acc->num, num);
        acc->den = __fadd_rn(acc->den, den);
    }
}

// One CTA per tile of 2 * kThreads units (two per thread): the block
// scheduler hands tiles to the SMs as they free up, which left fewer SMs idle
// than a resident grid striding over the units (P=16, b=4, 2^24: 0.265 ->
// 0.232 ms).
template <int B, bool kPacked, int kP>
__global__ void __launch_bounds__(kThreads, fused_min_blocks<B>()) thc_fused_kernel(const __grid_constant__ FusedParams p) {
    constexpr int E = unit_elems<B>();
    constexpr int G = E / 4;
    const Coder c = make_coder(p);
    const int64_t w_first = static_cast<int64_t>(blockIdx.x) * (2 * kThreads) + threadIdx.x;
#pragma unroll 1
    for (int u = 0; u < 2; ++u) {
        const int64_t w = w_first + u * kThreads;
        if (w >= p.nunits) break;
        const int64_t e0 = w * E;
        if (p.vec && e0 + E <= p.N) {
            fused_word_vec<B, kPacked, kP>(p, c, p.x, e0, p.packed, p.avg + e0, w);
        } else {  // ragged last word, or unaligned inputs: element by element
            uint32_t s[E];
#pragma unroll
            for (int i = 0; i < E; ++i) s[i] = 0;
            for (int wk = 0; wk < p.P; ++wk) {
                uint32_t word = 0;
                for (int g = 0; g < G; ++g) {
                    const int64_t eb = e0 + 4 * g;
                    if (eb >= p.N) break;
                    const uint4 r = philox_block(eb >> 2, p.wid[wk], p.keys);
                    for (int i = 0; i < 4 && eb + i < p.N; ++i) {
                        const uint32_t a = index_biased(p.x[wk][eb + i], c.m, c.sc, p.L, pick(r, i));
                        s[4 * g + i] += a;
                        word |= (a - kIndexBias) << ((4 * g + i) * B);
                    }
                }
                if (kPacked) reinterpret_cast<UnitT<B> *>(p.packed[wk])[w] = static_cast<UnitT<B>>(word);
            }
            for (int i = 0; i < E && e0 + i < p.N; ++i) {
                // elements never visited above kept s = 0; only in-range ones are stored
                p.avg[e0 + i] = __fmaf_rn(small_to_float(s[i] - c.bias), c.k, c.km);
            }
        }
    }
}

// ------------------------------------------- fused over a Tensor Fusion plan
// THC of one fusion buffer read straight from the workers' tensors ([H]
// "Tensor Fusion" with [T] Algorithm 1 on the fused buffer): element e of the
// buffer is element e - begin of the tensor whose slot [begin, end) holds it,
// or 0 in an alignment gap -- exactly the packed buffer's contents -- and its
// Philox draw is keyed by e, so indices, index sums, packed words and
// averages equal those of gar_thc_allreduce_fused over the packed buffer bit
// for bit.  The average of every tensor element goes straight to the output
// tensor (the unpack); gap elements are not written anywhere.
//
// Work decomposition (made on the host): a launch covers runs of words
// ("spans") of one or more fusion buffers, each with its own range and wire
// vectors.  A span's words are cut into pieces -- runs of whole words inside
// one tensor (loaded with 16-byte vectors when every pointer of the tensor is
// 16-byte aligned), and runs of the words between them (a tensor's first and
// last word shared with a neighbour or a gap, the buffer's ragged last word)
// taken element by element.  Pieces are cut into tiles of kPlanTileWords
// words, one CTA per tile; the piece of a tile, and so its buffer, range and
// coder, is found once per tile, uniform over the CTA.  Several buffers in one
// launch let a stream of small partitions (THC's 4 MB partitions, each with
// its own range) fill the GPU in one launch.
constexpr int kPlanSrcPtrs = 1792, kPlanPkPtrs = 256, kPlanSegs = 128, kPlanPieces = 2 * kPlanSegs + 1;
constexpr int kPlanBufs = 64;
// Words per tile: two per thread, so that the per-CTA set-up (the range's
// divisions, the piece search) is paid once per 2 x P x E element-workers.
constexpr int kPlanTileWords = 2 * kThreads;
constexpr int kPieceVec = 0, kPieceTensor = 1, kPieceMixed = 2;

struct PlanSeg {
    int64_t begin;  // first buffer element of the tensor
    int64_t end;    // one past its last
};

struct PlanPiece {
    int64_t w0, w1;  // words [w0, w1) of its buffer
    int32_t seg;     // the tensor holding every element of the words (kPieceVec, kPieceTensor), else -1
    int16_t kind;    // kPieceVec: 16-byte vectors; kPieceTensor: one tensor, element by element;
                     // kPieceMixed: each element looked up (tensor, gap or past the end)
    int16_t buf;     // its span: p.buf[buf]
};

struct PlanBuf {
    int64_t N;               // elements of the fusion buffer
    int32_t id;              // the buffer's index in the plan: its range is mM[2 id], mM[2 id + 1]
    int16_t seg_lo, seg_hi;  // the span's tensors: seg[seg_lo .. seg_hi), sorted by begin
    int32_t pk;              // its wire vectors: packed[pk + slot] (packed launches)
    int32_t pad;
};

struct ThcPlanParams {
    PhiloxKeys keys;
    int32_t wid[GAR_MAX_WORKERS];
    const float *mM;                         // the plan's ranges, two floats per fusion buffer
    int64_t total_tiles;
    int32_t P, nseg, npieces, nbuf;
    float L, fp;
    PlanBuf buf[kPlanBufs];
    PlanSeg seg[kPlanSegs];                  // every tensor meeting the launch's words, by span
    float *out[kPlanSegs];                   // output tensor of each segment
    const float *ref[kPlanSegs];             // NMSE reference tensor of each segment (NMSE launches)
    double *nmse_ws;                         // NMSE launches: this launch's per-CTA pairs of sums
    int64_t tile_start[kPlanPieces + 1];     // first tile of each piece; [npieces] = total
    PlanPiece piece[kPlanPieces];
    const float *src[kPlanSrcPtrs];          // src[k * P + slot]: worker slot's tensor of segment k
    uint32_t *packed[kPlanPkPtrs];           // packed[buf.pk + slot]: worker slot's wire vector of a span's buffer
};
static_assert(sizeof(ThcPlanParams) <= 32000, "plan parameters exceed the launch limit");

// Segment of buffer bf holding its element e, or -1 in a gap.
__device__ __forceinline__ int plan_find(const ThcPlanParams &p, const PlanBuf &bf, int64_t e) {
    int lo = bf.seg_lo, hi = bf.seg_hi - 1;
    if (hi < lo || p.seg[lo].begin > e) return -1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].begin <= e) lo = mid;
        else hi = mid - 1;
    }
    return e < p.seg[lo].end ? lo : -1;
}

// The buffer's ragged last unit (e0 + E > N), element by element: the
// missing elements pack as zero bits and get no output.
template <int B, bool kPacked, bool kNmse>
__device__ __noinline__ void plan_word_ragged(const ThcPlanParams &p, const PlanBuf &bf, const Coder &c, int64_t w,
                                              NmseAcc &acc) {
    constexpr int E = unit_elems<B>();
    constexpr int G = E / 4;
    const int64_t e0 = w * E;
    uint32_t s[E];
    for (int i = 0; i < E; ++i) s[i] = 0;
    for (int wk = 0; wk < p.P; ++wk) {
        uint32_t word = 0;
        for (int g = 0; g < G; ++g) {
            const int64_t eb = e0 + 4 * g;
            if (eb >= bf.N) break;
            const uint4 r = philox_block(eb >> 2, p.wid[wk], p.keys);
            for (int i = 0; i < 4 && eb + i < bf.N; ++i) {
                const int64_t e = eb + i;
                const int k = plan_find(p, bf, e);
                const float x = k < 0 ? 0.0f : p.src[k * p.P + wk][e - p.seg[k].begin];
                const uint32_t a = index_biased(x, c.m, c.sc, p.L, pick(r, i));
                s[4 * g + i] += a;
                word |= (a - kIndexBias) << ((4 * g + i) * B);
            }
        }
        if (kPacked) reinterpret_cast<UnitT<B> *>(p.packed[bf.pk + wk])[w] = static_cast<UnitT<B>>(word);
    }
    for (int i = 0; i < E && e0 + i < bf.N; ++i) {
        const int64_t e = e0 + i;
        const int k = plan_find(p, bf, e);
        if (k < 0) continue;
        const float a = __fmaf_rn(small_to_float(s[i] - c.bias), c.k, c.km);
        p.out[k][e - p.seg[k].begin] = a;
        if (kNmse) {
            const float r = p.ref[k][e - p.seg[k].begin], d = __fsub_rn(r, a);
            acc.num = __fadd_rn(acc.num, __fmul_rn(d, d));
            acc.den = __fadd_rn(acc.den, __fmul_rn(r, r));
        }
    }
}

// A whole word (e0 + E <= N) read element by element: a word shared by two
// tensors or a tensor and a gap (seg < 0: each element's tensor looked up
// once), or a word of a tensor whose pointers are not 16-byte aligned
// (seg >= 0).  Each worker's E values are gathered with independent loads,
// then quantized as a vector word.  Kept out of line: it serves only the few
// words at tensor ends and gaps, and the unaligned tensors.
template <int B, bool kPacked, bool kNmse>
__device__ __noinline__ void plan_word_gather(const ThcPlanParams &p, const PlanBuf &bf, const Coder &c, int64_t w,
                                              int seg, NmseAcc &acc) {
    constexpr int E = unit_elems<B>();
    constexpr int G = E / 4;
    const int64_t e0 = w * E;
    int ks[E];
    int64_t off[E];
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const int k = seg >= 0 ? seg : plan_find(p, bf, e0 + i);
        ks[i] = k;
        off[i] = k >= 0 ? e0 + i - p.seg[k].begin : 0;
    }
    uint32_t s[E];
#pragma unroll
    for (int i = 0; i < E; ++i) s[i] = 0;
    for (int wk = 0; wk < p.P; ++wk) {
        float x[E];
#pragma unroll
        for (int i = 0; i < E; ++i) x[i] = ks[i] >= 0 ? __ldcs(p.src[ks[i] * p.P + wk] + off[i]) : 0.0f;
        float4 v[G];
#pragma unroll
        for (int g = 0; g < G; ++g) v[g] = make_float4(x[4 * g], x[4 * g + 1], x[4 * g + 2], x[4 * g + 3]);
        fused_one_worker<B, kPacked>(v, s, e0, w, wk, kPacked ? p.packed[bf.pk + wk] : nullptr, p, c);
    }
#pragma unroll
    for (int i = 0; i < E; ++i) {
        if (ks[i] < 0) continue;
        const float a = __fmaf_rn(small_to_float(s[i] - c.bias), c.k, c.km);
        __stcs(p.out[ks[i]] + off[i], a);
        if (kNmse) {
            const float r = __ldcs(p.ref[ks[i]] + off[i]), d = __fsub_rn(r, a);
            acc.num = __fadd_rn(acc.num, __fmul_rn(d, d));
            acc.den = __fadd_rn(acc.den, __fmul_rn(r, r));
        }
    }
}

// kNmse: every CTA also writes its pair of NMSE sums (fp32 per thread and
// across a warp, fp64 across the warps in a fixed order) to
// p.nmse_ws[2 * blockIdx.x], p.nmse_ws[2 * blockIdx.x + 1].
template <int B, bool kPacked, int kP, bool kNmse>
__global__ void __launch_bounds__(kThreads, fused_min_blocks<B>()) thc_fused_plan_kernel(const __grid_constant__ ThcPlanParams p) {
    constexpr int E = unit_elems<B>();
    const int P = kP > 0 ? kP : p.P;
    NmseAcc acc;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        // the piece that owns tile t: largest i with tile_start[i] <= t (uniform per CTA)
        int lo = 0, hi = p.npieces - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.tile_start[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        const PlanPiece pc = p.piece[lo];
        const PlanBuf &bf = p.buf[pc.buf];
        const Coder c = make_coder_at(p.mM + 2 * bf.id, p.L, p.fp, P);
        const int64_t w0 = pc.w0 + (t - p.tile_start[lo]) * kPlanTileWords + threadIdx.x;
#pragma unroll 1
        for (int u = 0; u < kPlanTileWords / kThreads; ++u) {
            const int64_t w = w0 + u * kThreads;
            if (w >= pc.w1) break;
            if (pc.kind == kPieceVec) {
                const int64_t off = w * E - p.seg[pc.seg].begin;
                fused_word_vec<B, kPacked, kP, kNmse>(p, c, p.src + pc.seg * P, off, p.packed + bf.pk,
                                                      p.out[pc.seg] + off, w, kNmse ? p.ref[pc.seg] + off : nullptr,
                                                      &acc);
            } else if ((w + 1) * E <= bf.N) {
                plan_word_gather<B, kPacked, kNmse>(p, bf, c, w, pc.kind == kPieceTensor ? pc.seg : -1, acc);
            } else {
                plan_word_ragged<B, kPacked, kNmse>(p, bf, c, w, acc);
            }
        }
    }
    if constexpr (kNmse) {
        __shared__ float s_num[kThreads / 32], s_den[kThreads / 32];
        float num = acc.num, den = acc.den;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            num = __fadd_rn(num, __shfl_xor_sync(0xFFFFFFFFu, num, o));
            den = __fadd_rn(den, __shfl_xor_sync(0xFFFFFFFFu, den, o));
        }
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (lane == 0) {
            s_num[warp] = num;
            s_den[warp] = den;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            double dn = 0.0, dd = 0.0;
#pragma unroll
            for (int i = 0; i < kThreads / 32; ++i) {
                dn += static_cast<double>(s_num[i]);
                dd += static_cast<double>(s_den[i]);
            }
            p.nmse_ws[2 * blockIdx.x] = dn;
            p.nmse_ws[2 * blockIdx.x + 1] = dd;
        }
    }
}

template <typename K>
int grid_for(K kernel, int64_t work_items) {
    if (work_items <= 0) return 0;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0) != cudaSuccess || occ <= 0) occ = 2;
    int64_t g = static_cast<int64_t>(sm_count()) * occ;
    const int64_t need = ceil_div(work_items, kThreads);
    if (g > need) g = need;
    return static_cast<int>(g > 0 ? g : 1);
}


// Launchers: kernel grid (one CTA per tile of 2 * kThreads words), dispatch
// on b and on whether wire vectors are written.  kP = 0: any worker count;
// kP > 0: p.P == kP.
template <int kP>
int launch_fused(const FusedParams &p, int b, bool packed, cudaStream_t stream) {
#define GAR_FUSED_CASE(BB)                                                                                \
    case BB:                                                                                              \
        if (packed)                                                                                       \
            thc_fused_kernel<BB, true, kP><<<static_cast<unsigned>(ceil_div(p.nunits, 2 * kThreads)), kThreads, 0, \
                                             stream>>>(p);                                                \
        else                                                                                              \
            thc_fused_kernel<BB, false, kP><<<static_cast<unsigned>(ceil_div(p.nunits, 2 * kThreads)), kThreads, \
                                              0, stream>>>(p);                                            \
        break;
    switch (b) {
        GAR_FUSED_CASE(1)
        GAR_FUSED_CASE(2)
        GAR_FUSED_CASE(4)
        GAR_FUSED_CASE(8)
    }
#undef GAR_FUSED_CASE
    return check_launch("thc_fused_kernel");
}

// CTAs a plan launch runs (one per tile).
inline unsigned plan_grid(const ThcPlanParams &p) {
    return static_cast<unsigned>(p.total_tiles < 0x7FFFFFFF ? p.total_tiles : 0x7FFFFFFF);
}

template <int kP>
int launch_fused_plan(const ThcPlanParams &p, int b, bool packed, bool nmse, cudaStream_t stream) {
    if (p.total_tiles <= 0) return GAR_OK;
    // one CTA per tile: the block scheduler balances the SMs (see the ring kernel)
    const unsigned grid = plan_grid(p);
#define GAR_PLAN_KERNEL(BB, PK, NM) thc_fused_plan_kernel<BB, PK, kP, NM><<<grid, kThreads, 0, stream>>>(p)
#define GAR_PLAN_CASE(BB)                                                           \
    case BB:                                                                        \
        if (nmse) {                                                                 \
            if (packed) GAR_PLAN_KERNEL(BB, true, true);                            \
            else GAR_PLAN_KERNEL(BB, false, true);                                  \
        } else {                                                                    \
            if (packed) GAR_PLAN_KERNEL(BB, true, false);                           \
            else GAR_PLAN_KERNEL(BB, false, false);                                 \
        }                                                                           \
        break;
    switch (b) {
        GAR_PLAN_CASE(1)
        GAR_PLAN_CASE(2)
        GAR_PLAN_CASE(4)
        GAR_PLAN_CASE(8)
    }
#undef GAR_PLAN_CASE
#undef GAR_PLAN_KERNEL
    return check_launch("thc_fused_plan_kernel");
}

// the fixed worker counts live in thc_p4.cu, thc_p8.cu, thc_p16.cu, thc_p64.cu
extern template int launch_fused<4>(const FusedParams &, int, bool, cudaStream_t);
extern template int launch_fused<8>(const FusedParams &, int, bool, cudaStream_t);
extern template int launch_fused<16>(const FusedParams &, int, bool, cudaStream_t);
extern template int launch_fused<64>(const FusedParams &, int, bool, cudaStream_t);
extern template int launch_fused_plan<4>(const ThcPlanParams &, int, bool, bool, cudaStream_t);
extern template int launch_fused_plan<8>(const ThcPlanParams &, int, bool, bool, cudaStream_t);
extern template int launch_fused_plan<16>(const ThcPlanParams &, int, bool, bool, cudaStream_t);
extern template int launch_fused_plan<64>(const ThcPlanParams &, int, bool, bool, cudaStream_t);

// Index widths the packing supports.
inline bool valid_b(int b) { return b == 1 || b == 2 || b == 4 || b == 8; }

// The decode avg = m + (M - m)/steps * sums/P on a grid of `steps` steps
// (uniform THC: steps = 2^b - 1; non-uniform: the granularity g); arguments
// already checked by the caller.
int launch_grid_decode(const uint16_t *sums, int64_t N, const float *d_mM, int steps, int P, float *avg,
                       cudaStream_t stream);

}  // namespace thc
}  // namespace gar
