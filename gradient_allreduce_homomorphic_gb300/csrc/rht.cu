// rht.cu -- THC's pre- and post-processing ([T] section 5): the randomized
// Hadamard transform (1/sqrt(n)) H D x and its inverse (1/sqrt(n)) D H y,
// the norm-based range M = (t_p / sqrt(n)) max_w ||x_w||, m = -M, and the
// error-feedback updates x = grad + e and e = x - x_hat.
//
// The fast Walsh-Hadamard transform of n = 2^k elements is k butterfly
// stages ((a, b) -> (a + b, a - b) between elements whose indices differ in
// one bit); stages on different bits commute, so they may run in any order.
//
// Stages on index bits 0..11 run inside 4096-element tiles (one read and one
// write of HBM): a thread holds 16 elements (coalesced float4 loads give it
// bits 0, 1, 10, 11 in registers), does those four stages in registers, and
// two swizzled shared-memory transposes bring bits 2..5 and then 6..9 into
// its registers.  Higher bits go in passes of up to eight: a CTA holds 256
// rows of 16 consecutive elements, the rows 2^s apart (64-byte segments:
// whole DRAM sectors), and does the row bits in two register rounds around
// one transpose.  For n = 2^21 .. 2^24 one cluster pass does all the bits
// above 11 (clusters of up to 16 CTAs exchanging rows through distributed
// shared memory), so these sizes take two kernels, as does n = 2^20; larger
// n take the passes of eight (2^28: three kernels).
//
// The Rademacher signs D come from their own Philox stream (worker slot
// 0xFFFFFFFF): one 128-bit block per 128 elements, bit i mod 128 for
// element i.  The forward transform applies them as the first tile kernel
// loads; the inverse applies them as the last kernel stores.
#include <atomic>
#include <cmath>
#include <cstring>
#include <memory>

#include "common.cuh"

namespace gar {
namespace {

constexpr int kTile = 4096;  // elements per tile / per pass block
constexpr int kThreads = 256;
constexpr uint32_t kSignSlot = 0xFFFFFFFFu;

__device__ __forceinline__ uint4 sign_block(int64_t q, const PhiloxKeys &k) {
    return philox10(make_uint4(static_cast<uint32_t>(q), static_cast<uint32_t>(static_cast<uint64_t>(q) >> 32),
                               kSignSlot, 0u),
                    k);
}
__device__ __forceinline__ uint32_t word_of(const uint4 &b, int w) {
    return w == 0 ? b.x : (w == 1 ? b.y : (w == 2 ? b.z : b.w));
}

__device__ __forceinline__ uint64_t pair_bits(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void bits_pair(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

// L2 priorities of the transform's intermediate vector: the passes before the
// last write it with an evict-last policy (the next launch reads it back, so
// it should stay in L2 while the streams around it pass through) and the
// next launch reads it with an evict-first one (it is read once).
__device__ __forceinline__ uint64_t l2_keep_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_once_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_policy(float *a, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(a), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ float ld_policy(const float *a, uint64_t pol) {
    float v;
    asm volatile("ld.global.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(a), "l"(pol) : "memory");
    return v;
}

// Butterfly stages over v[0..15] on the register-index bits >= lo_bit.  The
// stages on bits 1..3 take the neighbouring registers (v[r], v[r + 1]) as
// one f32x2 operand (each lane rounded as the scalar add or subtract), two
// butterflies per instruction; bit 0 pairs the neighbours themselves and
// stays scalar.
__device__ __forceinline__ void butterfly16(float (&v)[16], int lo_bit = 0) {
    if (lo_bit <= 0) {
#pragma unroll
        for (int r = 0; r < 16; r += 2) {
            const float a = v[r], b = v[r + 1];
            v[r] = __fadd_rn(a, b);
            v[r + 1] = __fsub_rn(a, b);
        }
    }
#pragma unroll
    for (int bit = 1; bit < 4; ++bit) {
        if (bit < lo_bit) continue;
        const int h = 1 << bit;
#pragma unroll
        for (int r = 0; r < 16; r += 2) {
            if ((r & h) == 0) {
                const uint64_t a = pair_bits(v[r], v[r + 1]), b = pair_bits(v[r + h], v[r + h + 1]);
                uint64_t sum, dif;
                asm("add.rn.f32x2 %0, %1, %2;" : "=l"(sum) : "l"(a), "l"(b));
                asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dif) : "l"(a), "l"(b));
                bits_pair(sum, v[r], v[r + 1]);
                bits_pair(dif, v[r + h], v[r + h + 1]);
            }
        }
    }
}

struct RhtParams {
    PhiloxKeys keys;
    const float *in;
    float *out;
    int64_t n;
    int32_t inverse;  // 0: (1/sqrt n) H D x;  1: (1/sqrt n) D H y
    int32_t last;     // this launch writes the final values (scale, inverse signs)
    int32_t s;        // pass: log2 of the row stride
    int32_t lo_bit;   // pass: row bits below this were done by an earlier launch
    float scale;      // 1/sqrt(n) rounded to fp32
    // fused error feedback and decode (see the kIn / kEfOut kernel variants)
    const float *grad;       // kInEf: the input is grad + in; kEfOut: e = (grad + e) - result
    float *ef;               // kEfOut: the error vector e, read and rewritten
    const uint32_t *packed;  // kInPacked: a worker's b-bit indices
    const float *mM;         // kInPacked: their range [m, M]
    double *sumsq;           // kNorm: one sum of squares of the input per tile
    int32_t b;               // kInPacked: bits per index
    int32_t has_tab;         // kInPacked: index z stands for tab[z] (non-uniform THC), else for z
    float steps;             // kInPacked: grid steps between m and M (2^b - 1, or the granularity g)
    int32_t b_log;           // kInPacked: log2 b (indices per word 32 / b = 2^(5 - b_log))
    int32_t discard_in;      // kEfOut: the scratch p.out (128-byte aligned) may leave L2 unwritten once read
    uint16_t tab[256];       // kInPacked with has_tab: the table T
};

// What the first launch of a transform reads: the vector itself; grad + e
// (error feedback applied on the way in); or a worker's packed indices,
// decoded on the grid (its own quantized vector).
constexpr int kInPlain = 0, kInEf = 1, kInPacked = 2;

// Per-CTA set-up of the kInPacked decode: the table values as floats, and
// the decode step (M - m) / steps divided by one worker, as the grid decode
// takes them.
struct Decoder {
    float m, k;
};
__device__ __forceinline__ Decoder make_decoder(const RhtParams &p, float *s_tab) {
    if (p.has_tab)
        for (int z = threadIdx.x; z <= (1 << p.b) - 1; z += blockDim.x) s_tab[z] = static_cast<float>(p.tab[z]);
    Decoder d;
    d.m = p.mM[0];
    d.k = __fdiv_rn(__fdiv_rn(__fsub_rn(p.mM[1], d.m), p.steps), 1.0f);
    return d;
}
// The decoded value of index z: fma(S, k, m), S = tab[z] or z (exact floats).
__device__ __forceinline__ float decode_one(const RhtParams &p, const Decoder &d, const float *s_tab, uint32_t z) {
    const float S = p.has_tab ? s_tab[z] : static_cast<float>(z);
    return __fmaf_rn(S, d.k, d.m);
}
// Word of element e and the bit offset of its index in it (b a power of two:
// shifts, no division).
__device__ __forceinline__ uint32_t packed_word(const RhtParams &p, int64_t e, int &sh) {
    const int per_log = 5 - p.b_log;
    sh = static_cast<int>(e & ((int64_t{1} << per_log) - 1)) << p.b_log;
    return __ldcs(p.packed + (e >> per_log));
}
// Elements e .. e + 3 (e a multiple of 4) decoded from the packed indices.
__device__ __forceinline__ float4 decode4(const RhtParams &p, const Decoder &d, const float *s_tab, int64_t e) {
    int sh;
    const uint32_t w = packed_word(p, e, sh);
    const uint32_t mask = (1u << p.b) - 1u;
    return make_float4(decode_one(p, d, s_tab, (w >> sh) & mask), decode_one(p, d, s_tab, (w >> (sh + p.b)) & mask),
                       decode_one(p, d, s_tab, (w >> (sh + 2 * p.b)) & mask),
                       decode_one(p, d, s_tab, (w >> (sh + 3 * p.b)) & mask));
}
// Element i decoded from the packed indices.
__device__ __forceinline__ float decode_at(const RhtParams &p, const Decoder &d, const float *s_tab, int64_t i) {
    int sh;
    const uint32_t w = packed_word(p, i, sh);
    return decode_one(p, d, s_tab, (w >> sh) & ((1u << p.b) - 1u));
}

// e = (grad + e) - y for one element: the error-feedback update with x
// recomputed as gar_ef_apply forms it.
__device__ __forceinline__ void ef_out(const RhtParams &p, int64_t i, float y) {
    p.ef[i] = __fsub_rn(__fadd_rn(__ldcs(p.grad + i), p.ef[i]), y);
}

// Sum of squares of a thread's 16 values (fp32, pairwise), added over the
// CTA in fp64 in a fixed order; written by thread 0 to p.sumsq[tile].
__device__ __forceinline__ void tile_sumsq(const RhtParams &p, const float (&v)[16], int64_t tile) {
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fadd_rn(__fmul_rn(v[2 * i], v[2 * i]), __fmul_rn(v[2 * i + 1], v[2 * i + 1]));
    const float f = __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                              __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
    double a = static_cast<double>(f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
    __shared__ double s_part[kThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) s_part[warp] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
#pragma unroll
        for (int i = 0; i < kThreads / 32; ++i) t += s_part[i];
        p.sumsq[tile] = t;
    }
}

// Tile shared-memory layout: element i of the tile lives at i ^ (bits 6..8
// of i moved to bits 2..4).  Every warp access below then hits 32 distinct
// banks, and 16-byte groups stay whole for the float4 stores.
__device__ __forceinline__ int tile_swz(int i) { return i ^ (((i >> 6) & 7) << 2); }

// Index bits 0..11 of every 4096-element tile.  kIn: what the tile reads
// (the vector, grad + e, or packed indices to decode); kNorm: also the sum of
// squares of what it read, per tile; kEfOut (with p.last): instead of the
// result y, write e = (grad + e) - y.
template <int kIn, bool kNorm, bool kEfOut>
__global__ void __launch_bounds__(kThreads) rht_tile_kernel(const __grid_constant__ RhtParams p) {
    __shared__ __align__(16) float s[kTile];
    __shared__ uint32_t s_sign[kTile / 32];  // bit i: sign of tile element i (1 = negative)
    __shared__ float s_tab[kIn == kInPacked ? 256 : 1];
    const int t = threadIdx.x;
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kTile;
    float v[16];
    // v[4q + j] = tile element (q << 10) | (t << 2) | j
    if constexpr (kIn == kInPacked) {
        const Decoder d = make_decoder(p, s_tab);
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 a = decode4(p, d, s_tab, base + (q << 10) + (t << 2));
            v[4 * q] = a.x;
            v[4 * q + 1] = a.y;
            v[4 * q + 2] = a.z;
            v[4 * q + 3] = a.w;
        }
    } else {
        const float4 *src = reinterpret_cast<const float4 *>(p.in + base);
        const float4 *gsrc = reinterpret_cast<const float4 *>(kIn == kInEf ? p.grad + base : p.in + base);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float4 a = __ldcs(src + q * 256 + t);
            if constexpr (kIn == kInEf) {  // x = grad + e, as gar_ef_apply forms it
                const float4 gv = __ldcs(gsrc + q * 256 + t);
                a = make_float4(__fadd_rn(gv.x, a.x), __fadd_rn(gv.y, a.y), __fadd_rn(gv.z, a.z), __fadd_rn(gv.w, a.w));
            }
            v[4 * q] = a.x;
            v[4 * q + 1] = a.y;
            v[4 * q + 2] = a.z;
            v[4 * q + 3] = a.w;
        }
    }
    if constexpr (kNorm) tile_sumsq(p, v, blockIdx.x);
    const bool signs_in = !p.inverse;
    const bool signs_out = p.inverse && p.last;
    if (signs_in || signs_out) {
        if (t < kTile / 128) {
            const uint4 r = sign_block((base >> 7) + t, p.keys);
            s_sign[4 * t] = r.x;
            s_sign[4 * t + 1] = r.y;
            s_sign[4 * t + 2] = r.z;
            s_sign[4 * t + 3] = r.w;
        }
        __syncthreads();
    }
    if (signs_in) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t bits = s_sign[32 * q + (t >> 3)] >> (4 * (t & 7));
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if ((bits >> j) & 1u) v[4 * q + j] = -v[4 * q + j];
        }
    }
    butterfly16(v);  // bits 0, 1, 10, 11
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<float4 *>(&s[tile_swz((q << 10) | (t << 2))]) =
            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    __syncthreads();
    if constexpr (kEfOut && kIn == kInPlain) {
        // the last kernel of the update reads the scratch intermediate
        // (p.in == p.out == tmp) once, all of this tile by now: its dirty
        // lines leave L2 without being written back to DRAM.  (Where the
        // tile kernel is the only kernel, n = 4096, it decodes the packed
        // indices and there is no intermediate.)
        if (p.discard_in && t < kTile * 4 / 128)
            asm volatile("discard.global.L2 [%0], 128;" ::"l"(p.in + base + 32 * t) : "memory");
    }
    // bits 2..5 in registers: element (t & 3) | (r << 2) | ((t >> 2) << 6)
    const int b1 = (t & 3) | ((t >> 2) << 6);
#pragma unroll
    for (int r = 0; r < 16; ++r) v[r] = s[tile_swz(b1 | (r << 2))];
    butterfly16(v);
#pragma unroll
    for (int r = 0; r < 16; ++r) s[tile_swz(b1 | (r << 2))] = v[r];
    __syncthreads();
    // bits 6..9 in registers: element (t & 63) | (r << 6) | ((t >> 6) << 10)
    const int b2 = (t & 63) | ((t >> 6) << 10);
    float xr[kEfOut ? 16 : 1];  // kEfOut: x = grad + e of the elements this thread writes, loaded early
    if constexpr (kEfOut) {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int64_t i = base + (b2 | (r << 6));
            xr[r] = __fadd_rn(__ldcs(p.grad + i), p.ef[i]);
        }
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) v[r] = s[tile_swz(b2 | (r << 6))];
    butterfly16(v);
    float *dst = p.out + base;
    const uint64_t keep = l2_keep_policy();
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int e = b2 | (r << 6);
        float y = v[r];
        if (p.last) {
            if (signs_out && ((s_sign[e >> 5] >> (e & 31)) & 1u)) y = -y;
            y = __fmul_rn(y, p.scale);
        }
        if constexpr (kEfOut) __stcs(p.ef + base + e, __fsub_rn(xr[r], y));  // e = (grad + e) - x_hat
        else if (p.last) __stcs(dst + e, y);
        else st_policy(dst + e, y, keep);  // the next pass reads it back
    }
}

// Row bits [lo_bit, 8) of 256 rows 2^s apart (s >= 4), 16 columns each,
// read from p.in (kIn = kInPlain; p.in == p.out in place) or decoded from
// p.packed (kInPacked), written to p.out; with p.last scaled by 1/sqrt(n).
// Block -> (hi, column block cb): element of (row m, column c) =
// (hi << (s + 8)) | (m << s) | (cb << 4) | c.  Shared layout: row-major
// m * 16 + c with bit 8 folded into bit 4 (conflict-free both rounds).
__device__ __forceinline__ int pass_swz(int i) { return i ^ (((i >> 8) & 1) << 4); }

template <int kIn>
__global__ void __launch_bounds__(kThreads) rht_pass_kernel(const __grid_constant__ RhtParams p) {
    __shared__ float s[kTile];
    __shared__ float s_tab[kIn == kInPacked ? 256 : 1];
    const int t = threadIdx.x;
    const int c = t & 15, mh = t >> 4;
    const int64_t bid = blockIdx.x;
    const int cb_bits = p.s - 4;
    const int64_t cb = bid & ((int64_t{1} << cb_bits) - 1);
    const int64_t hi = bid >> cb_bits;
    const int64_t col0 = (hi << (p.s + 8)) | (cb << 4) | c;
    float v[16];
    // first stage: rows (mh << 4) | j
    if constexpr (kIn == kInPacked) {
        const Decoder d = make_decoder(p, s_tab);
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = decode_at(p, d, s_tab, col0 + (static_cast<int64_t>((mh << 4) | j) << p.s));
    } else {
        const float *x = p.in + col0;
        const uint64_t once = l2_once_policy();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = ld_policy(x + (static_cast<int64_t>((mh << 4) | j) << p.s), once);
    }
    butterfly16(v, p.lo_bit);
#pragma unroll
    for (int j = 0; j < 16; ++j) s[pass_swz((mh << 8) | (j << 4) | c)] = v[j];
    __syncthreads();
    // second stage: rows (j << 4) | mh
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = s[pass_swz((j << 8) | (mh << 4) | c)];
    butterfly16(v, p.lo_bit > 4 ? p.lo_bit - 4 : 0);
    float *y = p.out + col0;
    const uint64_t keep = l2_keep_policy();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int64_t off = static_cast<int64_t>((j << 4) | mh) << p.s;
        if (p.last) __stcs(y + off, __fmul_rn(v[j], p.scale));
        else st_policy(y + off, v[j], keep);  // the next launch reads it back
    }
}

// Row bits [0, 8 + RB) of 2^(8+RB) rows 2^s apart (s >= 12), 16 columns each,
// in place on p.out, by a cluster of K = 2^RB CTAs: the CTA of cluster rank q
// holds rows (q << 8) | m (m < 256) and does their bits 0..7 as
// rht_pass_kernel does, keeping the result in its shared memory; after a
// cluster barrier every thread takes positions (m, c) and reads that
// position from all K CTAs' shared memory (distributed shared memory), does
// the stages of row bits 8.. on the K values and stores rows (r << 8) | m.
// Cluster id -> (hi, column block cb): element of (row m, column c) =
// (hi << (s + 8 + RB)) | (m << s) | (cb << 4) | c.  With 16-CTA clusters one
// launch covers twelve index bits, so n = 2^21 .. 2^24 take two kernels.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The exit barrier orders nothing but the other CTAs' reads of this CTA's
// shared memory, which completed when their values arrived in registers: a
// relaxed arrive, so that the thread need not wait for its global stores.
__device__ __forceinline__ void cluster_sync_exit() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_cluster(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    return remote;
}
__device__ __forceinline__ float ld_cluster(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}

// The cluster pass always starts at index bit 12 (the tile pass has done bits
// 0..11) and n <= 2^24, so its row stride 2^12 is a constant and every
// element offset fits 32 bits: the 16 strided loads of a thread are one
// base register and immediate offsets.  kLast: this launch writes the final
// (scaled) values.
constexpr int kClusterRowBit = 12;

template <int RB, int kIn, bool kLast>
__global__ void __launch_bounds__(kThreads) rht_cluster_pass_kernel(const __grid_constant__ RhtParams p) {
    constexpr int K = 1 << RB;
    constexpr int S = kClusterRowBit;
    __shared__ float s[kTile];
    __shared__ float s_tab[kIn == kInPacked ? 256 : 1];
    const int t = threadIdx.x;
    const int c = t & 15, mh = t >> 4;
    const uint32_t q = cluster_rank();
    const int cid = static_cast<int>(blockIdx.x >> RB);
    const int cb = cid & ((1 << (S - 4)) - 1);
    const int hi = cid >> (S - 4);
    const int base = (hi << (S + 8 + RB)) | (cb << 4);  // row 0, column 0 of the cluster's block
    const int col0 = base + (static_cast<int>(q) << (S + 8)) + c;
    float v[16];
    if constexpr (kIn == kInPacked) {
        const Decoder d = make_decoder(p, s_tab);
        __syncthreads();
        // rows 2^12 apart hold their indices at the same bit offset of
        // words 2^(12 - log2(32 / b)) apart
        const int per_log = 5 - p.b_log;
        const int sh = (col0 & ((1 << per_log) - 1)) << p.b_log;
        const uint32_t mask = (1u << p.b) - 1u;
        const uint32_t *wp = p.packed + ((col0 + (mh << (S + 4))) >> per_log);
        const int wstride = 1 << (S - per_log);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = decode_one(p, d, s_tab, (__ldcs(wp + j * wstride) >> sh) & mask);
    } else {
        const float *x = p.in + (col0 + (mh << (S + 4)));
        const uint64_t once = l2_once_policy();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = ld_policy(x + (j << S), once);
    }
    butterfly16(v);
#pragma unroll
    for (int j = 0; j < 16; ++j) s[pass_swz((mh << 8) | (j << 4) | c)] = v[j];
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = s[pass_swz((j << 8) | (mh << 4) | c)];
    butterfly16(v);
#pragma unroll
    for (int j = 0; j < 16; ++j) s[pass_swz((j << 8) | (mh << 4) | c)] = v[j];
    cluster_sync_all();  // every CTA's rows are done and visible to the cluster
    // the cluster-window address of every CTA's array; an offset within the
    // array adds to it as to a local address
    uint32_t rbase[K];
    {
        const uint32_t s_addr = static_cast<uint32_t>(__cvta_generic_to_shared(s));
#pragma unroll
        for (int r = 0; r < K; ++r) rbase[r] = map_cluster(s_addr, r);
    }
#pragma unroll 1
    for (int i = 0; i < 16 / K; ++i) {
        const int pos = i * (K * 256) + static_cast<int>(q) * 256 + t;  // (m, c) = (pos >> 4, pos & 15)
        const int m = pos >> 4;
        float w[K];
#pragma unroll
        for (int r = 0; r < K; ++r) w[r] = ld_cluster(rbase[r] + 4u * static_cast<uint32_t>(pass_swz(pos)));
        // the K-point butterflies, paired in f32x2 from the second stage on
#pragma unroll
        for (int r = 0; r < K; r += 2) {
            const float a = w[r], b = w[r + 1];
            w[r] = __fadd_rn(a, b);
            w[r + 1] = __fsub_rn(a, b);
        }
#pragma unroll
        for (int h = 2; h < K; h <<= 1) {
#pragma unroll
            for (int r = 0; r < K; r += 2) {
                if ((r & h) == 0) {
                    const uint64_t a = pair_bits(w[r], w[r + 1]), b = pair_bits(w[r + h], w[r + h + 1]);
                    uint64_t sum, dif;
                    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(sum) : "l"(a), "l"(b));
                    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dif) : "l"(a), "l"(b));
                    bits_pair(sum, w[r], w[r + 1]);
                    bits_pair(dif, w[r + h], w[r + h + 1]);
                }
            }
        }
        float *y = p.out + (base + c + (m << S));
        const uint64_t keep = l2_keep_policy();
#pragma unroll
        for (int r = 0; r < K; ++r) {
            float *dst = y + (r << (S + 8));
            if constexpr (kLast) __stcs(dst, __fmul_rn(w[r], p.scale));
            else st_policy(dst, w[r], keep);  // the next launch reads it back
        }
    }
    cluster_sync_exit();  // no CTA leaves while another still reads its shared memory
}

// The cluster pass saves a launch where the vector stays in L2 between the
// launches (2^21: 0.0205 -> 0.0167 ms, 2^22: 0.027 -> 0.021, 2^24: equal);
// for vectors larger than L2 its barrier waits cost more than the extra plain
// pass (2^26: 0.25 -> 0.30 ms), so it serves n <= 2^24 only.
constexpr int kClusterMaxBits = 24;

// Launches the cluster pass with 2^RB-CTA clusters and sets *launched; where
// clusters of that size cannot be scheduled on this device (probed once) it
// launches nothing and returns GAR_OK with *launched false, and the caller
// takes the plain passes instead.
template <int RB, int kIn, bool kLast>
int launch_cluster_pass_as(const RhtParams &p, unsigned blocks, cudaStream_t stream, bool *launched) {
    static std::atomic<int> ok[64];  // 0: not probed, 1: schedulable, 2: not
    int dev = 0;
    *launched = false;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GAR_OK;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1u << RB;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int state = ok[dev].load(std::memory_order_relaxed);
    if (state == 0) {
        int clusters = 0;
        bool good = true;
        if (RB > 3)  // 16 CTAs: above the portable cluster size
            good = cudaFuncSetAttribute(rht_cluster_pass_kernel<RB, kIn, kLast>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        bool refused = !good;
        if (good) {
            refused = cudaOccupancyMaxActiveClusters(&clusters, rht_cluster_pass_kernel<RB, kIn, kLast>, &cfg) !=
                      cudaSuccess;
            good = !refused && clusters > 0;
        }
        if (refused) cudaGetLastError();  // a refused probe leaves no error behind
        state = good ? 1 : 2;
        ok[dev].store(state, std::memory_order_relaxed);
    }
    if (state != 1) return GAR_OK;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, rht_cluster_pass_kernel<RB, kIn, kLast>, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(GAR_ECUDA, "rht_cluster_pass_kernel: %s", cudaGetErrorString(e));
    }
    *launched = true;
    return check_launch("rht_cluster_pass_kernel");
}

// Launches the cluster pass with 2^RB-CTA clusters and sets *launched; where
// clusters of that size cannot be scheduled on this device (probed once) it
// launches nothing and returns GAR_OK with *launched false, and the caller
// takes the plain passes instead.  The pass must start at index bit 12.
template <int RB, int kIn>
int launch_cluster_pass(const RhtParams &p, unsigned blocks, cudaStream_t stream, bool *launched) {
    *launched = false;
    if (p.s != kClusterRowBit || p.n > (int64_t{1} << kClusterMaxBits)) return GAR_OK;
    return p.last ? launch_cluster_pass_as<RB, kIn, true>(p, blocks, stream, launched)
                  : launch_cluster_pass_as<RB, kIn, false>(p, blocks, stream, launched);
}

// n < 4096: one CTA, every stage in shared memory (the same kIn, kNorm and
// kEfOut variants as the tile kernel).
template <int kIn, bool kNorm, bool kEfOut>
__global__ void __launch_bounds__(kThreads) rht_small_kernel(const __grid_constant__ RhtParams p) {
    __shared__ float s[kTile];
    __shared__ float s_tab[kIn == kInPacked ? 256 : 1];
    const int n = static_cast<int>(p.n);
    Decoder d{0.0f, 0.0f};
    if constexpr (kIn == kInPacked) {
        d = make_decoder(p, s_tab);
        __syncthreads();
    }
    float sq = 0.0f;  // kNorm: this thread's squares, in element order
    for (int i = threadIdx.x; i < n; i += kThreads) {
        float x;
        if constexpr (kIn == kInPacked) {
            x = decode_at(p, d, s_tab, i);
        } else if constexpr (kIn == kInEf) {
            x = __fadd_rn(p.grad[i], p.in[i]);
        } else {
            x = p.in[i];
        }
        if (kNorm) sq = __fadd_rn(sq, __fmul_rn(x, x));
        if (!p.inverse && ((word_of(sign_block(i >> 7, p.keys), (i >> 5) & 3) >> (i & 31)) & 1u)) x = -x;
        s[i] = x;
    }
    if constexpr (kNorm) {
        double a = static_cast<double>(sq);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        __shared__ double s_part[kThreads / 32];
        if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = a;
        __syncthreads();
        if (threadIdx.x == 0) {
            double t = 0.0;
            for (int i = 0; i < kThreads / 32; ++i) t += s_part[i];
            p.sumsq[0] = t;
        }
    }
    __syncthreads();
    for (int h = 1; h < n; h <<= 1) {
        for (int j = threadIdx.x; j < n / 2; j += kThreads) {
            const int i = (j / h) * 2 * h + (j % h);
            const float a = s[i], b = s[i + h];
            s[i] = __fadd_rn(a, b);
            s[i + h] = __fsub_rn(a, b);
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < n; i += kThreads) {
        float y = s[i];
        if (p.inverse && ((word_of(sign_block(i >> 7, p.keys), (i >> 5) & 3) >> (i & 31)) & 1u)) y = -y;
        y = __fmul_rn(y, p.scale);
        if constexpr (kEfOut) ef_out(p, i, y);
        else p.out[i] = y;
    }
}

// ------------------------------------------------------------ norm range
constexpr int kNormBlocksMax = 256;  // per worker

struct NormParams {
    const float *x[GAR_MAX_WORKERS];
    double *ws;  // [P][blocks] partial sums of squares
    float *mM;
    int64_t n;
    int32_t P;
    int32_t blocks;
    double t_over_sqrt_n;
};

__device__ __forceinline__ double block_sum(double v) {
    __shared__ double s_v[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // s_v may still be read by a previous call
    if (lane == 0) s_v[warp] = v;
    __syncthreads();
    v = 0.0;
    if (warp == 0) {
        v = lane < kThreads / 32 ? s_v[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    }
    return v;  // valid in thread 0
}

__device__ __forceinline__ float sq4(const float4 &a) {
    return __fadd_rn(__fadd_rn(__fmul_rn(a.x, a.x), __fmul_rn(a.y, a.y)), __fadd_rn(__fmul_rn(a.z, a.z), __fmul_rn(a.w, a.w)));
}

// Partial sums of squares: grid (blocks, P).  Terms are formed in fp32 four
// at a time and accumulated in fp64 in a fixed order (deterministic).
__global__ void __launch_bounds__(kThreads) rht_norm_partial(const __grid_constant__ NormParams p) {
    const float *x = p.x[blockIdx.y];
    double acc = 0.0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    int64_t first = 0;
    if ((reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        // four vectors a step (i + k * stride: coalesced, all in flight), their
        // sixteen squares summed pairwise in fp32 before one fp64 add: fp64 runs
        // at a small fraction of the fp32 rate here, and one add per four
        // elements bounded the kernel (relative error of a step's sum < 3e-7)
        const int64_t nv = p.n / 4;
        const float4 *xv = reinterpret_cast<const float4 *>(x);
        int64_t i = tid;
        for (; i + 3 * stride < nv; i += 4 * stride) {
            float4 a[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) a[k] = __ldcs(xv + i + k * stride);
            acc += static_cast<double>(__fadd_rn(__fadd_rn(sq4(a[0]), sq4(a[1])), __fadd_rn(sq4(a[2]), sq4(a[3]))));
        }
        for (; i < nv; i += stride) acc += static_cast<double>(sq4(__ldcs(xv + i)));
        first = nv * 4;
    }
    for (int64_t i = first + tid; i < p.n; i += stride) {
        const float a = x[i];
        acc += static_cast<double>(__fmul_rn(a, a));
    }
    acc = block_sum(acc);
    if (threadIdx.x == 0) p.ws[static_cast<int64_t>(blockIdx.y) * p.blocks + blockIdx.x] = acc;
}

// max over workers of the summed partials -> (m, M)
__global__ void __launch_bounds__(kThreads) rht_norm_final(const __grid_constant__ NormParams p) {
    double best = 0.0;
    for (int w = 0; w < p.P; ++w) {
        double acc = 0.0;
        for (int b = threadIdx.x; b < p.blocks; b += kThreads) acc += p.ws[static_cast<int64_t>(w) * p.blocks + b];
        acc = block_sum(acc);
        if (threadIdx.x == 0 && acc > best) best = acc;
    }
    if (threadIdx.x == 0) {
        const float M = static_cast<float>(p.t_over_sqrt_n * sqrt(best));
        p.mM[0] = -M;
        p.mM[1] = M;
    }
}

// The range from per-tile sums of squares (gar_rht_ef_forward's): each
// worker's tiles added in a fixed order (fp64), the largest sum taken.
struct SumsRangeParams {
    const double *sums[GAR_MAX_WORKERS];
    float *mM;
    int64_t tiles;
    int32_t P;
    int32_t pad;
    double t_over_sqrt_n;
};

// One CTA per worker: each thread adds a fixed stride of the worker's tiles
// (four loads in flight), the CTA adds the threads' sums in a fixed order
// (fp64), and the worker's M = (t_p / sqrt(n)) l goes into d_mM by atomic
// max / min on the float bits (M >= 0: the bit patterns order as the values;
// the result does not depend on the order of the CTAs).  rht_range_init sets
// d_mM to (+0, +0) first.
constexpr int kRangeThreads = 1024;
__global__ void rht_range_init(float *mM) {
    mM[0] = 0.0f;
    mM[1] = 0.0f;
}

__global__ void __launch_bounds__(kRangeThreads) rht_range_from_sums(const __grid_constant__ SumsRangeParams p) {
    __shared__ double s_part[kRangeThreads / 32];
    const double *x = p.sums[blockIdx.x];
    double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
    int64_t i = threadIdx.x;
    constexpr int T = kRangeThreads;
    for (; i + 3 * T < p.tiles; i += 4 * T) {
        a0 += x[i];
        a1 += x[i + T];
        a2 += x[i + 2 * T];
        a3 += x[i + 3 * T];
    }
    for (; i < p.tiles; i += T) a0 += x[i];
    double acc = (a0 + a1) + (a2 + a3);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) s_part[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double l2 = 0.0;
        for (int w = 0; w < kRangeThreads / 32; ++w) l2 += s_part[w];
        const float M = static_cast<float>(p.t_over_sqrt_n * sqrt(l2));
        atomicMax(reinterpret_cast<int *>(p.mM + 1), __float_as_int(M));
        atomicMax(reinterpret_cast<unsigned int *>(p.mM), __float_as_uint(-M));  // negative floats: larger bits, smaller value
    }
}

int norm_blocks(int64_t n) {
    int64_t b = ceil_div(n, 4 * 2048);
    if (b > kNormBlocksMax) b = kNormBlocksMax;
    return static_cast<int>(b < 1 ? 1 : b);
}

// CTAs per worker of a launch: at most norm_blocks(n) (the workspace bound),
// and at most one resident wave over all P workers, so that no SM idles in a
// partial second wave (P=8, 2^24: 256 per worker were 1.7 waves).
int norm_grid(int64_t n, int P) {
    static std::atomic<int> cached[64];
    int dev = 0;
    int wave = kNormBlocksMax * 8;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        wave = cached[dev].load(std::memory_order_relaxed);
        if (wave == 0) {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rht_norm_partial, kThreads, 0) != cudaSuccess ||
                per_sm < 1)
                per_sm = 1;
            wave = sm_count() * per_sm;
            cached[dev].store(wave, std::memory_order_relaxed);
        }
    }
    const int per_worker = wave / P > 1 ? wave / P : 1;
    const int cap = norm_blocks(n);
    return cap < per_worker ? cap : per_worker;
}

// ---------------------------------------------------------- error feedback
// out = a + b (Sub = false) or a - b (Sub = true), one rounding each.
template <bool Sub>
__device__ __forceinline__ float ef_op(float a, float b) {
    return Sub ? __fsub_rn(a, b) : __fadd_rn(a, b);
}

template <bool Sub>
__global__ void __launch_bounds__(kThreads) ef_kernel(const float *a, const float *b, float *out, int64_t n, int vec) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    int64_t first = 0;
    if (vec) {
        const int64_t nv = n / 4;
        for (int64_t i = tid; i < nv; i += stride) {
            const float4 u = __ldcs(reinterpret_cast<const float4 *>(a) + i);
            const float4 w = __ldcs(reinterpret_cast<const float4 *>(b) + i);
            __stcs(reinterpret_cast<float4 *>(out) + i, make_float4(ef_op<Sub>(u.x, w.x), ef_op<Sub>(u.y, w.y),
                                                                    ef_op<Sub>(u.z, w.z), ef_op<Sub>(u.w, w.w)));
        }
        first = nv * 4;
    }
    for (int64_t i = first + tid; i < n; i += stride) out[i] = ef_op<Sub>(a[i], b[i]);
}

int ew_grid(int64_t items) {
    int64_t g = static_cast<int64_t>(sm_count()) * 8;
    const int64_t need = ceil_div(items, kThreads);
    if (g > need) g = need;
    return static_cast<int>(g < 1 ? 1 : g);
}

bool overlaps(const void *a, const void *b, int64_t bytes) {
    const char *x = static_cast<const char *>(a), *y = static_cast<const char *>(b);
    return x < y + bytes && y < x + bytes;
}

}  // namespace
}  // namespace gar

using namespace gar;

namespace gar {
namespace {

template <int kIn, bool kNorm, bool kEfOut>
int launch_first(const RhtParams &p, unsigned blocks, bool small, cudaStream_t stream) {
    if (small) {
        rht_small_kernel<kIn, kNorm, kEfOut><<<1, kThreads, 0, stream>>>(p);
        return check_launch("rht_small_kernel");
    }
    rht_tile_kernel<kIn, kNorm, kEfOut><<<blocks, kThreads, 0, stream>>>(p);
    return check_launch("rht_tile_kernel");
}

// Passes over index bits 12..k-1: for n <= 2^24, nine to twelve of them at
// once by a cluster pass where the clusters can be scheduled; else (and for
// the last eight or fewer) in passes of eight.  A plain pass that would run
// past bit k-1 is moved down (s = k - 8) and skips the row bits already
// done.  The first of them reads as kIn says (p.in, or p.packed); the others
// work in place on p.out.  fin: the last of them writes the final values.
template <int kIn>
int run_passes(const RhtParams &p0, int k, unsigned blocks, bool fin, cudaStream_t stream) {
    std::unique_ptr<RhtParams> q(new RhtParams(p0));
    int rc = GAR_OK;
    bool first = true;
    for (int done = 12; done < k && rc == GAR_OK; first = false) {
        if (!first) q->in = q->out;
        const int left = k - done;
        if (left > 8 && k <= kClusterMaxBits) {
            const int rb = left >= 12 ? 4 : left - 8;
            q->s = done;
            q->lo_bit = 0;
            q->last = fin && done + 8 + rb >= k ? 1 : 0;
            bool launched = false;
            if (first) {
                switch (rb) {
                    case 1: rc = launch_cluster_pass<1, kIn>(*q, blocks, stream, &launched); break;
                    case 2: rc = launch_cluster_pass<2, kIn>(*q, blocks, stream, &launched); break;
                    case 3: rc = launch_cluster_pass<3, kIn>(*q, blocks, stream, &launched); break;
                    default: rc = launch_cluster_pass<4, kIn>(*q, blocks, stream, &launched); break;
                }
            } else {
                switch (rb) {
                    case 1: rc = launch_cluster_pass<1, kInPlain>(*q, blocks, stream, &launched); break;
                    case 2: rc = launch_cluster_pass<2, kInPlain>(*q, blocks, stream, &launched); break;
                    case 3: rc = launch_cluster_pass<3, kInPlain>(*q, blocks, stream, &launched); break;
                    default: rc = launch_cluster_pass<4, kInPlain>(*q, blocks, stream, &launched); break;
                }
            }
            if (launched || rc != GAR_OK) {
                done += 8 + rb;
                continue;
            }
        }
        q->s = done < k - 8 ? done : k - 8;
        q->lo_bit = done - q->s;
        q->last = fin && q->s + 8 >= k ? 1 : 0;
        if (first) rht_pass_kernel<kIn><<<blocks, kThreads, 0, stream>>>(*q);
        else rht_pass_kernel<kInPlain><<<blocks, kThreads, 0, stream>>>(*q);
        rc = check_launch("rht_pass_kernel");
        done = q->s + 8;
    }
    return rc;
}

// The whole transform of p.n = 2^k elements.  The butterfly stages of
// different index bits commute, so the forward transform takes the
// 4096-element tiles (bits 0..11) first -- they apply the signs as they read,
// with error feedback (kInEf) and the norm's sums (kNorm) -- and the passes
// over the higher bits after, the last of them scaling; the inverse takes
// the passes first (reading p.in, or decoding p.packed) and the tiles last,
// where the signs, the scale and, with kEfOut, the error-feedback update are
// applied as contiguous tiles are written.
template <int kIn, bool kNorm, bool kEfOut>
int rht_run(RhtParams &p, cudaStream_t stream) {
    const int64_t n = p.n;
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(n)));
    int k = 0;
    while ((int64_t{1} << k) < n) ++k;
    if (n < kTile) {
        p.last = 1;
        return launch_first<kIn, kNorm, kEfOut>(p, 1, true, stream);
    }
    const unsigned blocks = static_cast<unsigned>(n / kTile);
    if (!p.inverse) {
        if constexpr (kEfOut) return fail(GAR_EINVAL, "the forward transform writes no error feedback");
        p.last = k == 12 ? 1 : 0;
        int rc = launch_first<kIn, kNorm, false>(p, blocks, false, stream);
        if (rc || k == 12) return rc;
        RhtParams &q = p;
        q.in = q.out;
        return run_passes<kInPlain>(q, k, blocks, true, stream);
    }
    if constexpr (kIn == kInEf || kNorm) return fail(GAR_EINVAL, "the inverse reads no error feedback and takes no norm");
    if (k == 12) {
        p.last = 1;
        return launch_first<kIn, false, kEfOut>(p, blocks, false, stream);
    }
    int rc = run_passes<kIn>(p, k, blocks, false, stream);
    if (rc) return rc;
    p.in = p.out;
    p.last = 1;
    p.s = 0;
    p.lo_bit = 0;
    return launch_first<kInPlain, false, kEfOut>(p, blocks, false, stream);
}

int check_n(int64_t n) {
    if (n < 1 || (n & (n - 1)) != 0) return fail(GAR_EINVAL, "n=%lld is not a power of two", static_cast<long long>(n));
    if (n > (int64_t{1} << 31)) return fail(GAR_EINVAL, "n=%lld above 2^31", static_cast<long long>(n));
    return GAR_OK;
}

}  // namespace
}  // namespace gar

extern "C" int gar_rht(const float *in, float *out, int64_t n, uint64_t seed, int32_t inverse, gar_stream_t stream_) {
    int rc = check_n(n);
    if (rc) return rc;
    if (!in || !out) return fail(GAR_EINVAL, "in or out is NULL");
    if (inverse != 0 && inverse != 1) return fail(GAR_EINVAL, "inverse must be 0 or 1");
    if (!aligned(in, 16) || !aligned(out, 16)) return fail(GAR_EALIGN, "in and out must be 16-byte aligned");
    if (in != out && overlaps(in, out, n * 4)) return fail(GAR_EINVAL, "in and out overlap without being equal");
    std::unique_ptr<RhtParams> p(new RhtParams);
    std::memset(p.get(), 0, sizeof(RhtParams));
    p->keys = philox_keys(seed);
    p->in = in;
    p->out = out;
    p->n = n;
    p->inverse = inverse;
    return rht_run<kInPlain, false, false>(*p, reinterpret_cast<cudaStream_t>(stream_));
}

extern "C" int64_t gar_rht_tiles(int64_t n) {
    if (check_n(n) != GAR_OK) return 0;
    return n < kTile ? 1 : n / kTile;
}

extern "C" int gar_rht_ef_forward(const float *grad, const float *e, float *y, int64_t n, uint64_t seed,
                                  double *d_sumsq, gar_stream_t stream_) {
    int rc = check_n(n);
    if (rc) return rc;
    if (!grad || !e || !y) return fail(GAR_EINVAL, "grad, e or y is NULL");
    if (!aligned(grad, 16) || !aligned(e, 16) || !aligned(y, 16))
        return fail(GAR_EALIGN, "grad, e and y must be 16-byte aligned");
    if (d_sumsq && !aligned(d_sumsq, 8)) return fail(GAR_EALIGN, "d_sumsq not 8-byte aligned");
    if (overlaps(y, grad, n * 4) || overlaps(y, e, n * 4)) return fail(GAR_EINVAL, "y overlaps grad or e");
    std::unique_ptr<RhtParams> p(new RhtParams);
    std::memset(p.get(), 0, sizeof(RhtParams));
    p->keys = philox_keys(seed);
    p->in = e;
    p->grad = grad;
    p->out = y;
    p->n = n;
    p->sumsq = d_sumsq;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    return d_sumsq ? rht_run<kInEf, true, false>(*p, stream) : rht_run<kInEf, false, false>(*p, stream);
}

extern "C" int gar_rht_ef_update(const uint32_t *packed, int32_t b, int32_t steps, const uint16_t *table,
                                 const float *d_mM, const float *grad, float *e, float *tmp, int64_t n,
                                 uint64_t seed, gar_stream_t stream_) {
    int rc = check_n(n);
    if (rc) return rc;
    if (b != 1 && b != 2 && b != 4 && b != 8) return fail(GAR_EINVAL, "b=%d not in {1, 2, 4, 8}", b);
    const int L = (1 << b) - 1;
    if (!packed || !d_mM || !grad || !e || !tmp) return fail(GAR_EINVAL, "NULL argument");
    if (!table && steps != L) return fail(GAR_EINVAL, "without a table the grid has 2^b - 1 = %d steps, not %d", L, steps);
    if (table) {
        if (table[0] != 0 || table[L] != steps) return fail(GAR_EINVAL, "table must start at 0 and end at %d", steps);
        for (int z = 0; z < L; ++z)
            if (table[z + 1] <= table[z]) return fail(GAR_EINVAL, "table not strictly increasing at %d", z);
    }
    if (steps < 1) return fail(GAR_EINVAL, "steps=%d < 1", steps);
    if (!aligned(packed, 4) || !aligned(d_mM, 4) || !aligned(grad, 16) || !aligned(e, 16) || !aligned(tmp, 16))
        return fail(GAR_EALIGN, "misaligned pointer (grad, e and tmp: 16 bytes; packed, d_mM: 4)");
    if (overlaps(tmp, grad, n * 4) || overlaps(tmp, e, n * 4) || overlaps(e, grad, n * 4))
        return fail(GAR_EINVAL, "tmp, grad and e must not overlap");
    std::unique_ptr<RhtParams> p(new RhtParams);
    std::memset(p.get(), 0, sizeof(RhtParams));
    p->keys = philox_keys(seed);
    p->out = tmp;
    p->n = n;
    p->inverse = 1;
    p->grad = grad;
    p->ef = e;
    p->packed = packed;
    p->mM = d_mM;
    p->b = b;
    p->b_log = b == 1 ? 0 : (b == 2 ? 1 : (b == 4 ? 2 : 3));
    p->steps = static_cast<float>(steps);
    p->has_tab = table ? 1 : 0;
    p->discard_in = aligned(tmp, 128) ? 1 : 0;
    if (table)
        for (int z = 0; z <= L; ++z) p->tab[z] = table[z];
    return rht_run<kInPacked, false, true>(*p, reinterpret_cast<cudaStream_t>(stream_));
}

extern "C" int gar_rht_norm_range_from_sums(const double *const *d_sumsq, int32_t P, int64_t n, double t_p,
                                            float *d_mM, gar_stream_t stream_) {
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    int rc = check_n(n);
    if (rc) return rc;
    if (!d_sumsq || !d_mM) return fail(GAR_EINVAL, "NULL argument");
    if (!(t_p > 0.0) || !std::isfinite(t_p)) return fail(GAR_EINVAL, "t_p must be positive and finite");
    if (!aligned(d_mM, 4)) return fail(GAR_EALIGN, "d_mM not 4-byte aligned");
    SumsRangeParams p;
    std::memset(&p, 0, sizeof(p));
    for (int w = 0; w < P; ++w) {
        if (!d_sumsq[w] || !aligned(d_sumsq[w], 8)) return fail(GAR_EINVAL, "sums of worker %d NULL or misaligned", w);
        p.sums[w] = d_sumsq[w];
    }
    p.P = P;
    p.tiles = gar_rht_tiles(n);
    p.mM = d_mM;
    p.t_over_sqrt_n = t_p / std::sqrt(static_cast<double>(n));
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    rht_range_init<<<1, 1, 0, stream>>>(d_mM);
    rc = check_launch("rht_range_init");
    if (rc) return rc;
    rht_range_from_sums<<<static_cast<unsigned>(P), kRangeThreads, 0, stream>>>(p);
    return check_launch("rht_range_from_sums");
}

extern "C" size_t gar_rht_norm_range_workspace_bytes(int32_t P, int64_t n) {
    if (P < 1 || P > GAR_MAX_WORKERS || n < 0) return 0;
    return static_cast<size_t>(P) * static_cast<size_t>(norm_blocks(n)) * sizeof(double);
}

extern "C" int gar_rht_norm_range(const float *const *x, int32_t P, int64_t n, double t_p, float *d_mM,
                                  void *d_workspace, size_t workspace_bytes, gar_stream_t stream_) {
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (n < 1) return fail(GAR_EINVAL, "n=%lld < 1", static_cast<long long>(n));
    if (!x || !d_mM || !d_workspace) return fail(GAR_EINVAL, "NULL argument");
    if (!(t_p > 0.0) || !std::isfinite(t_p)) return fail(GAR_EINVAL, "t_p must be positive and finite");
    const size_t need = gar_rht_norm_range_workspace_bytes(P, n);
    if (workspace_bytes < need) return fail(GAR_EINVAL, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
    if (!aligned(d_workspace, 8) || !aligned(d_mM, 4)) return fail(GAR_EALIGN, "misaligned workspace or d_mM");
    NormParams p;
    std::memset(&p, 0, sizeof(p));
    for (int w = 0; w < P; ++w) {
        if (!x[w]) return fail(GAR_EINVAL, "input %d is NULL", w);
        if (!aligned(x[w], 4)) return fail(GAR_EALIGN, "input %d not 4-byte aligned", w);
        p.x[w] = x[w];
    }
    p.ws = static_cast<double *>(d_workspace);
    p.mM = d_mM;
    p.n = n;
    p.P = P;
    p.blocks = norm_grid(n, P);
    p.t_over_sqrt_n = t_p / std::sqrt(static_cast<double>(n));
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    rht_norm_partial<<<dim3(static_cast<unsigned>(p.blocks), static_cast<unsigned>(P)), kThreads, 0, stream>>>(p);
    int rc = check_launch("rht_norm_partial");
    if (rc) return rc;
    rht_norm_final<<<1, kThreads, 0, stream>>>(p);
    return check_launch("rht_norm_final");
}

static int ef_launch(const float *a, const float *b, float *out, int64_t n, int subtract, gar_stream_t stream_) {
    if (n < 0) return fail(GAR_EINVAL, "n < 0");
    if (n == 0) return GAR_OK;
    if (!a || !b || !out) return fail(GAR_EINVAL, "NULL argument");
    if (!aligned(a, 4) || !aligned(b, 4) || !aligned(out, 4)) return fail(GAR_EALIGN, "pointer not 4-byte aligned");
    // out may be a or b exactly (each element is read before the same thread writes it)
    if ((out != a && overlaps(out, a, n * 4)) || (out != b && overlaps(out, b, n * 4)))
        return fail(GAR_EINVAL, "output overlaps an input without being equal to it");
    const int vec = aligned(a, 16) && aligned(b, 16) && aligned(out, 16);
    const int grid = ew_grid(vec ? ceil_div(n, 4) : n);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (subtract)
        ef_kernel<true><<<grid, kThreads, 0, stream>>>(a, b, out, n, vec);
    else
        ef_kernel<false><<<grid, kThreads, 0, stream>>>(a, b, out, n, vec);
    return check_launch("ef_kernel");
}

extern "C" int gar_ef_apply(const float *grad, const float *e, float *x, int64_t n, gar_stream_t stream) {
    return ef_launch(grad, e, x, n, 0, stream);
}

extern "C" int gar_ef_update(float *e, const float *x, const float *x_hat, int64_t n, gar_stream_t stream) {
    return ef_launch(x, x_hat, e, n, 1, stream);
}
