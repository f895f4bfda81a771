// nuhc.cu -- non-uniform Tensor Homomorphic Compression ([T] section 5,
// Algorithm 2): the worker's indices address a lookup table T of 2^b
// increasing points of a finer grid of g steps; the parameter server sums
// the table values T[index], and the sum decodes like uniform THC with the
// step (M - m) / g.
//
//   encode     Philox-driven stochastic quantization to the table's points
//   aggregate  sum of the workers' table values (the PS)
//   decode     the uniform decode with g steps
//   fused      encode (all workers) -> aggregate -> decode in one pass
#include <cstring>

#include "common.cuh"
#include "thc_fused.cuh"

namespace gar {
using namespace thc;
namespace {

// ([T] section 5, Algorithm 2.)  Granularity g >= 2^b - 1: the grid is
// m + k (M - m)/g, k = 0..g, and a worker may only send the 2^b points whose
// k is a table value T[z].  Decision in fp32, one rounding per op:
//   t = clamp((x - m) * (g / (M - m)), 0, g)
//   z = the largest z <= L - 1 with T[z] <= t  (= inv[min(floor(t), g - 1)])
//   up iff u < (t - T[z]) / (T[z + 1] - T[z]) exactly  (u as in uniform THC)
//   index = z + up; the PS sums T[index].
constexpr int kMaxGranularity = 16383;

struct NuhcTable {
    uint16_t t[256];
    int32_t L;
    int32_t g;
};

// Shared-memory tables: the pairs (T[z], T[z + 1]) as floats for z < L (one
// 8-byte load gives both neighbours), and the inverse of T on the integers
// 0..g-1 (z of the interval holding k).
constexpr int kNuhcPairBytes = 256 * 8;  // float2[255], rounded up
__device__ __forceinline__ void nuhc_load_tables(const NuhcTable &tab, float2 *s_pair, uint8_t *s_inv) {
    for (int z = threadIdx.x; z < tab.L; z += blockDim.x)
        s_pair[z] = make_float2(static_cast<float>(tab.t[z]), static_cast<float>(tab.t[z + 1]));
    for (int k = threadIdx.x; k < tab.g; k += blockDim.x) {
        int lo = 0, hi = tab.L - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tab.t[mid] <= k) lo = mid;
            else hi = mid - 1;
        }
        s_inv[k] = static_cast<uint8_t>(lo);
    }
    __syncthreads();
}

// Returns the index; tv receives the table value it stands for (an integer
// below 2^14, as a float).
__device__ __forceinline__ uint32_t nuhc_index(float x, float m, float sc, float G, int g, const float2 *s_pair,
                                               const uint8_t *s_inv, uint32_t r, float &tv) {
    float t = __fmul_rn(__fsub_rn(x, m), sc);
    t = fminf(fmaxf(t, 0.0f), G);
    int k = __float_as_int(__fadd_rd(t, 8388608.0f)) - 0x4B000000;  // floor(t)
    k = k < g - 1 ? k : g - 1;
    const int z = s_inv[k];
    const float2 lh = s_pair[z];  // T[z], T[z + 1]
    // up iff u < (t - lo) / (hi - lo) exactly, i.e. u * (hi - lo) < t - lo: t - lo and
    // hi - lo are exact (integer lo, hi below 2^14, t >= lo), u = (r mod 2^23) 2^-23 is
    // exact, and the sign of the once-rounded fma(-u, hi - lo, t - lo) is the sign of
    // the exact difference (a nonzero one is a multiple of 2^-149: never rounds to 0)
    const float u = __fsub_rn(__uint_as_float((r & 0x007FFFFFu) | 0x3F800000u), 1.0f);
    const bool up = __fmaf_rn(-u, __fsub_rn(lh.y, lh.x), __fsub_rn(t, lh.x)) > 0.0f;
    tv = up ? lh.y : lh.x;
    return static_cast<uint32_t>(z) + (up ? 1u : 0u);
}

// The same decision for two elements at once: the subtracts, the multiply,
// the rounded-down add and the FMA go through the packed f32x2 instructions
// (each lane rounded exactly as the scalar operation, subnormals kept); the
// clamp, the table lookups and the comparisons stay per element.  Bit for bit
// equal to two nuhc_index calls.
__device__ __forceinline__ uint64_t add_rn_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma_rm_f2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t fma_rn_f2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ void nuhc_index2(float x0, float x1, uint64_t m2, uint64_t sc2, float G, int g,
                                            const float2 *s_pair, const uint8_t *s_inv, uint32_t r0, uint32_t r1,
                                            uint32_t &i0, uint32_t &i1, float &tv0, float &tv1) {
    float2 t = unpack_f2(mul_rn_f2(sub_rn_f2(pack_f2(x0, x1), m2), sc2));
    t.x = fminf(fmaxf(t.x, 0.0f), G);
    t.y = fminf(fmaxf(t.y, 0.0f), G);
    const uint64_t t2 = pack_f2(t.x, t.y);
    const float2 jm = unpack_f2(add_rm_f2(t2, pack_f2(8388608.0f, 8388608.0f)));  // floor(t) + 2^23
    int k0 = __float_as_int(jm.x) - 0x4B000000, k1 = __float_as_int(jm.y) - 0x4B000000;
    k0 = k0 < g - 1 ? k0 : g - 1;
    k1 = k1 < g - 1 ? k1 : g - 1;
    const int z0 = s_inv[k0], z1 = s_inv[k1];
    const float2 p0 = s_pair[z0], p1 = s_pair[z1];  // (T[z], T[z + 1]) of each
    const uint64_t lo = pack_f2(p0.x, p1.x), hi = pack_f2(p0.y, p1.y);
    // -u = 1 - (1 + u), exact; then fma(-u, hi - lo, t - lo) as in nuhc_index
    const uint64_t one_u = pack_f2(__uint_as_float((r0 & 0x007FFFFFu) | 0x3F800000u),
                                   __uint_as_float((r1 & 0x007FFFFFu) | 0x3F800000u));
    const uint64_t neg_u = sub_rn_f2(pack_f2(1.0f, 1.0f), one_u);
    const float2 f = unpack_f2(fma_rn_f2(neg_u, sub_rn_f2(hi, lo), sub_rn_f2(t2, lo)));
    const bool up0 = f.x > 0.0f, up1 = f.y > 0.0f;
    tv0 = up0 ? p0.y : p0.x;
    tv1 = up1 ? p1.y : p1.x;
    i0 = static_cast<uint32_t>(z0) + (up0 ? 1u : 0u);
    i1 = static_cast<uint32_t>(z1) + (up1 ? 1u : 0u);
}

// Direct tables, for granularities up to kDirectMaxG: for every k = 0..g the
// lower end T[z] and the width T[z + 1] - T[z] of the interval holding k (as
// floats; the decision and the sum of table values need no more) and z itself
// (k = g belongs to the last interval).  One lookup by k replaces the two
// dependent ones k -> z -> (T[z], T[z + 1]); ends and widths sit in separate
// arrays, so that two elements' values load straight into the register pairs
// of the f32x2 instructions.  The result equals nuhc_index bit for bit:
// for k <= g - 1 the interval is the same, and for k = g (t = G) the old
// lookup clamps k to g - 1, which lies in the same last interval.
constexpr int kDirectMaxG = 1023;
constexpr int kDirectCap = kDirectMaxG + 1;
// s_lo[kDirectCap], s_w[kDirectCap], s_zb[kDirectCap] (floats: the interval's lower end T[z], its
// width w = T[z + 1] - T[z] and z + 2^23, all exact),
// s_z[kDirectCap] (bytes), then T itself
constexpr size_t kDirectBytes = kDirectCap * (3 * sizeof(float) + 1) + 256 * sizeof(uint16_t);
constexpr float kTwo23 = 8388608.0f;
constexpr uint32_t kTwo23Bits = 0x4B000000u;  // the bits of 2^23; of z + 2^23: kTwo23Bits + z

__device__ __forceinline__ void nuhc_load_direct(const NuhcTable &tab, unsigned char *mem, float *&s_lo,
                                                 uint8_t *&s_z) {
    s_lo = reinterpret_cast<float *>(mem);
    float *s_w = s_lo + kDirectCap;
    float *s_zb = s_w + kDirectCap;
    s_z = reinterpret_cast<uint8_t *>(s_zb + kDirectCap);
    uint16_t *s_t = reinterpret_cast<uint16_t *>(s_z + kDirectCap);
    for (int z = threadIdx.x; z <= tab.L; z += blockDim.x) s_t[z] = tab.t[z];
    __syncthreads();
    for (int k = threadIdx.x; k <= tab.g; k += blockDim.x) {
        int lo = 0, hi = tab.L - 1;  // the largest z <= L - 1 with T[z] <= k
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_t[mid] <= k) lo = mid;
            else hi = mid - 1;
        }
        s_lo[k] = static_cast<float>(s_t[lo]);
        s_w[k] = static_cast<float>(s_t[lo + 1] - s_t[lo]);
        s_zb[k] = kTwo23 + static_cast<float>(lo);
        s_z[k] = static_cast<uint8_t>(lo);
    }
    __syncthreads();
}

// nuhc_index over the direct tables (one element).
__device__ __forceinline__ uint32_t nuhc_direct(float x, float m, float sc, float G, const float *s_lo,
                                                const uint8_t *s_z, uint32_t r, float &tv) {
    float t = __fmul_rn(__fsub_rn(x, m), sc);
    t = fminf(fmaxf(t, 0.0f), G);
    const int k = __float_as_int(__fadd_rd(t, 8388608.0f)) - 0x4B000000;  // floor(t), 0..g
    const float lo = s_lo[k], w = s_lo[kDirectCap + k];
    const float u = __fsub_rn(__uint_as_float((r & 0x007FFFFFu) | 0x3F800000u), 1.0f);
    const bool up = __fmaf_rn(-u, w, __fsub_rn(t, lo)) > 0.0f;
    tv = up ? __fadd_rn(lo, w) : lo;  // T[z + 1], exact
    return static_cast<uint32_t>(s_z[k]) + (up ? 1u : 0u);
}

// nuhc_index2 over the direct tables; kZ: the indices are wanted (packed
// output), else only the table values.
template <bool kZ>
__device__ __forceinline__ void nuhc_direct2(float x0, float x1, uint64_t m2, uint64_t sc2, float G,
                                             const float *s_lo, const uint8_t *s_z, uint32_t r0, uint32_t r1,
                                             uint32_t &i0, uint32_t &i1, float &tv0, float &tv1) {
    float2 t = unpack_f2(mul_rn_f2(sub_rn_f2(pack_f2(x0, x1), m2), sc2));
    t.x = fminf(fmaxf(t.x, 0.0f), G);
    t.y = fminf(fmaxf(t.y, 0.0f), G);
    const uint64_t t2 = pack_f2(t.x, t.y);
    const float2 jm = unpack_f2(add_rm_f2(t2, pack_f2(8388608.0f, 8388608.0f)));  // floor(t) + 2^23
    const int k0 = __float_as_int(jm.x) - 0x4B000000, k1 = __float_as_int(jm.y) - 0x4B000000;  // 0..g
    const float lo0 = s_lo[k0], lo1 = s_lo[k1];
    const uint64_t lo = pack_f2(lo0, lo1), w = pack_f2(s_lo[kDirectCap + k0], s_lo[kDirectCap + k1]);
    const float2 hi2 = unpack_f2(add_rn_f2(lo, w));  // T[z + 1], exact
    const float hi0 = hi2.x, hi1 = hi2.y;
    const uint64_t one_u = pack_f2(__uint_as_float((r0 & 0x007FFFFFu) | 0x3F800000u),
                                   __uint_as_float((r1 & 0x007FFFFFu) | 0x3F800000u));
    // up iff lo + u w < t (w = hi - lo), decided exactly as (lo + u w) rounded
    // down < t: rounding down never passes the float t.  lo + u w is formed
    // with one rounding as fma((1 + u), w, lo - w); w and lo - w are exact
    // (integers below 2^15).  Equal to nuhc_index's fma(-u, w, t - lo) > 0.
    const float2 v = unpack_f2(fma_rm_f2(one_u, w, sub_rn_f2(lo, w)));
    const bool up0 = v.x < t.x, up1 = v.y < t.y;
    tv0 = up0 ? hi0 : lo0;
    tv1 = up1 ? hi1 : lo1;
    if (kZ) {
        i0 = static_cast<uint32_t>(s_z[k0]) + (up0 ? 1u : 0u);
        i1 = static_cast<uint32_t>(s_z[k1]) + (up1 ? 1u : 0u);
    }
}

// nuhc_direct2 for the fused kernel, adding the two elements' table values
// T[index] to their running sums (an f32x2 pair) as sum + lo + up * w, up =
// 1.0 or 0.0 the comparison's value: one add and one FMA, exact (integers
// below 2^24), with no select.  kZ: also the indices, biased: the bits of
// z + up + 2^23 (z + 2^23 from s_zb, exact) are kTwo23Bits + index.
template <bool kZ>
__device__ __forceinline__ void nuhc_direct2_sum(float x0, float x1, uint64_t m2, uint64_t sc2, float G,
                                                 const float *s_lo, uint32_t r0, uint32_t r1, uint64_t &sum,
                                                 uint32_t &a0, uint32_t &a1) {
    float2 t = unpack_f2(mul_rn_f2(sub_rn_f2(pack_f2(x0, x1), m2), sc2));
    t.x = fminf(fmaxf(t.x, 0.0f), G);
    t.y = fminf(fmaxf(t.y, 0.0f), G);
    const uint64_t t2 = pack_f2(t.x, t.y);
    const float2 jm = unpack_f2(add_rm_f2(t2, pack_f2(kTwo23, kTwo23)));  // floor(t) + 2^23
    const int k0 = __float_as_int(jm.x) - 0x4B000000, k1 = __float_as_int(jm.y) - 0x4B000000;  // 0..g
    const uint64_t lo = pack_f2(s_lo[k0], s_lo[k1]);
    const uint64_t w = pack_f2(s_lo[kDirectCap + k0], s_lo[kDirectCap + k1]);  // T[z + 1] - T[z]
    const uint64_t one_u = pack_f2(__uint_as_float((r0 & 0x007FFFFFu) | 0x3F800000u),
                                   __uint_as_float((r1 & 0x007FFFFFu) | 0x3F800000u));
    // up iff RD(lo + u w) < t, as in nuhc_direct2
    const float2 v = unpack_f2(fma_rm_f2(one_u, w, sub_rn_f2(lo, w)));
    float u0, u1;
    asm("set.lt.f32.f32 %0, %1, %2;" : "=f"(u0) : "f"(v.x), "f"(t.x));
    asm("set.lt.f32.f32 %0, %1, %2;" : "=f"(u1) : "f"(v.y), "f"(t.y));
    const uint64_t up = pack_f2(u0, u1);
    sum = fma_rn_f2(up, w, add_rn_f2(sum, lo));
    if (kZ) {
        const float2 ib =
            unpack_f2(add_rn_f2(pack_f2(s_lo[2 * kDirectCap + k0], s_lo[2 * kDirectCap + k1]), up));
        a0 = __float_as_uint(ib.x);
        a1 = __float_as_uint(ib.y);
    }
}

// Sum over the fields of a packed word of (kTwo23Bits << field shift), mod
// 2^32: the biased indices packed with plain shifted adds, minus this once,
// leave the exact word (the fields never overlap).
template <int B>
__host__ __device__ constexpr uint32_t zb_pack_bias() {
    uint32_t s = 0;
    for (int i = 0; i < 32 / B; ++i) s += (i * B < 32 ? kTwo23Bits << (i * B) : 0u);
    return s;
}

struct NuhcEncodeParams {
    PhiloxKeys keys;
    NuhcTable tab;
    const float *x;
    const float *mM;
    uint32_t *packed;
    int64_t N;
    int64_t nwords;
    int32_t worker;
    int32_t vec;
};

// kDirect: the direct tables (g <= kDirectMaxG), else the interval tables.
template <int B, bool kDirect>
__global__ void __launch_bounds__(kThreads) nuhc_encode_kernel(const __grid_constant__ NuhcEncodeParams p) {
    constexpr int E = 32 / B;
    extern __shared__ unsigned char s_mem[];
    float2 *s_pair;
    uint8_t *s_inv;
    float *s_lo = nullptr;
    if constexpr (kDirect) {
        nuhc_load_direct(p.tab, s_mem, s_lo, s_inv);
        s_pair = nullptr;
    } else {
        s_pair = reinterpret_cast<float2 *>(s_mem);
        s_inv = s_mem + kNuhcPairBytes;
        nuhc_load_tables(p.tab, s_pair, s_inv);
    }
    const float m = p.mM[0], M = p.mM[1];
    const float G = static_cast<float>(p.tab.g);
    const float sc = range_scale(m, M, G);
    const uint64_t m2 = pack_f2(m, m), sc2 = pack_f2(sc, sc);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; w < p.nwords; w += stride) {
        const int64_t e0 = w * E;
        uint32_t word = 0;
        float tv;
        for (int g4 = 0; g4 < E / 4; ++g4) {
            const int64_t eb = e0 + 4 * g4;
            if (eb >= p.N) break;
            const uint4 r = philox_block(eb >> 2, p.worker, p.keys);
            float4 v;
            if (p.vec && eb + 4 <= p.N) {
                v = __ldcs(reinterpret_cast<const float4 *>(p.x + eb));
            } else {
                v = make_float4(m, m, m, m);  // past N: index 0, masked out below
                if (eb < p.N) v.x = p.x[eb];
                if (eb + 1 < p.N) v.y = p.x[eb + 1];
                if (eb + 2 < p.N) v.z = p.x[eb + 2];
                if (eb + 3 < p.N) v.w = p.x[eb + 3];
            }
            uint32_t i0, i1, i2, i3;
            float tv1;
            if constexpr (kDirect) {
                nuhc_direct2<true>(v.x, v.y, m2, sc2, G, s_lo, s_inv, r.x, r.y, i0, i1, tv, tv1);
                nuhc_direct2<true>(v.z, v.w, m2, sc2, G, s_lo, s_inv, r.z, r.w, i2, i3, tv, tv1);
            } else {
                nuhc_index2(v.x, v.y, m2, sc2, G, p.tab.g, s_pair, s_inv, r.x, r.y, i0, i1, tv, tv1);
                nuhc_index2(v.z, v.w, m2, sc2, G, p.tab.g, s_pair, s_inv, r.z, r.w, i2, i3, tv, tv1);
            }
            uint32_t q = i0 | (i1 << B) | (i2 << (2 * B)) | (i3 << (3 * B));
            const int64_t valid = p.N - eb;  // elements of this group inside N
            if (valid < 4) q &= (1u << (B * valid)) - 1u;
            word |= q << (4 * g4 * B);
        }
        __stcs(p.packed + w, word);
    }
}

struct NuhcAggParams {
    NuhcTable tab;
    const uint32_t *packed[GAR_MAX_WORKERS];
    uint16_t *sums;
    int64_t N;
    int32_t P;
    int32_t pad;
};

// One packed word of every worker per thread: the PS looks each index up
// and adds the table values.
template <int B>
__global__ void __launch_bounds__(kThreads) nuhc_aggregate_kernel(const __grid_constant__ NuhcAggParams p) {
    constexpr int E = 32 / B;
    constexpr uint32_t kMask = (1u << B) - 1u;
    __shared__ uint16_t s_t[256];
    for (int z = threadIdx.x; z <= p.tab.L; z += blockDim.x) s_t[z] = p.tab.t[z];
    __syncthreads();
    const int64_t nwords = (p.N + E - 1) / E;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; w < nwords; w += stride) {
        uint32_t s[E];
#pragma unroll
        for (int i = 0; i < E; ++i) s[i] = 0;
        for (int k = 0; k < p.P; ++k) {
            const uint32_t word = __ldcs(p.packed[k] + w);
#pragma unroll
            for (int i = 0; i < E; ++i) s[i] += s_t[(word >> (B * i)) & kMask];
        }
        const int64_t e0 = w * E;
        if (e0 + E <= p.N && (E % 2 == 0)) {
#pragma unroll
            for (int i = 0; i < E; i += 2)
                *reinterpret_cast<uint32_t *>(p.sums + e0 + i) = (s[i] & 0xFFFFu) | (s[i + 1] << 16);
        } else {
            for (int i = 0; i < E && e0 + i < p.N; ++i) p.sums[e0 + i] = static_cast<uint16_t>(s[i]);
        }
    }
}

struct NuhcFusedParams {
    PhiloxKeys keys;
    NuhcTable tab;
    const float *x[GAR_MAX_WORKERS];    // the P contributing workers, slot by slot
    uint32_t *packed[GAR_MAX_WORKERS];
    int32_t wid[GAR_MAX_WORKERS];       // worker id of each slot (keys its Philox stream)
    const float *mM;
    float *avg;
    int64_t N;
    int64_t nwords;
    int32_t P;                          // contributing workers (the decode divides by this)
    int32_t vec;
};

// One worker's contribution to a whole word of E = 4 G4 elements: Philox
// draws, indices, the table values added to the running sums s, the packed
// word stored if wanted.
// (The sums of table values are integers below 2^24: exact in fp32.)
template <int B, bool kPacked, bool kDirect, int G4>
__device__ __forceinline__ void nuhc_one_worker(const float4 (&v)[G4], float (&s)[4 * G4], int64_t e0, int64_t w,
                                                int wk, int wid, const NuhcFusedParams &p, uint64_t m2,
                                                uint64_t sc2, float G, const float2 *s_pair, const uint8_t *s_inv) {
    uint32_t word = 0;
    if constexpr (kDirect) {
        // direct tables: s_pair holds s_lo (then s_w, s_zb)
        const float *s_lo = reinterpret_cast<const float *>(s_pair);
#pragma unroll
        for (int g4 = 0; g4 < G4; ++g4) {
            const uint4 r = philox_block((e0 >> 2) + g4, wid, p.keys);
            uint64_t s01 = pack_f2(s[4 * g4], s[4 * g4 + 1]), s23 = pack_f2(s[4 * g4 + 2], s[4 * g4 + 3]);
            uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
            nuhc_direct2_sum<kPacked>(v[g4].x, v[g4].y, m2, sc2, G, s_lo, r.x, r.y, s01, a0, a1);
            nuhc_direct2_sum<kPacked>(v[g4].z, v[g4].w, m2, sc2, G, s_lo, r.z, r.w, s23, a2, a3);
            const float2 f01 = unpack_f2(s01), f23 = unpack_f2(s23);
            s[4 * g4] = f01.x;
            s[4 * g4 + 1] = f01.y;
            s[4 * g4 + 2] = f23.x;
            s[4 * g4 + 3] = f23.y;
            if (kPacked)
                word += (a0 << (4 * g4 * B)) + (a1 << ((4 * g4 + 1) * B)) + (a2 << ((4 * g4 + 2) * B)) +
                        (a3 << ((4 * g4 + 3) * B));
        }
        if (kPacked) __stcs(p.packed[wk] + w, word - zb_pack_bias<B>());
        return;
    }
#pragma unroll
    for (int g4 = 0; g4 < G4; ++g4) {
        const uint4 r = philox_block((e0 >> 2) + g4, wid, p.keys);
        float t0, t1, t2, t3;
        uint32_t i0 = 0, i1 = 0, i2 = 0, i3 = 0;
        {
            nuhc_index2(v[g4].x, v[g4].y, m2, sc2, G, p.tab.g, s_pair, s_inv, r.x, r.y, i0, i1, t0, t1);
            nuhc_index2(v[g4].z, v[g4].w, m2, sc2, G, p.tab.g, s_pair, s_inv, r.z, r.w, i2, i3, t2, t3);
        }
        // the running sums, two per f32x2 add (each lane rounded as __fadd_rn)
        {
            float2 a = unpack_f2(add_rn_f2(pack_f2(s[4 * g4], s[4 * g4 + 1]), pack_f2(t0, t1)));
            float2 c = unpack_f2(add_rn_f2(pack_f2(s[4 * g4 + 2], s[4 * g4 + 3]), pack_f2(t2, t3)));
            s[4 * g4] = a.x;
            s[4 * g4 + 1] = a.y;
            s[4 * g4 + 2] = c.x;
            s[4 * g4 + 3] = c.y;
        }
        if (kPacked) word |= (i0 | (i1 << B) | (i2 << (2 * B)) | (i3 << (3 * B))) << (4 * g4 * B);
    }
    if (kPacked) __stcs(p.packed[wk] + w, word);
}

// kDirect (g <= kDirectMaxG): the direct tables (P=8, 2^24, packed output:
// b = 4 0.207 -> 0.190 ms, b = 8 0.208 -> 0.196, b = 1 0.262 -> 0.239 on a
// resident grid); else the interval tables (a larger g would not leave room
// for the direct ones).  The grid-stride loop serves a resident grid and one
// CTA per tile alike.
// kP > 0: built for exactly kP workers (the worker loop unrolls; pointers and
// worker ids come from fixed parameter offsets); 0: any P.
template <int B, bool kPacked, bool kDirect, int kP = 0>
__global__ void __launch_bounds__(kThreads, B == 4 ? 4 : 1) nuhc_fused_kernel(const __grid_constant__ NuhcFusedParams p) {
    constexpr int E = 32 / B;
    constexpr int G4 = E / 4;
    constexpr int kUnroll = kP > 0 ? kP : 1;
    const int P = kP > 0 ? kP : p.P;
    extern __shared__ unsigned char s_mem[];
    float2 *s_pair;
    uint8_t *s_inv;
    if constexpr (kDirect) {
        float *s_lo;
        nuhc_load_direct(p.tab, s_mem, s_lo, s_inv);
        s_pair = reinterpret_cast<float2 *>(s_lo);
    } else {
        s_pair = reinterpret_cast<float2 *>(s_mem);
        s_inv = s_mem + kNuhcPairBytes;
        nuhc_load_tables(p.tab, s_pair, s_inv);
    }
    const float m = p.mM[0], M = p.mM[1];
    const float G = static_cast<float>(p.tab.g);
    const float sc = range_scale(m, M, G);
    float km;
    const float k = decode_step(p.mM, G, static_cast<float>(p.P), km);
    const uint64_t m2 = pack_f2(m, m), sc2 = pack_f2(sc, sc);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; w < p.nwords; w += stride) {
        const int64_t e0 = w * E;
        float s[E];
#pragma unroll
        for (int i = 0; i < E; ++i) s[i] = 0.0f;
        if (p.vec && e0 + E <= p.N) {
            // two register buffers, the worker loop unrolled by two: one worker's
            // loads are in flight while the other is quantized
            float4 va[G4], vb[G4];
#pragma unroll
            for (int g4 = 0; g4 < G4; ++g4) va[g4] = __ldcs(reinterpret_cast<const float4 *>(p.x[0] + e0) + g4);
#pragma unroll(kUnroll)
            for (int wk = 0; wk < P; wk += 2) {
                const bool has1 = wk + 1 < P;
                if (has1) {
#pragma unroll
                    for (int g4 = 0; g4 < G4; ++g4) vb[g4] = __ldcs(reinterpret_cast<const float4 *>(p.x[wk + 1] + e0) + g4);
                }
                nuhc_one_worker<B, kPacked, kDirect>(va, s, e0, w, wk, kP > 0 ? wk : p.wid[wk], p, m2, sc2, G, s_pair,
                                                     s_inv);
                if (wk + 2 < P) {
#pragma unroll
                    for (int g4 = 0; g4 < G4; ++g4) va[g4] = __ldcs(reinterpret_cast<const float4 *>(p.x[wk + 2] + e0) + g4);
                }
                if (has1)
                    nuhc_one_worker<B, kPacked, kDirect>(vb, s, e0, w, wk + 1, kP > 0 ? wk + 1 : p.wid[wk + 1], p, m2,
                                                         sc2, G, s_pair, s_inv);
            }
            float4 *dst = reinterpret_cast<float4 *>(p.avg + e0);
#pragma unroll
            for (int g4 = 0; g4 < G4; ++g4)
                __stcs(dst + g4, make_float4(__fmaf_rn(s[4 * g4], k, km), __fmaf_rn(s[4 * g4 + 1], k, km),
                                             __fmaf_rn(s[4 * g4 + 2], k, km), __fmaf_rn(s[4 * g4 + 3], k, km)));
        } else {  // ragged last word, or unaligned pointers: element by element
            for (int wk = 0; wk < p.P; ++wk) {
                uint32_t word = 0;
                for (int g4 = 0; g4 < G4; ++g4) {
                    const int64_t eb = e0 + 4 * g4;
                    if (eb >= p.N) break;
                    const uint4 r = philox_block(eb >> 2, kP > 0 ? wk : p.wid[wk], p.keys);
                    for (int i = 0; i < 4 && eb + i < p.N; ++i) {
                        float tv;
                        const uint32_t idx =
                            kDirect ? nuhc_direct(p.x[wk][eb + i], m, sc, G, reinterpret_cast<const float *>(s_pair),
                                                  s_inv, pick(r, i), tv)
                                    : nuhc_index(p.x[wk][eb + i], m, sc, G, p.tab.g, s_pair, s_inv, pick(r, i), tv);
                        s[4 * g4 + i] = __fadd_rn(s[4 * g4 + i], tv);
                        word |= idx << ((4 * g4 + i) * B);
                    }
                }
                if (kPacked) p.packed[wk][w] = word;
            }
            for (int i = 0; i < E && e0 + i < p.N; ++i) p.avg[e0 + i] = __fmaf_rn(s[i], k, km);
        }
    }
}

// The fused kernel for one b and output kind.  b = 4 with the direct tables:
// one CTA per 2 x kThreads words (the grid-stride loop runs twice; P=8,
// 2^24: 0.190 -> 0.184 ms), and for 4, 8 or 16 workers the kernel built for
// that P (0.184 -> 0.166 ms with wire vectors, 0.162 -> 0.150 without).  The
// other widths, with 1.5 to 4 times the registers per thread or 8 words per
// worker and thread, ran faster on a resident grid (b = 2, P = 16: 0.413 ms
// resident, 0.440 ms one CTA per tile), and unrolling their worker loop
// raised their registers further (b = 2, P = 16: 255 and spills).
template <int BB, bool PK>
void launch_nuhc_fused(const NuhcFusedParams &p, bool direct, int P, unsigned tiles, size_t smem,
                       cudaStream_t stream) {
    if (!direct) {
        nuhc_fused_kernel<BB, PK, false><<<grid_for(nuhc_fused_kernel<BB, PK, false>, p.nwords), kThreads, smem,
                                           stream>>>(p);
    } else if constexpr (BB == 4) {
        switch (P) {
            case 4: nuhc_fused_kernel<BB, PK, true, 4><<<tiles, kThreads, smem, stream>>>(p); break;
            case 8: nuhc_fused_kernel<BB, PK, true, 8><<<tiles, kThreads, smem, stream>>>(p); break;
            case 16: nuhc_fused_kernel<BB, PK, true, 16><<<tiles, kThreads, smem, stream>>>(p); break;
            default: nuhc_fused_kernel<BB, PK, true><<<tiles, kThreads, smem, stream>>>(p); break;
        }
    } else {
        nuhc_fused_kernel<BB, PK, true><<<grid_for(nuhc_fused_kernel<BB, PK, true>, p.nwords), kThreads, smem,
                                          stream>>>(p);
    }
}

int nuhc_table(const uint16_t *table, int b, int g, NuhcTable &tab) {
    if (!table) return fail(GAR_EINVAL, "table is NULL");
    const int L = (1 << b) - 1;
    if (g < L || g > kMaxGranularity) return fail(GAR_EINVAL, "granularity %d outside [%d, %d]", g, L, kMaxGranularity);
    if (table[0] != 0 || table[L] != g) return fail(GAR_EINVAL, "table must start at 0 and end at g=%d", g);
    for (int z = 0; z < L; ++z)
        if (table[z + 1] <= table[z]) return fail(GAR_EINVAL, "table not strictly increasing at %d", z);
    std::memset(&tab, 0, sizeof(tab));
    for (int z = 0; z <= L; ++z) tab.t[z] = table[z];
    tab.L = L;
    tab.g = g;
    return GAR_OK;
}

}  // namespace
}  // namespace gar

using namespace gar;

extern "C" int gar_nuhc_encode(const float *x, int64_t N, const float *d_mM, int32_t b, int32_t g,
                               const uint16_t *table, uint64_t seed, int32_t worker, uint32_t *packed,
                               gar_stream_t stream_) {
    if (!valid_b(b)) return fail(GAR_EINVAL, "b=%d not in {1, 2, 4, 8}", b);
    NuhcEncodeParams p;
    std::memset(&p, 0, sizeof(p));
    int rc = nuhc_table(table, b, g, p.tab);
    if (rc) return rc;
    if (N < 0 || !d_mM) return fail(GAR_EINVAL, "N < 0 or d_mM NULL");
    if (N == 0) return GAR_OK;
    if (!x || !packed) return fail(GAR_EINVAL, "x or packed is NULL");
    if (worker < 0) return fail(GAR_EINVAL, "worker %d < 0", worker);
    if (!aligned(x, 4) || !aligned(packed, 4) || !aligned(d_mM, 4)) return fail(GAR_EALIGN, "misaligned pointer");
    p.keys = philox_keys(seed);
    p.x = x;
    p.mM = d_mM;
    p.packed = packed;
    p.N = N;
    p.nwords = gar_thc_words(N, b);
    p.worker = worker;
    p.vec = aligned(x, 16) ? 1 : 0;
    const bool direct = g <= kDirectMaxG;
    const size_t smem = direct ? kDirectBytes : kNuhcPairBytes + static_cast<size_t>(g);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
#define GAR_NUHC_ENC(BB)                                                                                            \
    case BB:                                                                                                        \
        if (direct)                                                                                                 \
            nuhc_encode_kernel<BB, true><<<grid_for(nuhc_encode_kernel<BB, true>, p.nwords), kThreads, smem, stream>>>(p); \
        else                                                                                                        \
            nuhc_encode_kernel<BB, false><<<grid_for(nuhc_encode_kernel<BB, false>, p.nwords), kThreads, smem,      \
                                            stream>>>(p);                                                           \
        break;
    switch (b) {
        GAR_NUHC_ENC(1)
        GAR_NUHC_ENC(2)
        GAR_NUHC_ENC(4)
        GAR_NUHC_ENC(8)
    }
#undef GAR_NUHC_ENC
    return check_launch("nuhc_encode_kernel");
}

extern "C" int gar_nuhc_aggregate(const uint32_t *const *packed, int32_t P, int64_t N, int32_t b,
                                  const uint16_t *table, uint16_t *sums, gar_stream_t stream_) {
    if (!valid_b(b)) return fail(GAR_EINVAL, "b=%d not in {1, 2, 4, 8}", b);
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    NuhcAggParams p;
    std::memset(&p, 0, sizeof(p));
    if (!table) return fail(GAR_EINVAL, "table is NULL");
    const int L = (1 << b) - 1;
    int rc = nuhc_table(table, b, table[L], p.tab);
    if (rc) return rc;
    if (static_cast<int64_t>(P) * p.tab.g > 65535) return fail(GAR_EOVERFLOW, "P * g > 65535");
    if (N < 0) return fail(GAR_EINVAL, "N < 0");
    if (N == 0) return GAR_OK;
    if (!packed || !sums) return fail(GAR_EINVAL, "packed or sums is NULL");
    if (!aligned(sums, 4)) return fail(GAR_EALIGN, "sums not 4-byte aligned");
    p.sums = sums;
    p.N = N;
    p.P = P;
    for (int w = 0; w < P; ++w) {
        if (!packed[w]) return fail(GAR_EINVAL, "packed vector %d is NULL", w);
        if (!aligned(packed[w], 4)) return fail(GAR_EALIGN, "packed vector %d not 4-byte aligned", w);
        p.packed[w] = packed[w];
    }
    const int64_t words = gar_thc_words(N, b);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    switch (b) {
        case 1: nuhc_aggregate_kernel<1><<<grid_for(nuhc_aggregate_kernel<1>, words), kThreads, 0, stream>>>(p); break;
        case 2: nuhc_aggregate_kernel<2><<<grid_for(nuhc_aggregate_kernel<2>, words), kThreads, 0, stream>>>(p); break;
        case 4: nuhc_aggregate_kernel<4><<<grid_for(nuhc_aggregate_kernel<4>, words), kThreads, 0, stream>>>(p); break;
        default: nuhc_aggregate_kernel<8><<<grid_for(nuhc_aggregate_kernel<8>, words), kThreads, 0, stream>>>(p); break;
    }
    return check_launch("nuhc_aggregate_kernel");
}

extern "C" int gar_nuhc_decode(const uint16_t *sums, int64_t N, const float *d_mM, int32_t g, int32_t P,
                               float *avg, gar_stream_t stream_) {
    if (g < 1 || g > kMaxGranularity) return fail(GAR_EINVAL, "granularity %d outside [1, %d]", g, kMaxGranularity);
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (N < 0 || !d_mM) return fail(GAR_EINVAL, "N < 0 or d_mM NULL");
    if (N == 0) return GAR_OK;
    if (!sums || !avg) return fail(GAR_EINVAL, "sums or avg is NULL");
    if (!aligned(sums, 2) || !aligned(avg, 4) || !aligned(d_mM, 4)) return fail(GAR_EALIGN, "misaligned pointer");
    // the uniform decode with the step (M - m) / g
    return launch_grid_decode(sums, N, d_mM, g, P, avg, reinterpret_cast<cudaStream_t>(stream_));
}

// The fused round over the workers whose bit is set in `arrived` (all of
// them for gar_nuhc_allreduce_fused): each arrived worker takes the next
// slot under its own worker id.  The kernels built for 4, 8 or 16 workers key
// Philox by the slot, so a round whose slots are not the ids 0 .. P-1 takes
// the build for any worker count, which reads the ids.
static int nuhc_fused_entry(const float *const *x, int32_t P, uint64_t arrived, int64_t N, int32_t b, int32_t g,
                            const uint16_t *table, uint64_t seed, const float *d_mM, float *avg,
                            uint32_t *const *packed, gar_stream_t stream_) {
    if (!valid_b(b)) return fail(GAR_EINVAL, "b=%d not in {1, 2, 4, 8}", b);
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (P < 64) arrived &= (uint64_t{1} << P) - 1u;
    const int p_eff = __builtin_popcountll(arrived);
    if (p_eff == 0) return fail(GAR_EINVAL, "no worker arrived");
    NuhcFusedParams p;
    std::memset(&p, 0, sizeof(p));
    int rc = nuhc_table(table, b, g, p.tab);
    if (rc) return rc;
    if (static_cast<int64_t>(p_eff) * g > 65535) return fail(GAR_EOVERFLOW, "P * g > 65535");
    if (N < 0 || !d_mM || !x) return fail(GAR_EINVAL, "N < 0 or NULL argument");
    if (N == 0) return GAR_OK;
    if (!avg) return fail(GAR_EINVAL, "avg is NULL");
    if (!aligned(avg, 4) || !aligned(d_mM, 4)) return fail(GAR_EALIGN, "misaligned pointer");
    p.keys = philox_keys(seed);
    p.mM = d_mM;
    p.avg = avg;
    p.N = N;
    p.nwords = gar_thc_words(N, b);
    p.P = p_eff;
    p.vec = aligned(avg, 16) ? 1 : 0;
    bool ids_are_slots = true;
    int slot = 0;
    for (int w = 0; w < P; ++w) {
        if (!((arrived >> w) & 1u)) continue;
        if (!x[w]) return fail(GAR_EINVAL, "input %d is NULL", w);
        if (!aligned(x[w], 4)) return fail(GAR_EALIGN, "input %d not 4-byte aligned", w);
        p.x[slot] = x[w];
        p.wid[slot] = w;
        ids_are_slots = ids_are_slots && w == slot;
        p.vec = p.vec && aligned(x[w], 16);
        if (packed) {
            if (!packed[w]) return fail(GAR_EINVAL, "packed vector %d is NULL", w);
            if (!aligned(packed[w], 4)) return fail(GAR_EALIGN, "packed vector %d not 4-byte aligned", w);
            p.packed[slot] = packed[w];
        }
        ++slot;
    }
    const int P_build = ids_are_slots ? p_eff : 0;  // 0: the build for any worker count
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const bool direct = g <= kDirectMaxG;
    const size_t smem = direct ? kDirectBytes : kNuhcPairBytes + static_cast<size_t>(g);
    const unsigned tiles = static_cast<unsigned>(ceil_div(p.nwords, int64_t{2 * kThreads}));
#define GAR_NUHC_LAUNCH(BB, PK) launch_nuhc_fused<BB, PK>(p, direct, P_build, tiles, smem, stream);
#define GAR_NUHC_CASE(BB)                 \
    case BB:                              \
        if (packed) {                     \
            GAR_NUHC_LAUNCH(BB, true)     \
        } else {                          \
            GAR_NUHC_LAUNCH(BB, false)    \
        }                                 \
        break;
    switch (b) {
        GAR_NUHC_CASE(1)
        GAR_NUHC_CASE(2)
        GAR_NUHC_CASE(4)
        GAR_NUHC_CASE(8)
    }
#undef GAR_NUHC_CASE
#undef GAR_NUHC_LAUNCH
    return check_launch("nuhc_fused_kernel");
}

extern "C" int gar_nuhc_allreduce_fused(const float *const *x, int32_t P, int64_t N, int32_t b, int32_t g,
                                        const uint16_t *table, uint64_t seed, const float *d_mM, float *avg,
                                        uint32_t *const *packed, gar_stream_t stream) {
    return nuhc_fused_entry(x, P, ~uint64_t{0}, N, b, g, table, seed, d_mM, avg, packed, stream);
}

extern "C" int gar_nuhc_allreduce_fused_masked(const float *const *x, int32_t P, uint64_t arrived, int64_t N,
                                               int32_t b, int32_t g, const uint16_t *table, uint64_t seed,
                                               const float *d_mM, float *avg, uint32_t *const *packed,
                                               gar_stream_t stream) {
    return nuhc_fused_entry(x, P, arrived, N, b, g, table, seed, d_mM, avg, packed, stream);
}
