// thc.cu -- uniform Tensor Homomorphic Compression ([T] section 4, Uniform
// THC / Algorithm 1; section 5 for the index vectors the PS sums).
//
//   range      the preliminary round: global min / max over all workers
//   encode     Philox-driven stochastic quantization to packed b-bit indices
//   aggregate  integer sum of the workers' indices, never decoded (the PS)
//   decode     index sum / P mapped back onto the grid (each worker)
//   fused      encode (all workers) -> aggregate -> decode in one pass
//
// Index decision in fp32 (shared by encode and fused; one rounding per op):
//   t = clamp((x - m) * sc, 0, L),  sc = L / (M - m)  (0 when M == m)
//   up iff u < f = t - j, j = min(floor t, L - 1), u = (r mod 2^23) / 2^23,
//   so the index is ceil(t - u).  It is formed as bits((t - (1 + u) rounded
//   up) + 1.5 * 2^23 rounded up) - (bits(1.5 * 2^23) - 1), where 1 + u is the
//   float with mantissa r mod 2^23 (see index_biased in thc_fused.cuh).
// No integer<->float conversion is needed per element.
#include <algorithm>
#include <cstring>
#include <memory>
#include <vector>

#include "common.cuh"
#include "thc_fused.cuh"

namespace gar {
using namespace thc;
namespace {

// ------------------------------------------------------------------ range
__device__ __forceinline__ void atomic_min_float(float *a, float v) {
    if ((__float_as_uint(v) >> 31) == 0u) atomicMin(reinterpret_cast<int *>(a), __float_as_int(v));
    else atomicMax(reinterpret_cast<unsigned int *>(a), __float_as_uint(v));
}
__device__ __forceinline__ void atomic_max_float(float *a, float v) {
    if ((__float_as_uint(v) >> 31) == 0u) atomicMax(reinterpret_cast<int *>(a), __float_as_int(v));
    else atomicMin(reinterpret_cast<unsigned int *>(a), __float_as_uint(v));
}

__global__ void thc_range_init(float *mM) {
    mM[0] = __int_as_float(0x7F800000);   // +inf
    mM[1] = __int_as_float(0xFF800000u);  // -inf
}

struct RangeParams {
    const float *x[GAR_MAX_WORKERS];
    int64_t N;
    float *mM;
    unsigned int *status;  // GAR_STATUS_NONFINITE raised here
    int32_t vec;  // all inputs 16-byte aligned
    int32_t pad;
};

__global__ void __launch_bounds__(kThreads) thc_range_kernel(const __grid_constant__ RangeParams p) {
    const float *x = p.x[blockIdx.y];
    float lo = __int_as_float(0x7F800000), hi = __int_as_float(0xFF800000u);
    float chk = 0.0f;  // NaN once a non-finite input is seen
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    int64_t scalar_from = 0;
    if (p.vec) {
        const int64_t nv = p.N / 4;
        const float4 *xv = reinterpret_cast<const float4 *>(x);
        int64_t i = tid;
        for (; i + stride < nv; i += 2 * stride) {  // two loads in flight
            const float4 a = __ldcs(xv + i), b = __ldcs(xv + i + stride);
            lo = fminf(lo, fminf(fminf(a.x, a.y), fminf(a.z, a.w)));
            hi = fmaxf(hi, fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)));
            lo = fminf(lo, fminf(fminf(b.x, b.y), fminf(b.z, b.w)));
            hi = fmaxf(hi, fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w)));
            chk = nonfinite_acc(nonfinite_acc(nonfinite_acc(nonfinite_acc(chk, a.x), a.y), a.z), a.w);
            chk = nonfinite_acc(nonfinite_acc(nonfinite_acc(nonfinite_acc(chk, b.x), b.y), b.z), b.w);
        }
        if (i < nv) {
            const float4 a = __ldcs(xv + i);
            lo = fminf(lo, fminf(fminf(a.x, a.y), fminf(a.z, a.w)));
            hi = fmaxf(hi, fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)));
            chk = nonfinite_acc(nonfinite_acc(nonfinite_acc(nonfinite_acc(chk, a.x), a.y), a.z), a.w);
        }
        scalar_from = nv * 4;
    }
    for (int64_t k = scalar_from + tid; k < p.N; k += stride) {
        const float v = __ldcs(x + k);
        lo = fminf(lo, v);
        hi = fmaxf(hi, v);
        chk = nonfinite_acc(chk, v);
    }
    flag_nonfinite_warp(p.status, chk);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
    }
    __shared__ float s_lo[kThreads / 32], s_hi[kThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        s_lo[warp] = lo;
        s_hi[warp] = hi;
    }
    __syncthreads();
    if (warp == 0) {
        lo = lane < kThreads / 32 ? s_lo[lane] : __int_as_float(0x7F800000);
        hi = lane < kThreads / 32 ? s_hi[lane] : __int_as_float(0xFF800000u);
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
        }
        if (lane == 0) {
            if (lo == lo) atomic_min_float(p.mM, lo);  // NaN only if the slice was empty of numbers
            if (hi == hi) atomic_max_float(p.mM + 1, hi);
        }
    }
}

// ----------------------------------------------------------------- encode
struct EncodeParams {
    PhiloxKeys keys;
    const float *x;
    const float *mM;
    uint32_t *packed;
    int64_t N;
    int64_t nwords;
    int32_t worker;
    int32_t vec;
    float L;
    int32_t pad;
};

// One full word of E = 32 / B elements (four per float4 group): indices
// packed LSB first, the decision as in the fused kernels.
template <int B>
__device__ __forceinline__ uint32_t encode_word(const float4 (&v)[32 / B / 4], int64_t e0, const EncodeParams &p,
                                                float m, float sc, uint64_t m2, uint64_t sc2) {
    constexpr int G = 32 / B / 4;
    uint32_t word = 0;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 r = philox_block((e0 >> 2) + g, p.worker, p.keys);
        uint32_t a0, a1, a2, a3;
        if constexpr (B == 1) {
            a0 = index_biased(v[g].x, m, sc, p.L, r.x);
            a1 = index_biased(v[g].y, m, sc, p.L, r.y);
            a2 = index_biased(v[g].z, m, sc, p.L, r.z);
            a3 = index_biased(v[g].w, m, sc, p.L, r.w);
        } else {
            index_biased2(v[g].x, v[g].y, m2, sc2, p.L, r.x, r.y, a0, a1);
            index_biased2(v[g].z, v[g].w, m2, sc2, p.L, r.z, r.w, a2, a3);
        }
        word += (a0 << (4 * g * B)) + (a1 << ((4 * g + 1) * B)) + (a2 << ((4 * g + 2) * B)) +
                (a3 << ((4 * g + 3) * B));
    }
    return word - pack_bias<B>();
}

template <int B>
__global__ void __launch_bounds__(kThreads) thc_encode_kernel(const __grid_constant__ EncodeParams p) {
    constexpr int E = 32 / B;  // elements per packed word
    constexpr int G = E / 4;
    const float m = p.mM[0], M = p.mM[1];
    const float sc = range_scale(m, M, p.L);
    const uint64_t m2 = pack_f2(m, m), sc2 = pack_f2(sc, sc);
    // one CTA per tile of 2 * kThreads words: words w and w + kThreads of a
    // thread, both words' loads in flight before either is quantized
    const int64_t w = static_cast<int64_t>(blockIdx.x) * (2 * kThreads) + threadIdx.x;
    const int64_t w2 = w + kThreads;
    const int64_t nfull = p.vec ? (p.N / E < p.nwords ? p.N / E : p.nwords) : 0;
    if (w2 < nfull) {
        float4 a[G], b[G];
#pragma unroll
        for (int g = 0; g < G; ++g) a[g] = __ldcs(reinterpret_cast<const float4 *>(p.x + w * E) + g);
#pragma unroll
        for (int g = 0; g < G; ++g) b[g] = __ldcs(reinterpret_cast<const float4 *>(p.x + w2 * E) + g);
        __stcs(p.packed + w, encode_word<B>(a, w * E, p, m, sc, m2, sc2));
        __stcs(p.packed + w2, encode_word<B>(b, w2 * E, p, m, sc, m2, sc2));
        return;
    }
    for (int u = 0; u < 2; ++u) {
        const int64_t wu = u == 0 ? w : w2;
        if (wu >= nfull) break;
        float4 a[G];
#pragma unroll
        for (int g = 0; g < G; ++g) a[g] = __ldcs(reinterpret_cast<const float4 *>(p.x + wu * E) + g);
        __stcs(p.packed + wu, encode_word<B>(a, wu * E, p, m, sc, m2, sc2));
    }
    // the ragged last word, or unaligned inputs: element by element
    for (int u = 0; u < 2; ++u) {
        const int64_t wr = u == 0 ? w : w2;
        if (wr < nfull || wr >= p.nwords) continue;
        const int64_t ww = wr;
        const int64_t e0 = ww * E;
        uint32_t word = 0;
        for (int g = 0; g < G; ++g) {
            const int64_t eb = e0 + 4 * g;
            if (eb >= p.N) break;
            const uint4 r = philox_block(eb >> 2, p.worker, p.keys);
            for (int i = 0; i < 4 && eb + i < p.N; ++i) {
                const uint32_t idx = index_biased(p.x[eb + i], m, sc, p.L, pick(r, i)) - kIndexBias;
                word |= idx << ((4 * g + i) * B);
            }
        }
        __stcs(p.packed + ww, word);
    }
}

// -------------------------------------------------------------- aggregate
struct AggParams {
    const uint32_t *packed[GAR_MAX_WORKERS];
    uint16_t *sums;
    int64_t N;
    int64_t nwords;
    int32_t P;
    int32_t vec;  // every packed vector and sums 16-byte aligned
};

// Sixteen-bit lanes: word bits [B*i, B*i + B) hold element i and bits
// [16 + B*i, ...) element i + 16/B, so masking with the pair mask and
// adding sums two elements per 32-bit add without carries (P*L <= 65535).
template <int B>
__global__ void __launch_bounds__(kThreads) thc_aggregate_kernel(const __grid_constant__ AggParams p) {
    constexpr int E = 32 / B;
    constexpr int K = 16 / B;  // lane-pair accumulators per word
    constexpr uint32_t kPair = ((1u << B) - 1u) | (((1u << B) - 1u) << 16);
    const int64_t ngroups = p.nwords / 4;  // whole 16-byte groups of words
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (p.vec) {
        for (int64_t g = tid; g < ngroups; g += stride) {
            if ((g + 1) * 4 * E > p.N) break;  // the group holding the tail is done below
            uint32_t acc[4][K];
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < K; ++i) acc[j][i] = 0;
            for (int w = 0; w < p.P; ++w) {
                const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(p.packed[w]) + g);
                const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int i = 0; i < K; ++i) acc[j][i] += (words[j] >> (B * i)) & kPair;
            }
            // element j*E + i is the low half of acc[j][i], element j*E + K + i the high half
            uint32_t out[4 * E / 2];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int i = 0; i < K; i += 2) {
                    out[(j * E + i) / 2] = __byte_perm(acc[j][i], acc[j][i + 1], 0x5410);
                    out[(j * E + K + i) / 2] = __byte_perm(acc[j][i], acc[j][i + 1], 0x7632);
                }
            }
            uint4 *dst = reinterpret_cast<uint4 *>(p.sums + g * 4 * E);
#pragma unroll
            for (int q = 0; q < 4 * E / 8; ++q)
                __stcs(dst + q, make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]));
        }
    }
    // elements not covered above: one element per thread
    int64_t first = 0;
    if (p.vec) {
        first = (p.N / (4 * E)) * 4 * E;
        if (first > ngroups * 4 * E) first = ngroups * 4 * E;
    }
    const uint32_t L = (1u << B) - 1u;
    for (int64_t e = first + tid; e < p.N; e += stride) {
        uint32_t s = 0;
        for (int w = 0; w < p.P; ++w) s += (p.packed[w][e / E] >> ((e % E) * B)) & L;
        p.sums[e] = static_cast<uint16_t>(s);
    }
}

// ----------------------------------------------------------------- decode
struct DecodeParams {
    const uint16_t *sums;
    const float *mM;
    float *avg;
    int64_t N;
    float L;
    float fp;  // P
    int32_t vec;
    int32_t pad;
};

__global__ void __launch_bounds__(kThreads) thc_decode_kernel(const __grid_constant__ DecodeParams p) {
    float m;
    const float k = decode_step(p.mM, p.L, p.fp, m);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    int64_t first = 0;
    if (p.vec) {
        // eight sums per 16-byte load; four loads a thread in flight before
        // the first is decoded
        const int64_t n8 = p.N / 8;
        auto decode8 = [&](const uint4 &sv, int64_t i) {
            const uint32_t w[4] = {sv.x, sv.y, sv.z, sv.w};
            float o[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                o[2 * q] = __fmaf_rn(small_to_float(w[q] & 0xFFFFu), k, m);
                o[2 * q + 1] = __fmaf_rn(small_to_float(w[q] >> 16), k, m);
            }
            float4 *dst = reinterpret_cast<float4 *>(p.avg) + 2 * i;
            __stcs(dst, make_float4(o[0], o[1], o[2], o[3]));
            __stcs(dst + 1, make_float4(o[4], o[5], o[6], o[7]));
        };
        // one CTA per tile of 4 * kThreads groups of eight: a thread's four
        // groups i, i + kThreads, ... loaded before the first is decoded
        const int64_t i = static_cast<int64_t>(blockIdx.x) * (4 * kThreads) + threadIdx.x;
        if (i + 3 * kThreads < n8) {
            uint4 sv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) sv[u] = __ldcs(reinterpret_cast<const uint4 *>(p.sums) + i + u * kThreads);
#pragma unroll
            for (int u = 0; u < 4; ++u) decode8(sv[u], i + u * kThreads);
        } else {
            for (int u = 0; u < 4; ++u)
                if (i + u * kThreads < n8) decode8(__ldcs(reinterpret_cast<const uint4 *>(p.sums) + i + u * kThreads),
                                                   i + u * kThreads);
        }
        first = n8 * 8;
    }
    for (int64_t e = first + tid; e < p.N; e += stride)  // the tail past the groups, or unaligned
        p.avg[e] = __fmaf_rn(small_to_float(p.sums[e]), k, m);
}

// The launch for p.P workers: the build fixed to that count when there is one.
int dispatch_fused(const FusedParams &p, int b, bool packed, cudaStream_t stream) {
    switch (p.P) {
        case 4: return launch_fused<4>(p, b, packed, stream);
        case 8: return launch_fused<8>(p, b, packed, stream);
        case 16: return launch_fused<16>(p, b, packed, stream);
        case 64: return launch_fused<64>(p, b, packed, stream);
        default: return launch_fused<0>(p, b, packed, stream);
    }
}
int dispatch_fused_plan(const ThcPlanParams &p, int b, bool packed, bool nmse, cudaStream_t stream) {
    switch (p.P) {
        case 4: return launch_fused_plan<4>(p, b, packed, nmse, stream);
        case 8: return launch_fused_plan<8>(p, b, packed, nmse, stream);
        case 16: return launch_fused_plan<16>(p, b, packed, nmse, stream);
        case 64: return launch_fused_plan<64>(p, b, packed, nmse, stream);
        default: return launch_fused_plan<0>(p, b, packed, nmse, stream);
    }
}

// The NMSE pair of a plan call: the n per-CTA pairs of its launches added in
// index order (fp64; each thread a fixed stride, then a fixed-order tree).
__global__ void __launch_bounds__(kThreads) thc_nmse_pair_kernel(const double *ws, int64_t n, double *pair) {
    double num = 0.0, den = 0.0;
    for (int64_t i = threadIdx.x; i < n; i += kThreads) {
        num += ws[2 * i];
        den += ws[2 * i + 1];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        num += __shfl_xor_sync(0xFFFFFFFFu, num, o);
        den += __shfl_xor_sync(0xFFFFFFFFu, den, o);
    }
    __shared__ double s_num[kThreads / 32], s_den[kThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        s_num[warp] = num;
        s_den[warp] = den;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        num = 0.0;
        den = 0.0;
        for (int i = 0; i < kThreads / 32; ++i) {
            num += s_num[i];
            den += s_den[i];
        }
        pair[0] = num;
        pair[1] = den;
    }
}

// Upper bound on the CTAs (one pair each) all launches of one plan call run:
// every piece adds at most one partial tile to the buffers' whole tiles.  A
// span of k tensors makes at most 2 k + 1 pieces; the spans hold at most
// count + S tensors in all (a tensor appears twice only across a span
// boundary), and there are at most S <= count + 2 n_buffers spans (every
// launch holds a tensor, and a buffer's last span may hold none), so at most
// 5 count + 6 n_buffers pieces.
int64_t plan_nmse_pairs_bound(const int64_t *buf_numel, int32_t n_buffers, int32_t count, int32_t b) {
    int64_t tiles = 0;
    for (int i = 0; i < n_buffers; ++i)
        tiles += ceil_div(thc_units(gar_thc_words(buf_numel[i] > 0 ? buf_numel[i] : 0, b), b), kPlanTileWords);
    return tiles + 5 * static_cast<int64_t>(count) + 6 * static_cast<int64_t>(n_buffers) + 1;
}


}  // namespace
}  // namespace gar

using namespace gar;

extern "C" int64_t gar_thc_words(int64_t N, int32_t b) {
    if (!valid_b(b) || N < 0) return 0;
    const int64_t per = 32 / b;
    return (N + per - 1) / per;
}

extern "C" int gar_thc_range(const float *const *x, int32_t P, int64_t N, float *d_mM, gar_stream_t stream_) {
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (N < 0 || !x || !d_mM) return fail(GAR_EINVAL, "N < 0 or NULL argument");
    if (!aligned(d_mM, 4)) return fail(GAR_EALIGN, "d_mM not 4-byte aligned");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    RangeParams p;
    std::memset(&p, 0, sizeof(p));
    p.N = N;
    p.mM = d_mM;
    p.status = device_status();
    p.vec = 1;
    for (int w = 0; w < P; ++w) {
        if (!x[w] && N > 0) return fail(GAR_EINVAL, "input %d is NULL", w);
        if (!aligned(x[w], 4)) return fail(GAR_EALIGN, "input %d not 4-byte aligned", w);
        p.x[w] = x[w];
        p.vec = p.vec && aligned(x[w], 16);
    }
    thc_range_init<<<1, 1, 0, stream>>>(d_mM);
    int rc = check_launch("thc_range_init");
    if (rc || N == 0) return rc;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, thc_range_kernel, kThreads, 0) != cudaSuccess || occ <= 0)
        occ = 4;
    int64_t per_worker = static_cast<int64_t>(sm_count()) * occ / P;
    const int64_t need = ceil_div(ceil_div(N, 8), kThreads);  // two float4 per thread
    if (per_worker > need) per_worker = need;
    if (per_worker < 1) per_worker = 1;
    thc_range_kernel<<<dim3(static_cast<unsigned>(per_worker), static_cast<unsigned>(P)), kThreads, 0, stream>>>(p);
    return check_launch("thc_range_kernel");
}

extern "C" int gar_thc_encode(const float *x, int64_t N, const float *d_mM, int32_t b, uint64_t seed, int32_t worker,
                              uint32_t *packed, gar_stream_t stream_) {
    if (!valid_b(b)) return fail(GAR_EINVAL, "b=%d not in {1, 2, 4, 8}", b);
    if (N < 0 || !d_mM) return fail(GAR_EINVAL, "N < 0 or d_mM NULL");
    if (N == 0) return GAR_OK;
    if (!x || !packed) return fail(GAR_EINVAL, "x or packed is NULL");
    if (worker < 0) return fail(GAR_EINVAL, "worker %d < 0", worker);
    if (!aligned(x, 4) || !aligned(packed, 4) || !aligned(d_mM, 4)) return fail(GAR_EALIGN, "misaligned pointer");
    EncodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.keys = philox_keys(seed);
    p.x = x;
    p.mM = d_mM;
    p.packed = packed;
    p.N = N;
    p.nwords = gar_thc_words(N, b);
    p.worker = worker;
    const unsigned enc_grid = static_cast<unsigned>(ceil_div(p.nwords, 2 * kThreads));
    p.vec = aligned(x, 16) ? 1 : 0;
    p.L = static_cast<float>((1 << b) - 1);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    switch (b) {
        case 1: thc_encode_kernel<1><<<enc_grid, kThreads, 0, stream>>>(p); break;
        case 2: thc_encode_kernel<2><<<enc_grid, kThreads, 0, stream>>>(p); break;
        case 4: thc_encode_kernel<4><<<enc_grid, kThreads, 0, stream>>>(p); break;
        default: thc_encode_kernel<8><<<enc_grid, kThreads, 0, stream>>>(p); break;
    }
    return check_launch("thc_encode_kernel");
}

extern "C" int gar_thc_aggregate(const uint32_t *const *packed, int32_t P, int64_t N, int32_t b, uint16_t *sums,
                                 gar_stream_t stream_) {
    if (!valid_b(b)) return fail(GAR_EINVAL, "b=%d not in {1, 2, 4, 8}", b);
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (static_cast<int64_t>(P) * ((1 << b) - 1) > 65535) return fail(GAR_EOVERFLOW, "P * (2^b - 1) > 65535");
    if (N < 0) return fail(GAR_EINVAL, "N < 0");
    if (N == 0) return GAR_OK;
    if (!packed || !sums) return fail(GAR_EINVAL, "packed or sums is NULL");
    if (!aligned(sums, 2)) return fail(GAR_EALIGN, "sums not 2-byte aligned");
    AggParams p;
    std::memset(&p, 0, sizeof(p));
    p.sums = sums;
    p.N = N;
    p.nwords = gar_thc_words(N, b);
    p.P = P;
    p.vec = aligned(sums, 16) ? 1 : 0;
    for (int w = 0; w < P; ++w) {
        if (!packed[w]) return fail(GAR_EINVAL, "packed vector %d is NULL", w);
        if (!aligned(packed[w], 4)) return fail(GAR_EALIGN, "packed vector %d not 4-byte aligned", w);
        p.packed[w] = packed[w];
        p.vec = p.vec && aligned(packed[w], 16);
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const int64_t items = p.vec ? p.nwords / 4 + 4 * (32 / b) : N;
    switch (b) {
        case 1: thc_aggregate_kernel<1><<<grid_for(thc_aggregate_kernel<1>, items), kThreads, 0, stream>>>(p); break;
        case 2: thc_aggregate_kernel<2><<<grid_for(thc_aggregate_kernel<2>, items), kThreads, 0, stream>>>(p); break;
        case 4: thc_aggregate_kernel<4><<<grid_for(thc_aggregate_kernel<4>, items), kThreads, 0, stream>>>(p); break;
        default: thc_aggregate_kernel<8><<<grid_for(thc_aggregate_kernel<8>, items), kThreads, 0, stream>>>(p); break;
    }
    return check_launch("thc_aggregate_kernel");
}

namespace gar {
namespace thc {
int launch_grid_decode(const uint16_t *sums, int64_t N, const float *d_mM, int steps, int P, float *avg,
                       cudaStream_t stream) {
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.sums = sums;
    p.mM = d_mM;
    p.avg = avg;
    p.N = N;
    p.L = static_cast<float>(steps);
    p.fp = static_cast<float>(P);
    p.vec = aligned(sums, 16) && aligned(avg, 16);
    // vector path: one CTA per 4 * kThreads groups of eight; else a resident grid
    const int64_t grid = p.vec ? std::max<int64_t>(ceil_div(ceil_div(N, 8), 4 * kThreads), 1)
                               : grid_for(thc_decode_kernel, N);
    thc_decode_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
    return check_launch("thc_decode_kernel");
}
}  // namespace thc
}  // namespace gar

extern "C" int gar_thc_decode(const uint16_t *sums, int64_t N, const float *d_mM, int32_t b, int32_t P, float *avg,
                              gar_stream_t stream_) {
    if (!valid_b(b)) return fail(GAR_EINVAL, "b=%d not in {1, 2, 4, 8}", b);
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (N < 0 || !d_mM) return fail(GAR_EINVAL, "N < 0 or d_mM NULL");
    if (N == 0) return GAR_OK;
    if (!sums || !avg) return fail(GAR_EINVAL, "sums or avg is NULL");
    if (!aligned(sums, 2) || !aligned(avg, 4) || !aligned(d_mM, 4)) return fail(GAR_EALIGN, "misaligned pointer");
    return launch_grid_decode(sums, N, d_mM, (1 << b) - 1, P, avg, reinterpret_cast<cudaStream_t>(stream_));
}

// Shared by the plain and the straggler-masked fused entry points: the
// workers whose bit is set in `arrived` contribute, each under its own id.
static int thc_fused_entry(const float *const *x, int32_t P, uint64_t arrived, int64_t N, int32_t b, uint64_t seed,
                           const float *d_mM, float *avg, uint32_t *const *packed, gar_stream_t stream_) {
    if (!valid_b(b)) return fail(GAR_EINVAL, "b=%d not in {1, 2, 4, 8}", b);
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (P < 64) arrived &= (uint64_t{1} << P) - 1u;
    const int p_eff = __builtin_popcountll(arrived);
    if (p_eff == 0) return fail(GAR_EINVAL, "no worker arrived");
    if (static_cast<int64_t>(p_eff) * ((1 << b) - 1) > 65535) return fail(GAR_EOVERFLOW, "P * (2^b - 1) > 65535");
    if (N < 0 || !d_mM || !x) return fail(GAR_EINVAL, "N < 0 or NULL argument");
    if (N == 0) return GAR_OK;
    if (!avg) return fail(GAR_EINVAL, "avg is NULL");
    if (!aligned(avg, 4) || !aligned(d_mM, 4)) return fail(GAR_EALIGN, "misaligned pointer");
    FusedParams p;
    std::memset(&p, 0, sizeof(p));
    p.keys = philox_keys(seed);
    p.mM = d_mM;
    p.avg = avg;
    p.N = N;
    p.nunits = thc_units(gar_thc_words(N, b), b);
    p.P = p_eff;
    p.L = static_cast<float>((1 << b) - 1);
    p.fp = static_cast<float>(p_eff);
    p.vec = aligned(avg, 16) ? 1 : 0;
    int slot = 0;
    for (int w = 0; w < P; ++w) {
        if (!((arrived >> w) & 1u)) continue;
        if (!x[w]) return fail(GAR_EINVAL, "input %d is NULL", w);
        if (!aligned(x[w], 4)) return fail(GAR_EALIGN, "input %d not 4-byte aligned", w);
        p.x[slot] = x[w];
        p.wid[slot] = w;
        p.vec = p.vec && aligned(x[w], 16);
        if (packed) {
            if (!packed[w]) return fail(GAR_EINVAL, "packed vector %d is NULL", w);
            if (!aligned(packed[w], 4)) return fail(GAR_EALIGN, "packed vector %d not 4-byte aligned", w);
            p.packed[slot] = packed[w];
        }
        ++slot;
    }
    return dispatch_fused(p, b, packed != nullptr, reinterpret_cast<cudaStream_t>(stream_));
}

extern "C" int gar_thc_allreduce_fused(const float *const *x, int32_t P, int64_t N, int32_t b, uint64_t seed,
                                       const float *d_mM, float *avg, uint32_t *const *packed, gar_stream_t stream) {
    return thc_fused_entry(x, P, ~uint64_t{0}, N, b, seed, d_mM, avg, packed, stream);
}

extern "C" int gar_thc_allreduce_fused_masked(const float *const *x, int32_t P, uint64_t arrived, int64_t N,
                                              int32_t b, uint64_t seed, const float *d_mM, float *avg,
                                              uint32_t *const *packed, gar_stream_t stream) {
    return thc_fused_entry(x, P, arrived, N, b, seed, d_mM, avg, packed, stream);
}

// ------------------------------------------- fused over a Tensor Fusion plan
// Builds the launches of one plan call.  A launch holds spans -- runs of
// words [w0, w1) of one fusion buffer with every tensor meeting them -- of
// as many buffers as its tables allow, so that many small buffers (a stream
// of THC partitions, each with its own range) go out in one launch, and a
// buffer with more tensors than one table holds is cut into several spans
// over several launches.
class PlanLaunches {
  public:
    PlanLaunches(ThcPlanParams &p, int P, int E, bool nmse, bool packed, double *ws, cudaStream_t stream, int b)
        : p_(p), P_(P), E_(E), nmse_(nmse), packed_(packed), ws_(ws), stream_(stream), b_(b) {
        reset();
    }

    // Tensors that one more span of this launch may hold (0: flush first).
    int seg_room() const {
        if (p_.nbuf >= kPlanBufs) return 0;
        if (packed_ && (p_.nbuf + 1) * P_ > kPlanPkPtrs) return 0;
        int room = std::min(kPlanSegs - p_.nseg, kPlanSrcPtrs / P_ - p_.nseg);
        room = std::min(room, (kPlanPieces - nraw_ - 1) / 2);  // a span of k tensors makes at most 2 k + 1 pieces
        return std::max(room, 0);
    }
    bool empty() const { return p_.nbuf == 0; }

    // One span: words [w0, w1) of buffer `bf` (N elements, wire vectors pk[slot]) and its tensors
    // idx[0 .. k) (plan order), with their source, output and reference pointers.
    void add_span(int bf, int64_t N, int64_t w0, int64_t w1, uint32_t *const *pk, const int *idx, int k,
                  const gar_seg *segs, const float *const *src, int32_t count, float *const *out,
                  const float *const *ref) {
        PlanBuf &B = p_.buf[p_.nbuf];
        B.N = N;
        B.id = bf;
        B.seg_lo = static_cast<int16_t>(p_.nseg);
        B.seg_hi = static_cast<int16_t>(p_.nseg + k);
        B.pk = packed_ ? p_.nbuf * P_ : 0;
        if (packed_)
            for (int w = 0; w < P_; ++w) p_.packed[B.pk + w] = pk[w];
        for (int j = 0; j < k; ++j) {
            const int i = idx[j], ks = p_.nseg + j;
            PlanSeg &sg = p_.seg[ks];
            sg.begin = segs[i].offset;
            sg.end = segs[i].offset + segs[i].numel;
            bool v = (sg.begin % 4 == 0) && aligned(out[i], 16) && (!nmse_ || aligned(ref[i], 16));
            for (int w = 0; w < P_; ++w) {
                const float *sp = src[static_cast<int64_t>(w) * count + i];
                p_.src[ks * P_ + w] = sp;
                v = v && aligned(sp, 16);
            }
            vec_[ks] = v;
            p_.out[ks] = out[i];
            p_.ref[ks] = nmse_ ? ref[i] : nullptr;
        }
        // pieces: per tensor its whole words, and the words between them
        int64_t cur = w0;
        const int16_t slot = static_cast<int16_t>(p_.nbuf);
        auto add = [&](int64_t a, int64_t z, int seg, int kind) {
            raw_[nraw_++] = PlanPiece{a, z, seg, static_cast<int16_t>(kind), slot};
        };
        for (int ks = B.seg_lo; ks < B.seg_hi; ++ks) {
            const int64_t fw0 = std::max(ceil_div(p_.seg[ks].begin, E_), w0);
            const int64_t fw1 = std::min(p_.seg[ks].end / E_, w1);
            if (fw0 >= fw1) continue;
            if (cur < fw0) add(cur, fw0, -1, kPieceMixed);
            add(fw0, fw1, ks, vec_[ks] ? kPieceVec : kPieceTensor);
            cur = fw1;
        }
        if (cur < w1) add(cur, w1, -1, kPieceMixed);
        p_.nseg += k;
        p_.nbuf += 1;
    }

    // Launch what has been added.  The element-by-element pieces come first
    // in tile order: a word of theirs costs many times a vector word, and
    // taking them in the first round of tiles lets the vector tiles even out
    // when the CTAs finish.
    int flush() {
        if (empty()) return GAR_OK;
        int m = 0;
        int64_t tiles = 0;
        for (int pass = 0; pass < 2; ++pass) {
            for (int i = 0; i < nraw_; ++i) {
                if ((raw_[i].kind == kPieceVec) != (pass == 1)) continue;
                p_.piece[m] = raw_[i];
                p_.tile_start[m] = tiles;
                tiles += ceil_div(raw_[i].w1 - raw_[i].w0, kPlanTileWords);
                ++m;
            }
        }
        p_.npieces = m;
        p_.tile_start[m] = tiles;
        p_.total_tiles = tiles;
        int rc = GAR_OK;
        if (tiles > 0) {
            if (nmse_) p_.nmse_ws = ws_ + 2 * used_;
            rc = dispatch_fused_plan(p_, b_, packed_, nmse_, stream_);
            used_ += plan_grid(p_);
        }
        reset();
        return rc;
    }

    int64_t used() const { return used_; }  // NMSE pairs written so far (one per CTA)

  private:
    void reset() {
        p_.nseg = 0;
        p_.nbuf = 0;
        p_.npieces = 0;
        p_.total_tiles = 0;
        nraw_ = 0;
    }
    ThcPlanParams &p_;
    int P_, E_;
    bool nmse_, packed_;
    double *ws_;
    cudaStream_t stream_;
    int b_;
    int64_t used_ = 0;
    bool vec_[kPlanSegs];
    PlanPiece raw_[kPlanPieces];
    int nraw_ = 0;
};

// Uniform THC over a plan; with ref != NULL also the NMSE pair of the call
// (per-CTA pairs in ws, added by one more kernel into d_pair).
static int thc_plan_impl(const float *const *src, int32_t P, const gar_seg *segs, const int32_t *dtype,
                         int32_t count, const int64_t *buf_numel, int32_t n_buffers, int32_t b, uint64_t seed,
                         const float *d_mM, float *const *out, uint32_t *const *packed, const float *const *ref,
                         double *d_pair, double *ws, size_t ws_bytes, gar_stream_t stream_) {
    if (!valid_b(b)) return fail(GAR_EINVAL, "b=%d not in {1, 2, 4, 8}", b);
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (static_cast<int64_t>(P) * ((1 << b) - 1) > 65535) return fail(GAR_EOVERFLOW, "P * (2^b - 1) > 65535");
    if (count < 0 || n_buffers < 0) return fail(GAR_EINVAL, "count or n_buffers < 0");
    const bool nmse = ref != nullptr;
    if (nmse) {
        if (!d_pair || !ws) return fail(GAR_EINVAL, "d_pair or the workspace is NULL");
        if (!aligned(d_pair, 8) || !aligned(ws, 8)) return fail(GAR_EALIGN, "d_pair or the workspace not 8-byte aligned");
        if (count > 0 && !buf_numel) return fail(GAR_EINVAL, "NULL argument");
        const size_t need = 16 * static_cast<size_t>(plan_nmse_pairs_bound(buf_numel, n_buffers, count, b));
        if (ws_bytes < need) return fail(GAR_EINVAL, "workspace of %zu bytes < %zu needed", ws_bytes, need);
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (count == 0) {
        if (!nmse) return GAR_OK;
        thc_nmse_pair_kernel<<<1, kThreads, 0, stream>>>(ws, 0, d_pair);  // no elements: (0, 0)
        return check_launch("thc_nmse_pair_kernel");
    }
    if (!src || !segs || !dtype || !buf_numel || !d_mM || !out) return fail(GAR_EINVAL, "NULL argument");
    if (!aligned(d_mM, 4)) return fail(GAR_EALIGN, "d_mM not 4-byte aligned");
    std::vector<int64_t> cursor(n_buffers, 0);
    std::vector<std::vector<int>> members(n_buffers);
    for (int i = 0; i < count; ++i) {
        const gar_seg &sg = segs[i];
        if (dtype[i] != GAR_F32) return fail(GAR_EDTYPE, "tensor %d is not fp32", i);
        if (sg.buffer < 0 || sg.buffer >= n_buffers) return fail(GAR_EINVAL, "tensor %d has buffer id %d", i, sg.buffer);
        if (sg.numel < 0 || sg.offset < cursor[sg.buffer] || sg.offset + sg.numel > buf_numel[sg.buffer])
            return fail(GAR_EINVAL, "tensor %d does not lie in order inside buffer %d", i, sg.buffer);
        cursor[sg.buffer] = sg.offset + sg.numel;
        if (sg.numel == 0) continue;
        if (!out[i] || !aligned(out[i], 4)) return fail(out[i] ? GAR_EALIGN : GAR_EINVAL, "output %d NULL or misaligned", i);
        for (int w = 0; w < P; ++w) {
            const float *sp = src[static_cast<int64_t>(w) * count + i];
            if (!sp) return fail(GAR_EINVAL, "worker %d tensor %d pointer is NULL", w, i);
            if (!aligned(sp, 4)) return fail(GAR_EALIGN, "worker %d tensor %d not 4-byte aligned", w, i);
        }
        if (nmse && (!ref[i] || !aligned(ref[i], 4)))
            return fail(ref[i] ? GAR_EALIGN : GAR_EINVAL, "reference %d NULL or not 4-byte aligned", i);
        members[sg.buffer].push_back(i);
    }
    std::vector<uint32_t *> pk(P, nullptr);
    if (packed) {
        for (int bf = 0; bf < n_buffers; ++bf) {
            if (members[bf].empty()) continue;
            for (int w = 0; w < P; ++w) {
                uint32_t *q = packed[static_cast<int64_t>(w) * n_buffers + bf];
                if (!q || !aligned(q, 4))
                    return fail(q ? GAR_EALIGN : GAR_EINVAL, "packed vector of worker %d buffer %d NULL or misaligned", w, bf);
            }
        }
    }
    std::unique_ptr<ThcPlanParams> p(new ThcPlanParams);  // ~30 KB: keep it off the stack
    std::memset(p.get(), 0, sizeof(ThcPlanParams));
    p->keys = philox_keys(seed);
    p->P = P;
    p->L = static_cast<float>((1 << b) - 1);
    p->fp = static_cast<float>(P);
    p->mM = d_mM;
    for (int w = 0; w < P; ++w) p->wid[w] = w;
    const int E = unit_elems_of(b);  // elements of a unit of work
    std::unique_ptr<PlanLaunches> L(new PlanLaunches(*p, P, E, nmse, packed != nullptr, ws, stream, b));
    int rc = GAR_OK;
    for (int bf = 0; bf < n_buffers && rc == GAR_OK; ++bf) {
        const std::vector<int> &mem = members[bf];
        if (mem.empty()) continue;
        if (packed)
            for (int w = 0; w < P; ++w) pk[w] = packed[static_cast<int64_t>(w) * n_buffers + bf];
        const int64_t nwords = thc_units(gar_thc_words(buf_numel[bf], b), b);  // in units
        // spans over consecutive word ranges; each one's table holds every
        // tensor that meets its words (those before `lo` end before them, those
        // from `hi` on begin after them)
        int lo = 0;
        int64_t w0 = 0;
        const int n = static_cast<int>(mem.size());
        while (w0 < nwords && rc == GAR_OK) {
            while (lo < n && segs[mem[lo]].offset + segs[mem[lo]].numel <= w0 * E) ++lo;
            const int room = L->seg_room();
            if (room == 0) {  // this launch's tables are full (never the case for an empty one)
                rc = L->flush();
                continue;
            }
            const int hi = std::min(lo + room, n);
            const int64_t w1 = hi == n ? nwords : segs[mem[hi]].offset / E;
            if (w1 <= w0) {
                if (!L->empty()) {  // a fresh launch has room for more tensors
                    rc = L->flush();
                    continue;
                }
                rc = fail(GAR_EINVAL, "more than %d tensors meet one unit of buffer %d", room, bf);
                break;
            }
            L->add_span(bf, buf_numel[bf], w0, w1, pk.data(), mem.data() + lo, hi - lo, segs, src, count, out, ref);
            w0 = w1;
        }
    }
    if (rc == GAR_OK) rc = L->flush();
    if (rc == GAR_OK && nmse) {
        thc_nmse_pair_kernel<<<1, kThreads, 0, stream>>>(ws, L->used(), d_pair);
        rc = check_launch("thc_nmse_pair_kernel");
    }
    return rc;
}

extern "C" int gar_thc_allreduce_fused_plan(const float *const *src, int32_t P, const gar_seg *segs,
                                            const int32_t *dtype, int32_t count, const int64_t *buf_numel,
                                            int32_t n_buffers, int32_t b, uint64_t seed, const float *d_mM,
                                            float *const *out, uint32_t *const *packed, gar_stream_t stream) {
    return thc_plan_impl(src, P, segs, dtype, count, buf_numel, n_buffers, b, seed, d_mM, out, packed, nullptr,
                         nullptr, nullptr, 0, stream);
}

extern "C" size_t gar_thc_plan_nmse_workspace_bytes(const int64_t *buf_numel, int32_t n_buffers, int32_t count,
                                                    int32_t b) {
    if (!valid_b(b) || n_buffers < 0 || count < 0 || (n_buffers > 0 && !buf_numel)) return 0;
    return 16 * static_cast<size_t>(plan_nmse_pairs_bound(buf_numel, n_buffers, count, b));
}

extern "C" int gar_thc_allreduce_fused_plan_nmse(const float *const *src, int32_t P, const gar_seg *segs,
                                                 const int32_t *dtype, int32_t count, const int64_t *buf_numel,
                                                 int32_t n_buffers, int32_t b, uint64_t seed, const float *d_mM,
                                                 float *const *out, uint32_t *const *packed,
                                                 const float *const *ref, double *d_pair, void *d_workspace,
                                                 size_t workspace_bytes, gar_stream_t stream) {
    if (!ref) return fail(GAR_EINVAL, "ref is NULL");
    return thc_plan_impl(src, P, segs, dtype, count, buf_numel, n_buffers, b, seed, d_mM, out, packed, ref, d_pair,
                         static_cast<double *>(d_workspace), workspace_bytes, stream);
}
