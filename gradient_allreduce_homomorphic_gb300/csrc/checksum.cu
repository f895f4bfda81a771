// checksum.cu -- checksum of a vector of 32-bit words, for silent-data-
// corruption checks of THC's wire vectors (the packed indices a worker sends
// and the parameter server receives): s1 = sum w_i and s2 = sum (i + 1) w_i,
// both mod 2^32, returned as (s2 << 32) | s1.  A flipped bit changes s1; a
// swap of words i and j changes s2 by (j - i)(w_i - w_j) mod 2^32, so it goes
// unseen only when that product is 0 mod 2^32 (e.g. words 2^16 apart whose
// values differ by a multiple of 2^16).  Both sums are associative and commutative
// mod 2^32, so the CTAs' partial sums are added with atomics and the result
// does not depend on the order.
#include "common.cuh"

namespace gar {
namespace {

constexpr int kThreads = 256;

__global__ void checksum_init(unsigned long long *out) { *out = 0ull; }

__device__ __forceinline__ void sum_word(uint32_t w, uint64_t i, uint32_t &s1, uint32_t &s2) {
    s1 += w;
    s2 += static_cast<uint32_t>(i + 1) * w;
}

// One CTA per tile of 4 * U * kThreads words (U 16-byte groups per thread);
// vec: the words are 16-byte aligned.  Every CTA ends in two same-address
// atomics, whose serial rate bounds a grid of many small tiles (at 1 GB,
// 4096-word tiles ran at half the copy rate, 16384-word tiles at the copy
// rate), so large vectors take U = 16.
template <int U>
__global__ void __launch_bounds__(kThreads) checksum_kernel(const uint32_t *w, int64_t n, int vec,
                                                            unsigned long long *out) {
    constexpr int kTileWords = 4 * U * kThreads;
    uint32_t s1 = 0, s2 = 0;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTileWords;
    if (vec && t0 + kTileWords <= n) {
        uint4 g[U];
#pragma unroll
        for (int u = 0; u < U; ++u) g[u] = ld16(w + t0 + 4 * (u * kThreads + threadIdx.x));
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t i = static_cast<uint64_t>(t0 + 4 * (u * kThreads + threadIdx.x));
            sum_word(g[u].x, i, s1, s2);
            sum_word(g[u].y, i + 1, s1, s2);
            sum_word(g[u].z, i + 2, s1, s2);
            sum_word(g[u].w, i + 3, s1, s2);
        }
    } else {  // the last tile, or unaligned words
        for (int64_t i = t0 + threadIdx.x; i < n && i < t0 + kTileWords; i += kThreads)
            sum_word(w[i], static_cast<uint64_t>(i), s1, s2);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, o);
        s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, o);
    }
    __shared__ uint32_t a1[kThreads / 32], a2[kThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        a1[warp] = s1;
        a2[warp] = s2;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int k = 1; k < kThreads / 32; ++k) {
            s1 += a1[k];
            s2 += a2[k];
        }
        // both halves wrap mod 2^32 on their own: add them as separate 32-bit words
        unsigned int *o = reinterpret_cast<unsigned int *>(out);
        atomicAdd(o, s1);      // low word: s1
        atomicAdd(o + 1, s2);  // high word: s2
    }
}

}  // namespace
}  // namespace gar

using namespace gar;

extern "C" int gar_checksum(const uint32_t *d_words, int64_t n, uint64_t *d_out, gar_stream_t stream_) {
    if (n < 0 || !d_out || (n > 0 && !d_words)) return fail(GAR_EINVAL, "n < 0 or NULL argument");
    if (!aligned(d_out, 8) || (d_words && !aligned(d_words, 4))) return fail(GAR_EALIGN, "misaligned pointer");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    unsigned long long *out = reinterpret_cast<unsigned long long *>(d_out);
    checksum_init<<<1, 1, 0, stream>>>(out);
    int rc = check_launch("checksum_init");
    if (rc || n == 0) return rc;
    const int vec = aligned(d_words, 16) ? 1 : 0;
    if (n <= (int64_t{1} << 26)) {  // up to 256 MB: 8192-word tiles keep more CTAs in flight
        checksum_kernel<8><<<static_cast<unsigned>(ceil_div(n, int64_t{4 * 8 * kThreads})), kThreads, 0, stream>>>(
            d_words, n, vec, out);
    } else {
        const int64_t blocks = ceil_div(n, int64_t{4 * 16 * kThreads});
        if (blocks > 0x7FFFFFFF) return fail(GAR_EINVAL, "n=%lld too large", static_cast<long long>(n));
        checksum_kernel<16><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(d_words, n, vec, out);
    }
    return check_launch("checksum_kernel");
}
