// nmse.cu -- NMSE(x, x_hat) = ||x - x_hat||^2 / ||x||^2 ([T] section 2).
//
// Two launches, deterministic on a given GPU (the grid is one wave of it):
// (1) each CTA folds its grid-stride slice into
// one (sum (x - x_hat)^2, sum x^2) pair of doubles in the caller's
// workspace; (2) one CTA adds the pairs in a fixed order and divides.
// Per-element terms are formed in fp32 (sixteen at a time, summed pairwise)
// and accumulated in fp64: fp64 throughput on this part is a small fraction
// of fp32, and the few fp32 roundings per term (at most 2 + 4 on the way to
// the fp64 sum, about 4e-7 relative) keep the result within 2e-6 of an
// all-fp64 sum.
#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace gar {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxBlocks = 1024;

int nmse_blocks(int64_t N) {
    int64_t g = ceil_div(ceil_div(N, 4), kThreads);
    if (g > kMaxBlocks) g = kMaxBlocks;
    return static_cast<int>(g < 1 ? 1 : g);
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Block-wide sum of two doubles in a fixed order; result valid in thread 0.
__device__ __forceinline__ void block_sum2(double &a, double &b) {
    __shared__ double s_a[kThreads / 32], s_b[kThreads / 32];
    a = warp_sum(a);
    b = warp_sum(b);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        s_a[warp] = a;
        s_b[warp] = b;
    }
    __syncthreads();
    if (warp == 0) {
        a = lane < kThreads / 32 ? s_a[lane] : 0.0;
        b = lane < kThreads / 32 ? s_b[lane] : 0.0;
        a = warp_sum(a);
        b = warp_sum(b);
    }
}

// (a - b)^2 and a^2 over the four lanes, summed pairwise in fp32
__device__ __forceinline__ float sq_diff4(const float4 &a, const float4 &b) {
    const float d0 = __fsub_rn(a.x, b.x), d1 = __fsub_rn(a.y, b.y);
    const float d2 = __fsub_rn(a.z, b.z), d3 = __fsub_rn(a.w, b.w);
    return __fadd_rn(__fadd_rn(__fmul_rn(d0, d0), __fmul_rn(d1, d1)), __fadd_rn(__fmul_rn(d2, d2), __fmul_rn(d3, d3)));
}
__device__ __forceinline__ float sq4(const float4 &a) {
    return __fadd_rn(__fadd_rn(__fmul_rn(a.x, a.x), __fmul_rn(a.y, a.y)), __fadd_rn(__fmul_rn(a.z, a.z), __fmul_rn(a.w, a.w)));
}

__global__ void __launch_bounds__(kThreads)
nmse_partial_kernel(const float *__restrict__ x, const float *__restrict__ xh, int64_t N, int vec, double *ws) {
    double num = 0.0, den = 0.0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    int64_t first = 0;
    if (vec) {
        // four float4 pairs per iteration (i + k * stride, k < 4: every load
        // coalesced, eight in flight), sixteen terms summed pairwise in fp32
        // before each fp64 accumulation: fp64 adds and conversions run at a
        // small fraction of the fp32 rate on this part, and at one per eight
        // terms they, not HBM, bounded the kernel
        const int64_t nv = N / 4;
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
        const float4 *h4 = reinterpret_cast<const float4 *>(xh);
        int64_t i = tid;
        for (; i + 3 * stride < nv; i += 4 * stride) {
            float4 a[4], b[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                a[k] = __ldcs(x4 + i + k * stride);
                b[k] = __ldcs(h4 + i + k * stride);
            }
            num += static_cast<double>(__fadd_rn(__fadd_rn(sq_diff4(a[0], b[0]), sq_diff4(a[1], b[1])),
                                                 __fadd_rn(sq_diff4(a[2], b[2]), sq_diff4(a[3], b[3]))));
            den += static_cast<double>(__fadd_rn(__fadd_rn(sq4(a[0]), sq4(a[1])), __fadd_rn(sq4(a[2]), sq4(a[3]))));
        }
        for (; i < nv; i += stride) {
            const float4 a0 = __ldcs(x4 + i), b0 = __ldcs(h4 + i);
            num += static_cast<double>(sq_diff4(a0, b0));
            den += static_cast<double>(sq4(a0));
        }
        first = nv * 4;
    }
    for (int64_t k = first + tid; k < N; k += stride) {
        const float a = x[k], d = __fsub_rn(a, xh[k]);
        num += static_cast<double>(__fmul_rn(d, d));
        den += static_cast<double>(__fmul_rn(a, a));
    }
    block_sum2(num, den);
    if (threadIdx.x == 0) {
        ws[2 * blockIdx.x] = num;
        ws[2 * blockIdx.x + 1] = den;
    }
}

// Grid of the partial kernel: one wave of the CTAs that fit on the GPU at once
// (a whole number per SM, so that every SM gets the same share of the
// grid-stride loop), never more than the workspace bound nmse_blocks(N).
// Cached per device.
int nmse_grid(int64_t N) {
    static std::atomic<int> cached[64];
    int dev = 0;
    int wave = kMaxBlocks;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        wave = cached[dev].load(std::memory_order_relaxed);
        if (wave == 0) {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, nmse_partial_kernel, kThreads, 0) !=
                    cudaSuccess ||
                per_sm < 1)
                per_sm = 1;
            const int sms = sm_count();
            const int fit = kMaxBlocks / sms;  // whole CTAs per SM within the bound
            wave = sms * (per_sm < fit ? per_sm : (fit > 0 ? fit : 1));
            if (wave > kMaxBlocks) wave = kMaxBlocks;
            cached[dev].store(wave, std::memory_order_relaxed);
        }
    }
    const int cap = nmse_blocks(N);
    return cap < wave ? cap : wave;
}

__global__ void __launch_bounds__(kThreads) nmse_final_kernel(const double *ws, int nblocks, double *out) {
    double num = 0.0, den = 0.0;
    for (int i = threadIdx.x; i < nblocks; i += kThreads) {
        num += ws[2 * i];
        den += ws[2 * i + 1];
    }
    block_sum2(num, den);
    if (threadIdx.x == 0) *out = den == 0.0 ? __longlong_as_double(0x7FF8000000000000ll) : num / den;
}

// The two sums of one range, (sum (x - x_hat)^2, sum x^2), added in the same
// fixed order as nmse_final_kernel but not divided.
__global__ void __launch_bounds__(kThreads) nmse_pair_kernel(const double *ws, int nblocks, double *pair) {
    double num = 0.0, den = 0.0;
    for (int i = threadIdx.x; i < nblocks; i += kThreads) {
        num += ws[2 * i];
        den += ws[2 * i + 1];
    }
    block_sum2(num, den);
    if (threadIdx.x == 0) {
        pair[0] = num;
        pair[1] = den;
    }
}

// NMSE from n pairs: both sums added in pair order (one thread: n is small),
// then divided.
__global__ void nmse_combine_kernel(const double *pairs, int n, double *out) {
    double num = 0.0, den = 0.0;
    for (int i = 0; i < n; ++i) {
        num += pairs[2 * i];
        den += pairs[2 * i + 1];
    }
    *out = den == 0.0 ? __longlong_as_double(0x7FF8000000000000ll) : num / den;
}

}  // namespace
}  // namespace gar

using namespace gar;

extern "C" size_t gar_nmse_workspace_bytes(int64_t N) {
    return static_cast<size_t>(nmse_blocks(N < 0 ? 0 : N)) * 2 * sizeof(double);
}

extern "C" int gar_nmse(const float *x, const float *x_hat, int64_t N, double *d_out, void *d_workspace,
                        size_t workspace_bytes, gar_stream_t stream_) {
    if (N < 0 || !d_out || !d_workspace) return fail(GAR_EINVAL, "N < 0 or NULL argument");
    if (N > 0 && (!x || !x_hat)) return fail(GAR_EINVAL, "x or x_hat is NULL");
    if (workspace_bytes < gar_nmse_workspace_bytes(N))
        return fail(GAR_EINVAL, "workspace of %zu bytes < %zu needed", workspace_bytes, gar_nmse_workspace_bytes(N));
    if (!aligned(d_workspace, 8) || !aligned(d_out, 8)) return fail(GAR_EALIGN, "workspace or d_out not 8-byte aligned");
    if ((x && !aligned(x, 4)) || (x_hat && !aligned(x_hat, 4))) return fail(GAR_EALIGN, "x or x_hat not 4-byte aligned");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const int g = nmse_grid(N);
    const int vec = aligned(x, 16) && aligned(x_hat, 16);
    double *ws = static_cast<double *>(d_workspace);
    nmse_partial_kernel<<<g, kThreads, 0, stream>>>(x, x_hat, N, vec, ws);
    int rc = check_launch("nmse_partial_kernel");
    if (rc) return rc;
    nmse_final_kernel<<<1, kThreads, 0, stream>>>(ws, g, d_out);
    return check_launch("nmse_final_kernel");
}

extern "C" int gar_nmse_sums(const float *x, const float *x_hat, int64_t N, double *d_pair, void *d_workspace,
                             size_t workspace_bytes, gar_stream_t stream_) {
    if (N < 0 || !d_pair || !d_workspace) return fail(GAR_EINVAL, "N < 0 or NULL argument");
    if (N > 0 && (!x || !x_hat)) return fail(GAR_EINVAL, "x or x_hat is NULL");
    if (workspace_bytes < gar_nmse_workspace_bytes(N))
        return fail(GAR_EINVAL, "workspace of %zu bytes < %zu needed", workspace_bytes, gar_nmse_workspace_bytes(N));
    if (!aligned(d_workspace, 8) || !aligned(d_pair, 8)) return fail(GAR_EALIGN, "workspace or d_pair not 8-byte aligned");
    if ((x && !aligned(x, 4)) || (x_hat && !aligned(x_hat, 4))) return fail(GAR_EALIGN, "x or x_hat not 4-byte aligned");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const int g = nmse_grid(N);
    const int vec = aligned(x, 16) && aligned(x_hat, 16);
    double *ws = static_cast<double *>(d_workspace);
    nmse_partial_kernel<<<g, kThreads, 0, stream>>>(x, x_hat, N, vec, ws);
    int rc = check_launch("nmse_partial_kernel");
    if (rc) return rc;
    nmse_pair_kernel<<<1, kThreads, 0, stream>>>(ws, g, d_pair);
    return check_launch("nmse_pair_kernel");
}

extern "C" int gar_nmse_combine(const double *d_pairs, int32_t n, double *d_out, gar_stream_t stream_) {
    if (n < 1 || !d_pairs || !d_out) return fail(GAR_EINVAL, "n < 1 or NULL argument");
    if (!aligned(d_pairs, 8) || !aligned(d_out, 8)) return fail(GAR_EALIGN, "d_pairs or d_out not 8-byte aligned");
    nmse_combine_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream_)>>>(d_pairs, n, d_out);
    return check_launch("nmse_combine_kernel");
}

// ---------------------------------------------------------------------------
// Allocation-free NMSE.  Some callers cannot hand this library a workspace:
// they are given their input and output buffers by someone else and may not
// call cudaMalloc themselves -- e.g. a plug-in inside a host framework whose
// allocator owns all of the device's memory, or a latency-critical path that
// must not pay cudaMalloc's implicit device-wide synchronisation.  For them the
// per-block partial sums live in the fixed array below, which is part of the
// library's image: every GPU that loads the library holds these 16 KiB until
// the process exits.  The array is shared by every call on a device and keeps
// the last call's contents; nothing in it needs to start at zero, because each
// CTA of the first kernel overwrites its own pair before the second kernel
// reads it.  Calls that overlap on the GPU (e.g. on two streams) race on it.
namespace {

constexpr int kStaticPairs = 1024;  // (sum (x - x_hat)^2, sum x^2) per CTA, at most 1024 CTAs
static_assert(kStaticPairs >= kMaxBlocks, "the static scratch must hold one pair per CTA");
static __device__ __align__(256) double g_nmse_scratch[2 * kStaticPairs];

std::mutex g_scratch_mutex;
double *g_scratch_addr[64] = {};

// Device address of g_nmse_scratch on the current device, looked up once per
// device (host code cannot use the symbol itself as a device pointer).
int static_scratch(double **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GAR_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(GAR_EINVAL, "device ordinal %d outside [0, 64)", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_nmse_scratch);
        if (e != cudaSuccess || !p)
            return fail(GAR_ECUDA, "cudaGetSymbolAddress(nmse scratch): %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = static_cast<double *>(p);
    }
    *out = g_scratch_addr[dev];
    return GAR_OK;
}

}  // namespace

extern "C" int gar_nmse_noalloc(const float *x, const float *x_hat, int64_t N, double *d_out, gar_stream_t stream_) {
    if (N < 0 || !d_out) return fail(GAR_EINVAL, "N < 0 or d_out is NULL");
    if (N > 0 && (!x || !x_hat)) return fail(GAR_EINVAL, "x or x_hat is NULL");
    const int g = nmse_grid(N);
    if (g > kStaticPairs)  // cannot happen while nmse_grid caps the grid at kMaxBlocks
        return fail(GAR_EINVAL, "N=%lld needs %d partial sums, the static scratch holds %d",
                    static_cast<long long>(N), g, kStaticPairs);
    if (!aligned(d_out, 8)) return fail(GAR_EALIGN, "d_out not 8-byte aligned");
    if ((x && !aligned(x, 4)) || (x_hat && !aligned(x_hat, 4))) return fail(GAR_EALIGN, "x or x_hat not 4-byte aligned");
    double *ws = nullptr;
    int rc = static_scratch(&ws);
    if (rc) return rc;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const int vec = aligned(x, 16) && aligned(x_hat, 16);
    nmse_partial_kernel<<<g, kThreads, 0, stream>>>(x, x_hat, N, vec, ws);
    rc = check_launch("nmse_partial_kernel");
    if (rc) return rc;
    nmse_final_kernel<<<1, kThreads, 0, stream>>>(ws, g, d_out);
    return check_launch("nmse_final_kernel");
}
