// fusion.cu -- Tensor Fusion ([H] "Tensor Fusion: Why Small Tensors Break
// Ring-Allreduce", steps 1-6): the fusion plan (host), the copy into and out
// of fusion buffers (steps 3 and 5) and the plan-driven one-pass all-reduce.
//
// Copies run as a list of byte-range jobs (a tensor into its slot, a slot
// back into a tensor, or a zero fill of an alignment gap).  Jobs are cut
// into tiles of 512 x 16-byte vectors, one CTA per tile, so a launch moves
// hundreds of tensors of any size mix at streaming bandwidth.
#include <cstring>
#include <memory>
#include <vector>

#include "common.cuh"
#include "ring.cuh"

namespace gar {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;
constexpr int kTileUnits = kThreads * kUnroll;
constexpr int kMaxJobs = 256;

struct CopyJob {
    const unsigned char *src;  // NULL: zero fill
    unsigned char *dst;
    int64_t bytes;
    int32_t unit;  // 16, 4, 2 or 1: the widest access both addresses allow
    int32_t pad;
};

struct CopyParams {
    int32_t njobs;
    int32_t pad;
    int64_t total_tiles;
    int64_t tile_start[kMaxJobs + 1];
    CopyJob job[kMaxJobs];
};
static_assert(sizeof(CopyParams) <= 32000, "copy parameters exceed the launch limit");

template <int U>
struct Word;
template <>
struct Word<16> {
    using T = uint4;
};
template <>
struct Word<4> {
    using T = uint32_t;
};
template <>
struct Word<2> {
    using T = uint16_t;
};
template <>
struct Word<1> {
    using T = unsigned char;
};

template <int U>
__device__ __forceinline__ void copy_units(const CopyJob &j, int64_t lt) {
    using T = typename Word<U>::T;
    const int64_t n = j.bytes / U;
    const T *s = reinterpret_cast<const T *>(j.src);
    T *d = reinterpret_cast<T *>(j.dst);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = lt * kTileUnits + u * kThreads + threadIdx.x;
        if (i < n) {
            T v;
            if (s) {
                if constexpr (U == 16) v = __ldcs(s + i);
                else v = s[i];
            } else {
                v = T{};
            }
            if constexpr (U == 16) __stcs(d + i, v);
            else d[i] = v;
        }
    }
    if (lt == 0) {  // bytes past the last whole unit
        const int64_t rem = j.bytes - n * U;
        if (threadIdx.x < rem) {
            const int64_t k = n * U + threadIdx.x;
            j.dst[k] = j.src ? j.src[k] : static_cast<unsigned char>(0);
        }
    }
}

__global__ void __launch_bounds__(kThreads) copy_jobs_kernel(const __grid_constant__ CopyParams p) {
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        int lo = 0, hi = p.njobs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.tile_start[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        const CopyJob &j = p.job[lo];
        const int64_t lt = t - p.tile_start[lo];
        switch (j.unit) {
            case 16: copy_units<16>(j, lt); break;
            case 4: copy_units<4>(j, lt); break;
            case 2: copy_units<2>(j, lt); break;
            default: copy_units<1>(j, lt); break;
        }
    }
}

int widest_unit(const void *s, const void *d) {
    for (int u : {16, 4, 2}) {
        if ((!s || aligned(s, u)) && aligned(d, u)) return u;
    }
    return 1;
}

class CopyBatch {
  public:
    explicit CopyBatch(cudaStream_t s) : stream_(s), p_(new CopyParams) { std::memset(p_, 0, sizeof(CopyParams)); }
    ~CopyBatch() { delete p_; }
    int add(const void *src, void *dst, int64_t bytes) {
        if (bytes <= 0) return GAR_OK;
        if (p_->njobs == kMaxJobs) {
            const int rc = flush();
            if (rc) return rc;
        }
        CopyJob &j = p_->job[p_->njobs++];
        j.src = static_cast<const unsigned char *>(src);
        j.dst = static_cast<unsigned char *>(dst);
        j.bytes = bytes;
        j.unit = widest_unit(src, dst);
        j.pad = 0;
        return GAR_OK;
    }
    int flush() {
        if (p_->njobs == 0) return GAR_OK;
        int64_t tiles = 0;
        for (int i = 0; i < p_->njobs; ++i) {
            p_->tile_start[i] = tiles;
            const int64_t t = ceil_div(p_->job[i].bytes / p_->job[i].unit, kTileUnits);
            tiles += t > 0 ? t : 1;
        }
        p_->tile_start[p_->njobs] = tiles;
        p_->total_tiles = tiles;
        // one CTA per tile: the block scheduler balances the SMs (as for the ring fold)
        const int64_t grid = tiles < 0x7FFFFFFF ? tiles : 0x7FFFFFFF;
        copy_jobs_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream_>>>(*p_);
        p_->njobs = 0;
        return check_launch("copy_jobs_kernel");
    }

  private:
    cudaStream_t stream_;
    CopyParams *p_;
};

// ------------------------------------------------- all workers, one pass
// One row per tensor: P source pointers (the workers' copies of the tensor)
// and P destination pointers (each worker's fusion buffer at the tensor's
// offset).  Tile 0 of a row also zero-fills the row's alignment gap.  With
// a range output every tile folds its values (and the gap zeros) into the
// buffer's global [min, max], THC's preliminary round, while copying.
struct PackRow {
    int32_t buffer;
    int32_t vec;   // every pointer of the row 16-byte aligned
    int32_t gap;   // zero elements after the tensor, up to the next one's offset
    int32_t pad;
    int64_t numel;
};

constexpr int kPackPtrs = 1024, kPackRows = 256;
struct PackAllParams {
    int32_t P;
    int32_t nrows;
    int32_t pad0;
    int32_t pad1;
    float *mM;  // [n_buffers][2] or NULL
    unsigned int *status;  // with a range: GAR_STATUS_NONFINITE raised here
    int64_t total_tiles;
    int64_t tile_start[kPackRows + 1];
    PackRow row[kPackRows];
    const void *src[kPackPtrs];  // src[row * P + w]
    void *dst[kPackPtrs];        // dst[row * P + w]
};
static_assert(sizeof(PackAllParams) <= 32000, "pack parameters exceed the launch limit");

constexpr int kPackBatch = 8;  // worker vectors in flight per thread

template <typename T>
struct PackElem;
template <>
struct PackElem<float> {
    static constexpr int kVec = 4;
    __device__ static void range(const uint4 &r, float &lo, float &hi, float &chk) {
        const float a = __uint_as_float(r.x), b = __uint_as_float(r.y), c = __uint_as_float(r.z),
                    d = __uint_as_float(r.w);
        lo = fminf(lo, fminf(fminf(a, b), fminf(c, d)));
        hi = fmaxf(hi, fmaxf(fmaxf(a, b), fmaxf(c, d)));
        chk = nonfinite_acc(nonfinite_acc(nonfinite_acc(nonfinite_acc(chk, a), b), c), d);
    }
};
template <>
struct PackElem<uint16_t> {
    static constexpr int kVec = 8;
    __device__ static void range(const uint4 &, float &, float &, float &) {}
};

__device__ __forceinline__ void atomic_min_f(float *a, float v) {
    if ((__float_as_uint(v) >> 31) == 0u) atomicMin(reinterpret_cast<int *>(a), __float_as_int(v));
    else atomicMax(reinterpret_cast<unsigned int *>(a), __float_as_uint(v));
}
__device__ __forceinline__ void atomic_max_f(float *a, float v) {
    if ((__float_as_uint(v) >> 31) == 0u) atomicMax(reinterpret_cast<int *>(a), __float_as_int(v));
    else atomicMin(reinterpret_cast<unsigned int *>(a), __float_as_uint(v));
}

struct RangeInitParams {
    float *mM;
    int32_t n;
    int32_t ids[255];  // buffers whose range entries are reset
};

__global__ void pack_range_init(const __grid_constant__ RangeInitParams p) {
    for (int i = threadIdx.x; i < p.n; i += blockDim.x) {
        p.mM[2 * p.ids[i]] = __int_as_float(0x7F800000);       // +inf
        p.mM[2 * p.ids[i] + 1] = __int_as_float(0xFF800000u);  // -inf
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) pack_all_kernel(const __grid_constant__ PackAllParams p) {
    constexpr int V = PackElem<T>::kVec;
    const bool want_range = p.mM != nullptr;
    __shared__ float s_lo[kThreads / 32], s_hi[kThreads / 32];
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        int lo_i = 0, hi_i = p.nrows - 1;
        while (lo_i < hi_i) {
            const int mid = (lo_i + hi_i + 1) >> 1;
            if (p.tile_start[mid] <= t) lo_i = mid;
            else hi_i = mid - 1;
        }
        const PackRow r = p.row[lo_i];
        const int64_t lt = t - p.tile_start[lo_i];
        const void *const *src = p.src + static_cast<int64_t>(lo_i) * p.P;
        void *const *dst = p.dst + static_cast<int64_t>(lo_i) * p.P;
        float lo = __int_as_float(0x7F800000), hi = __int_as_float(0xFF800000u);
        float chk = 0.0f;  // NaN once a non-finite input is seen
        const int64_t nvec = r.vec ? r.numel / V : 0;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = lt * kTileUnits + u * kThreads + threadIdx.x;
            if (i < nvec) {
                for (int w0 = 0; w0 < p.P; w0 += kPackBatch) {
                    uint4 v[kPackBatch];
#pragma unroll
                    for (int j = 0; j < kPackBatch; ++j)
                        if (w0 + j < p.P) v[j] = ld16(static_cast<const T *>(src[w0 + j]) + i * V);
#pragma unroll
                    for (int j = 0; j < kPackBatch; ++j) {
                        if (w0 + j < p.P) {
                            st16(static_cast<T *>(dst[w0 + j]) + i * V, v[j]);
                            if (want_range) PackElem<T>::range(v[j], lo, hi, chk);
                        }
                    }
                }
            }
        }
        if (!r.vec) {  // unaligned row: element by element
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t e = lt * kTileUnits + u * kThreads + threadIdx.x;
                if (e < r.numel) {
                    for (int w = 0; w < p.P; ++w) {
                        const T v = static_cast<const T *>(src[w])[e];
                        static_cast<T *>(dst[w])[e] = v;
                        if constexpr (sizeof(T) == 4) {
                            lo = fminf(lo, v);
                            hi = fmaxf(hi, v);
                            chk = nonfinite_acc(chk, v);
                        }
                    }
                }
            }
        }
        if (lt == 0) {  // vector tail of the tensor, then the zero gap after it
            // (an unaligned row has copied every element above: no tail, the gap starts at numel)
            const int64_t tail0 = r.vec ? nvec * V : r.numel;
            const int64_t ntail = r.numel - tail0;
            for (int64_t k = threadIdx.x; k < ntail + r.gap; k += kThreads) {
                for (int w = 0; w < p.P; ++w) {
                    T v;
                    if (k < ntail) {
                        v = static_cast<const T *>(src[w])[tail0 + k];
                    } else {
                        v = T{};
                    }
                    static_cast<T *>(dst[w])[tail0 + k] = v;
                    if constexpr (sizeof(T) == 4) {
                        lo = fminf(lo, static_cast<float>(v));
                        hi = fmaxf(hi, static_cast<float>(v));
                        chk = nonfinite_acc(chk, static_cast<float>(v));
                    }
                }
            }
        }
        if (want_range) {  // uniform branch: one pair of atomics per tile
            flag_nonfinite_warp(p.status, chk);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
                hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
            }
            const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
            __syncthreads();  // the previous tile's readers are done with s_lo/s_hi
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
                    if (lo == lo) atomic_min_f(p.mM + 2 * r.buffer, lo);
                    if (hi == hi) atomic_max_f(p.mM + 2 * r.buffer + 1, hi);
                }
            }
        }
    }
}

template <typename T>
int launch_pack_all(PackAllParams &p, cudaStream_t stream) {
    constexpr int V = PackElem<T>::kVec;
    int64_t tiles = 0;
    for (int i = 0; i < p.nrows; ++i) {
        p.tile_start[i] = tiles;
        const int64_t units = p.row[i].vec ? p.row[i].numel / V : p.row[i].numel;
        const int64_t t = ceil_div(units, kTileUnits);
        tiles += t > 0 ? t : 1;
    }
    p.tile_start[p.nrows] = tiles;
    p.total_tiles = tiles;
    // one CTA per tile: the block scheduler balances the SMs (as for the ring fold)
    const int64_t grid = tiles < 0x7FFFFFFF ? tiles : 0x7FFFFFFF;
    pack_all_kernel<T><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
    return check_launch("pack_all_kernel");
}

// Checks shared by pack / unpack: the buffer's tensors, their common dtype.
int buffer_members(const gar_seg *segs, const int32_t *dtype, int32_t count, int32_t buffer,
                   std::vector<int> &members, int &es) {
    if (!segs || !dtype || count < 0) return fail(GAR_EINVAL, "segs/dtype NULL or count < 0");
    if (buffer < 0) return fail(GAR_EINVAL, "buffer id %d < 0", buffer);
    int dt = -1;
    for (int i = 0; i < count; ++i) {
        if (segs[i].buffer != buffer) continue;
        if (elem_bytes(dtype[i]) < 0) return fail(GAR_EDTYPE, "tensor %d has unknown dtype %d", i, dtype[i]);
        if (dt >= 0 && dtype[i] != dt) return fail(GAR_EDTYPE, "buffer %d mixes dtypes", buffer);
        if (segs[i].offset < 0 || segs[i].numel < 0) return fail(GAR_EINVAL, "tensor %d has a negative offset/numel", i);
        dt = dtype[i];
        members.push_back(i);
    }
    es = dt >= 0 ? elem_bytes(dt) : 4;
    return GAR_OK;
}

}  // namespace
}  // namespace gar

using namespace gar;

extern "C" int gar_fusion_plan(const int64_t *numel, const int32_t *dtype, int32_t count, int64_t capacity_bytes,
                               int32_t align_bytes, gar_seg *segs, int32_t *n_buffers, int64_t *buf_numel) {
    if (count < 0) return fail(GAR_EINVAL, "count %d < 0", count);
    if (count > 0 && (!numel || !dtype || !segs || !buf_numel)) return fail(GAR_EINVAL, "NULL plan array");
    if (!n_buffers) return fail(GAR_EINVAL, "n_buffers is NULL");
    if (capacity_bytes <= 0) return fail(GAR_EINVAL, "capacity %lld <= 0", static_cast<long long>(capacity_bytes));
    if (align_bytes <= 0) return fail(GAR_EINVAL, "alignment %d <= 0", align_bytes);
    int32_t open = -1;       // id of the open buffer
    int32_t open_dtype = -1;
    int64_t fill = 0;        // bytes used in the open buffer
    for (int32_t i = 0; i < count; ++i) {
        const int es = elem_bytes(dtype[i]);
        if (es < 0) return fail(GAR_EDTYPE, "tensor %d has unknown dtype %d", i, dtype[i]);
        if (numel[i] < 0) return fail(GAR_EINVAL, "tensor %d has numel < 0", i);
        if (align_bytes % es) return fail(GAR_EINVAL, "alignment %d is not a multiple of %d", align_bytes, es);
        const int64_t bytes = numel[i] * es;
        const int64_t at = ceil_div(fill, align_bytes) * align_bytes;
        const bool joins = open >= 0 && dtype[i] == open_dtype && at + bytes <= capacity_bytes;
        int64_t start = at;
        if (!joins) {  // close the open buffer (if any), open the next one
            ++open;
            open_dtype = dtype[i];
            start = 0;
        }
        segs[i].buffer = open;
        segs[i].reserved = 0;
        segs[i].offset = start / es;
        segs[i].numel = numel[i];
        fill = start + bytes;
        buf_numel[open] = fill / es;
    }
    *n_buffers = open + 1;
    return GAR_OK;
}

extern "C" int gar_fusion_pack(const void *const *src, const gar_seg *segs, const int32_t *dtype, int32_t count,
                               int32_t buffer, void *fusion_buf, int64_t buf_numel, gar_stream_t stream) {
    std::vector<int> members;
    int es = 4;
    int rc = buffer_members(segs, dtype, count, buffer, members, es);
    if (rc) return rc;
    if (buf_numel < 0) return fail(GAR_EINVAL, "buf_numel < 0");
    if (buf_numel > 0 && !fusion_buf) return fail(GAR_EINVAL, "fusion_buf is NULL");
    if (!members.empty() && !src) return fail(GAR_EINVAL, "src is NULL");
    if (fusion_buf && !aligned(fusion_buf, es)) return fail(GAR_EALIGN, "fusion_buf not aligned to %d bytes", es);
    CopyBatch batch(reinterpret_cast<cudaStream_t>(stream));
    unsigned char *base = static_cast<unsigned char *>(fusion_buf);
    int64_t cursor = 0;  // element where the next zero gap starts
    for (int i : members) {
        const gar_seg &s = segs[i];
        if (s.offset < cursor || s.offset + s.numel > buf_numel)
            return fail(GAR_EINVAL, "tensor %d does not lie in order inside buffer %d", i, buffer);
        if (s.numel > 0 && !src[i]) return fail(GAR_EINVAL, "source tensor %d is NULL", i);
        if (s.numel > 0 && !aligned(src[i], es)) return fail(GAR_EALIGN, "source tensor %d not aligned", i);
    }
    for (int i : members) {
        const gar_seg &s = segs[i];
        if ((rc = batch.add(nullptr, base + cursor * es, (s.offset - cursor) * es))) return rc;
        if ((rc = batch.add(src[i], base + s.offset * es, s.numel * es))) return rc;
        cursor = s.offset + s.numel;
    }
    if ((rc = batch.add(nullptr, base + cursor * es, (buf_numel - cursor) * es))) return rc;
    return batch.flush();
}

extern "C" int gar_fusion_unpack(const void *fusion_buf, const gar_seg *segs, const int32_t *dtype, int32_t count,
                                 int32_t buffer, void *const *dst, gar_stream_t stream) {
    std::vector<int> members;
    int es = 4;
    int rc = buffer_members(segs, dtype, count, buffer, members, es);
    if (rc) return rc;
    if (members.empty()) return GAR_OK;
    if (!fusion_buf || !dst) return fail(GAR_EINVAL, "fusion_buf or dst is NULL");
    if (!aligned(fusion_buf, es)) return fail(GAR_EALIGN, "fusion_buf not aligned to %d bytes", es);
    for (int i : members) {
        if (segs[i].numel > 0 && !dst[i]) return fail(GAR_EINVAL, "destination tensor %d is NULL", i);
        if (segs[i].numel > 0 && !aligned(dst[i], es)) return fail(GAR_EALIGN, "destination tensor %d not aligned", i);
    }
    CopyBatch batch(reinterpret_cast<cudaStream_t>(stream));
    const unsigned char *base = static_cast<const unsigned char *>(fusion_buf);
    for (int i : members)
        if ((rc = batch.add(base + segs[i].offset * es, dst[i], segs[i].numel * es))) return rc;
    return batch.flush();
}

extern "C" int gar_fusion_pack_all(const void *const *src, int32_t P, const gar_seg *segs, const int32_t *dtype,
                                   int32_t count, void *const *fusion_bufs, const int64_t *buf_numel,
                                   int32_t n_buffers, float *d_mM, gar_stream_t stream_) {
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (count < 0 || n_buffers < 0) return fail(GAR_EINVAL, "count or n_buffers < 0");
    if (count > 0 && (!src || !segs || !dtype || !fusion_bufs || !buf_numel)) return fail(GAR_EINVAL, "NULL argument");
    if (d_mM && !aligned(d_mM, 4)) return fail(GAR_EALIGN, "d_mM not 4-byte aligned");
    std::vector<int32_t> buf_dt(n_buffers, -1);
    std::vector<int> last(n_buffers, -1);  // last tensor of each buffer so far
    std::vector<int> first(n_buffers, -1);
    for (int i = 0; i < count; ++i) {
        const gar_seg &s = segs[i];
        const int es = elem_bytes(dtype[i]);
        if (es < 0) return fail(GAR_EDTYPE, "tensor %d has unknown dtype %d", i, dtype[i]);
        if (s.buffer < 0 || s.buffer >= n_buffers) return fail(GAR_EINVAL, "tensor %d has buffer id %d", i, s.buffer);
        if (buf_dt[s.buffer] >= 0 && buf_dt[s.buffer] != dtype[i]) return fail(GAR_EDTYPE, "buffer %d mixes dtypes", s.buffer);
        if (d_mM && dtype[i] != GAR_F32) return fail(GAR_EDTYPE, "a range is only computed over fp32 buffers");
        buf_dt[s.buffer] = dtype[i];
        const int prev = last[s.buffer];
        const int64_t cursor = prev < 0 ? 0 : segs[prev].offset + segs[prev].numel;
        if (s.numel < 0 || s.offset < cursor || s.offset + s.numel > buf_numel[s.buffer])
            return fail(GAR_EINVAL, "tensor %d does not lie in order inside buffer %d", i, s.buffer);
        if (first[s.buffer] < 0) first[s.buffer] = i;
        last[s.buffer] = i;
        for (int w = 0; w < P; ++w) {
            const void *sp = src[static_cast<int64_t>(w) * count + i];
            if (s.numel > 0 && !sp) return fail(GAR_EINVAL, "worker %d tensor %d pointer is NULL", w, i);
            if (!aligned(sp, es)) return fail(GAR_EALIGN, "worker %d tensor %d not aligned", w, i);
        }
    }
    for (int b = 0; b < n_buffers; ++b) {
        if (buf_numel[b] < 0) return fail(GAR_EINVAL, "buffer %d has negative length", b);
        const int es = buf_dt[b] >= 0 ? elem_bytes(buf_dt[b]) : 4;
        for (int w = 0; w < P; ++w) {
            void *fb = fusion_bufs[static_cast<int64_t>(w) * n_buffers + b];
            if (buf_numel[b] > 0 && !fb) return fail(GAR_EINVAL, "worker %d fusion buffer %d is NULL", w, b);
            if (!aligned(fb, es)) return fail(GAR_EALIGN, "worker %d fusion buffer %d not aligned", w, b);
        }
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (d_mM) {  // reset the range entries of the buffers this call packs
        RangeInitParams ip;
        std::memset(&ip, 0, sizeof(ip));
        ip.mM = d_mM;
        for (int b = 0; b <= n_buffers; ++b) {
            const bool last = b == n_buffers;
            if (!last && first[b] >= 0) ip.ids[ip.n++] = b;
            if (ip.n > 0 && (last || ip.n == 255)) {
                pack_range_init<<<1, 256, 0, stream>>>(ip);
                const int rc = check_launch("pack_range_init");
                if (rc) return rc;
                ip.n = 0;
            }
        }
    }
    std::unique_ptr<PackAllParams> p(new PackAllParams);  // ~30 KB: keep it off the stack
    int rc = GAR_OK;
    for (int pass_dtype = 0; pass_dtype < 2 && rc == GAR_OK; ++pass_dtype) {
        std::memset(p.get(), 0, sizeof(PackAllParams));
        p->P = P;
        p->mM = d_mM;
        p->status = d_mM ? device_status() : nullptr;
        const int es = elem_bytes(pass_dtype);
        auto flush = [&]() -> int {
            if (p->nrows == 0) return GAR_OK;
            const int r = pass_dtype == GAR_F32 ? launch_pack_all<float>(*p, stream) : launch_pack_all<uint16_t>(*p, stream);
            p->nrows = 0;
            return r;
        };
        auto add_row = [&](int buffer, int64_t dst_elem, int64_t numel, int64_t gap, int tensor) -> int {
            if ((p->nrows + 1) * P > kPackPtrs || p->nrows + 1 > kPackRows) {
                const int r = flush();
                if (r) return r;
            }
            PackRow &row = p->row[p->nrows];
            row.buffer = buffer;
            row.numel = numel;
            row.gap = static_cast<int32_t>(gap);
            row.pad = 0;
            bool vec = true;
            for (int w = 0; w < P; ++w) {
                const void *sp = tensor >= 0 ? src[static_cast<int64_t>(w) * count + tensor] : nullptr;
                unsigned char *fb = static_cast<unsigned char *>(fusion_bufs[static_cast<int64_t>(w) * n_buffers + buffer]);
                void *dp = fb + dst_elem * es;
                vec = vec && aligned(sp, 16) && aligned(dp, 16);
                p->src[p->nrows * P + w] = sp;
                p->dst[p->nrows * P + w] = dp;
            }
            row.vec = vec ? 1 : 0;
            ++p->nrows;
            return GAR_OK;
        };
        for (int b = 0; b < n_buffers && rc == GAR_OK; ++b) {
            // buffers that none of the given tensors belong to are left untouched,
            // so a caller can pack one buffer at a time with a slice of the plan
            if (buf_dt[b] != pass_dtype || first[b] < 0) continue;
            const int f = first[b];
            const int64_t lead = segs[f].offset;
            if (lead > 0) {  // zeros before the buffer's first tensor (none in plans from gar_fusion_plan)
                for (int64_t z = 0; z < lead && rc == GAR_OK; z += (1 << 30))
                    rc = add_row(b, z, 0, lead - z < (1 << 30) ? lead - z : (1 << 30), -1);
            }
        }
        for (int i = 0; i < count && rc == GAR_OK; ++i) {
            if (dtype[i] != pass_dtype) continue;
            const gar_seg &s = segs[i];
            // the gap runs to the next tensor of the same buffer, or to the buffer's end
            int64_t next = buf_numel[s.buffer];
            for (int j = i + 1; j < count; ++j)
                if (segs[j].buffer == s.buffer) {
                    next = segs[j].offset;
                    break;
                }
            const int64_t gap = next - (s.offset + s.numel);
            if (gap >= (1 << 30)) {
                rc = fail(GAR_EINVAL, "gap after tensor %d too large", i);
                break;
            }
            rc = add_row(s.buffer, s.offset, s.numel, gap, i);
        }
        if (rc == GAR_OK) rc = flush();
    }
    return rc;
}

static int fused_allreduce_entry(const void *const *src, void *const *dst, int32_t P, const gar_seg *segs,
                                 const int32_t *dtype, int32_t count, const int64_t *buf_numel, int32_t n_buffers,
                                 int32_t op, float *d_mM, gar_stream_t stream) {
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (op != GAR_SUM && op != GAR_AVG) return fail(GAR_EINVAL, "unknown op %d", op);
    if (count < 0 || n_buffers < 0) return fail(GAR_EINVAL, "count or n_buffers < 0");
    if (count == 0) return GAR_OK;
    if (!src || !dst || !segs || !dtype || !buf_numel) return fail(GAR_EINVAL, "NULL argument");
    std::vector<int32_t> buf_dt(n_buffers, -1);
    std::vector<int64_t> cursor(n_buffers, 0);
    for (int i = 0; i < count; ++i) {
        const gar_seg &s = segs[i];
        const int es = elem_bytes(dtype[i]);
        if (es < 0) return fail(GAR_EDTYPE, "tensor %d has unknown dtype %d", i, dtype[i]);
        if (s.buffer < 0 || s.buffer >= n_buffers) return fail(GAR_EINVAL, "tensor %d has buffer id %d", i, s.buffer);
        if (buf_dt[s.buffer] >= 0 && buf_dt[s.buffer] != dtype[i]) return fail(GAR_EDTYPE, "buffer %d mixes dtypes", s.buffer);
        if (d_mM && dtype[i] != GAR_F32) return fail(GAR_EDTYPE, "a range is only computed over fp32 buffers");
        buf_dt[s.buffer] = dtype[i];
        if (s.numel < 0 || s.offset < cursor[s.buffer] || s.offset + s.numel > buf_numel[s.buffer])
            return fail(GAR_EINVAL, "tensor %d does not lie in order inside buffer %d", i, s.buffer);
        cursor[s.buffer] = s.offset + s.numel;
        if (s.numel == 0) continue;
        for (int w = 0; w < P; ++w) {
            const void *sp = src[static_cast<int64_t>(w) * count + i];
            const void *dp = dst[static_cast<int64_t>(w) * count + i];
            if (!sp || !dp) return fail(GAR_EINVAL, "worker %d tensor %d pointer is NULL", w, i);
            if (!aligned(sp, es) || !aligned(dp, es)) return fail(GAR_EALIGN, "worker %d tensor %d not aligned", w, i);
        }
    }
    if (d_mM && !aligned(d_mM, 4)) return fail(GAR_EALIGN, "d_mM not 4-byte aligned");
    return fused_allreduce_impl(src, dst, P, segs, dtype, count, buf_numel, n_buffers, op, d_mM,
                                reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int gar_fused_allreduce(const void *const *src, void *const *dst, int32_t P, const gar_seg *segs,
                                   const int32_t *dtype, int32_t count, const int64_t *buf_numel, int32_t n_buffers,
                                   int32_t op, gar_stream_t stream) {
    return fused_allreduce_entry(src, dst, P, segs, dtype, count, buf_numel, n_buffers, op, nullptr, stream);
}

extern "C" int gar_fused_allreduce_range(const void *const *src, void *const *dst, int32_t P, const gar_seg *segs,
                                         const int32_t *dtype, int32_t count, const int64_t *buf_numel,
                                         int32_t n_buffers, int32_t op, float *d_mM, gar_stream_t stream) {
    if (!d_mM && count > 0) return fail(GAR_EINVAL, "d_mM is NULL");
    return fused_allreduce_entry(src, dst, P, segs, dtype, count, buf_numel, n_buffers, op, d_mM, stream);
}
