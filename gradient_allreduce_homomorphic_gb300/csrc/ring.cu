// ring.cu -- ring all-reduce of P worker buffers held in one GPU's HBM.
//
// Ring all-reduce ([H] "The Ring-Allreduce Algorithm"; [R] sections 4, 5, 7):
// the buffer is cut into P chunks; in P-1 scatter-reduce steps chunk c
// travels c -> c+1 -> ... gaining each worker's addend, and in P-1
// all-gather steps the finished chunk is copied around the ring.  On one
// GPU the "wire" is HBM, so the whole schedule collapses into one pass: for
// every element, load the P workers' values, fold them in fp32 in the ring
// order of the element's chunk (x_c, x_{c+1}, ..., x_{c+P-1}, indices mod P)
// and store the result to every destination.  IEEE addition is commutative,
// so this matches the literal schedule bit for bit; its traffic is the
// minimum (each input read once, each output written once).
//
// Work decomposition: the element range is cut into "pieces" -- runs of one
// tensor that lie in one ring chunk -- so the chunk (the fold's starting
// worker) is uniform over a piece and never computed per element.  Pieces are
// cut into tiles of 512 x 16-byte vectors; CTAs stride over the flattened
// tile list.  The same kernel serves a single buffer (one tensor, P pieces)
// and a whole Tensor Fusion plan (every tensor of every fusion buffer, split
// at that buffer's chunk boundaries), where it reads the workers' tensors and
// writes their results directly: pack, all-reduce and unpack in one pass.
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
constexpr int kLoadBatch = 8;  // worker vectors in flight per thread before folding
constexpr int kRangeMinBlocks = 4;  // CTAs per SM the range variant is built for

template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static constexpr int kVec = 4;  // elements per 16 bytes
    __device__ static void unpack(const uint4 &r, float (&v)[4]) {
        v[0] = __uint_as_float(r.x);
        v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z);
        v[3] = __uint_as_float(r.w);
    }
    __device__ static uint4 pack(const float (&v)[4]) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
    }
    __device__ static float load1(const void *p, int64_t e) { return __ldcs(static_cast<const float *>(p) + e); }
    __device__ static void store1(void *p, int64_t e, float v) { __stcs(static_cast<float *>(p) + e, v); }
};
template <>
struct Elem<uint16_t> {  // bf16 storage
    static constexpr int kVec = 8;
    __device__ static void unpack(const uint4 &r, float (&v)[8]) {
        v[0] = bf16_lo(r.x);
        v[1] = bf16_hi(r.x);
        v[2] = bf16_lo(r.y);
        v[3] = bf16_hi(r.y);
        v[4] = bf16_lo(r.z);
        v[5] = bf16_hi(r.z);
        v[6] = bf16_lo(r.w);
        v[7] = bf16_hi(r.w);
    }
    __device__ static uint4 pack(const float (&v)[8]) {
        return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                          pack_bf16x2(v[6], v[7]));
    }
    __device__ static float load1(const void *p, int64_t e) {
        return bf16_one(__ldcs(reinterpret_cast<const unsigned short *>(p) + e));
    }
    __device__ static void store1(void *p, int64_t e, float v) {
        __stcs(reinterpret_cast<unsigned short *>(p) + e, static_cast<unsigned short>(to_bf16(v)));
    }
};

template <class Prm>
__device__ __forceinline__ float finish(const Prm &p, float s) {
    if (p.mode == kModeMulInv) return __fmul_rn(s, p.inv_p);  // exact: P is a power of two
    if (p.mode == kModeDiv) return __fdiv_rn(s, p.fp);
    return s;
}

// Worker at position k of the fold that starts at worker c: c + k, or c - k
// on the counter-clockwise ring (indices mod P).
__device__ __forceinline__ int ring_worker(int c, int k, int ccw, int P) {
    int w = ccw ? c - k : c + k;
    w += (w < 0) ? P : 0;
    w -= (w >= P) ? P : 0;
    return w;
}

// min / max over every input value seen, for the THC range of a fusion buffer
// (fminf / fmaxf: NaN inputs are skipped, as in the packing kernel)
struct Range {
    float lo, hi;
    float chk;  // NaN once a non-finite input is seen
    __device__ __forceinline__ Range() {
        lo = __int_as_float(0x7F800000);   // +inf
        hi = __int_as_float(0xFF800000u);  // -inf
        chk = 0.0f;
    }
    __device__ __forceinline__ void add(float v) {
        lo = fminf(lo, v);
        hi = fmaxf(hi, v);
        chk = nonfinite_acc(chk, v);
    }
    // two values per instruction: sm_100's three-input min / max (NaN
    // inputs are skipped, as by fminf / fmaxf)
    __device__ __forceinline__ void add2(float a, float b) {
        asm("min.f32 %0, %0, %1, %2;" : "+f"(lo) : "f"(a), "f"(b));
        asm("max.f32 %0, %0, %1, %2;" : "+f"(hi) : "f"(a), "f"(b));
        chk = nonfinite_acc(nonfinite_acc(chk, a), b);
    }
    template <int V>
    __device__ __forceinline__ void add_vec(const float (&v)[V]) {
#pragma unroll
        for (int q = 0; q < V; q += 2) add2(v[q], v[q + 1]);
    }
};

// The workers of one tile's fold, in ring order from the piece's chunk
// (src[k] = the input of worker (c + k) mod P, or (c - k) mod P on the
// counter-clockwise ring), and the row's destinations: set once per tile in
// shared memory, so that each load and store takes one broadcast shared load
// for its pointer instead of the ring index arithmetic and an indexed
// parameter load.
struct TileTables {
    const void *src[GAR_MAX_WORKERS];
    void *dst[GAR_MAX_WORKERS];
};

// Fold one 16-byte vector at element e of the tile's row, in ring order:
// acc = x_0 + x_1 + ... + x_{P-1} over tt.src, left to right in fp32.
template <typename T, bool kRange, class Prm>
__device__ __forceinline__ void fold_vec(const Prm &p, const TileTables &tt, int64_t e, Range &rg) {
    constexpr int V = Elem<T>::kVec;
    const int P = p.P;
    float acc[V];
    uint4 raw[kLoadBatch];
    // first batch, its first worker peeled off (it starts the sum)
#pragma unroll
    for (int j = 0; j < kLoadBatch; ++j)
        if (j < P) raw[j] = ld16(static_cast<const T *>(tt.src[j]) + e);
    Elem<T>::unpack(raw[0], acc);
    if (kRange) rg.add_vec(acc);
#pragma unroll
    for (int j = 1; j < kLoadBatch; ++j) {
        if (j < P) {
            float v[V];
            Elem<T>::unpack(raw[j], v);
            if (kRange) rg.add_vec(v);
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] = __fadd_rn(acc[q], v[q]);
        }
    }
    for (int k0 = kLoadBatch; k0 < P; k0 += kLoadBatch) {
#pragma unroll
        for (int j = 0; j < kLoadBatch; ++j)
            if (k0 + j < P) raw[j] = ld16(static_cast<const T *>(tt.src[k0 + j]) + e);
#pragma unroll
        for (int j = 0; j < kLoadBatch; ++j) {
            if (k0 + j < P) {
                float v[V];
                Elem<T>::unpack(raw[j], v);
                if (kRange) rg.add_vec(v);
#pragma unroll
                for (int q = 0; q < V; ++q) acc[q] = __fadd_rn(acc[q], v[q]);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = finish(p, acc[q]);
    const uint4 out = Elem<T>::pack(acc);
#pragma unroll 4
    for (int k = 0; k < p.n_out; ++k) st16(static_cast<T *>(tt.dst[k]) + e, out);
}

template <typename T, bool kRange, class Prm>
__device__ __forceinline__ void fold_one(const Prm &p, const TileTables &tt, int64_t e, Range &rg) {
    const int P = p.P;
    float acc = Elem<T>::load1(tt.src[0], e);
    if (kRange) rg.add(acc);
    for (int k = 1; k < P; ++k) {
        const float v = Elem<T>::load1(tt.src[k], e);
        if (kRange) rg.add(v);
        acc = __fadd_rn(acc, v);
    }
    acc = finish(p, acc);
    for (int k = 0; k < p.n_out; ++k) Elem<T>::store1(tt.dst[k], e, acc);
}

__device__ __forceinline__ void atomic_min_f(float *a, float v) {
    if ((__float_as_uint(v) >> 31) == 0u) atomicMin(reinterpret_cast<int *>(a), __float_as_int(v));
    else atomicMax(reinterpret_cast<unsigned int *>(a), __float_as_uint(v));
}
__device__ __forceinline__ void atomic_max_f(float *a, float v) {
    if ((__float_as_uint(v) >> 31) == 0u) atomicMax(reinterpret_cast<int *>(a), __float_as_int(v));
    else atomicMin(reinterpret_cast<unsigned int *>(a), __float_as_uint(v));
}

// Block-wide min / max of rg merged into range[slot] (one pair of atomics).
__device__ __forceinline__ void flush_range(Range rg, float *range, int slot, unsigned int *status) {
    __shared__ float s_lo[kThreads / 32], s_hi[kThreads / 32];
    flag_nonfinite_warp(status, rg.chk);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        rg.lo = fminf(rg.lo, __shfl_xor_sync(0xFFFFFFFFu, rg.lo, o));
        rg.hi = fmaxf(rg.hi, __shfl_xor_sync(0xFFFFFFFFu, rg.hi, o));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // an earlier flush's readers are done with s_lo / s_hi
    if (lane == 0) {
        s_lo[warp] = rg.lo;
        s_hi[warp] = rg.hi;
    }
    __syncthreads();
    if (warp == 0) {
        rg.lo = lane < kThreads / 32 ? s_lo[lane] : __int_as_float(0x7F800000);
        rg.hi = lane < kThreads / 32 ? s_hi[lane] : __int_as_float(0xFF800000u);
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
            rg.lo = fminf(rg.lo, __shfl_xor_sync(0xFFFFFFFFu, rg.lo, o));
            rg.hi = fmaxf(rg.hi, __shfl_xor_sync(0xFFFFFFFFu, rg.hi, o));
        }
        if (lane == 0) {
            if (rg.lo == rg.lo) atomic_min_f(range + 2 * slot, rg.lo);
            if (rg.hi == rg.hi) atomic_max_f(range + 2 * slot + 1, rg.hi);
        }
    }
}

// kRange: also fold the inputs into their buffer's [min, max]; a CTA merges
// its partial range when the buffer of its next tile differs, and at the end.
template <typename T, class Prm, bool kRange>
__global__ void __launch_bounds__(kThreads, kRange ? kRangeMinBlocks : 4) ring_fold_kernel(const __grid_constant__ Prm p) {
    constexpr int V = Elem<T>::kVec;
    __shared__ TileTables tt;
    Range rg;
    int slot = -1;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        // the piece that owns tile t: largest i with tile_start[i] <= t (uniform per CTA)
        int lo = 0, hi = p.npieces - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.tile_start[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        const Piece pc = p.piece[lo];
        if (kRange && p.slot[lo] != slot) {
            if (slot >= 0) flush_range(rg, p.range, slot, p.status);
            rg = Range();
            slot = p.slot[lo];
        }
        const int64_t lt = t - p.tile_start[lo];
        __syncthreads();  // the previous tile's readers are done with tt
        if (threadIdx.x < p.P)
            tt.src[threadIdx.x] = p.src[static_cast<int64_t>(pc.row) * p.P + ring_worker(pc.chunk, threadIdx.x, pc.ccw, p.P)];
        if (threadIdx.x < p.n_out) tt.dst[threadIdx.x] = p.dst[static_cast<int64_t>(pc.row) * p.n_out + threadIdx.x];
        __syncthreads();
        if (pc.vec) {
            const int sh = pc.vec - 1;  // the row's pointers' common phase
            int64_t vb = (pc.begin + sh + V - 1) / V * V - sh;
            if (vb > pc.end) vb = pc.end;
            int64_t ve = (pc.end + sh) / V * V - sh;
            if (ve < vb) ve = vb;
            const int64_t nvec = (ve - vb) / V;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t i = lt * kTileUnits + u * kThreads + threadIdx.x;
                if (i < nvec) fold_vec<T, kRange>(p, tt, vb + i * V, rg);
            }
            if (lt == 0) {  // ragged head and tail of the piece (fewer than V each)
                const int head = static_cast<int>(vb - pc.begin);
                const int tail = static_cast<int>(pc.end - ve);
                if (threadIdx.x < head) fold_one<T, kRange>(p, tt, pc.begin + threadIdx.x, rg);
                else if (threadIdx.x >= 32 && threadIdx.x < 32 + tail)
                    fold_one<T, kRange>(p, tt, ve + (threadIdx.x - 32), rg);
            }
        } else {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t e = pc.begin + lt * kTileUnits + u * kThreads + threadIdx.x;
                if (e < pc.end) fold_one<T, kRange>(p, tt, e, rg);
            }
        }
    }
    if (kRange && slot >= 0) flush_range(rg, p.range, slot, p.status);
}

// Range entries of the buffers a call covers start at (+inf, -inf), or at
// (0, 0) when the packed buffer would hold zero gaps.
struct RangeResetParams {
    float *mM;
    int32_t n;
    int32_t ids[255];
    uint8_t zero[256];
};

__global__ void range_reset_kernel(const __grid_constant__ RangeResetParams p) {
    for (int i = threadIdx.x; i < p.n; i += blockDim.x) {
        p.mM[2 * p.ids[i]] = p.zero[i] ? 0.0f : __int_as_float(0x7F800000);
        p.mM[2 * p.ids[i] + 1] = p.zero[i] ? 0.0f : __int_as_float(0xFF800000u);
    }
}

// Launch configuration: one CTA per tile.  The hardware block scheduler hands
// the next tile to whichever SM frees a slot first, so SMs that draw less
// bandwidth finish no later than the rest; a persistent grid striding over the
// tiles left single SMs busy up to 13% past the average (ncu), and one CTA per
// tile measured 6.3 TB/s against 5.7 TB/s for the fp32 ring of 8 x 2^24.
template <typename T, class Prm, bool kRange>
int launch_fold_as(const Prm &p, cudaStream_t stream) {
    const int64_t grid = p.total_tiles < 0x7FFFFFFF ? p.total_tiles : 0x7FFFFFFF;
    ring_fold_kernel<T, Prm, kRange><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
    return check_launch("ring_fold_kernel");
}

template <typename T, class Prm>
int launch_fold(const Prm &p, cudaStream_t stream) {
    if (p.total_tiles <= 0) return GAR_OK;
    if (p.range) return launch_fold_as<T, Prm, true>(p, stream);
    return launch_fold_as<T, Prm, false>(p, stream);
}

template <class Prm>
void set_mode(Prm &p, int op, int P) {
    p.fp = static_cast<float>(P);
    p.inv_p = 1.0f / static_cast<float>(P);
    if (op == GAR_SUM || P == 1) p.mode = kModeSum;
    else if ((P & (P - 1)) == 0) p.mode = kModeMulInv;
    else p.mode = kModeDiv;
}

}  // namespace

// ------------------------------------------------------------------ host
// Number of tiles a piece needs (at least one: tile 0 also folds the ragged
// head and tail).
static int64_t piece_tiles(const Piece &pc, int V) {
    if (!pc.vec) {
        const int64_t t = ceil_div(pc.end - pc.begin, kTileUnits);
        return t > 0 ? t : 1;
    }
    const int sh = pc.vec - 1;
    int64_t vb = (pc.begin + sh + V - 1) / V * V - sh;
    if (vb > pc.end) vb = pc.end;
    int64_t ve = (pc.end + sh) / V * V - sh;
    if (ve < vb) ve = vb;
    const int64_t t = ceil_div((ve - vb) / V, kTileUnits);
    return t > 0 ? t : 1;
}

// Common phase of a row's pointers: 1 + s when every pointer lies s elements
// (of es bytes) past a 16-byte line, the same s for all; 0 when they differ.
struct PhaseOf {
    int es;
    int sh = -1;  // -1 before the first pointer, -2 once two differ
    void add(const void *ptr) {
        const int s = static_cast<int>((reinterpret_cast<uintptr_t>(ptr) & 15) / es);
        sh = sh == -1 ? s : (sh == s ? sh : -2);
    }
    int vec() const { return sh >= 0 ? 1 + sh : 0; }
};

template <class Prm>
static void finalize_tiles(Prm &p, int V) {
    int64_t tiles = 0;
    for (int i = 0; i < p.npieces; ++i) {
        p.tile_start[i] = tiles;
        tiles += piece_tiles(p.piece[i], V);
    }
    p.tile_start[p.npieces] = tiles;
    p.total_tiles = tiles;
}

template <class Prm>
static int launch_dtype(const Prm &p, int32_t dtype, cudaStream_t stream) {
    if (dtype == GAR_F32) return launch_fold<float>(p, stream);
    Prm q = p;  // a range is only ever asked of fp32 buffers
    q.range = nullptr;
    return launch_fold<uint16_t>(q, stream);
}

static int check_common(int32_t P, int64_t N, int32_t dtype, int32_t op) {
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (N < 0) return fail(GAR_EINVAL, "N=%lld < 0", static_cast<long long>(N));
    if (elem_bytes(dtype) < 0) return fail(GAR_EDTYPE, "unknown dtype %d", dtype);
    if (op != GAR_SUM && op != GAR_AVG) return fail(GAR_EINVAL, "unknown op %d", op);
    return GAR_OK;
}

// Ring all-reduce of one buffer per worker: n_out destinations.  rings = 1:
// P chunks on the clockwise ring; rings = 2: 2P sub-chunks, the first P on
// the clockwise ring, the last P on the counter-clockwise ring.
template <class Prm>
static int ring_single_impl(Prm &p, const void *const *src, void *const *dst, int n_out, int32_t P, int64_t N,
                            int32_t dtype, int32_t op, int rings, cudaStream_t stream) {
    std::memset(&p, 0, sizeof(p));
    p.P = P;
    p.n_out = n_out;
    set_mode(p, op, P);
    const int es = elem_bytes(dtype);
    if (N == 0) return GAR_OK;  // nothing is read or written: pointers may be NULL
    PhaseOf phase{es};
    for (int w = 0; w < P; ++w) {
        if (!src[w]) return fail(GAR_EINVAL, "input buffer %d is NULL", w);
        if (!aligned(src[w], es)) return fail(GAR_EALIGN, "input buffer %d not aligned to %d bytes", w, es);
        phase.add(src[w]);
        p.src[w] = src[w];
    }
    for (int k = 0; k < n_out; ++k) {
        if (!dst[k]) return fail(GAR_EINVAL, "output buffer %d is NULL", k);
        if (!aligned(dst[k], es)) return fail(GAR_EALIGN, "output buffer %d not aligned to %d bytes", k, es);
        phase.add(dst[k]);
        p.dst[k] = dst[k];
    }
    if (N == 0) return GAR_OK;
    const int nchunks = rings * P;
    const int64_t clen = ceil_div(N, nchunks);
    for (int k = 0; k < nchunks; ++k) {
        const int64_t b = static_cast<int64_t>(k) * clen;
        if (b >= N) break;
        const int64_t e = b + clen < N ? b + clen : N;
        Piece &pc = p.piece[p.npieces++];
        pc.row = 0;
        pc.chunk = k < P ? k : k - P;
        pc.vec = phase.vec();
        pc.ccw = k < P ? 0 : 1;
        pc.begin = b;
        pc.end = e;
    }
    finalize_tiles(p, 16 / es);
    return launch_dtype(p, dtype, stream);
}

static int ring_single(const void *const *src, void *const *dst, int n_out, int32_t P, int64_t N, int32_t dtype,
                       int32_t op, int rings, cudaStream_t stream) {
    if (rings * P <= kSmallPieces) {
        FoldParamsSmall p;
        return ring_single_impl(p, src, dst, n_out, P, N, dtype, op, rings, stream);
    }
    std::unique_ptr<FoldParamsLarge> p(new FoldParamsLarge);  // ~25 KB: keep it off the stack
    return ring_single_impl(*p, src, dst, n_out, P, N, dtype, op, rings, stream);
}

extern "C" int gar_ring_allreduce_sim(void *const *bufs, int32_t P, int64_t N, int32_t dtype, int32_t op,
                                      gar_stream_t stream) {
    int rc = check_common(P, N, dtype, op);
    if (rc) return rc;
    if (!bufs) return fail(GAR_EINVAL, "bufs is NULL");
    for (int a = 0; a < P && N > 0; ++a)
        for (int b = a + 1; b < P; ++b)
            if (bufs[a] == bufs[b]) return fail(GAR_EINVAL, "workers %d and %d share a buffer", a, b);
    return ring_single(reinterpret_cast<const void *const *>(bufs), bufs, P, P, N, dtype, op, 1,
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int gar_ring_allreduce_bidir(void *const *bufs, int32_t P, int64_t N, int32_t dtype, int32_t op,
                                        gar_stream_t stream) {
    int rc = check_common(P, N, dtype, op);
    if (rc) return rc;
    if (!bufs) return fail(GAR_EINVAL, "bufs is NULL");
    for (int a = 0; a < P && N > 0; ++a)
        for (int b = a + 1; b < P; ++b)
            if (bufs[a] == bufs[b]) return fail(GAR_EINVAL, "workers %d and %d share a buffer", a, b);
    return ring_single(reinterpret_cast<const void *const *>(bufs), bufs, P, P, N, dtype, op, 2,
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int gar_ring_allreduce_sim_out(const void *const *bufs, int32_t P, int64_t N, int32_t dtype, int32_t op,
                                          void *const *out, int32_t n_out, gar_stream_t stream) {
    int rc = check_common(P, N, dtype, op);
    if (rc) return rc;
    if (!bufs || !out) return fail(GAR_EINVAL, "bufs or out is NULL");
    if (n_out < 1 || n_out > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "n_out=%d outside [1, %d]", n_out, GAR_MAX_WORKERS);
    return ring_single(bufs, out, n_out, P, N, dtype, op, 1, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------- plan-driven (fused) launch
// Reset the range entries of the buffers the call covers.  A buffer starts at
// (0, 0) when its packed form would hold zeros: an alignment gap after one of
// the given tensors (up to the next given tensor of the buffer, or the end).
static int reset_ranges(const gar_seg *segs, int32_t count, const int64_t *buf_numel, int32_t n_buffers,
                        float *d_mM, cudaStream_t stream) {
    std::vector<int8_t> state(n_buffers, -1);  // -1 not covered, 0 no zeros, 1 zeros
    std::vector<int64_t> last_end(n_buffers, 0);
    for (int i = 0; i < count; ++i) {
        const gar_seg &s = segs[i];
        if (state[s.buffer] < 0) state[s.buffer] = 0;
        else if (s.offset > last_end[s.buffer]) state[s.buffer] = 1;  // gap before this tensor
        last_end[s.buffer] = s.offset + s.numel;
    }
    for (int b = 0; b < n_buffers; ++b)
        if (state[b] == 0 && last_end[b] < buf_numel[b]) state[b] = 1;  // gap up to the buffer's end
    RangeResetParams rp;
    std::memset(&rp, 0, sizeof(rp));
    rp.mM = d_mM;
    for (int b = 0; b <= n_buffers; ++b) {
        if (b < n_buffers && state[b] >= 0) {
            rp.ids[rp.n] = b;
            rp.zero[rp.n] = static_cast<uint8_t>(state[b]);
            ++rp.n;
        }
        if (rp.n > 0 && (rp.n == 255 || b == n_buffers)) {
            range_reset_kernel<<<1, 256, 0, stream>>>(rp);
            const int rc = check_launch("range_reset_kernel");
            if (rc) return rc;
            rp.n = 0;
        }
    }
    return GAR_OK;
}

int fused_allreduce_impl(const void *const *src, void *const *dst, int32_t P, const gar_seg *segs,
                         const int32_t *dtype, int32_t count, const int64_t *buf_numel, int32_t n_buffers,
                         int32_t op, float *d_mM, cudaStream_t stream) {
    using Prm = FoldParamsLarge;
    int rc = GAR_OK;
    if (d_mM) {
        rc = reset_ranges(segs, count, buf_numel, n_buffers, d_mM, stream);
        if (rc) return rc;
    }
    std::unique_ptr<Prm> p(new Prm);  // ~25 KB: keep it off the stack
    for (int pass_dtype = 0; pass_dtype < 2 && rc == GAR_OK; ++pass_dtype) {
        const int es = elem_bytes(pass_dtype);
        std::memset(p.get(), 0, sizeof(Prm));
        p->P = P;
        p->n_out = P;
        p->range = pass_dtype == GAR_F32 ? d_mM : nullptr;
        p->status = p->range ? device_status() : nullptr;
        set_mode(*p, op, P);
        int rows = 0;
        auto flush = [&]() -> int {
            if (p->npieces == 0) return GAR_OK;
            finalize_tiles(*p, 16 / es);
            const int r = launch_dtype(*p, pass_dtype, stream);
            p->npieces = 0;
            rows = 0;
            return r;
        };
        for (int i = 0; i < count && rc == GAR_OK; ++i) {
            if (dtype[i] != pass_dtype || segs[i].numel == 0) continue;
            const int b = segs[i].buffer;
            const int64_t clen = ceil_div(buf_numel[b], P);
            const int64_t first_chunk = segs[i].offset / clen;
            const int64_t last_chunk = (segs[i].offset + segs[i].numel - 1) / clen;
            const int need = static_cast<int>(last_chunk - first_chunk + 1);
            if ((rows + 1) * P > kLargePtrs || p->npieces + need > kLargePieces) rc = flush();
            if (rc) break;
            PhaseOf phase{elem_bytes(pass_dtype)};
            for (int w = 0; w < P; ++w) {
                const void *s = src[static_cast<int64_t>(w) * count + i];
                void *d = dst[static_cast<int64_t>(w) * count + i];
                phase.add(s);
                phase.add(d);
                p->src[rows * P + w] = s;
                p->dst[rows * P + w] = d;
            }
            int64_t pos = 0;
            const int64_t off = segs[i].offset, n = segs[i].numel;
            while (pos < n) {
                const int64_t c = (off + pos) / clen;
                int64_t stop = (c + 1) * clen - off;
                if (stop > n) stop = n;
                Piece &pc = p->piece[p->npieces++];
                pc.row = rows;
                pc.chunk = static_cast<int32_t>(c);
                pc.vec = phase.vec();
                pc.ccw = 0;
                p->slot[p->npieces - 1] = b;
                pc.begin = pos;
                pc.end = stop;
                pos = stop;
            }
            ++rows;
        }
        if (rc == GAR_OK) rc = flush();
    }
    return rc;
}

// ------------------------------------------------- literal step schedule
namespace {

__global__ void ring_step_kernel(const __grid_constant__ StepParams p) {
    // worker i = blockIdx.y receives from i - 1 into chunk (i - s - 1) mod P
    // (scatter-reduce) or (i - s) mod P (all-gather)
    const int P = p.P;
    const int i = blockIdx.y;
    const int from = (i - 1 + P) % P;
    const int c = p.gather ? ((i - p.step) % P + P) % P : ((i - p.step - 1) % P + 2 * P) % P;
    const int64_t b = static_cast<int64_t>(c) * p.clen;
    int64_t e = b + p.clen;
    if (e > p.N) e = p.N;
    float *mine = p.buf[i];
    const float *recv = p.buf[from];
    for (int64_t k = b + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < e;
         k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        mine[k] = p.gather ? recv[k] : __fadd_rn(mine[k], recv[k]);
    }
}

__global__ void ring_divide_kernel(const __grid_constant__ StepParams p) {
    float *x = p.buf[blockIdx.y];
    const float fp = static_cast<float>(p.P);
    for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < p.N;
         k += static_cast<int64_t>(gridDim.x) * blockDim.x)
        x[k] = __fdiv_rn(x[k], fp);
}

}  // namespace

extern "C" int gar_ring_allreduce_steps(void *const *bufs, int32_t P, int64_t N, int32_t op, int32_t *steps,
                                        int64_t *sent_elems, gar_stream_t stream_) {
    int rc = check_common(P, N, GAR_F32, op);
    if (rc) return rc;
    if (!bufs) return fail(GAR_EINVAL, "bufs is NULL");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    StepParams p;
    std::memset(&p, 0, sizeof(p));
    p.P = P;
    p.N = N;
    p.clen = N > 0 ? ceil_div(N, P) : 0;
    for (int w = 0; w < P; ++w) {
        if (!bufs[w] && N > 0) return fail(GAR_EINVAL, "buffer %d is NULL", w);
        if (!aligned(bufs[w], 4)) return fail(GAR_EALIGN, "buffer %d not 4-byte aligned", w);
        p.buf[w] = static_cast<float *>(bufs[w]);
    }
    for (int a = 0; a < P && N > 0; ++a)
        for (int b = a + 1; b < P; ++b)
            if (bufs[a] == bufs[b]) return fail(GAR_EINVAL, "workers %d and %d share a buffer", a, b);
    std::vector<int64_t> sent(P, 0);
    auto chunk_len = [&](int c) -> int64_t {
        const int64_t b = static_cast<int64_t>(c) * p.clen;
        if (b >= N) return 0;
        return (b + p.clen < N ? b + p.clen : N) - b;
    };
    const int64_t per_block = 256 * 8;
    int64_t gx = p.clen > 0 ? ceil_div(p.clen, per_block) : 1;
    if (gx > 65535) gx = 65535;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(P));
    int nsteps = 0;
    for (int phase = 0; phase < 2; ++phase) {
        for (int s = 0; s < P - 1; ++s) {
            p.step = s;
            p.gather = phase;
            if (N > 0) {
                ring_step_kernel<<<grid, 256, 0, stream>>>(p);
                rc = check_launch("ring_step_kernel");
                if (rc) return rc;
            }
            for (int i = 0; i < P; ++i) {
                // worker i sends chunk (i - s) mod P, or (i - s + 1) mod P while gathering
                const int c = phase ? ((i - s + 1) % P + P) % P : ((i - s) % P + P) % P;
                sent[i] += chunk_len(c);
            }
            ++nsteps;
        }
    }
    if (op == GAR_AVG && P > 1 && N > 0) {
        int64_t gd = ceil_div(N, per_block);
        if (gd > 65535) gd = 65535;
        ring_divide_kernel<<<dim3(static_cast<unsigned>(gd), static_cast<unsigned>(P)), 256, 0, stream>>>(p);
        rc = check_launch("ring_divide_kernel");
        if (rc) return rc;
    }
    if (steps) *steps = nsteps;
    if (sent_elems)
        for (int i = 0; i < P; ++i) sent_elems[i] = sent[i];
    return GAR_OK;
}

}  // namespace gar
