// dbtree.cu -- double-binary-tree all-reduce of P worker buffers held in one
// GPU's HBM, computed as a fold order ([R] "Design Alternatives & Collective
// Comparison Matrix: Ring vs. Tree vs. NVLS"; the two trees of [ST]).
//
// Two trees of one shape carry half of the buffer each.  The shape is the
// in-order binary tree on the labels 1..P: a run of labels is rooted at its
// label with the most trailing zero bits, with the runs below and above it
// as its subtrees.  For elements [0, ceil(N/2)) label l sits on rank l - 1;
// for the rest on rank P - l (P even: the mirror image) or (l - 2) mod P
// (P odd: shifted by one), so that no rank is interior in both trees.  A
// node's partial sum is its own value plus its left child's partial sum,
// then plus its right child's (fp32); the root's sum, divided by P for
// GAR_AVG, is broadcast down the tree.  On one GPU the reduce and the
// broadcast collapse into one pass: for every element, load the P values,
// fold them in that order, store the result to every buffer.
//
// The fold streams the labels in increasing order (the in-order walk) and
// keeps one pending value per tree level.  Label l with k trailing zeros
// closes its left subtree -- the pending nodes of levels k-1 .. 0, each
// (own + its left subtree), summed from level 0 upwards -- and becomes the
// pending node of level k, holding x_l + that sum.  After label P the
// pending nodes on the levels of P's set bits are the tree's right spine,
// and summed the same way they give the root's sum.  Labels are loaded in
// batches b + 1 .. b + 8 with b a multiple of 8: all but the last have the
// trailing zeros of 1 .. 7, template constants, and the last one's level is
// chosen by predicates, so every pending value keeps a fixed register.
#include <cstring>

#include "common.cuh"

namespace gar {
namespace {

constexpr int kThreads = 256;
constexpr int kGroupsPerThread = 2;
constexpr int kTileGroups = kThreads * kGroupsPerThread;
enum { kSum = 0, kMulInv = 1, kDiv = 2 };

struct DbtreeParams {
    const void *src[2][GAR_MAX_WORKERS];  // [tree][label - 1]: the buffer of the rank on that label
    void *dst[GAR_MAX_WORKERS];           // every worker's buffer (all receive the result)
    int64_t N;
    int64_t half;    // elements [0, half) go over tree 0
    int64_t groups;  // 16-byte groups (vec) or elements
    int32_t P;
    int32_t vec;     // every buffer 16-byte aligned
    int32_t mode;
    float fp;
    float inv_p;
    int32_t pad;
};

constexpr int trailing_zeros(int v) { return (v & 1) ? 0 : 1 + trailing_zeros(v >> 1); }

template <typename T>
struct Lanes;
template <>
struct Lanes<float> {
    static constexpr int kVec = 4;
    __device__ static void unpack(const uint4 &r, float (&v)[4]) {
        v[0] = __uint_as_float(r.x);
        v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z);
        v[3] = __uint_as_float(r.w);
    }
    __device__ static void store(void *p, int64_t e, const float (&v)[4]) {
        st16(static_cast<float *>(p) + e,
             make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3])));
    }
    __device__ static float load1(const void *p, int64_t e) { return __ldcs(static_cast<const float *>(p) + e); }
    __device__ static void store1(void *p, int64_t e, float v) { __stcs(static_cast<float *>(p) + e, v); }
};
template <>
struct Lanes<uint16_t> {  // bf16 storage: widened exactly, folded in fp32, rounded once
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
    __device__ static void store(void *p, int64_t e, const float (&v)[8]) {
        st16(static_cast<uint16_t *>(p) + e, make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                        pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7])));
    }
    __device__ static float load1(const void *p, int64_t e) {
        return bf16_one(__ldcs(reinterpret_cast<const unsigned short *>(p) + e));
    }
    __device__ static void store1(void *p, int64_t e, float v) {
        __stcs(reinterpret_cast<unsigned short *>(p) + e, static_cast<unsigned short>(to_bf16(v)));
    }
};

// A batch keeps its loads as raw 16-byte words (4 registers each, whatever
// the element type) and widens one label at a time as it is folded.
template <typename T>
struct VecLoader {
    static constexpr int V = Lanes<T>::kVec;
    using Raw = uint4;
    int64_t e;
    __device__ Raw load(const void *p) const { return ld16(static_cast<const T *>(p) + e); }
    __device__ void unpack(const Raw &r, float (&v)[V]) const { Lanes<T>::unpack(r, v); }
};
template <typename T>
struct OneLoader {
    using Raw = float;
    int64_t e;
    __device__ Raw load(const void *p) const { return Lanes<T>::load1(p, e); }
    __device__ void unpack(const Raw &r, float (&v)[1]) const { v[0] = r; }
};

// Register budget of the fold for P <= M (M a power of two): pending values
// on levels 0 .. log2(M), loads in batches of min(8, M) labels, and the CTAs
// per SM the build asks for (more for small P and fp32, whose folds hold
// fewer live values).
template <typename T, int M>
struct Shape {
    static constexpr int kLevels = trailing_zeros(M) + 1;
    static constexpr int kBatch = M < 8 ? M : 8;
    static constexpr bool kWide = Lanes<T>::kVec == 8;
    static constexpr int kMinBlocks = M <= 4 ? (kWide ? 3 : 4) : (M <= 16 && !kWide ? 3 : 2);
};

// Label with K trailing zeros arrives with value x: close its left subtree
// (levels K-1 .. 0 of the pending chain) and make it the pending node of level K.
template <int K, int L, int V>
__device__ __forceinline__ void take_label(float (&pend)[L][V], const float (&x)[V]) {
    if constexpr (K == 0) {
#pragma unroll
        for (int q = 0; q < V; ++q) pend[0][q] = x[q];
    } else {
        float s[V];
#pragma unroll
        for (int q = 0; q < V; ++q) s[q] = pend[0][q];
#pragma unroll
        for (int lev = 1; lev < K; ++lev)
#pragma unroll
            for (int q = 0; q < V; ++q) s[q] = __fadd_rn(pend[lev][q], s[q]);
#pragma unroll
        for (int q = 0; q < V; ++q) pend[K][q] = __fadd_rn(x[q], s[q]);
    }
}

// Labels b + J .. b + B - 1 of a batch (b a multiple of B): their trailing
// zeros are those of J, fixed at compile time.
template <int J, int B, class Ld, int L, int V>
__device__ __forceinline__ void take_fixed(float (&pend)[L][V], const typename Ld::Raw (&raw)[B], const Ld &ld,
                                           int b, int P) {
    if constexpr (J < B) {
        if (b + J <= P) {
            float x[V];
            ld.unpack(raw[J - 1], x);
            take_label<trailing_zeros(J)>(pend, x);
            take_fixed<J + 1, B>(pend, raw, ld, b, P);
        }
    }
}

// Label l = b + B: at least log2(B) trailing zeros, the exact count known
// only at run time; predicated on every level so that the pending values
// keep fixed registers.
template <int B, int L, int V>
__device__ __forceinline__ void take_top(float (&pend)[L][V], const float (&x)[V], int l) {
    constexpr int kMin = trailing_zeros(B);
    const int k = __ffs(l) - 1;
    float s[V];
#pragma unroll
    for (int q = 0; q < V; ++q) s[q] = pend[0][q];
#pragma unroll
    for (int lev = 1; lev < L - 1; ++lev)
        if (lev < k)
#pragma unroll
            for (int q = 0; q < V; ++q) s[q] = __fadd_rn(pend[lev][q], s[q]);
#pragma unroll
    for (int lev = kMin; lev < L; ++lev)
        if (lev == k)
#pragma unroll
            for (int q = 0; q < V; ++q) pend[lev][q] = __fadd_rn(x[q], s[q]);
}

// The root's sum of the P values (src[l - 1] = the buffer on label l), after
// the division the op asks for.
template <class S, class Ld, int V>
__device__ __forceinline__ void tree_fold(const DbtreeParams &p, const void *const *src, const Ld &ld,
                                          float (&out)[V]) {
    constexpr int L = S::kLevels, B = S::kBatch;
    float pend[L][V];
#pragma unroll
    for (int lev = 0; lev < L; ++lev)
#pragma unroll
        for (int q = 0; q < V; ++q) pend[lev][q] = 0.0f;
    const int P = p.P;
#pragma unroll 1
    for (int b = 0; b < P; b += B) {
        typename Ld::Raw raw[B];
#pragma unroll
        for (int j = 0; j < B; ++j)
            if (b + j < P) raw[j] = ld.load(src[b + j]);
        take_fixed<1, B>(pend, raw, ld, b, P);
        if (b + B <= P) {
            float x[V];
            ld.unpack(raw[B - 1], x);
            take_top<B>(pend, x, b + B);
        }
    }
    bool have = false;  // the right spine, from its lowest node (label P) up to the root
#pragma unroll
    for (int lev = 0; lev < L; ++lev) {
        if ((P >> lev) & 1) {
#pragma unroll
            for (int q = 0; q < V; ++q) out[q] = have ? __fadd_rn(pend[lev][q], out[q]) : pend[lev][q];
            have = true;
        }
    }
#pragma unroll
    for (int q = 0; q < V; ++q) {
        if (p.mode == kMulInv) out[q] = __fmul_rn(out[q], p.inv_p);  // exact: P is a power of two
        else if (p.mode == kDiv) out[q] = __fdiv_rn(out[q], p.fp);
    }
}

template <class S, typename T, int M>
__device__ __forceinline__ void fold_element(const DbtreeParams &p, const void *const (&src)[2][M],
                                             void *const *dst, int64_t e) {
    const void *const *s = src[e < p.half ? 0 : 1];
    float r[1];
    tree_fold<S>(p, s, OneLoader<T>{e}, r);
    for (int k = 0; k < p.P; ++k) Lanes<T>::store1(dst[k], e, r[0]);
}

// One CTA per tile of 512 groups of 16 bytes (two per thread), P <= M.
template <typename T, int M>
__global__ void __launch_bounds__(kThreads, Shape<T, M>::kMinBlocks)
    dbtree_fold_kernel(const __grid_constant__ DbtreeParams p) {
    using S = Shape<T, M>;
    constexpr int V = Lanes<T>::kVec;
    __shared__ const void *s_src[2][M];
    __shared__ void *s_dst[M];
    if (threadIdx.x < p.P) {
        s_src[0][threadIdx.x] = p.src[0][threadIdx.x];
        s_src[1][threadIdx.x] = p.src[1][threadIdx.x];
        s_dst[threadIdx.x] = p.dst[threadIdx.x];
    }
    __syncthreads();
    const int64_t g0 = static_cast<int64_t>(blockIdx.x) * kTileGroups + threadIdx.x;
#pragma unroll 1
    for (int u = 0; u < kGroupsPerThread; ++u) {
        const int64_t g = g0 + static_cast<int64_t>(u) * kThreads;
        if (g >= p.groups) break;
        if (!p.vec) {
            fold_element<S, T>(p, s_src, s_dst, g);
            continue;
        }
        const int64_t e = g * V;
        if (e + V <= p.half || (e >= p.half && e + V <= p.N)) {
            float r[V];
            tree_fold<S>(p, s_src[e < p.half ? 0 : 1], VecLoader<T>{e}, r);
#pragma unroll 4
            for (int k = 0; k < p.P; ++k) Lanes<T>::store(s_dst[k], e, r);
        } else {  // the group that straddles the two halves, or the ragged last one
            for (int i = 0; i < V && e + i < p.N; ++i) fold_element<S, T>(p, s_src, s_dst, e + i);
        }
    }
}

template <typename T>
void launch_fold(const DbtreeParams &p, unsigned blocks, cudaStream_t s) {
    if (p.P <= 4) dbtree_fold_kernel<T, 4><<<blocks, kThreads, 0, s>>>(p);
    else if (p.P <= 8) dbtree_fold_kernel<T, 8><<<blocks, kThreads, 0, s>>>(p);
    else if (p.P <= 16) dbtree_fold_kernel<T, 16><<<blocks, kThreads, 0, s>>>(p);
    else dbtree_fold_kernel<T, GAR_MAX_WORKERS><<<blocks, kThreads, 0, s>>>(p);
}

// Rank on `label` (1-based) of tree 0 or 1.
int rank_of(int P, int tree, int label) {
    if (tree == 0) return label - 1;
    if (P % 2 == 0) return P - label;
    return ((label - 2) % P + P) % P;
}

// Parent label of `label` in the in-order tree on 1..P (0: the root): of the
// nearest labels with more trailing zeros, label -/+ 2^k, the one in 1..P
// with fewer trailing zeros.
int parent_label(int P, int label) {
    const int low = label & -label;
    const int lo = label - low, hi = label + low;
    const bool lo_ok = lo >= 1, hi_ok = hi <= P;
    if (lo_ok && hi_ok) return (lo & -lo) < (hi & -hi) ? lo : hi;
    if (lo_ok) return lo;
    if (hi_ok) return hi;
    return 0;
}

}  // namespace
}  // namespace gar

using namespace gar;

extern "C" int gar_dbtree_parents(int32_t P, int32_t tree, int32_t *parent) {
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (tree != 0 && tree != 1) return fail(GAR_EINVAL, "tree %d is not 0 or 1", tree);
    if (!parent) return fail(GAR_EINVAL, "parent is NULL");
    for (int l = 1; l <= P; ++l) {
        const int up = parent_label(P, l);
        parent[rank_of(P, tree, l)] = up ? rank_of(P, tree, up) : -1;
    }
    return GAR_OK;
}

extern "C" int gar_dbtree_allreduce(void *const *bufs, int32_t P, int64_t N, int32_t dtype, int32_t op,
                                    gar_stream_t stream) {
    if (P < 1 || P > GAR_MAX_WORKERS) return fail(GAR_EINVAL, "P=%d outside [1, %d]", P, GAR_MAX_WORKERS);
    if (N < 0) return fail(GAR_EINVAL, "N=%lld < 0", static_cast<long long>(N));
    const int es = elem_bytes(dtype);
    if (es < 0) return fail(GAR_EDTYPE, "unknown dtype %d", dtype);
    if (op != GAR_SUM && op != GAR_AVG) return fail(GAR_EINVAL, "unknown op %d", op);
    if (N == 0) return GAR_OK;  // nothing is read or written
    if (!bufs) return fail(GAR_EINVAL, "bufs is NULL");
    DbtreeParams p;
    std::memset(&p, 0, sizeof(p));
    p.P = P;
    p.N = N;
    p.half = (N + 1) / 2;
    p.vec = 1;
    for (int w = 0; w < P; ++w) {
        if (!bufs[w]) return fail(GAR_EINVAL, "buffer %d is NULL", w);
        if (!aligned(bufs[w], es)) return fail(GAR_EALIGN, "buffer %d not aligned to %d bytes", w, es);
        for (int v = 0; v < w; ++v)
            if (bufs[v] == bufs[w]) return fail(GAR_EINVAL, "workers %d and %d share a buffer", v, w);
        p.vec = p.vec && aligned(bufs[w], 16);
        p.dst[w] = bufs[w];
    }
    for (int tree = 0; tree < 2; ++tree)
        for (int l = 1; l <= P; ++l) p.src[tree][l - 1] = bufs[rank_of(P, tree, l)];
    p.fp = static_cast<float>(P);
    p.inv_p = 1.0f / static_cast<float>(P);
    p.mode = op == GAR_SUM ? kSum : ((P & (P - 1)) == 0 ? kMulInv : kDiv);
    p.groups = p.vec ? ceil_div(N, 16 / es) : N;
    const int64_t blocks = ceil_div(p.groups, kTileGroups);
    if (blocks > 0x7FFFFFFF) return fail(GAR_EINVAL, "N=%lld too large", static_cast<long long>(N));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == GAR_F32) launch_fold<float>(p, static_cast<unsigned>(blocks), s);
    else launch_fold<uint16_t>(p, static_cast<unsigned>(blocks), s);
    return check_launch("dbtree_fold_kernel");
}
