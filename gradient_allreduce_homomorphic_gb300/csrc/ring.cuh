// ring.cuh -- kernel-parameter layouts of the ring all-reduce kernels.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace gar {

// A run of one tensor's elements that lies inside one ring chunk: the fold
// of every element of the run starts at worker `chunk`.
struct Piece {
    int32_t row;    // row of the pointer tables (one tensor)
    int32_t chunk;  // ring chunk id = first worker of the fold
    int32_t vec;    // 0: element by element; 1 + s: every pointer of the row lies s elements past a
                    // 16-byte line (the same s for all), so element e is on a line iff (e + s) % V == 0
    int32_t ccw;    // 1: the fold runs x_c, x_{c-1}, ... (counter-clockwise ring)
    int64_t begin;  // first element, in the tensor's own indexing
    int64_t end;    // one past the last element
};

enum { kModeSum = 0, kModeMulInv = 1, kModeDiv = 2 };

// Passed by value (kernel parameter space): no device-side tables to upload.
template <int NPTR, int NPIECE>
struct FoldParams {
    int32_t P;        // workers
    int32_t n_out;    // destinations per row
    int32_t npieces;
    int32_t mode;     // kMode*
    float inv_p;      // 1/P (exact when P is a power of two)
    float fp;         // P
    float *range;     // [slot][2] min / max of the inputs, or NULL
    unsigned int *status;  // range launches: GAR_STATUS_NONFINITE raised here
    int64_t total_tiles;
    int64_t tile_start[NPIECE + 1];  // first tile of each piece; [npieces] = total
    Piece piece[NPIECE];
    int32_t slot[NPIECE];  // range launches: fusion buffer each piece's inputs are folded into
    const void *src[NPTR];  // src[row * P + w]
    void *dst[NPTR];        // dst[row * n_out + k]
};

constexpr int kSmallPtrs = 64, kSmallPieces = 64;
constexpr int kLargePtrs = 1024, kLargePieces = 256;
using FoldParamsSmall = FoldParams<kSmallPtrs, kSmallPieces>;  // < 4 KB
using FoldParamsLarge = FoldParams<kLargePtrs, kLargePieces>;  // < 32 KB (large-parameter launch)
static_assert(sizeof(FoldParamsSmall) <= 4096, "small fold parameters exceed 4 KB");
static_assert(sizeof(FoldParamsLarge) <= 32000, "large fold parameters exceed the 32 KB launch limit");

struct StepParams {
    int32_t P, step, gather, pad;
    int64_t N, clen;
    float *buf[GAR_MAX_WORKERS];
};

// Plan-driven all-reduce over the workers' tensors (validated by the caller).
// d_mM (NULL, or [n_buffers][2] device floats): also fold every fp32 input
// into its buffer's [min, max], as the THC range of the packed buffer.
int fused_allreduce_impl(const void *const *src, void *const *dst, int32_t P, const gar_seg *segs,
                         const int32_t *dtype, int32_t count, const int64_t *buf_numel, int32_t n_buffers,
                         int32_t op, float *d_mM, cudaStream_t stream);

}  // namespace gar
