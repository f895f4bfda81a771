// common.cuh -- internal helpers shared by the library's translation units.
//
// Host side: error reporting (thread-local message + status), launch checks,
// SM count.  Device side: 16-byte streaming loads/stores, bf16 <-> fp32
// conversion, and the Philox4x32-10 counter-based generator.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "gar.h"

namespace gar {

// ------------------------------------------------------------------ host
// Record `msg` as this thread's last error and return `status`.
int fail(int status, const char *fmt, ...);
// GAR_ECUDA (with the runtime's message) if the last launch failed, else GAR_OK.
int check_launch(const char *what);
// Multiprocessor count of the current device (cached per device).
int sm_count();
// Device address of the library's status word on the current device (bits
// that kernels set for conditions found on the device, GAR_STATUS_*), or
// NULL if it cannot be had; looked up once per device.
unsigned int *device_status();

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline int elem_bytes(int32_t dtype) { return dtype == GAR_F32 ? 4 : (dtype == GAR_BF16 ? 2 : -1); }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- device
// Non-finite check at one FMA per value: chk = fma(v, 0, chk) stays 0 for
// finite values and becomes NaN for good once a NaN or an infinity is seen.
__device__ __forceinline__ float nonfinite_acc(float chk, float v) { return __fmaf_rn(v, 0.0f, chk); }
// Raise GAR_STATUS_NONFINITE if any lane of the warp saw a non-finite value
// (call with every lane of the warp; one atomic per warp at most).
__device__ __forceinline__ void flag_nonfinite_warp(unsigned int *status, float chk) {
    if (__any_sync(0xFFFFFFFFu, chk != chk) && (threadIdx.x & 31) == 0 && status)
        atomicOr(status, static_cast<unsigned int>(GAR_STATUS_NONFINITE));
}

// 16-byte loads and stores with the streaming ("evict first") cache hint:
// every byte of the hot path is touched once per pass.
__device__ __forceinline__ uint4 ld16(const void *p) { return __ldcs(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void st16(void *p, uint4 v) { __stcs(reinterpret_cast<uint4 *>(p), v); }

// bf16 is the upper half of an IEEE binary32: widening is exact.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_one(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }
// Two fp32 values rounded to nearest-even bf16 and packed (lo in bits 0-15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint16_t to_bf16(float v) { return static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xFFFFu); }

// Philox4x32 round keys for a 64-bit seed: round r uses
// (seed_lo + r * 0x9E3779B9, seed_hi + r * 0xBB67AE85) (mod 2^32), [S].
struct PhiloxKeys {
    uint32_t lo[10];
    uint32_t hi[10];
};
inline PhiloxKeys philox_keys(uint64_t seed) {
    PhiloxKeys k;
    uint32_t a = static_cast<uint32_t>(seed), b = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        k.lo[r] = a;
        k.hi[r] = b;
        a += 0x9E3779B9u;
        b += 0xBB67AE85u;
    }
    return k;
}

// Philox4x32-10 [S]: ten rounds; each multiplies counter words 0 and 2 by
// the two round constants (full 64-bit products), then the next counter is
// (hi(B*c2) ^ c1 ^ k_lo, lo(B*c2), hi(A*c0) ^ c3 ^ k_hi, lo(A*c0)).
__device__ __forceinline__ uint4 philox10(uint4 c, const PhiloxKeys &k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t pa = static_cast<uint64_t>(c.x) * 0xD2511F53ull;
        const uint64_t pb = static_cast<uint64_t>(c.z) * 0xCD9E8D57ull;
        c = make_uint4(static_cast<uint32_t>(pb >> 32) ^ c.y ^ k.lo[r], static_cast<uint32_t>(pb),
                       static_cast<uint32_t>(pa >> 32) ^ c.w ^ k.hi[r], static_cast<uint32_t>(pa));
    }
    return c;
}

}  // namespace gar
