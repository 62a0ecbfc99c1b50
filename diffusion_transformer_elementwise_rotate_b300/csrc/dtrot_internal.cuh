// Private helpers shared by the sm_103a kernels of libdtrot.
//
// bf16 arithmetic uses the packed bf16x2 instructions with an explicit .rn
// modifier: each op rounds its exact result once to bf16 (round to nearest
// even), and PTX never contracts an op that carries an explicit rounding
// modifier into a fused multiply-add.  That is the per-op rounding of the
// eager chain that the rotate-half RoPE, GEGLU and the residual add must
// reproduce.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dtrot {

// ------------------------------------------------------------ bf16x2 ops

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t badd2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// bf16 bits -> fp32 (exact)
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf1(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// RN16 of an fp32 value (cvt.rn.bf16.f32: round to nearest even, NaN stays NaN)
__device__ __forceinline__ uint16_t rn16f(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

// Pack two fp32 values as RN16(lo) | RN16(hi) << 16.
__device__ __forceinline__ uint32_t rn16x2f(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Distance, in fp32 ulps, from an fp32 value to the nearest bf16 rounding
// midpoint.  bf16 keeps the top 16 bits of an fp32 pattern, so a midpoint is
// a pattern whose low 16 bits are 0x8000; this holds for subnormals too.
__device__ __forceinline__ int ulps_to_bf16_midpoint(float f) {
    int low = (int)(__float_as_uint(f) & 0xFFFFu);
    return abs(low - 0x8000);
}

// RN16 of a double.  The double is first rounded to fp32 towards zero and the
// lost bits are folded into the last fp32 bit ("round to odd"); rounding that
// to bf16 then equals rounding the double directly, because fp32 carries more
// than 8 + 2 significant bits.  Values below the fp32 normal range are scaled
// by 2^64 first (exact), rounded onto the scaled bf16 subnormal grid with an
// integer rint, and encoded directly.
__device__ __forceinline__ uint16_t rn16d(double d) {
    double a = fabs(d);
    uint16_t sign = (__double2hiint(d) < 0) ? 0x8000u : 0u;
    if (!(a == a)) return (uint16_t)(sign | 0x7FC0u);
    if (a < 0x1p-126) {
        // bf16 subnormal grid: multiples of 2^-133, up to 2^-126 (=128 steps)
        double k = rint(a * 0x1p133);  // exact scaling, ties to even
        return (uint16_t)(sign | (uint16_t)k);  // k = 128 encodes 2^-126 exactly
    }
    float fz = __double2float_rz(d);
    if ((double)fz != d) {
        uint32_t u = __float_as_uint(fz) | 1u;  // sticky bit: round to odd
        fz = __uint_as_float(u);
    }
    return rn16f(fz);
}

// ------------------------------------------------------------ rotary tables

// One table entry: c16 = RN16(RN32(cos f)), s16 = RN16(RN32(sin f)) with the
// fp32 cos/sin taken as correctly rounded.  sincosf (fp32, within 2 ulps of
// the exact value) decides the bf16 rounding unless its result lies within
// kCosSinMargin fp32 ulps of a bf16 rounding midpoint; only then is the value
// recomputed from the fp64 cos/sin (within 2 double ulps), rounded to fp32 and
// then to bf16.  A few in 10^4 entries take that path, so the fp64 units stay
// idle almost always.
constexpr int kCosSinMargin = 4;

__device__ __forceinline__ void cos_sin_entry(float f, uint16_t& c16, uint16_t& s16) {
    float s32, c32;
    sincosf(f, &s32, &c32);
    if (ulps_to_bf16_midpoint(c32) <= kCosSinMargin) {
        c32 = __double2float_rn(cos((double)f));
    }
    if (ulps_to_bf16_midpoint(s32) <= kCosSinMargin) {
        s32 = __double2float_rn(sin((double)f));
    }
    c16 = rn16f(c32);
    s16 = rn16f(s32);
}

// ------------------------------------------------------------ launchers

struct RopeParams {
    const uint16_t* x;
    uint16_t* out;
    const uint16_t* cos;
    const uint16_t* sin;
    int64_t B, S, H, D, rot;
    int64_t sx_b, sx_s, sx_h;
    int64_t so_b, so_s, so_h;
    int in_place;
};

struct RopeQKParams {
    uint16_t* q;             // (B, S, Hq, D), strides sq_*, rotated in place
    uint16_t* k;             // (B, S, Hk, D), strides sk_*, rotated in place
    const uint16_t* cos;     // (B*S, rot) tables, or NULL when freqs is given
    const uint16_t* sin;
    const float* freqs;      // (S, B, 1, rot) angles, or NULL when tables are given
    int64_t B, S, Hq, Hk, D, rot;
    int64_t sq_b, sq_s, sq_h;
    int64_t sk_b, sk_s, sk_h;
};

struct GegluParams {
    const uint16_t* gate;
    const uint16_t* up;
    uint16_t* out;
    int64_t s_gate, s_up, s_out, T, F;
};

struct RmsParams {
    const uint16_t* x;
    uint16_t* residual;
    const uint16_t* w;
    uint16_t* out;
    int64_t sx, sr, so, T, C;
    float eps;
};

int num_sms();  // SM count of the current device (cached)

cudaError_t launch_rope_cos_sin(const float* freqs, int64_t S, int64_t B, int64_t R,
                                uint16_t* cos_out, uint16_t* sin_out, cudaStream_t st);
cudaError_t launch_rope_rotate_half(const RopeParams& p, cudaStream_t st);
cudaError_t launch_rope_qk(const RopeQKParams& p, cudaStream_t st);
size_t gelu_table_bytes();  // workspace the GEGLU launch needs for its activation table
cudaError_t launch_gelu_and_mul(const GegluParams& p, uint16_t* table, cudaStream_t st);
// Device address and size of the library-owned activation table of the
// current device (looked up on the first call per device).
cudaError_t noalloc_gelu_table(uint16_t** table, size_t* capacity);
cudaError_t launch_rmsnorm_residual(const RmsParams& p, cudaStream_t st);

}  // namespace dtrot
