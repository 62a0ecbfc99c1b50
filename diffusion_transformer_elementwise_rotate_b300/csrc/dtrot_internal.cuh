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

// The fp64 recomputations, out of line: they run for a few entries in 10^4,
// and inlined at every call site they made the table kernel's code large
// enough to stall on instruction fetch.
static __device__ __noinline__ float cos_exact_f32(float f) { return __double2float_rn(cos((double)f)); }
static __device__ __noinline__ float sin_exact_f32(float f) { return __double2float_rn(sin((double)f)); }

__device__ __forceinline__ void cos_sin_entry(float f, uint16_t& c16, uint16_t& s16) {
    float s32, c32;
    sincosf(f, &s32, &c32);
    if (ulps_to_bf16_midpoint(c32) <= kCosSinMargin) c32 = cos_exact_f32(f);
    if (ulps_to_bf16_midpoint(s32) <= kCosSinMargin) s32 = sin_exact_f32(f);
    c16 = rn16f(c32);
    s16 = rn16f(s32);
}

// The same entry through a call (for paths that rarely need it).
static __device__ __noinline__ uint32_t cos_sin_entry_call(float f) {
    uint16_t c, s;
    cos_sin_entry(f, c, s);
    return (uint32_t)c | ((uint32_t)s << 16);
}

// ------------------------------------------------------------ GELU table entries

// RN16(RN32(gelu(x))) for the bf16 value with bit pattern `bits`, gelu(x) =
// x/2 * erfc(-x/sqrt 2) (the erf form's exact equal, without its cancellation
// for x << 0).  fp32 erfcf decides the rounding unless the fp32 value lies
// within an error margin of a bf16 rounding midpoint (the margin grows with
// erfc's condition number 2z^2 for z = -x/sqrt 2 > 0); those entries, and the
// far negative tail x in (-20, -9) where the fp32 erfc result loses precision
// to underflow, are recomputed in fp64 and rounded to fp32, then to bf16.
__device__ inline uint16_t gelu_entry(uint32_t bits) {
    const float x = __uint_as_float(bits << 16);
    const float z = __fmul_rn(x, -0.70710678118654752440f);  // -x / sqrt 2
    bool slow = (x < -9.0f) && (x > -20.0f);
    float y = 0.0f;
    if (!slow) {
        const float e = erfcf(z);
        y = __fmul_rn(__fmul_rn(0.5f, x), e);
        const float zz = z > 0.0f ? fminf(z, 16.0f) : 0.0f;
        const int margin = 8 + (int)(4.0f * zz * zz);
        slow = ulps_to_bf16_midpoint(y) <= margin;
    }
    if (slow) {
        const double xd = (double)x;
        y = __double2float_rn(0.5 * xd * erfc(-xd * 0.70710678118654752440));
    }
    return rn16f(y);
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
    const uint16_t* q;       // (B, S, Hq, D), strides sq_*
    const uint16_t* k;       // (B, S, Hk, D), strides sk_*
    uint16_t* qo;            // rotated q, strides sqo_* (== q, sq_* in place)
    uint16_t* ko;            // rotated k, strides sko_* (== k, sk_* in place)
    const uint16_t* cos;     // (B*S, rot) tables, or NULL when freqs is given
    const uint16_t* sin;
    const float* freqs;      // (S, B, 1, rot) angles, or NULL when tables are given
    int64_t B, S, Hq, Hk, D, rot;
    int64_t sq_b, sq_s, sq_h;
    int64_t sk_b, sk_s, sk_h;
    int64_t sqo_b, sqo_s, sqo_h;
    int64_t sko_b, sko_s, sko_h;
    int copy_tail;           // out of place: columns [rot, D) are copied to the outputs
};

struct GemmGegluArgs {
    const uint16_t* x;   // (T, C) row-major
    const uint16_t* w;   // (2F, C) row-major, gate rows first
    int64_t T, C, F;
    uint16_t* out;       // (T, F), row stride s_out
    int64_t s_out;
    uint16_t* gate_up;   // optional (T, 2F), row stride s_gate_up
    int64_t s_gate_up;
    void* workspace;     // gemm_geglu_workspace_bytes()
    int withhold_last_stage = 0;  // diagnostic (see dtrot_gemm_gelu_and_mul_withhold_last_stage)
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

// ------------------------------------------------------------ launch order
//
// The library's kernels are launched as programmatic dependents of the
// previous kernel in the stream.  None of the elementwise kernels triggers its
// dependents early: the next launch is scheduled as this kernel's CTAs exit,
// which overlaps its launch latency and ramp-up with this kernel's drain, and
// its CTAs never sit on an SM beside running CTAs of this kernel (an early
// trigger was measured equal on the video layer and 1-1.5% slower on the image
// and CFG layers).  Every kernel executes pdl_wait() before its first
// global-memory access, read or write; pdl_wait returns once the predecessor
// has completed and its writes are visible (at once when the launch has no
// programmatic predecessor), so every memory effect keeps plain stream order.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

int num_sms();  // SM count of the current device (cached)
// Process-unique id of the CUDA context current on this thread (cuCtxGetId),
// 0 if none is current.  Per-device set-up (function attributes, symbol
// addresses) is cached against it, so it is redone after cudaDeviceReset
// gives the device a new primary context.
uint64_t current_context_id();

cudaError_t launch_rope_cos_sin(const float* freqs, int64_t S, int64_t B, int64_t R,
                                uint16_t* cos_out, uint16_t* sin_out, cudaStream_t st);
cudaError_t launch_rope_rotate_half(const RopeParams& p, cudaStream_t st);
cudaError_t launch_rope_qk(const RopeQKParams& p, cudaStream_t st);
size_t gemm_geglu_workspace_bytes();
size_t gemm_geglu_error_offset();  // byte offset of the error word in that workspace
cudaError_t launch_gemm_geglu(const GemmGegluArgs& a, cudaStream_t st);
size_t gelu_table_bytes();  // workspace the GEGLU launch needs for its activation table
cudaError_t launch_gelu_and_mul(const GegluParams& p, uint16_t* table, cudaStream_t st);
cudaError_t launch_gelu_table(uint16_t* table, cudaStream_t st);
// The streaming kernel alone, on a table already built (or being built by the
// previous launch in the stream).
cudaError_t launch_gelu_stream(const GegluParams& p, const uint16_t* table, cudaStream_t st);
// Device address and size of the library-owned activation table of the
// current device (looked up on the first call per device).
cudaError_t noalloc_gelu_table(uint16_t** table, size_t* capacity);
cudaError_t launch_rmsnorm_residual(const RmsParams& p, cudaStream_t st);

}  // namespace dtrot
