// Rotary cos/sin tables, computed once per forward.
//
// ERNIE-Image fusion page (sglang PR #34306 analysis), section 1: freqs is the
// (S, B, 1, R) fp32 angle tensor; the tables are cos/sin in fp32 cast to bf16,
// laid out as (B*S, R) rows, row b*S + s.  The entry is defined as
// RN16(RN32(cos f)) with the fp32 cos correctly rounded.
//
// Evaluation (cos_sin_entry, shared with the fused q/k kernel): sincosf
// decides the bf16 rounding unless its result lies near a bf16 rounding
// midpoint, where the entry is recomputed in fp64.
//
// Layout: one thread per group of VEC consecutive columns of an output row;
// the permute is index arithmetic on the read side.  The table is a few tens
// of MB at most, so the kernel is bound by the sincosf arithmetic and by the
// launch, not by HBM.
#include "dtrot_internal.cuh"

namespace dtrot {
namespace {

__device__ __forceinline__ uint4 pack8(const uint16_t (&v)[8]) {
    return make_uint4(v[0] | ((uint32_t)v[1] << 16), v[2] | ((uint32_t)v[3] << 16),
                      v[4] | ((uint32_t)v[5] << 16), v[6] | ((uint32_t)v[7] << 16));
}

// Eight consecutive angles -> their cos and sin entries.
__device__ __forceinline__ void entries8(const float (&f)[8], uint16_t (&c)[8],
                                         uint16_t (&sn)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) cos_sin_entry(f[k], c[k], sn[k]);
}

__device__ __forceinline__ void load8(const float* src, float (&f)[8]) {
    const float4 f0 = __ldg(reinterpret_cast<const float4*>(src));
    const float4 f1 = __ldg(reinterpret_cast<const float4*>(src) + 1);
    f[0] = f0.x; f[1] = f0.y; f[2] = f0.z; f[3] = f0.w;
    f[4] = f1.x; f[5] = f1.y; f[6] = f1.z; f[7] = f1.w;
}

// VEC = 8: R % 8 == 0 and every base pointer 16-byte aligned (freqs 32-byte).
// PAIR (R % 16 == 0): a thread takes columns j..j+7 of the first half of the
// row and the same columns of the second half, j+R/2..; a second-half angle
// whose bits equal its first-half partner's has the same entry, which is then
// copied instead of evaluated again (a rotate-half table built from per-axis
// angles repeats its half-row, so this halves the arithmetic there; any other
// angle is evaluated, so nothing is assumed about the layout).  Loading the
// second half's angles only after evaluating the first half cost a second
// wait for memory per thread: 16.4 against 12.3 us per launch on the video
// layer after a streaming kernel, 8.0 against 6.5 us back to back.
template <int VEC, bool PAIR>
__global__ void __launch_bounds__(256) rope_cos_sin_kernel(const float* __restrict__ freqs,
                                                          int64_t S, int64_t B, int64_t R,
                                                          uint16_t* __restrict__ cos_out,
                                                          uint16_t* __restrict__ sin_out) {
    pdl_wait();
    const int64_t span = PAIR ? R / 2 : R;  // columns whose groups a thread starts at
    const int64_t groups_per_row = span / VEC;
    const int64_t total = B * S * groups_per_row;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < total;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = g / groups_per_row;
        const int64_t j = (g - row * groups_per_row) * VEC;
        const int64_t b = row / S;
        const int64_t s = row - b * S;
        const float* src = freqs + (s * B + b) * R + j;
        const int64_t dst = row * R + j;
        if constexpr (VEC == 8) {
            // both halves' angles are loaded before any is evaluated, so the
            // thread waits for memory once
            float f[8], f2[8];
            uint16_t c[8], sn[8];
            load8(src, f);
            if constexpr (PAIR) load8(src + R / 2, f2);
            entries8(f, c, sn);
            *reinterpret_cast<uint4*>(cos_out + dst) = pack8(c);
            *reinterpret_cast<uint4*>(sin_out + dst) = pack8(sn);
            if constexpr (PAIR) {
                const int64_t h = R / 2;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (__float_as_uint(f2[k]) != __float_as_uint(f[k])) {
                        const uint32_t e = cos_sin_entry_call(f2[k]);
                        c[k] = (uint16_t)e;
                        sn[k] = (uint16_t)(e >> 16);
                    }
                }
                *reinterpret_cast<uint4*>(cos_out + dst + h) = pack8(c);
                *reinterpret_cast<uint4*>(sin_out + dst + h) = pack8(sn);
            }
        } else {
            uint16_t c, sn;
            cos_sin_entry(__ldg(src), c, sn);
            cos_out[dst] = c;
            sin_out[dst] = sn;
        }
    }
}

bool aligned(const void* p, int bytes) { return ((uintptr_t)p % bytes) == 0; }

}  // namespace

cudaError_t launch_rope_cos_sin(const float* freqs, int64_t S, int64_t B, int64_t R,
                                uint16_t* cos_out, uint16_t* sin_out, cudaStream_t st) {
    const bool vec = (R % 8 == 0) && aligned(freqs, 32) && aligned(cos_out, 16) &&
                     aligned(sin_out, 16);
    const bool pair = vec && (R % 16 == 0);
    const int64_t work = B * S * (pair ? R / 16 : vec ? R / 8 : R);
    const int threads = 256;
    int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 8;  // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (pair)
        return launch_pdl(rope_cos_sin_kernel<8, true>, dim3((unsigned)blocks), dim3(threads), 0,
                          st, freqs, S, B, R, cos_out, sin_out);
    return vec ? launch_pdl(rope_cos_sin_kernel<8, false>, dim3((unsigned)blocks), dim3(threads),
                            0, st, freqs, S, B, R, cos_out, sin_out)
               : launch_pdl(rope_cos_sin_kernel<1, false>, dim3((unsigned)blocks), dim3(threads),
                            0, st, freqs, S, B, R, cos_out, sin_out);
}

}  // namespace dtrot
