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

// VEC = 8: R % 8 == 0 and every base pointer 16-byte aligned (freqs 32-byte).
template <int VEC>
__global__ void __launch_bounds__(256) rope_cos_sin_kernel(const float* __restrict__ freqs,
                                                          int64_t S, int64_t B, int64_t R,
                                                          uint16_t* __restrict__ cos_out,
                                                          uint16_t* __restrict__ sin_out) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t groups_per_row = R / VEC;
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
            float4 f0 = __ldg(reinterpret_cast<const float4*>(src));
            float4 f1 = __ldg(reinterpret_cast<const float4*>(src) + 1);
            float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
            uint16_t c[8], sn[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) cos_sin_entry(f[k], c[k], sn[k]);
            uint4 cv, sv;
            cv.x = c[0] | ((uint32_t)c[1] << 16);
            cv.y = c[2] | ((uint32_t)c[3] << 16);
            cv.z = c[4] | ((uint32_t)c[5] << 16);
            cv.w = c[6] | ((uint32_t)c[7] << 16);
            sv.x = sn[0] | ((uint32_t)sn[1] << 16);
            sv.y = sn[2] | ((uint32_t)sn[3] << 16);
            sv.z = sn[4] | ((uint32_t)sn[5] << 16);
            sv.w = sn[6] | ((uint32_t)sn[7] << 16);
            *reinterpret_cast<uint4*>(cos_out + dst) = cv;
            *reinterpret_cast<uint4*>(sin_out + dst) = sv;
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
    const int64_t work = B * S * (vec ? R / 8 : R);
    const int threads = 256;
    int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 8;  // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return vec ? launch_pdl(rope_cos_sin_kernel<8>, dim3((unsigned)blocks), dim3(threads), 0, st,
                            freqs, S, B, R, cos_out, sin_out)
               : launch_pdl(rope_cos_sin_kernel<1>, dim3((unsigned)blocks), dim3(threads), 0, st,
                            freqs, S, B, R, cos_out, sin_out);
}

}  // namespace dtrot
