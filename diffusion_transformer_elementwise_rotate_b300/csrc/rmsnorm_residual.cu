// Token-wise RMSNorm fused with the residual add (Pre-Norm order):
//   h = RN16(x + residual);  residual := h;
//   out = RN16(h * (mean(h^2) + eps)^(-1/2) * w)
//
// Sequence-parallelism post, section on per-token normalisation and residual
// add: RMSNorm rescales a token by that token's own features and the residual
// add pairs the same features of the same token, so a row is independent of
// every other row.  The Pre-Norm layer figure adds the residual, then
// normalises.
//
// Design.  One CTA per token row; each thread holds VPT 8-column vectors of
// the row in registers (one HBM read of x and residual, one write of h and
// out; w is re-read from L1/L2).
//   - h = one add.rn.bf16x2 per packed pair (the bf16 rounding of x + r);
//   - sum of h^2: each square is exact in fp32 (a bf16 has 8 significant
//     bits), accumulated per thread with TwoSum compensation, combined across
//     the warp as fp32 pairs with warp shuffles, and across warps in double by
//     one thread, which also forms inv = (sum/C + eps)^(-1/2) in double;
//   - out: h*w is exact in fp32; RN32(h*w*inv32) decides the bf16 rounding
//     unless it lies within 3 fp32 ulps of a bf16 midpoint (or h*w left the
//     fp32 normal range), where the value is recomputed as h*w*inv in double
//     and rounded once.  So the output is the rounding of the fp64 result
//     except in the rare rows where fp32-vs-fp64 summation order moves it
//     across a midpoint.
//   - rows whose fp32 sum of squares overflowed or is below 2^-60 (where
//     squares may have underflowed) redo the sum in double.
// A generic kernel (any alignment or width) loops over the row twice instead
// of keeping it in registers.
#include "dtrot_internal.cuh"

namespace dtrot {
namespace {

constexpr int kMaxWarps = 32;

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// acc (hi, lo) += v
__device__ __forceinline__ void acc_add(float& hi, float& lo, float v) {
    float e;
    two_sum(hi, v, hi, e);
    lo = __fadd_rn(lo, e);
}

// (hi, lo) += (hi2, lo2)
__device__ __forceinline__ void acc_merge(float& hi, float& lo, float hi2, float lo2) {
    float e;
    two_sum(hi, hi2, hi, e);
    lo = __fadd_rn(__fadd_rn(lo, lo2), e);
}

struct RowShared {
    float hi[kMaxWarps];
    float lo[kMaxWarps];
    double dsum[kMaxWarps];
    double inv_d;
    float inv_f;
    int redo;
};

// Block-wide reduction of the per-thread (hi, lo) pair; on return every
// thread sees inv (double and fp32) and whether the row must redo its sum of
// squares in double (then inv is not yet valid).
__device__ __forceinline__ void block_sumsq(RowShared& sh, float hi, float lo) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
        acc_merge(hi, lo, h2, l2);
    }
    if (lane == 0) {
        sh.hi[warp] = hi;
        sh.lo[warp] = lo;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0, fp32_mag = 0.0;
        const int nw = (blockDim.x + 31) >> 5;
        for (int w = 0; w < nw; ++w) {
            t += (double)sh.hi[w] + (double)sh.lo[w];
            fp32_mag += (double)sh.hi[w];
        }
        // an overflowed square makes hi inf (t inf or NaN); a tiny total may
        // have lost underflowed squares
        sh.redo = !(fabs(fp32_mag) < 1e38) || (t < 0x1p-60);
        sh.dsum[0] = t;
    }
    __syncthreads();
}

__device__ __forceinline__ void finish_inv(RowShared& sh, double total, int64_t C, float eps) {
    const double inv = 1.0 / sqrt(total / (double)C + (double)eps);
    sh.inv_d = inv;
    sh.inv_f = __double2float_rn(inv);
}

// Block-wide double sum of per-thread partials (the redo path).
__device__ __forceinline__ double block_sum_double(RowShared& sh, double v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();  // everyone has read dsum[0] of the fp32 pass
    if (lane == 0) sh.dsum[warp] = v;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        for (int w = 0; w < nw; ++w) t += sh.dsum[w];
    }
    return t;
}

// One output element from h and w (bf16 bits), with the midpoint check.
__device__ __forceinline__ uint16_t norm_out(uint32_t hb, uint32_t wb, float inv_f,
                                             double inv_d) {
    const float h = __uint_as_float(hb << 16);
    const float w = __uint_as_float(wb << 16);
    const float hw = __fmul_rn(h, w);
    const float y = __fmul_rn(hw, inv_f);
    const float ahw = fabsf(hw);
    const bool risky = (hw != 0.0f && !(ahw >= 0x1p-126f && ahw <= 0x1p127f)) ||
                       !(fabsf(y) <= 0x1p127f) || ulps_to_bf16_midpoint(y) <= 3;
    if (risky) return rn16d((double)h * (double)w * inv_d);  // NaN/inf follow IEEE here
    return rn16f(y);
}

__device__ __forceinline__ uint32_t norm_out2(uint32_t h2, uint32_t w2, float inv_f,
                                              double inv_d) {
    const uint32_t lo = norm_out(h2 & 0xFFFFu, w2 & 0xFFFFu, inv_f, inv_d);
    const uint32_t hi = norm_out(h2 >> 16, w2 >> 16, inv_f, inv_d);
    return lo | (hi << 16);
}

__device__ __forceinline__ void sq_acc2(uint32_t h2, float& hi, float& lo) {
    const float a = bf_lo(h2), b = bf_hi(h2);
    acc_add(hi, lo, __fmul_rn(a, a));
    acc_add(hi, lo, __fmul_rn(b, b));
}

__device__ __forceinline__ double sq_d2(uint32_t h2) {
    const double a = (double)bf_lo(h2), b = (double)bf_hi(h2);
    return a * a + b * b;
}

// Vector path: C % 8 == 0, strides % 8 == 0, pointers 16-byte aligned,
// C <= 8 * VPT * blockDim.
// Threads per CTA are at most 256 for VPT <= 4 and 512 for VPT = 8, which
// leaves 128 registers per thread for the row (x, residual and h vectors).
template <int VPT>
__global__ void __launch_bounds__(VPT == 8 ? 512 : 256) rms_vec_kernel(RmsParams p) {
    __shared__ RowShared sh;
    const int64_t nv = p.C >> 3;
    for (int64_t row = blockIdx.x; row < p.T; row += gridDim.x) {
        const uint16_t* xr = p.x + row * p.sx;
        uint16_t* rr = p.residual + row * p.sr;
        uint16_t* orow = p.out + row * p.so;
        uint4 hv[VPT];
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t v = (int64_t)k * blockDim.x + threadIdx.x;
            if (v < nv) {
                xv[k] = *reinterpret_cast<const uint4*>(xr + v * 8);
                rv[k] = *reinterpret_cast<const uint4*>(rr + v * 8);
            }
        }
        float hi = 0.0f, lo = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t v = (int64_t)k * blockDim.x + threadIdx.x;
            if (v < nv) {
                hv[k].x = badd2(xv[k].x, rv[k].x);
                hv[k].y = badd2(xv[k].y, rv[k].y);
                hv[k].z = badd2(xv[k].z, rv[k].z);
                hv[k].w = badd2(xv[k].w, rv[k].w);
                *reinterpret_cast<uint4*>(rr + v * 8) = hv[k];
                sq_acc2(hv[k].x, hi, lo);
                sq_acc2(hv[k].y, hi, lo);
                sq_acc2(hv[k].z, hi, lo);
                sq_acc2(hv[k].w, hi, lo);
            }
        }
        block_sumsq(sh, hi, lo);
        if (sh.redo) {  // uniform across the block
            double d = 0.0;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int64_t v = (int64_t)k * blockDim.x + threadIdx.x;
                if (v < nv) d += sq_d2(hv[k].x) + sq_d2(hv[k].y) + sq_d2(hv[k].z) + sq_d2(hv[k].w);
            }
            const double t = block_sum_double(sh, d);
            if (threadIdx.x == 0) finish_inv(sh, t, p.C, p.eps);
        } else if (threadIdx.x == 0) {
            finish_inv(sh, sh.dsum[0], p.C, p.eps);
        }
        __syncthreads();
        const float inv_f = sh.inv_f;
        const double inv_d = sh.inv_d;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int64_t v = (int64_t)k * blockDim.x + threadIdx.x;
            if (v < nv) {
                const uint4 wv = __ldg(reinterpret_cast<const uint4*>(p.w + v * 8));
                uint4 o;
                o.x = norm_out2(hv[k].x, wv.x, inv_f, inv_d);
                o.y = norm_out2(hv[k].y, wv.y, inv_f, inv_d);
                o.z = norm_out2(hv[k].z, wv.z, inv_f, inv_d);
                o.w = norm_out2(hv[k].w, wv.w, inv_f, inv_d);
                *reinterpret_cast<uint4*>(orow + v * 8) = o;
            }
        }
        __syncthreads();  // sh is reused by the next row
    }
}

// Generic path: any alignment and any C.  Pass 1 writes h into residual and
// accumulates; pass 2 re-reads the thread's own h values.
__global__ void __launch_bounds__(256) rms_generic_kernel(RmsParams p) {
    __shared__ RowShared sh;
    for (int64_t row = blockIdx.x; row < p.T; row += gridDim.x) {
        const uint16_t* xr = p.x + row * p.sx;
        uint16_t* rr = p.residual + row * p.sr;
        uint16_t* orow = p.out + row * p.so;
        float hi = 0.0f, lo = 0.0f;
        for (int64_t c = threadIdx.x; c < p.C; c += blockDim.x) {
            const uint32_t h = badd2(xr[c], rr[c]) & 0xFFFFu;
            rr[c] = (uint16_t)h;
            const float hf = bf_lo(h);
            acc_add(hi, lo, __fmul_rn(hf, hf));
        }
        block_sumsq(sh, hi, lo);
        if (sh.redo) {
            double d = 0.0;
            for (int64_t c = threadIdx.x; c < p.C; c += blockDim.x) {
                const double hf = (double)bf1(rr[c]);
                d += hf * hf;
            }
            const double t = block_sum_double(sh, d);
            if (threadIdx.x == 0) finish_inv(sh, t, p.C, p.eps);
        } else if (threadIdx.x == 0) {
            finish_inv(sh, sh.dsum[0], p.C, p.eps);
        }
        __syncthreads();
        const float inv_f = sh.inv_f;
        const double inv_d = sh.inv_d;
        for (int64_t c = threadIdx.x; c < p.C; c += blockDim.x) {
            orow[c] = norm_out(rr[c], p.w[c], inv_f, inv_d);
        }
        __syncthreads();
    }
}

bool aligned(const void* ptr, int bytes) { return ((uintptr_t)ptr % bytes) == 0; }

template <int VPT>
cudaError_t launch_vec(const RmsParams& p, int threads, cudaStream_t st) {
    int64_t blocks = p.T;
    if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
    rms_vec_kernel<VPT><<<(unsigned)blocks, threads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm_residual(const RmsParams& p, cudaStream_t st) {
    const bool vec = (p.C % 8 == 0) && (p.sx % 8 == 0) && (p.sr % 8 == 0) && (p.so % 8 == 0) &&
                     aligned(p.x, 16) && aligned(p.residual, 16) && aligned(p.w, 16) &&
                     aligned(p.out, 16);
    const int64_t nv = p.C / 8;
    if (vec && nv <= 8 * 512) {
        int vpt = 8;
        for (int c : {1, 2, 4, 8}) {
            if ((nv + c - 1) / c <= 256) {
                vpt = c;
                break;
            }
        }
        int threads = (int)((nv + vpt - 1) / vpt);
        threads = (threads + 31) / 32 * 32;
        switch (vpt) {
            case 1: return launch_vec<1>(p, threads, st);
            case 2: return launch_vec<2>(p, threads, st);
            case 4: return launch_vec<4>(p, threads, st);
            default: return launch_vec<8>(p, threads, st);
        }
    }
    int64_t blocks = p.T;
    if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
    rms_generic_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace dtrot
