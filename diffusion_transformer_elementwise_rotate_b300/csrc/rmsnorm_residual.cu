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
// Design.  Persistent CTAs (as many as fit on the device), each working on one
// token row at a time: thread t owns the 8-column vectors k * blockDim + t of
// every row (VPT of them), keeps its w vectors in registers for the whole
// launch, and loads the next row's x and residual vectors into registers while
// it works on the current one.  Rows of at most 1280 columns go to one warp
// each instead (lane l owns the vectors k * 32 + l), so their sums need no
// shared memory or barrier.  One HBM read of x and residual, one write of h
// and out per row.  No fp64 on the common path (this part's fp64 rate is a
// small fraction of its fp32 rate), so the row statistics are carried in fp32
// pairs ("double-float", value = hi + lo):
//   - h = one add.rn.bf16x2 per packed pair (the bf16 rounding of x + r);
//   - sum of h^2: each square is exact in fp32 (a bf16 has 8 significant
//     bits); accumulated with TwoSum on packed fp32x2 lanes, merged across the
//     warp with shuffles and across warps through shared memory (every thread
//     merges the warp partials in the same order, so all see the same total;
//     with a warp per row, the shuffle butterfly alone gives every lane the
//     same total);
//   - inv = (sum/C + eps)^(-1/2) as a double-float: rsqrtf seed plus one
//     Newton step with an exactly computed residual (relative error ~2^-43);
//   - out: h*w is exact in fp32; RN32(h*w*inv_hi) decides the bf16 rounding
//     unless it lies within 2 fp32 ulps of a bf16 midpoint or outside
//     [2^-90, 2^100]; there the product is formed as an exact fp32 pair (fma
//     error term) and a midpoint is resolved by the sign of the low part.
//   Only rows whose fp32 sum of squares overflowed or is tiny (< 2^-60, where
//   squares may have underflowed) and elements outside the fp32 normal range
//   (NaN, inf, |h*w| or |out| beyond 2^+-100) fall back to fp64.
// The exact path runs out of line: inlined at every packed word of a thread's
// vectors it made the kernel large enough to stall on instruction fetch (233
// against 218 us per call on 32760 x 5120), and rows that exactly fill the CTA
// (every width of the workloads) take a variant without bounds checks.
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

// |a| >= |b| (or a == 0)
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
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

// Per-row statistics exchanged between warps; two slots alternate by row so a
// warp starting the next row never overwrites values another warp still reads.
struct RowShared {
    float hi[2][kMaxWarps];
    float lo[2][kMaxWarps];
    double dsum[kMaxWarps];
};

// inv = (q + eps)^(-1/2) with q = (hi + lo) / C, as inv_hi + inv_lo.
__device__ __forceinline__ void inv_rms_df(float hi, float lo, int64_t C, float eps,
                                           float& inv_hi, float& inv_lo) {
    const float Cf = (float)C;                       // exact for C < 2^24
    const float q_hi = __fdiv_rn(hi, Cf);
    const float rem = __fmaf_rn(-q_hi, Cf, hi);      // exact: hi - q_hi * C
    const float q_lo = __fdiv_rn(__fadd_rn(rem, lo), Cf);
    float s_hi, e;
    two_sum(q_hi, eps, s_hi, e);
    float s_lo = __fadd_rn(e, q_lo);
    fast_two_sum(s_hi, s_lo, s_hi, s_lo);
    const float y0 = rsqrtf(s_hi);
    // residual 1 - s * y0^2, with y0^2 and s_hi * y0^2 formed exactly
    const float p_hi = __fmul_rn(y0, y0);
    const float p_lo = __fmaf_rn(y0, y0, -p_hi);
    const float t_hi = __fmul_rn(s_hi, p_hi);
    const float t_lo = __fmaf_rn(s_hi, p_hi, -t_hi);
    float rr = __fsub_rn(1.0f, t_hi);                // exact: t_hi is close to 1
    rr = __fsub_rn(rr, t_lo);
    rr = __fsub_rn(rr, __fmaf_rn(s_hi, p_lo, __fmul_rn(s_lo, p_hi)));
    const float corr = __fmul_rn(__fmul_rn(y0, rr), 0.5f);
    fast_two_sum(y0, corr, inv_hi, inv_lo);
}

// Block-wide sum of squares.  Returns false when the row must redo the sum in
// double (fp32 overflow, or a total small enough that squares may have
// underflowed); the result is identical in every thread.
__device__ __forceinline__ bool block_sumsq(RowShared& sh, int slot, float hi, float lo,
                                            float& tot_hi, float& tot_lo) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
        acc_merge(hi, lo, h2, l2);
    }
    if (lane == 0) {
        sh.hi[slot][warp] = hi;
        sh.lo[slot][warp] = lo;
    }
    __syncthreads();
    const int nw = (blockDim.x + 31) >> 5;
    float th = sh.hi[slot][0], tl = sh.lo[slot][0];
    for (int w = 1; w < nw; ++w) acc_merge(th, tl, sh.hi[slot][w], sh.lo[slot][w]);
    fast_two_sum(th, tl, tot_hi, tot_lo);
    return (tot_hi <= 1e37f) && (tot_hi >= 0x1p-60f);  // false for NaN too
}

// Block-wide double sum of per-thread partials (the rare redo path).
__device__ __forceinline__ double block_sum_double(RowShared& sh, double v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sh.dsum[warp] = v;
    __syncthreads();
    const int nw = (blockDim.x + 31) >> 5;
    double t = 0.0;
    for (int w = 0; w < nw; ++w) t += sh.dsum[w];
    __syncthreads();  // dsum is reused by the next redo row
    return t;
}

// Warp-wide versions for rows that one warp owns: the xor butterfly merges
// the same two values at every step (the merge is symmetric in its operands),
// so every lane ends with the same bits.
__device__ __forceinline__ bool warp_sumsq(float hi, float lo, float& tot_hi, float& tot_lo) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
        acc_merge(hi, lo, h2, l2);
    }
    fast_two_sum(hi, lo, tot_hi, tot_lo);
    return (tot_hi <= 1e37f) && (tot_hi >= 0x1p-60f);  // false for NaN too
}

__device__ __forceinline__ double warp_sum_double(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void inv_from_double(double total, int64_t C, float eps,
                                                float& inv_hi, float& inv_lo) {
    const double inv = 1.0 / sqrt(total / (double)C + (double)eps);
    inv_hi = __double2float_rn(inv);
    inv_lo = __double2float_rn(inv - (double)inv_hi);
}

// NaN, inf and extreme magnitudes: IEEE double (kept out of line so the
// common path's register allocation does not carry it).
__device__ __noinline__ uint16_t norm_out_rare(float h, float w, float inv_hi, float inv_lo) {
    return rn16d((double)h * (double)w * ((double)inv_hi + (double)inv_lo));
}

// One output element from h and w (bf16 bits).
__device__ __forceinline__ uint16_t norm_out(uint32_t hb, uint32_t wb, float inv_hi,
                                             float inv_lo) {
    const float h = __uint_as_float(hb << 16);
    const float w = __uint_as_float(wb << 16);
    const float hw = __fmul_rn(h, w);                 // exact in the normal range
    const float y = __fmul_rn(hw, inv_hi);
    const float ahw = fabsf(hw), ay = fabsf(y);
    const bool normal = (ahw >= 0x1p-100f && ahw <= 0x1p100f && ay >= 0x1p-100f &&
                         ay <= 0x1p100f);
    if (normal) {
        if (ulps_to_bf16_midpoint(y) > 2) return rn16f(y);
        // exact pair for hw * inv_hi, plus hw * inv_lo
        const float p_lo = __fmaf_rn(hw, inv_hi, -y);
        const float y_lo = __fmaf_rn(hw, inv_lo, p_lo);
        float y2, y2lo;
        fast_two_sum(y, y_lo, y2, y2lo);
        const uint32_t u = __float_as_uint(y2);
        if ((u & 0xFFFFu) == 0x8000u && y2lo != 0.0f) {
            // exactly on a midpoint in fp32: the low part decides
            const bool away = (y2lo > 0.0f) == (y2 > 0.0f);
            return (uint16_t)((u >> 16) + (away ? 1u : 0u));
        }
        return rn16f(y2);
    }
    if (hw == 0.0f && ay == 0.0f) return rn16f(y);    // exact zero (h or w is 0)
    return norm_out_rare(h, w, inv_hi, inv_lo);
}

// Two output elements by the exact path, out of line: the vector kernel runs it
// for a few elements in 10^4, and inlined at each of its call sites (one per
// packed word of a thread's vectors) it made the kernel's code large enough
// to stall on instruction fetch.
__device__ __noinline__ uint32_t norm_out2(uint32_t h2, uint32_t w2, float inv_hi,
                                           float inv_lo) {
    const uint32_t lo = norm_out(h2 & 0xFFFFu, w2 & 0xFFFFu, inv_hi, inv_lo);
    const uint32_t hi = norm_out(h2 >> 16, w2 >> 16, inv_hi, inv_lo);
    return lo | (hi << 16);
}

__device__ __forceinline__ double sq_d2(uint32_t h2) {
    const double a = (double)bf_lo(h2), b = (double)bf_hi(h2);
    return a * a + b * b;
}

// Row statistics: inv = (mean(h^2) + eps)^(-1/2) as a double-float, from the
// thread's compensated partial sum; `redo_sq` recomputes the thread's partial
// in double when the fp32 total is out of range (uniform across the row's
// threads).  WARP: the row belongs to one warp (sh is not used).
template <bool WARP, typename RedoSq>
__device__ __forceinline__ void row_inv(RowShared* sh, int slot, float hi, float lo, int64_t C,
                                        float eps, RedoSq redo_sq, float& inv_hi,
                                        float& inv_lo) {
    float th, tl;
    const bool ok = WARP ? warp_sumsq(hi, lo, th, tl) : block_sumsq(*sh, slot, hi, lo, th, tl);
    if (ok && C < (1 << 24)) {
        inv_rms_df(th, tl, C, eps, inv_hi, inv_lo);
    } else {
        const double t = WARP ? warp_sum_double(redo_sq()) : block_sum_double(*sh, redo_sq());
        inv_from_double(t, C, eps, inv_hi, inv_lo);
    }
}

// ---- packed fp32 pairs (two lanes per 64-bit register, one .rn rounding per lane)

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float f2lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t add_x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub_x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul_x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// bf16x2 word -> its two values as an exact fp32 pair
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
    return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// (hi, lo) += v lane-wise, TwoSum: hi + lo + v == new hi + new lo exactly up
// to the rounding of the lo accumulation.
__device__ __forceinline__ void acc_add_x2(uint64_t& hi, uint64_t& lo, uint64_t v) {
    const uint64_t s = add_x2(hi, v);
    const uint64_t bb = sub_x2(s, hi);
    const uint64_t e = add_x2(sub_x2(hi, sub_x2(s, bb)), sub_x2(v, bb));
    lo = add_x2(lo, e);
    hi = s;
}

// Fast-path acceptance test for y = RN32(h * w * inv_hi): the bf16 rounding of
// y is final when y is at least 3 fp32 ulps from a bf16 rounding midpoint and
// 2^-90 <= |y| <= 2^100 (h * w exact, y normal).  NaN fails the range test.
__device__ __forceinline__ bool y_settled(float y) {
    const float a = fabsf(y);
    const bool mid = ((__float_as_uint(y) + 0x8002u) & 0xFFFFu) <= 4u;
    return (a >= 0x1p-90f) && (a <= 0x1p100f) && !mid;
}

// The 8-column vectors of a row that a thread owns: v = k * row_stride + idx
// for k < VPT (and v < nv), the row spread over the CTA (idx = thread) or,
// WARP, over one warp (idx = lane).
template <bool WARP>
__device__ __forceinline__ int row_idx() { return WARP ? (int)(threadIdx.x & 31) : (int)threadIdx.x; }
template <bool WARP>
__device__ __forceinline__ int row_stride() { return WARP ? 32 : (int)blockDim.x; }

// One token row on the vector path.  The thread owns the vectors
// v = k * row_stride + row_idx (k < VPT, v < nv); xc, rc hold its x and
// residual vectors of the row and wv its w vectors.  FULL: nv == VPT *
// row_stride (every thread owns VPT vectors, so no access needs a bounds
// check).
template <int VPT, bool FULL, bool WARP>
__device__ __forceinline__ void rms_row(const RmsParams& p, RowShared* sh, int slot, int64_t row,
                                        int nv, const uint4 (&xc)[VPT], const uint4 (&rc)[VPT],
                                        const uint4 (&wv)[VPT]) {
    const int tid = row_idx<WARP>();
    const int stride = row_stride<WARP>();
    // h = RN16(x + r), written back to the residual stream; exact squares
    // accumulated lane-wise with TwoSum
    uint4 hv[VPT];
    uint64_t hi = 0, lo = 0;
    uint4* rrow = reinterpret_cast<uint4*>(p.residual + row * p.sr);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * stride + tid;
        if (FULL || v < nv) {
            hv[k].x = badd2(xc[k].x, rc[k].x);
            hv[k].y = badd2(xc[k].y, rc[k].y);
            hv[k].z = badd2(xc[k].z, rc[k].z);
            hv[k].w = badd2(xc[k].w, rc[k].w);
            rrow[v] = hv[k];
            uint64_t f;
            f = bf2_to_f2(hv[k].x);
            acc_add_x2(hi, lo, mul_x2(f, f));
            f = bf2_to_f2(hv[k].y);
            acc_add_x2(hi, lo, mul_x2(f, f));
            f = bf2_to_f2(hv[k].z);
            acc_add_x2(hi, lo, mul_x2(f, f));
            f = bf2_to_f2(hv[k].w);
            acc_add_x2(hi, lo, mul_x2(f, f));
        }
    }
    float shi = f2lo(hi), slo = f2lo(lo);
    acc_merge(shi, slo, f2hi(hi), f2hi(lo));

    float inv_hi, inv_lo;
    row_inv<WARP>(sh, slot, shi, slo, p.C, p.eps,
            [&]() {
                double d = 0.0;
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = k * stride + tid;
                    if (FULL || v < nv)
                        d += sq_d2(hv[k].x) + sq_d2(hv[k].y) + sq_d2(hv[k].z) + sq_d2(hv[k].w);
                }
                return d;
            },
            inv_hi, inv_lo);

    // out = RN16(h * w * inv): RN32(RN32(h * w) * inv_hi) decides unless it is
    // near a bf16 midpoint or outside the safe range (then the exact path).
    // With inv <= 2^40, |y| >= 2^-90 implies |h * w| >= 2^-130, where the
    // product of two bf16 values is exact in fp32; rows with a larger inverse
    // (only possible through the double re-sum) take the exact path.
    const bool fast_row = inv_hi <= 0x1p40f;
    const uint64_t inv2 = f2(inv_hi, inv_hi);
    uint4* orow = reinterpret_cast<uint4*>(p.out + row * p.so);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * stride + tid;
        if (FULL || v < nv) {
            const uint32_t hw[4] = {hv[k].x, hv[k].y, hv[k].z, hv[k].w};
            const uint32_t ww[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint64_t y = mul_x2(mul_x2(bf2_to_f2(hw[q]), bf2_to_f2(ww[q])), inv2);
                const float y0 = f2lo(y), y1 = f2hi(y);
                if (fast_row && y_settled(y0) && y_settled(y1))
                    o[q] = rn16x2f(y0, y1);
                else
                    o[q] = norm_out2(hw[q], ww[q], inv_hi, inv_lo);
            }
            orow[v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

template <int VPT, bool FULL, bool WARP>
__device__ __forceinline__ void load_w(const RmsParams& p, int nv, uint4 (&wv)[VPT]) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * row_stride<WARP>() + row_idx<WARP>();
        if (FULL || v < nv) wv[k] = __ldg(reinterpret_cast<const uint4*>(p.w) + v);
    }
}

// A row's x and residual vectors into registers.
template <int VPT, bool FULL, bool WARP>
__device__ __forceinline__ void load_row(const RmsParams& p, int nv, int64_t r, uint4 (&xs)[VPT],
                                         uint4 (&rs)[VPT]) {
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + r * p.sx);
    const uint4* rr = reinterpret_cast<const uint4*>(p.residual + r * p.sr);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * row_stride<WARP>() + row_idx<WARP>();
        if (FULL || v < nv) {
            xs[k] = xr[v];
            rs[k] = rr[v];
        }
    }
}

// Vector path: C % 8 == 0, strides % 8 == 0, pointers 16-byte aligned,
// C <= 8 * VPT * blockDim.  Persistent CTAs, one token row at a time;
// each thread keeps its w vectors in registers for the whole launch and
// prefetches the next row's x and residual vectors into registers while it
// works on the current row.  Register budgets: the launcher gives VPT 2 and 4
// at most 160 threads, and the bounds below keep 5 and 3 such CTAs per SM
// (unbounded, the guard-free FULL variant of VPT 2 took 118 registers and fit
// 3, 5% slower at C = 2560; bounding VPT 1 the same way made C = 768 6%
// slower, so VPT 1 and 8 keep the compiler's choice: a minimum of 0 CTAs
// leaves the register count unconstrained).
constexpr int rms_max_threads(int vpt) { return (vpt == 2 || vpt == 4) ? 160 : 256; }
constexpr int rms_min_blocks(int vpt) { return vpt == 2 ? 5 : vpt == 4 ? 3 : 0; }

template <int VPT, bool FULL>
__global__ void __launch_bounds__(rms_max_threads(VPT), rms_min_blocks(VPT))
    rms_vec_kernel(RmsParams p) {
    __shared__ RowShared sh;
    pdl_wait();
    const int nv = (int)(p.C >> 3);
    uint4 wv[VPT], xc[VPT], rc[VPT];
    load_w<VPT, FULL, false>(p, nv, wv);
    int64_t row = blockIdx.x;
    if (row < p.T) load_row<VPT, FULL, false>(p, nv, row, xc, rc);
    int slot = 0;
    for (; row < p.T; row += gridDim.x, slot ^= 1) {
        uint4 xn[VPT], rn[VPT];
        const int64_t nrow = row + gridDim.x;
        if (nrow < p.T) load_row<VPT, FULL, false>(p, nv, nrow, xn, rn);
        rms_row<VPT, FULL, false>(p, &sh, slot, row, nv, xc, rc, wv);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            xc[k] = xn[k];
            rc[k] = rn[k];
        }
    }
}

// Narrow rows (at most 32 * VPT vectors): one warp per row, so the row's sum
// needs shuffles only, no shared memory and no barrier; the warps of a CTA
// work on different rows independently.  Persistent warps, each prefetching
// its next row like the CTA-wide kernel (up to 4 vectors per lane), in CTAs
// of 4 warps.  Measured per call at ~1.34 GB (32 * VPT a multiple of C / 8 or
// not): C = 768 225 us and C = 1024 215 us against 288 and 277 us with a CTA
// per row; C = 1152 (5 vectors per lane, no prefetch) 241 against 346 us.
// The variant without bounds checks for rows that fill the warp, and 8-warp
// CTAs, were slower at some widths (C = 768: 452 us), so every width takes
// this one.  From C = 1288 up a CTA per row is faster (C = 1536: 230 against
// 249 us with 6 vectors per lane; C = 2048: 226 against 237 us).
constexpr int kWarpRowThreads = 128;
constexpr int kWarpPrefetchVpt = 4;  // up to this many vectors per lane, prefetch the next row
constexpr int kWarpMaxVpt = 5;       // rows of up to 32 * 5 vectors (C <= 1280) take a warp

template <int VPT>
__global__ void __launch_bounds__(kWarpRowThreads) rms_warp_kernel(RmsParams p) {
    pdl_wait();
    const int nv = (int)(p.C >> 3);
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    uint4 wv[VPT], xc[VPT], rc[VPT];
    load_w<VPT, false, true>(p, nv, wv);
    int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if constexpr (VPT > kWarpPrefetchVpt) {
        // wider rows: the row's own 2 * VPT loads per lane are enough in flight
        for (; row < p.T; row += warps) {
            load_row<VPT, false, true>(p, nv, row, xc, rc);
            rms_row<VPT, false, true>(p, nullptr, 0, row, nv, xc, rc, wv);
        }
        return;
    }
    if (row < p.T) load_row<VPT, false, true>(p, nv, row, xc, rc);
    for (; row < p.T; row += warps) {
        uint4 xn[VPT], rn[VPT];
        const int64_t nrow = row + warps;
        if (nrow < p.T) load_row<VPT, false, true>(p, nv, nrow, xn, rn);
        rms_row<VPT, false, true>(p, nullptr, 0, row, nv, xc, rc, wv);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            xc[k] = xn[k];
            rc[k] = rn[k];
        }
    }
}

// Generic path: any alignment and any C.  Pass 1 writes h into residual and
// accumulates; pass 2 re-reads the thread's own h values.
__global__ void __launch_bounds__(256) rms_generic_kernel(RmsParams p) {
    __shared__ RowShared sh;
    pdl_wait();
    int slot = 0;
    for (int64_t row = blockIdx.x; row < p.T; row += gridDim.x, slot ^= 1) {
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
        float inv_hi, inv_lo;
        row_inv<false>(&sh, slot, hi, lo, p.C, p.eps,
                [&]() {
                    double d = 0.0;
                    for (int64_t c = threadIdx.x; c < p.C; c += blockDim.x) {
                        const double hf = (double)bf1(rr[c]);
                        d += hf * hf;
                    }
                    return d;
                },
                inv_hi, inv_lo);
        for (int64_t c = threadIdx.x; c < p.C; c += blockDim.x) {
            orow[c] = norm_out(rr[c], p.w[c], inv_hi, inv_lo);
        }
    }
}

bool aligned(const void* ptr, int bytes) { return ((uintptr_t)ptr % bytes) == 0; }

// CTAs of `kernel` that fit on one SM at once (at least 1).
template <typename K>
cudaError_t per_sm_blocks(K kernel, int threads, size_t smem, int* n) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kernel, threads, smem);
    if (*n < 1) *n = 1;
    return e;
}

template <int VPT, bool FULL>
cudaError_t launch_vec_as(const RmsParams& p, int threads, cudaStream_t st) {
    // persistent grid: as many CTAs as fit on the device at once, at most T
    int per_sm = 0;
    cudaError_t e = per_sm_blocks(rms_vec_kernel<VPT, FULL>, threads, 0, &per_sm);
    if (e != cudaSuccess) return e;
    int64_t blocks = (int64_t)num_sms() * per_sm;
    if (blocks > p.T) blocks = p.T;
    return launch_pdl(rms_vec_kernel<VPT, FULL>, dim3((unsigned)blocks), dim3(threads), 0, st,
                      p);
}

template <int VPT>
cudaError_t launch_vec(const RmsParams& p, int threads, cudaStream_t st) {
    return (p.C / 8 == (int64_t)VPT * threads) ? launch_vec_as<VPT, true>(p, threads, st)
                                               : launch_vec_as<VPT, false>(p, threads, st);
}

template <int VPT>
cudaError_t launch_warp(const RmsParams& p, cudaStream_t st) {
    // persistent warps: as many CTAs as fit on the device, at most one warp per row
    int per_sm = 0;
    cudaError_t e = per_sm_blocks(rms_warp_kernel<VPT>, kWarpRowThreads, 0, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t rows_per_cta = kWarpRowThreads / 32;
    int64_t blocks = (int64_t)num_sms() * per_sm;
    const int64_t need = (p.T + rows_per_cta - 1) / rows_per_cta;
    if (blocks > need) blocks = need;
    return launch_pdl(rms_warp_kernel<VPT>, dim3((unsigned)blocks), dim3(kWarpRowThreads), 0,
                      st, p);
}

}  // namespace

cudaError_t launch_rmsnorm_residual(const RmsParams& p, cudaStream_t st) {
    const bool vec = (p.C % 8 == 0) && (p.sx % 8 == 0) && (p.sr % 8 == 0) && (p.so % 8 == 0) &&
                     aligned(p.x, 16) && aligned(p.residual, 16) && aligned(p.w, 16) &&
                     aligned(p.out, 16);
    const int64_t nv = p.C / 8;
    // rows of at most 160 vectors (C <= 1280): one warp per row, VPT = nv / 32
    // rounded up
    if (vec && nv <= kWarpMaxVpt * 32) {
        switch ((nv + 31) / 32) {
            case 1: return launch_warp<1>(p, st);
            case 2: return launch_warp<2>(p, st);
            case 3: return launch_warp<3>(p, st);
            case 4: return launch_warp<4>(p, st);
            default: return launch_warp<5>(p, st);
        }
    }
    // VPT vectors per thread: the smallest of 1, 2, 4 that keeps a row within
    // 160 threads, else 8 (up to 256 threads, C <= 16384)
    if (vec && nv <= 8 * 256) {
        int vpt = 8;
        for (int c : {1, 2, 4}) {
            if ((nv + c - 1) / c <= 160) {
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
    return launch_pdl(rms_generic_kernel, dim3((unsigned)blocks), dim3(256), 0, st, p);
}

}  // namespace dtrot
