// Rotate-half RoPE over the leading rot_dim columns of x (B, S, H, D).
//
// ERNIE-Image fusion page (sglang PR #34306 analysis), section 2: the eager
// chain chunk / neg / cat / mul / add rounds every product and the sum to
// bf16, round(round(x1*cos1) + round(-x2*sin1)); the fused kernel must give
// the same bits, with the tail columns [rot_dim, D) passed through.  Each
// product and the sum is one bf16x2 instruction with .rn rounding, so the
// per-op rounding is the hardware's and nothing can be contracted.
//
// Fast path (the pair half-width h and D are multiples of the vector width VW,
// and a head row has at most 32 vector items):
//   - one warp per token (b, s); a head row is split into NI items: NP = h/VW
//     "pair" items (columns j..j+VW and their partners j+h..j+h+VW) followed by
//     NT = (D-rot)/VW "tail" items (plain copies);
//   - lane -> (ri, it) with it = lane % NI, ri = lane / NI: lanes keep fixed
//     columns and walk heads ri, ri + RPW, ... (RPW = 32 / NI rows per pass),
//     so each lane loads its cos/sin vectors of the token once into registers
//     and reuses them for all H / RPW heads it visits;
//   - heads are processed in batches of U: all loads of a batch are issued
//     before any store, which keeps U * 2 vector loads in flight per lane and
//     stays correct in place (every element belongs to exactly one item).
// Generic path (any alignment / width): one thread per (token, head, item),
// items = h pair columns plus the tail columns, scalar bf16 ops.
#include "dtrot_internal.cuh"

namespace dtrot {
namespace {

template <int VW>
struct VecT;
template <>
struct VecT<8> { using T = uint4; };
template <>
struct VecT<4> { using T = uint2; };
template <>
struct VecT<2> { using T = uint32_t; };

template <int VW>
__device__ __forceinline__ typename VecT<VW>::T ldv(const uint16_t* p) {
    return *reinterpret_cast<const typename VecT<VW>::T*>(p);
}
template <int VW>
__device__ __forceinline__ void stv(uint16_t* p, typename VecT<VW>::T v) {
    *reinterpret_cast<typename VecT<VW>::T*>(p) = v;
}

// Apply the rotation to one packed word (2 bf16 lanes) of the first and the
// second half.
__device__ __forceinline__ void rot_word(uint32_t x1, uint32_t x2, uint32_t c1, uint32_t s1,
                                         uint32_t c2, uint32_t s2, uint32_t& o1,
                                         uint32_t& o2) {
    o1 = bsub2(bmul2(x1, c1), bmul2(x2, s1));  // R(R(x1 c1) + R(-x2 s1))
    o2 = badd2(bmul2(x2, c2), bmul2(x1, s2));  // R(R(x2 c2) + R( x1 s2))
}

__device__ __forceinline__ void rot_vec(uint4 a, uint4 b, uint4 c1, uint4 s1, uint4 c2,
                                        uint4 s2, uint4& o1, uint4& o2) {
    rot_word(a.x, b.x, c1.x, s1.x, c2.x, s2.x, o1.x, o2.x);
    rot_word(a.y, b.y, c1.y, s1.y, c2.y, s2.y, o1.y, o2.y);
    rot_word(a.z, b.z, c1.z, s1.z, c2.z, s2.z, o1.z, o2.z);
    rot_word(a.w, b.w, c1.w, s1.w, c2.w, s2.w, o1.w, o2.w);
}
__device__ __forceinline__ void rot_vec(uint2 a, uint2 b, uint2 c1, uint2 s1, uint2 c2,
                                        uint2 s2, uint2& o1, uint2& o2) {
    rot_word(a.x, b.x, c1.x, s1.x, c2.x, s2.x, o1.x, o2.x);
    rot_word(a.y, b.y, c1.y, s1.y, c2.y, s2.y, o1.y, o2.y);
}
__device__ __forceinline__ void rot_vec(uint32_t a, uint32_t b, uint32_t c1, uint32_t s1,
                                        uint32_t c2, uint32_t s2, uint32_t& o1,
                                        uint32_t& o2) {
    rot_word(a, b, c1, s1, c2, s2, o1, o2);
}

struct FastArgs {
    RopeParams p;
    int NP;   // pair items per head row
    int NI;   // items per head row (NP + tail items)
    int RPW;  // head rows per warp pass
};

template <int VW, int U>
__global__ void __launch_bounds__(256) rope_fast_kernel(FastArgs a) {
    pdl_wait();
    using V = typename VecT<VW>::T;
    const RopeParams& p = a.p;
    const int lane = threadIdx.x & 31;
    const int ri = lane / a.NI;
    const int it = lane - ri * a.NI;
    if (ri >= a.RPW) return;  // idle lanes (32 is not a multiple of NI)
    const int64_t ntok = p.B * p.S;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t hh = p.rot >> 1;
    const bool pair = it < a.NP;
    const int64_t j = pair ? (int64_t)it * VW : p.rot + (int64_t)(it - a.NP) * VW;

    for (int64_t tok = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         tok < ntok; tok += warps) {
        const int64_t b = tok / p.S;
        const int64_t s = tok - b * p.S;
        const uint16_t* xr = p.x + b * p.sx_b + s * p.sx_s + j;
        uint16_t* orow = p.out + b * p.so_b + s * p.so_s + j;
        if (pair) {
            const uint16_t* ct = p.cos + tok * p.rot + j;
            const uint16_t* st = p.sin + tok * p.rot + j;
            const V c1 = ldv<VW>(ct), c2 = ldv<VW>(ct + hh);
            const V s1 = ldv<VW>(st), s2 = ldv<VW>(st + hh);
            for (int64_t h0 = ri; h0 < p.H; h0 += (int64_t)U * a.RPW) {
                V xa[U], xb[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t h = h0 + (int64_t)u * a.RPW;
                    if (h < p.H) {
                        xa[u] = ldv<VW>(xr + h * p.sx_h);
                        xb[u] = ldv<VW>(xr + h * p.sx_h + hh);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t h = h0 + (int64_t)u * a.RPW;
                    if (h < p.H) {
                        V o1, o2;
                        rot_vec(xa[u], xb[u], c1, s1, c2, s2, o1, o2);
                        stv<VW>(orow + h * p.so_h, o1);
                        stv<VW>(orow + h * p.so_h + hh, o2);
                    }
                }
            }
        } else {
            for (int64_t h0 = ri; h0 < p.H; h0 += (int64_t)U * a.RPW) {
                V xa[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t h = h0 + (int64_t)u * a.RPW;
                    if (h < p.H) xa[u] = ldv<VW>(xr + h * p.sx_h);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t h = h0 + (int64_t)u * a.RPW;
                    if (h < p.H) stv<VW>(orow + h * p.so_h, xa[u]);
                }
            }
        }
    }
}

// Generic path: one thread per (token, head, item); item < h is the pair
// (j, j + h), item >= h is tail column rot + (item - h).
__global__ void __launch_bounds__(256) rope_generic_kernel(RopeParams p, int64_t items) {
    pdl_wait();
    const int64_t hh = p.rot >> 1;
    const int64_t per_tok = p.H * items;
    const int64_t total = p.B * p.S * per_tok;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < total;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tok = g / per_tok;
        const int64_t rem = g - tok * per_tok;
        const int64_t h = rem / items;
        const int64_t it = rem - h * items;
        const int64_t b = tok / p.S;
        const int64_t s = tok - b * p.S;
        const uint16_t* xr = p.x + b * p.sx_b + s * p.sx_s + h * p.sx_h;
        uint16_t* orow = p.out + b * p.so_b + s * p.so_s + h * p.so_h;
        if (it < hh) {
            const uint16_t* ct = p.cos + tok * p.rot;
            const uint16_t* st = p.sin + tok * p.rot;
            const uint32_t x1 = xr[it], x2 = xr[it + hh];
            uint32_t o1, o2;
            rot_word(x1, x2, ct[it], st[it], ct[it + hh], st[it + hh], o1, o2);
            orow[it] = (uint16_t)o1;
            orow[it + hh] = (uint16_t)o2;
        } else {
            const int64_t c = p.rot + (it - hh);
            orow[c] = xr[c];
        }
    }
}

bool aligned(const void* p, int bytes) { return ((uintptr_t)p % bytes) == 0; }

// Largest vector width VW in {8, 4, 2} that every offset and pointer allows.
int pick_vw(const RopeParams& p) {
    for (int vw = 8; vw >= 2; vw >>= 1) {
        const int64_t hh = p.rot / 2;
        if (hh % vw || p.D % vw) continue;
        if (p.sx_b % vw || p.sx_s % vw || p.sx_h % vw) continue;
        if (p.so_b % vw || p.so_s % vw || p.so_h % vw) continue;
        const int bytes = 2 * vw;
        if (!aligned(p.x, bytes) || !aligned(p.out, bytes) || !aligned(p.cos, bytes) ||
            !aligned(p.sin, bytes))
            continue;
        return vw;
    }
    return 1;
}

template <int VW>
cudaError_t launch_fast(const FastArgs& a, cudaStream_t st) {
    const int threads = 256;
    const int64_t ntok = a.p.B * a.p.S;
    int64_t blocks = (ntok + (threads / 32) - 1) / (threads / 32);
    if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
    return launch_pdl(rope_fast_kernel<VW, 4>, dim3((unsigned)blocks), dim3(threads), 0, st, a);
}

}  // namespace

cudaError_t launch_rope_rotate_half(const RopeParams& p, cudaStream_t st) {
    const int vw = pick_vw(p);
    if (vw >= 2) {
        FastArgs a;
        a.p = p;
        a.NP = (int)(p.rot / 2 / vw);
        const int nt = p.in_place ? 0 : (int)((p.D - p.rot) / vw);
        a.NI = a.NP + nt;
        if (a.NI <= 32) {
            a.RPW = 32 / a.NI;
            switch (vw) {
                case 8: return launch_fast<8>(a, st);
                case 4: return launch_fast<4>(a, st);
                default: return launch_fast<2>(a, st);
            }
        }
    }
    const int64_t items = p.rot / 2 + (p.in_place ? 0 : p.D - p.rot);
    const int64_t total = p.B * p.S * p.H * items;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(rope_generic_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, p,
                      items);
}

}  // namespace dtrot
