// Rotate-half RoPE on q and k of one attention layer in a single launch, in
// place or into separate outputs, with the cos/sin rows either read from the
// (B*S, rot_dim) tables or computed on the fly from the rotary angles.
//
// ERNIE-Image fusion page (sglang PR #34306 analysis): section 2 gives the
// per-op bf16 rounding of the rotation, round(round(x1*cos1) + round(-x2*sin1)),
// applied to q and to k of every layer; section 1 hoists the cos/sin
// computation out of the per-projection path.  This kernel goes one step
// further on both counts: q and k (for example the q and k head ranges of one
// fused QKV buffer) are rotated by one launch, so a token's cos/sin row is
// fetched once for both; and with angles given instead of tables the row is
// evaluated per token inside the kernel (cos_sin_entry, the same evaluation as
// the table kernel, hence the same bits) and never written to HBM.
//
// Fast path (hh = rot_dim / 2 and every stride and pointer a multiple of the
// vector width VW, at most 32 pair and tail items per head row, and
// rot_dim <= kMaxRot with angles):
//   - one warp per token (b, s); lanes own NP = hh / VW pair items (columns
//     j..j+VW and j+hh..j+hh+VW) and walk the q rows and then the k rows,
//     RPW = 32 / NP rows per pass, U rows per batch with all loads of a batch
//     issued before any of its stores; the first batch is loaded before the
//     token's cos/sin row is fetched or evaluated;
//   - with angles, the warp first evaluates the token's rot_dim (cos, sin)
//     pairs into its slot of shared memory: each lane loads the angles of its
//     first-half columns and of their second-half partners, then evaluates
//     them (a partner's entry copied when its angle has the same bits); the
//     lanes then read their vectors from there, and the same registers serve
//     every q and k head of the token;
//   - tail columns [rot_dim, D) are not touched in place (they already hold
//     x); out of place, NT = (D - rot_dim) / VW more items per head row copy
//     them, so a lane's item is a pair (it < NP) or a tail vector, and NP + NT
//     items share the warp's 32 lanes.
// Generic path: one thread per (token, head row of q or k, item), items being
// the pair indices and, out of place, the tail columns.
#include "dtrot_internal.cuh"

namespace dtrot {
namespace {

constexpr int kMaxRot = 256;  // angle-mode fast path: rot_dim <= kMaxRot
constexpr int kAngIt = kMaxRot / 64;  // first-half angle columns per lane (32 lanes)
constexpr int kWarps = 8;     // warps per CTA of the fast kernel

template <int VW>
struct QKVec;
template <>
struct QKVec<8> { using T = uint4; };
template <>
struct QKVec<4> { using T = uint2; };
template <>
struct QKVec<2> { using T = uint32_t; };

template <int VW>
__device__ __forceinline__ typename QKVec<VW>::T qk_ld(const uint16_t* p) {
    return *reinterpret_cast<const typename QKVec<VW>::T*>(p);
}
template <int VW>
__device__ __forceinline__ void qk_st(uint16_t* p, typename QKVec<VW>::T v) {
    *reinterpret_cast<typename QKVec<VW>::T*>(p) = v;
}

// o1 = R(R(x1 c1) + R(-x2 s1)), o2 = R(R(x2 c2) + R(x1 s2)) on packed words
__device__ __forceinline__ void qk_rot_word(uint32_t x1, uint32_t x2, uint32_t c1, uint32_t s1,
                                            uint32_t c2, uint32_t s2, uint32_t& o1,
                                            uint32_t& o2) {
    o1 = bsub2(bmul2(x1, c1), bmul2(x2, s1));
    o2 = badd2(bmul2(x2, c2), bmul2(x1, s2));
}
__device__ __forceinline__ void qk_rot(uint4 a, uint4 b, uint4 c1, uint4 s1, uint4 c2, uint4 s2,
                                       uint4& o1, uint4& o2) {
    qk_rot_word(a.x, b.x, c1.x, s1.x, c2.x, s2.x, o1.x, o2.x);
    qk_rot_word(a.y, b.y, c1.y, s1.y, c2.y, s2.y, o1.y, o2.y);
    qk_rot_word(a.z, b.z, c1.z, s1.z, c2.z, s2.z, o1.z, o2.z);
    qk_rot_word(a.w, b.w, c1.w, s1.w, c2.w, s2.w, o1.w, o2.w);
}
__device__ __forceinline__ void qk_rot(uint2 a, uint2 b, uint2 c1, uint2 s1, uint2 c2, uint2 s2,
                                       uint2& o1, uint2& o2) {
    qk_rot_word(a.x, b.x, c1.x, s1.x, c2.x, s2.x, o1.x, o2.x);
    qk_rot_word(a.y, b.y, c1.y, s1.y, c2.y, s2.y, o1.y, o2.y);
}
__device__ __forceinline__ void qk_rot(uint32_t a, uint32_t b, uint32_t c1, uint32_t s1,
                                       uint32_t c2, uint32_t s2, uint32_t& o1, uint32_t& o2) {
    qk_rot_word(a, b, c1, s1, c2, s2, o1, o2);
}

struct QKArgs {
    RopeQKParams p;
    int NP;   // pair items per head row
    int NI;   // items per head row: the NP pairs, then the tail items
    int RPW;  // head rows per warp pass
};

// TAIL: out of place with tail columns, so some lanes copy instead of rotate.
template <int VW, int U, bool ANGLES, bool TAIL>
__global__ void __launch_bounds__(kWarps * 32) rope_qk_kernel(QKArgs a) {
    using V = typename QKVec<VW>::T;
    __shared__ __align__(16) uint16_t cs[kWarps][2][kMaxRot];  // angle mode: cos, sin row
    pdl_wait();
    const RopeQKParams& p = a.p;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int ri = lane / a.NI;
    const int it = lane - ri * a.NI;
    const bool active = ri < a.RPW;  // 32 may not be a multiple of NI
    const bool pair = !TAIL || it < a.NP;
    const int64_t ntok = p.B * p.S;
    const int64_t warps = (int64_t)gridDim.x * kWarps;
    const int64_t hh = p.rot >> 1;
    const int64_t j = pair ? (int64_t)it * VW : p.rot + (int64_t)(it - a.NP) * VW;
    const int64_t rows = p.Hq + p.Hk;  // q rows, then k rows
    const int64_t step = (int64_t)U * a.RPW;
    for (int64_t tok = (int64_t)blockIdx.x * kWarps + w; tok < ntok; tok += warps) {
        const int64_t b = tok / p.S;
        const int64_t s = tok - b * p.S;
        const uint16_t* qb = p.q + b * p.sq_b + s * p.sq_s + j;
        const uint16_t* kb = p.k + b * p.sk_b + s * p.sk_s + j;
        uint16_t* qob = p.qo + b * p.sqo_b + s * p.sqo_s + j;
        uint16_t* kob = p.ko + b * p.sko_b + s * p.sko_s + j;
        auto in_row = [&](int64_t r) {
            return r < p.Hq ? qb + r * p.sq_h : kb + (r - p.Hq) * p.sk_h;
        };
        auto out_row = [&](int64_t r) {
            return r < p.Hq ? qob + r * p.sqo_h : kob + (r - p.Hq) * p.sko_h;
        };
        // the first batch of head rows is loaded before the cos/sin row is
        // fetched or evaluated, so its memory latency overlaps that work
        V xa[U], xb[U];
        auto load_batch = [&](int64_t r0) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t r = r0 + (int64_t)u * a.RPW;
                if (active && r < rows) {
                    const uint16_t* ptr = in_row(r);
                    xa[u] = qk_ld<VW>(ptr);
                    if (pair) xb[u] = qk_ld<VW>(ptr + hh);
                }
            }
        };
        load_batch(ri);
        V c1{}, c2{}, s1{}, s2{};
        if constexpr (ANGLES) {
            // column c of the first half and its partner c + hh: a partner
            // angle with the same bits has the same entry, which is copied
            // (per-axis rotate-half angles repeat their half-row); any other
            // is evaluated
            // a lane's angles (at most kAngIt columns and their partners) are
            // all loaded before any is evaluated, so it waits for memory once
            const float* fr = p.freqs + (s * p.B + b) * p.rot;
            float a1[kAngIt], a2[kAngIt];
#pragma unroll
            for (int i = 0; i < kAngIt; ++i) {
                const int64_t c = lane + 32 * i;
                if (c < hh) {
                    a1[i] = __ldg(fr + c);
                    a2[i] = __ldg(fr + c + hh);
                }
            }
#pragma unroll
            for (int i = 0; i < kAngIt; ++i) {
                const int64_t c = lane + 32 * i;
                if (c < hh) {
                    uint16_t cv, sv;
                    cos_sin_entry(a1[i], cv, sv);
                    cs[w][0][c] = cv;
                    cs[w][1][c] = sv;
                    if (__float_as_uint(a2[i]) != __float_as_uint(a1[i])) {
                        const uint32_t e = cos_sin_entry_call(a2[i]);
                        cv = (uint16_t)e;
                        sv = (uint16_t)(e >> 16);
                    }
                    cs[w][0][c + hh] = cv;
                    cs[w][1][c + hh] = sv;
                }
            }
            __syncwarp();
            if (active && pair) {
                c1 = qk_ld<VW>(&cs[w][0][j]);
                c2 = qk_ld<VW>(&cs[w][0][j + hh]);
                s1 = qk_ld<VW>(&cs[w][1][j]);
                s2 = qk_ld<VW>(&cs[w][1][j + hh]);
            }
            __syncwarp();  // every lane has its row before the next token overwrites it
        } else {
            if (active && pair) {
                const uint16_t* ct = p.cos + tok * p.rot + j;
                const uint16_t* st = p.sin + tok * p.rot + j;
                c1 = qk_ld<VW>(ct);
                c2 = qk_ld<VW>(ct + hh);
                s1 = qk_ld<VW>(st);
                s2 = qk_ld<VW>(st + hh);
            }
        }
        if (!active) continue;
        for (int64_t r0 = ri;;) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t r = r0 + (int64_t)u * a.RPW;
                if (r < rows) {
                    uint16_t* ptr = out_row(r);
                    if (pair) {
                        V o1, o2;
                        qk_rot(xa[u], xb[u], c1, s1, c2, s2, o1, o2);
                        qk_st<VW>(ptr, o1);
                        qk_st<VW>(ptr + hh, o2);
                    } else {
                        qk_st<VW>(ptr, xa[u]);
                    }
                }
            }
            r0 += step;
            if (r0 >= rows) break;
            load_batch(r0);
        }
    }
}

// Generic path: one thread per (token, head row, item); head rows [0, Hq) are
// q's, [Hq, Hq + Hk) k's; item i < hh is the pair (i, i + hh), item i >= hh
// (out of place only) copies tail column rot + (i - hh).
template <bool ANGLES>
__global__ void __launch_bounds__(256) rope_qk_generic_kernel(RopeQKParams p) {
    pdl_wait();
    const int64_t hh = p.rot >> 1;
    const int64_t rows = p.Hq + p.Hk;
    const int64_t items = hh + (p.copy_tail ? p.D - p.rot : 0);
    const int64_t per_tok = rows * items;
    const int64_t total = p.B * p.S * per_tok;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < total;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tok = g / per_tok;
        const int64_t rem = g - tok * per_tok;
        const int64_t r = rem / items;
        const int64_t i = rem - r * items;
        const int64_t b = tok / p.S;
        const int64_t s = tok - b * p.S;
        const uint16_t* row = r < p.Hq ? p.q + b * p.sq_b + s * p.sq_s + r * p.sq_h
                                       : p.k + b * p.sk_b + s * p.sk_s + (r - p.Hq) * p.sk_h;
        uint16_t* orow = r < p.Hq ? p.qo + b * p.sqo_b + s * p.sqo_s + r * p.sqo_h
                                  : p.ko + b * p.sko_b + s * p.sko_s + (r - p.Hq) * p.sko_h;
        if (i >= hh) {
            const int64_t c = p.rot + (i - hh);
            orow[c] = row[c];
            continue;
        }
        uint32_t c1, c2, s1, s2;
        if constexpr (ANGLES) {
            const float* fr = p.freqs + (s * p.B + b) * p.rot;
            uint16_t a0, b0, a1, b1;
            cos_sin_entry(__ldg(fr + i), a0, b0);
            cos_sin_entry(__ldg(fr + i + hh), a1, b1);
            c1 = a0, s1 = b0, c2 = a1, s2 = b1;
        } else {
            c1 = p.cos[tok * p.rot + i];
            c2 = p.cos[tok * p.rot + i + hh];
            s1 = p.sin[tok * p.rot + i];
            s2 = p.sin[tok * p.rot + i + hh];
        }
        uint32_t o1, o2;
        qk_rot_word(row[i], row[i + hh], c1, s1, c2, s2, o1, o2);
        orow[i] = (uint16_t)o1;
        orow[i + hh] = (uint16_t)o2;
    }
}

bool aligned(const void* ptr, int bytes) { return ((uintptr_t)ptr % bytes) == 0; }

// Every pointer and stride of the q side (and of the k side) a multiple of vw
// elements, for a tensor whose head count is n.
bool vec_ok(int vw, int64_t n, const void* ptr, int64_t sb, int64_t ss, int64_t sh) {
    return n == 0 || (sb % vw == 0 && ss % vw == 0 && sh % vw == 0 && aligned(ptr, 2 * vw));
}

int pick_qk_vw(const RopeQKParams& p) {
    const int64_t hh = p.rot / 2;
    for (int vw = 8; vw >= 2; vw >>= 1) {
        if (hh % vw || (p.copy_tail && p.D % vw)) continue;
        if (!vec_ok(vw, p.Hq, p.q, p.sq_b, p.sq_s, p.sq_h) ||
            !vec_ok(vw, p.Hq, p.qo, p.sqo_b, p.sqo_s, p.sqo_h) ||
            !vec_ok(vw, p.Hk, p.k, p.sk_b, p.sk_s, p.sk_h) ||
            !vec_ok(vw, p.Hk, p.ko, p.sko_b, p.sko_s, p.sko_h))
            continue;
        if (!p.freqs && (!aligned(p.cos, 2 * vw) || !aligned(p.sin, 2 * vw))) continue;
        return vw;
    }
    return 1;
}

template <int VW, bool ANGLES, bool TAIL>
cudaError_t launch_qk_fast(const QKArgs& a, cudaStream_t st) {
    const int64_t ntok = a.p.B * a.p.S;
    int64_t blocks = (ntok + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
    return launch_pdl(rope_qk_kernel<VW, 4, ANGLES, TAIL>, dim3((unsigned)blocks),
                      dim3(kWarps * 32), 0, st, a);
}

template <int VW, bool ANGLES>
cudaError_t launch_qk_fast(const QKArgs& a, cudaStream_t st) {
    return a.NI > a.NP ? launch_qk_fast<VW, ANGLES, true>(a, st)
                       : launch_qk_fast<VW, ANGLES, false>(a, st);
}

template <bool ANGLES>
cudaError_t launch_qk(const RopeQKParams& p, cudaStream_t st) {
    const int vw = pick_qk_vw(p);
    const int64_t hh = p.rot / 2;
    if (vw >= 2 && (!ANGLES || p.rot <= kMaxRot)) {
        QKArgs a;
        a.p = p;
        a.NP = (int)(hh / vw);
        const int64_t ni = hh / vw + (p.copy_tail ? (p.D - p.rot) / vw : 0);
        if (ni <= 32) {
            a.NI = (int)ni;
            a.RPW = 32 / a.NI;
            switch (vw) {
                case 8: return launch_qk_fast<8, ANGLES>(a, st);
                case 4: return launch_qk_fast<4, ANGLES>(a, st);
                default: return launch_qk_fast<2, ANGLES>(a, st);
            }
        }
    }
    const int64_t total =
        p.B * p.S * (p.Hq + p.Hk) * (hh + (p.copy_tail ? p.D - p.rot : 0));
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(rope_qk_generic_kernel<ANGLES>, dim3((unsigned)blocks), dim3(256), 0, st, p);
}

}  // namespace

cudaError_t launch_rope_qk(const RopeQKParams& p, cudaStream_t st) {
    return p.freqs ? launch_qk<true>(p, st) : launch_qk<false>(p, st);
}

}  // namespace dtrot
