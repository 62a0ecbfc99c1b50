// extern "C" entry points of libdtrot: host-side argument validation, then one
// kernel launch on the caller's stream.  The declarations, with the meaning,
// layout, ownership and error behaviour of every argument, are in dtrot.h.
#include <cuda.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/dtrot.h"
#include "dtrot_internal.cuh"

#define DTROT_API extern "C" __attribute__((visibility("default")))

namespace dtrot {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_arch_ok[kMaxDevices];  // 0 unknown, 1 ok, 2 wrong arch

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}

bool device_ok() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return false;
    int st = g_arch_ok[dev].load(std::memory_order_relaxed);
    if (st == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        g_sms[dev].store(sms, std::memory_order_relaxed);
        st = (major == 10 && minor == 3) ? 1 : 2;
        g_arch_ok[dev].store(st, std::memory_order_relaxed);
    }
    return st == 1;
}

// ---- shape / stride / overlap helpers (element counts, int64) ----

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }

// Byte range [lo, hi) touched by a strided view with positive strides.
struct Range {
    uintptr_t lo, hi;
};

bool span(const void* base, int elem, const int64_t* size, const int64_t* stride, int n,
          Range* r) {
    int64_t last = 0;
    for (int i = 0; i < n; ++i) {
        int64_t t;
        if (!mul_ok(size[i] - 1, stride[i], &t)) return false;
        if (__builtin_add_overflow(last, t, &last)) return false;
    }
    int64_t bytes;
    if (!mul_ok(last + 1, elem, &bytes)) return false;
    r->lo = (uintptr_t)base;
    r->hi = r->lo + (uintptr_t)bytes;
    return true;
}

bool overlap(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }

// True if no two distinct index tuples of the view share an element.
bool non_self_overlapping(const int64_t* size, const int64_t* stride, int n) {
    constexpr int kMaxDims = 8;
    if (n < 0 || n > kMaxDims) return false;
    int idx[kMaxDims];
    int m = 0;
    for (int i = 0; i < n; ++i)
        if (size[i] > 1) idx[m++] = i;
    for (int k = 1; k < m; ++k) {  // insertion sort by stride (m <= 8)
        const int v = idx[k];
        int j = k;
        for (; j > 0 && stride[idx[j - 1]] > stride[v]; --j) idx[j] = idx[j - 1];
        idx[j] = v;
    }
    int64_t extent = 0;  // elements spanned by the dims already placed, minus one
    for (int k = 0; k < m; ++k) {
        const int i = idx[k];
        if (stride[i] <= extent) return false;
        int64_t t;
        if (!mul_ok(size[i] - 1, stride[i], &t)) return false;
        extent += t;
    }
    return true;
}

// Two (rows, cols) views with row strides sa, sb: element-disjoint?
bool views2d_disjoint(const uint16_t* a, int64_t sa, const uint16_t* b, int64_t sb,
                      int64_t rows, int64_t cols) {
    int64_t sz[2] = {rows, cols};
    int64_t st_a[2] = {sa, 1}, st_b[2] = {sb, 1};
    Range ra, rb;
    if (!span(a, 2, sz, st_a, 2, &ra) || !span(b, 2, sz, st_b, 2, &rb)) return false;
    if (!overlap(ra, rb)) return true;
    if (sa != sb || rows == 1) return false;
    const intptr_t dbytes = (intptr_t)((uintptr_t)b - (uintptr_t)a);
    if (dbytes % 2) return false;
    const int64_t d = (int64_t)(dbytes / 2);
    const int64_t m = ((d % sa) + sa) % sa;
    return m >= cols && m <= sa - cols;
}

// A single row [w, w + cols) against a (rows, cols) view with row stride sv.
// Disjoint if the byte ranges are, or if w's offset from the view, taken
// modulo sv, falls in a gap between rows (checked on w repeated every sv).
bool row_disjoint(const uint16_t* w, int64_t cols, const uint16_t* v, int64_t sv,
                  int64_t rows) {
    int64_t sz[2] = {rows, cols}, st[2] = {sv, 1};
    Range rv;
    if (!span(v, 2, sz, st, 2, &rv)) return false;
    const Range rw{(uintptr_t)w, (uintptr_t)w + (uintptr_t)cols * 2};
    if (!overlap(rw, rv)) return true;
    return views2d_disjoint(v, sv, w, sv, rows, cols);
}

// A byte range [p, p + bytes) against a (rows, cols) bf16 view with row
// stride sv: disjoint if the byte ranges are, or if the range lies wholly in
// the gap after one row (element-aligned offsets only; otherwise reported as
// overlapping).
bool range_disjoint(const void* p, int64_t bytes, const uint16_t* v, int64_t sv, int64_t rows,
                    int64_t cols) {
    int64_t sz[2] = {rows, cols}, st[2] = {sv, 1};
    Range rv;
    if (!span(v, 2, sz, st, 2, &rv)) return false;
    const Range rp{(uintptr_t)p, (uintptr_t)p + (uintptr_t)bytes};
    if (!overlap(rp, rv)) return true;
    if (rows == 1 || sv <= cols) return false;
    const intptr_t dbytes = (intptr_t)((uintptr_t)p - (uintptr_t)v);
    if (dbytes < 0 || dbytes % 2 || bytes % 2) return false;
    const int64_t d = (int64_t)(dbytes / 2), len = bytes / 2;
    const int64_t t0 = d / sv;
    return d - t0 * sv >= cols && d + len <= (t0 + 1) * sv;
}

dtrot_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return DTROT_OK;
    return DTROT_ERR_LAUNCH;
}

}  // namespace

uint64_t current_context_id() {
    // cuCtxGetCurrent / cuCtxGetId through the runtime's driver entry points
    // (no link-time dependency on libcuda)
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static std::atomic<GetCurrent> s_cur{nullptr};
    static std::atomic<GetId> s_id{nullptr};
    static std::atomic<int> s_missing{0};
    if (s_missing.load(std::memory_order_relaxed)) return 0;
    GetCurrent cur = s_cur.load(std::memory_order_acquire);
    GetId gid = s_id.load(std::memory_order_acquire);
    if (!cur || !gid) {
        void* p1 = nullptr;
        void* p2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p1, 12000, cudaEnableDefault,
                                             &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || !p1 ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &p2, 12000, cudaEnableDefault, &q2) !=
                cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess || !p2) {
            s_missing.store(1, std::memory_order_relaxed);
            return 0;
        }
        cur = reinterpret_cast<GetCurrent>(p1);
        gid = reinterpret_cast<GetId>(p2);
        s_cur.store(cur, std::memory_order_release);
        s_id.store(gid, std::memory_order_release);
    }
    CUcontext ctx = nullptr;
    if (cur(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (gid(ctx, &id) != CUDA_SUCCESS) return 0;
    return (uint64_t)id;
}

int num_sms() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 148;
    int s = g_sms[dev].load(std::memory_order_relaxed);
    if (s <= 0) {
        if (cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            s = 148;
        }
        g_sms[dev].store(s, std::memory_order_relaxed);
    }
    return s;
}

}  // namespace dtrot

using namespace dtrot;

DTROT_API const char* dtrot_status_str(dtrot_status s) {
    switch (s) {
        case DTROT_OK: return "DTROT_OK";
        case DTROT_ERR_NULL: return "DTROT_ERR_NULL: a required pointer is NULL";
        case DTROT_ERR_SHAPE: return "DTROT_ERR_SHAPE: a size is negative or too large";
        case DTROT_ERR_ROTDIM: return "DTROT_ERR_ROTDIM: rot_dim must be even, > 0 and <= D";
        case DTROT_ERR_STRIDE: return "DTROT_ERR_STRIDE: a stride is invalid";
        case DTROT_ERR_ALIAS: return "DTROT_ERR_ALIAS: an output overlaps an input";
        case DTROT_ERR_LAUNCH: return "DTROT_ERR_LAUNCH: the CUDA launch failed";
        case DTROT_ERR_DEVICE: return "DTROT_ERR_DEVICE: no sm_103 CUDA device is current";
        case DTROT_ERR_VALUE: return "DTROT_ERR_VALUE: a scalar argument is out of range";
        case DTROT_ERR_WORKSPACE:
            return "DTROT_ERR_WORKSPACE: the workspace is too small or not 16-byte aligned";
        case DTROT_ERR_ALIGN:
            return "DTROT_ERR_ALIGN: a pointer, stride or size misses the op's alignment";
    }
    return "DTROT_ERR_UNKNOWN";
}

DTROT_API int dtrot_version(void) { return 200; }  // 0.2.0

DTROT_API int64_t dtrot_gelu_and_mul_workspace_bytes(void) {
    return (int64_t)gelu_table_bytes();
}

DTROT_API dtrot_status dtrot_rope_cos_sin_precompute(const float* freqs, int64_t S, int64_t B,
                                                     int64_t R, uint16_t* cos_out,
                                                     uint16_t* sin_out, void* stream) {
    if (S < 0 || B < 0 || R < 0) return DTROT_ERR_SHAPE;
    int64_t n, n2;
    if (!mul_ok(S, B, &n) || !mul_ok(n, R, &n) || !mul_ok(n, 8, &n2)) return DTROT_ERR_SHAPE;
    if (n == 0) return DTROT_OK;
    if (!freqs || !cos_out || !sin_out) return DTROT_ERR_NULL;
    const Range rf{(uintptr_t)freqs, (uintptr_t)freqs + (uintptr_t)n * 4};
    const Range rc{(uintptr_t)cos_out, (uintptr_t)cos_out + (uintptr_t)n * 2};
    const Range rs{(uintptr_t)sin_out, (uintptr_t)sin_out + (uintptr_t)n * 2};
    if (overlap(rc, rs) || overlap(rc, rf) || overlap(rs, rf)) return DTROT_ERR_ALIAS;
    if (!device_ok()) return DTROT_ERR_DEVICE;
    return launch_status(
        launch_rope_cos_sin(freqs, S, B, R, cos_out, sin_out, (cudaStream_t)stream));
}

DTROT_API dtrot_status dtrot_rope_rotate_half(const uint16_t* x, int64_t B, int64_t S,
                                              int64_t H, int64_t D, int64_t sx_b,
                                              int64_t sx_s, int64_t sx_h, const uint16_t* cos,
                                              const uint16_t* sin, int64_t rot_dim,
                                              uint16_t* out, int64_t so_b, int64_t so_s,
                                              int64_t so_h, void* stream) {
    if (B < 0 || S < 0 || H < 0 || D < 0) return DTROT_ERR_SHAPE;
    int64_t ntok, n;
    if (!mul_ok(B, S, &ntok) || !mul_ok(ntok, H, &n) || !mul_ok(n, D, &n) ||
        !mul_ok(n, 16, &n))
        return DTROT_ERR_SHAPE;
    if (n == 0) return DTROT_OK;
    if (!x || !cos || !sin || !out) return DTROT_ERR_NULL;
    if (rot_dim <= 0 || rot_dim % 2 || rot_dim > D) return DTROT_ERR_ROTDIM;
    int64_t tab;
    if (!mul_ok(ntok, rot_dim, &tab)) return DTROT_ERR_SHAPE;
    const int64_t size[4] = {B, S, H, D};
    const int64_t sxs[4] = {sx_b, sx_s, sx_h, 1};
    const int64_t sos[4] = {so_b, so_s, so_h, 1};
    for (int i = 0; i < 3; ++i)
        if ((size[i] > 1 && (sxs[i] <= 0 || sos[i] <= 0)) || sxs[i] < 0 || sos[i] < 0)
            return DTROT_ERR_STRIDE;
    if (!non_self_overlapping(size, sos, 4)) return DTROT_ERR_STRIDE;
    Range rx, ro;
    if (!span(x, 2, size, sxs, 4, &rx) || !span(out, 2, size, sos, 4, &ro)) return DTROT_ERR_SHAPE;
    const Range rc{(uintptr_t)cos, (uintptr_t)cos + (uintptr_t)tab * 2};
    const Range rs{(uintptr_t)sin, (uintptr_t)sin + (uintptr_t)tab * 2};
    bool in_place = false;
    if (overlap(rx, ro)) {
        bool same = (x == out);
        for (int i = 0; i < 3; ++i)
            if (size[i] > 1 && sxs[i] != sos[i]) same = false;
        if (!same) return DTROT_ERR_ALIAS;
        in_place = true;
    }
    if (overlap(ro, rc) || overlap(ro, rs)) return DTROT_ERR_ALIAS;
    if (!device_ok()) return DTROT_ERR_DEVICE;
    RopeParams p;
    p.x = x;
    p.out = out;
    p.cos = cos;
    p.sin = sin;
    p.B = B;
    p.S = S;
    p.H = H;
    p.D = D;
    p.rot = rot_dim;
    p.sx_b = sx_b;
    p.sx_s = sx_s;
    p.sx_h = sx_h;
    p.so_b = so_b;
    p.so_s = so_s;
    p.so_h = so_h;
    p.in_place = in_place ? 1 : 0;
    return launch_status(launch_rope_rotate_half(p, (cudaStream_t)stream));
}

// The q and k views of a fused q+k RoPE call, (B, S, Hq, D) and (B, S, Hk, D)
// with element strides qst, kst (the D stride 1): strides valid, and for the
// views written (`written`) rows that do not overlap and no element shared
// between q and k, whose byte ranges are then disjoint or the two head ranges
// of one (B, S, Hq + Hk, D) view, in either order (the q and k parts of a
// fused QKV buffer).  Fills the byte spans rq, rk (empty for no heads).
static dtrot_status qk_views(const uint16_t* q, int64_t Hq, const int64_t* qst,
                             const uint16_t* k, int64_t Hk, const int64_t* kst, int64_t B,
                             int64_t S, int64_t D, bool written, Range* rq, Range* rk) {
    const int64_t qsz[4] = {B, S, Hq, D}, ksz[4] = {B, S, Hk, D};
    for (int i = 0; i < 3; ++i) {
        if (Hq > 0 && (qst[i] < 0 || (qsz[i] > 1 && qst[i] == 0))) return DTROT_ERR_STRIDE;
        if (Hk > 0 && (kst[i] < 0 || (ksz[i] > 1 && kst[i] == 0))) return DTROT_ERR_STRIDE;
    }
    if (written && ((Hq > 0 && !non_self_overlapping(qsz, qst, 4)) ||
                    (Hk > 0 && !non_self_overlapping(ksz, kst, 4))))
        return DTROT_ERR_STRIDE;
    *rq = Range{0, 0};
    *rk = Range{0, 0};
    if ((Hq > 0 && !span(q, 2, qsz, qst, 4, rq)) || (Hk > 0 && !span(k, 2, ksz, kst, 4, rk)))
        return DTROT_ERR_SHAPE;
    if (written && Hq > 0 && Hk > 0 && overlap(*rq, *rk)) {
        bool ok = qst[0] == kst[0] && qst[1] == kst[1] && qst[2] == kst[2];
        if (ok) {
            const uint16_t* first = q < k ? q : k;
            const uint16_t* second = q < k ? k : q;
            const int64_t h_first = q < k ? Hq : Hk;
            int64_t off;
            ok = mul_ok(h_first, qst[2], &off) && second == first + off;
            const int64_t usz[4] = {B, S, Hq + Hk, D};
            ok = ok && non_self_overlapping(usz, qst, 4);
        }
        if (!ok) return DTROT_ERR_ALIAS;
    }
    return DTROT_OK;
}

// A fused q+k RoPE call: q, k read (with their strides), qo, ko written
// (qo == q and ko == k with the same strides in place).
static dtrot_status rope_qk_call(const uint16_t* q, int64_t Hq, const int64_t* qst,
                                 const uint16_t* k, int64_t Hk, const int64_t* kst, int64_t B,
                                 int64_t S, int64_t D, const uint16_t* cos, const uint16_t* sin,
                                 const float* freqs, int64_t rot_dim, uint16_t* qo,
                                 const int64_t* qost, uint16_t* ko, const int64_t* kost,
                                 bool in_place, void* stream) {
    if (B < 0 || S < 0 || Hq < 0 || Hk < 0 || D < 0) return DTROT_ERR_SHAPE;
    int64_t ntok, rows, n;
    if (!mul_ok(B, S, &ntok) || __builtin_add_overflow(Hq, Hk, &rows) ||
        !mul_ok(ntok, rows, &n) || !mul_ok(n, D, &n) || !mul_ok(n, 16, &n))
        return DTROT_ERR_SHAPE;
    if (n == 0) return DTROT_OK;
    if ((Hq > 0 && (!q || !qo)) || (Hk > 0 && (!k || !ko))) return DTROT_ERR_NULL;
    if (freqs && (cos || sin)) return DTROT_ERR_VALUE;  // tables or angles, not both
    if (!freqs && (!cos || !sin)) return DTROT_ERR_NULL;
    if (rot_dim <= 0 || rot_dim % 2 || rot_dim > D) return DTROT_ERR_ROTDIM;
    int64_t tab;
    if (!mul_ok(ntok, rot_dim, &tab) || !mul_ok(tab, 4, &tab)) return DTROT_ERR_SHAPE;
    tab /= 4;
    Range rq, rk, rqo, rko;
    dtrot_status st = qk_views(q, Hq, qst, k, Hk, kst, B, S, D, in_place, &rq, &rk);
    if (st != DTROT_OK) return st;
    if (in_place) {
        rqo = rq;
        rko = rk;
    } else {
        st = qk_views(qo, Hq, qost, ko, Hk, kost, B, S, D, true, &rqo, &rko);
        if (st != DTROT_OK) return st;
    }
    // nothing read may overlap what is written (in place, q and k themselves)
    Range rin[4] = {{0, 0}, {0, 0}, {0, 0}, {0, 0}};
    if (freqs) {
        rin[0] = Range{(uintptr_t)freqs, (uintptr_t)freqs + (uintptr_t)tab * 4};
    } else {
        rin[0] = Range{(uintptr_t)cos, (uintptr_t)cos + (uintptr_t)tab * 2};
        rin[1] = Range{(uintptr_t)sin, (uintptr_t)sin + (uintptr_t)tab * 2};
    }
    if (!in_place) {
        rin[2] = rq;
        rin[3] = rk;
    }
    for (const Range* w : {&rqo, &rko})
        for (const Range& r : rin)
            if (w->hi > w->lo && r.hi > r.lo && overlap(*w, r)) return DTROT_ERR_ALIAS;
    if (!device_ok()) return DTROT_ERR_DEVICE;
    RopeQKParams p;
    p.q = q;
    p.k = k;
    p.qo = qo;
    p.ko = ko;
    p.cos = freqs ? nullptr : cos;
    p.sin = freqs ? nullptr : sin;
    p.freqs = freqs;
    p.B = B;
    p.S = S;
    p.Hq = Hq;
    p.Hk = Hk;
    p.D = D;
    p.rot = rot_dim;
    p.sq_b = qst[0];
    p.sq_s = qst[1];
    p.sq_h = qst[2];
    p.sk_b = kst[0];
    p.sk_s = kst[1];
    p.sk_h = kst[2];
    p.sqo_b = qost[0];
    p.sqo_s = qost[1];
    p.sqo_h = qost[2];
    p.sko_b = kost[0];
    p.sko_s = kost[1];
    p.sko_h = kost[2];
    p.copy_tail = in_place ? 0 : 1;
    return launch_status(launch_rope_qk(p, (cudaStream_t)stream));
}

DTROT_API dtrot_status dtrot_rope_rotate_half_qk(uint16_t* q, int64_t Hq, int64_t sq_b,
                                                 int64_t sq_s, int64_t sq_h, uint16_t* k,
                                                 int64_t Hk, int64_t sk_b, int64_t sk_s,
                                                 int64_t sk_h, int64_t B, int64_t S, int64_t D,
                                                 const uint16_t* cos, const uint16_t* sin,
                                                 const float* freqs, int64_t rot_dim,
                                                 void* stream) {
    const int64_t qst[4] = {sq_b, sq_s, sq_h, 1}, kst[4] = {sk_b, sk_s, sk_h, 1};
    return rope_qk_call(q, Hq, qst, k, Hk, kst, B, S, D, cos, sin, freqs, rot_dim, q, qst, k,
                        kst, true, stream);
}

DTROT_API dtrot_status dtrot_rope_rotate_half_qk_out(
    const uint16_t* q, int64_t Hq, int64_t sq_b, int64_t sq_s, int64_t sq_h, const uint16_t* k,
    int64_t Hk, int64_t sk_b, int64_t sk_s, int64_t sk_h, int64_t B, int64_t S, int64_t D,
    const uint16_t* cos, const uint16_t* sin, const float* freqs, int64_t rot_dim,
    uint16_t* q_out, int64_t soq_b, int64_t soq_s, int64_t soq_h, uint16_t* k_out,
    int64_t sok_b, int64_t sok_s, int64_t sok_h, void* stream) {
    const int64_t qst[4] = {sq_b, sq_s, sq_h, 1}, kst[4] = {sk_b, sk_s, sk_h, 1};
    const int64_t qost[4] = {soq_b, soq_s, soq_h, 1}, kost[4] = {sok_b, sok_s, sok_h, 1};
    return rope_qk_call(q, Hq, qst, k, Hk, kst, B, S, D, cos, sin, freqs, rot_dim, q_out, qost,
                        k_out, kost, false, stream);
}

// Strides, spans and overlaps of a GEGLU call's gate, up and out; fills p.
static dtrot_status geglu_views(const uint16_t* gate, int64_t s_gate, const uint16_t* up, int64_t s_up,
                         uint16_t* out, int64_t s_out, int64_t T, int64_t F, GegluParams* p) {
    if (T > 1 && (s_gate < F || s_up < F || s_out < F)) return DTROT_ERR_STRIDE;
    if (s_gate < 0 || s_up < 0 || s_out < 0) return DTROT_ERR_STRIDE;
    const int64_t sg = T > 1 ? s_gate : F, su = T > 1 ? s_up : F, so = T > 1 ? s_out : F;
    {
        int64_t size[2] = {T, F}, a[2] = {sg, 1}, b[2] = {su, 1}, c[2] = {so, 1};
        Range r;
        if (!span(gate, 2, size, a, 2, &r) || !span(up, 2, size, b, 2, &r) ||
            !span(out, 2, size, c, 2, &r))
            return DTROT_ERR_SHAPE;
    }
    const bool in_place = (out == gate) && (so == sg);
    if (!in_place && !views2d_disjoint(out, so, gate, sg, T, F)) return DTROT_ERR_ALIAS;
    if (!views2d_disjoint(out, so, up, su, T, F)) return DTROT_ERR_ALIAS;
    p->gate = gate;
    p->up = up;
    p->out = out;
    p->s_gate = sg;
    p->s_up = su;
    p->s_out = so;
    p->T = T;
    p->F = F;
    return DTROT_OK;
}

DTROT_API dtrot_status dtrot_gelu_and_mul(const uint16_t* gate, int64_t s_gate,
                                          const uint16_t* up, int64_t s_up, uint16_t* out,
                                          int64_t s_out, int64_t T, int64_t F, void* workspace,
                                          int64_t workspace_bytes, void* stream) {
    if (T < 0 || F < 0) return DTROT_ERR_SHAPE;
    int64_t n;
    if (!mul_ok(T, F, &n) || !mul_ok(n, 8, &n)) return DTROT_ERR_SHAPE;
    if (n == 0) return DTROT_OK;
    if (!gate || !up || !out || !workspace) return DTROT_ERR_NULL;
    if (workspace_bytes < (int64_t)gelu_table_bytes() || (uintptr_t)workspace % 16)
        return DTROT_ERR_WORKSPACE;
    GegluParams p;
    const dtrot_status v = geglu_views(gate, s_gate, up, s_up, out, s_out, T, F, &p);
    if (v != DTROT_OK) return v;
    {
        // the workspace is written: it must not overlap gate, up or out
        const int64_t wb = (int64_t)gelu_table_bytes();
        if (!range_disjoint(workspace, wb, gate, p.s_gate, T, F) ||
            !range_disjoint(workspace, wb, up, p.s_up, T, F) ||
            !range_disjoint(workspace, wb, out, p.s_out, T, F))
            return DTROT_ERR_ALIAS;
    }
    if (!device_ok()) return DTROT_ERR_DEVICE;
    return launch_status(launch_gelu_and_mul(p, (uint16_t*)workspace, (cudaStream_t)stream));
}

DTROT_API dtrot_status dtrot_gelu_table_build(void* table, int64_t table_bytes, void* stream) {
    if (!table) return DTROT_ERR_NULL;
    if (table_bytes < (int64_t)gelu_table_bytes() || (uintptr_t)table % 16)
        return DTROT_ERR_WORKSPACE;
    if (!device_ok()) return DTROT_ERR_DEVICE;
    return launch_status(launch_gelu_table((uint16_t*)table, (cudaStream_t)stream));
}

DTROT_API dtrot_status dtrot_gelu_and_mul_with_table(const uint16_t* gate, int64_t s_gate,
                                                     const uint16_t* up, int64_t s_up,
                                                     uint16_t* out, int64_t s_out, int64_t T,
                                                     int64_t F, const void* table,
                                                     int64_t table_bytes, void* stream) {
    if (T < 0 || F < 0) return DTROT_ERR_SHAPE;
    int64_t n;
    if (!mul_ok(T, F, &n) || !mul_ok(n, 8, &n)) return DTROT_ERR_SHAPE;
    if (n == 0) return DTROT_OK;
    if (!gate || !up || !out || !table) return DTROT_ERR_NULL;
    if (table_bytes < (int64_t)gelu_table_bytes() || (uintptr_t)table % 16)
        return DTROT_ERR_WORKSPACE;
    GegluParams p;
    const dtrot_status v = geglu_views(gate, s_gate, up, s_up, out, s_out, T, F, &p);
    if (v != DTROT_OK) return v;
    // the table is only read: it must not overlap out, which is written
    if (!range_disjoint(table, (int64_t)gelu_table_bytes(), out, p.s_out, T, F))
        return DTROT_ERR_ALIAS;
    if (!device_ok()) return DTROT_ERR_DEVICE;
    return launch_status(
        launch_gelu_stream(p, (const uint16_t*)table, (cudaStream_t)stream));
}

// GEGLU for callers that cannot allocate device memory: the same computation
// as dtrot_gelu_and_mul, with the activation table kept in the library's own
// static device array instead of a caller workspace.  Every argument is
// checked, in the order dtrot_gelu_and_mul checks them, before the device is
// queried or the array's address looked up, so the two entry points return
// the same status for the same invalid call.
DTROT_API dtrot_status dtrot_gelu_and_mul_noalloc(const uint16_t* gate, int64_t s_gate,
                                                  const uint16_t* up, int64_t s_up, uint16_t* out,
                                                  int64_t s_out, int64_t T, int64_t F,
                                                  void* stream) {
    if (T < 0 || F < 0) return DTROT_ERR_SHAPE;
    int64_t n;
    if (!mul_ok(T, F, &n) || !mul_ok(n, 8, &n)) return DTROT_ERR_SHAPE;
    if (n == 0) return DTROT_OK;
    if (!gate || !up || !out) return DTROT_ERR_NULL;
    GegluParams p;
    const dtrot_status v = geglu_views(gate, s_gate, up, s_up, out, s_out, T, F, &p);
    if (v != DTROT_OK) return v;
    if (!device_ok()) return DTROT_ERR_DEVICE;
    uint16_t* table = nullptr;
    size_t capacity = 0;
    const cudaError_t pending = cudaPeekAtLastError();
    if (noalloc_gelu_table(&table, &capacity) != cudaSuccess) {
        // clear the lookup's own error, but leave an error the caller already
        // had pending in place
        if (pending == cudaSuccess) cudaGetLastError();
        return DTROT_ERR_DEVICE;
    }
    // the table's size is fixed (it does not grow with T or F); a library
    // whose table outgrew the static array would refuse every call here
    if (gelu_table_bytes() > capacity) return DTROT_ERR_WORKSPACE;
    const int64_t wb = (int64_t)gelu_table_bytes();
    if (!range_disjoint(table, wb, gate, p.s_gate, T, F) ||
        !range_disjoint(table, wb, up, p.s_up, T, F) ||
        !range_disjoint(table, wb, out, p.s_out, T, F))
        return DTROT_ERR_ALIAS;
    return launch_status(launch_gelu_and_mul(p, table, (cudaStream_t)stream));
}

DTROT_API int64_t dtrot_gemm_gelu_and_mul_workspace_bytes(void) {
    return (int64_t)gemm_geglu_workspace_bytes();
}

// Validation and launch of the projection with GEGLU in its epilogue;
// `withhold` selects the diagnostic run whose last pipeline stage is withheld.
static dtrot_status gemm_call(const uint16_t* x, int64_t T, int64_t C, const uint16_t* w,
                              int64_t F, uint16_t* out, int64_t s_out, uint16_t* gate_up,
                              int64_t s_gate_up, void* workspace, int64_t workspace_bytes,
                              void* stream, int withhold) {
    if (T < 0 || C < 0 || F < 0) return DTROT_ERR_SHAPE;
    int64_t n, f2, nw;
    if (!mul_ok(T, C, &n) || !mul_ok(n, 2, &n) || !mul_ok(F, 2, &f2) || !mul_ok(f2, C, &nw) ||
        !mul_ok(nw, 2, &nw) || !mul_ok(T, F, &n) || !mul_ok(n, 2, &n))
        return DTROT_ERR_SHAPE;
    if (T == 0 || F == 0) return DTROT_OK;
    if (C == 0) return DTROT_ERR_SHAPE;  // no projection to take
    if (T > 0x7FFFFFFF || f2 > 0x7FFFFFFF) return DTROT_ERR_SHAPE;
    if (!x || !w || !out || !workspace) return DTROT_ERR_NULL;
    if (T > 1 && (s_out < F || (gate_up && s_gate_up < 2 * F))) return DTROT_ERR_STRIDE;
    const int64_t so = T > 1 ? s_out : F;
    const int64_t sg = T > 1 ? s_gate_up : 2 * F;
    if (C % 8 || F % 8 || so % 8 || (uintptr_t)x % 16 || (uintptr_t)w % 16 ||
        (uintptr_t)out % 16 || (gate_up && (sg % 8 || (uintptr_t)gate_up % 16)))
        return DTROT_ERR_ALIGN;
    if (workspace_bytes < (int64_t)gemm_geglu_workspace_bytes() || (uintptr_t)workspace % 16)
        return DTROT_ERR_WORKSPACE;
    {
        int64_t size[2] = {T, F}, st[2] = {so, 1};
        Range ro;
        if (!span(out, 2, size, st, 2, &ro)) return DTROT_ERR_SHAPE;
        const Range rx{(uintptr_t)x, (uintptr_t)x + (uintptr_t)(T * C * 2)};
        const Range rw{(uintptr_t)w, (uintptr_t)w + (uintptr_t)nw};
        const Range rws{(uintptr_t)workspace,
                        (uintptr_t)workspace + (uintptr_t)gemm_geglu_workspace_bytes()};
        if (overlap(ro, rx) || overlap(ro, rw) || overlap(ro, rws) || overlap(rws, rx) ||
            overlap(rws, rw))
            return DTROT_ERR_ALIAS;
        if (gate_up) {
            int64_t gsize[2] = {T, 2 * F}, gst[2] = {sg, 1};
            Range rg;
            if (!span(gate_up, 2, gsize, gst, 2, &rg)) return DTROT_ERR_SHAPE;
            if (overlap(rg, rx) || overlap(rg, rw) || overlap(rg, rws) || overlap(rg, ro))
                return DTROT_ERR_ALIAS;
        }
    }
    if (!device_ok()) return DTROT_ERR_DEVICE;
    GemmGegluArgs a;
    a.x = x;
    a.w = w;
    a.T = T;
    a.C = C;
    a.F = F;
    a.out = out;
    a.s_out = so;
    a.gate_up = gate_up;
    a.s_gate_up = sg;
    a.workspace = workspace;
    a.withhold_last_stage = withhold;
    return launch_status(launch_gemm_geglu(a, (cudaStream_t)stream));
}

DTROT_API dtrot_status dtrot_gemm_gelu_and_mul(const uint16_t* x, int64_t T, int64_t C,
                                               const uint16_t* w, int64_t F, uint16_t* out,
                                               int64_t s_out, uint16_t* gate_up,
                                               int64_t s_gate_up, void* workspace,
                                               int64_t workspace_bytes, void* stream) {
    return gemm_call(x, T, C, w, F, out, s_out, gate_up, s_gate_up, workspace, workspace_bytes,
                     stream, 0);
}

DTROT_API dtrot_status dtrot_gemm_gelu_and_mul_withhold_last_stage(
    const uint16_t* x, int64_t T, int64_t C, const uint16_t* w, int64_t F, uint16_t* out,
    int64_t s_out, uint16_t* gate_up, int64_t s_gate_up, void* workspace,
    int64_t workspace_bytes, void* stream) {
    return gemm_call(x, T, C, w, F, out, s_out, gate_up, s_gate_up, workspace, workspace_bytes,
                     stream, 1);
}

DTROT_API dtrot_status dtrot_gemm_gelu_and_mul_error(const void* workspace, uint32_t* host_word,
                                                     void* stream) {
    if (!workspace || !host_word) return DTROT_ERR_NULL;
    if ((uintptr_t)workspace % 16) return DTROT_ERR_WORKSPACE;
    if (!device_ok()) return DTROT_ERR_DEVICE;
    const uint8_t* src = static_cast<const uint8_t*>(workspace) + gemm_geglu_error_offset();
    return launch_status(cudaMemcpyAsync(host_word, src, sizeof(uint32_t),
                                         cudaMemcpyDeviceToHost, (cudaStream_t)stream));
}

DTROT_API dtrot_status dtrot_rmsnorm_residual(const uint16_t* x, int64_t sx, uint16_t* residual,
                                              int64_t sr, const uint16_t* w, float eps,
                                              uint16_t* out, int64_t so, int64_t T, int64_t C,
                                              void* stream) {
    if (T < 0 || C < 0) return DTROT_ERR_SHAPE;
    int64_t n;
    if (!mul_ok(T, C, &n) || !mul_ok(n, 8, &n)) return DTROT_ERR_SHAPE;
    if (n == 0) return DTROT_OK;
    if (!x || !residual || !w || !out) return DTROT_ERR_NULL;
    if (!(eps >= 0.0f) || !(eps <= 3.4028235e38f)) return DTROT_ERR_VALUE;
    if (T > 1 && (sx < C || sr < C || so < C)) return DTROT_ERR_STRIDE;
    if (sx < 0 || sr < 0 || so < 0) return DTROT_ERR_STRIDE;
    const int64_t ssx = T > 1 ? sx : C, ssr = T > 1 ? sr : C, sso = T > 1 ? so : C;
    {
        int64_t size[2] = {T, C}, a[2] = {ssx, 1}, b[2] = {ssr, 1}, c[2] = {sso, 1};
        Range r;
        if (!span(x, 2, size, a, 2, &r) || !span(residual, 2, size, b, 2, &r) ||
            !span(out, 2, size, c, 2, &r))
            return DTROT_ERR_SHAPE;
    }
    const bool x_is_res = (x == residual) && (ssx == ssr);
    if (!x_is_res && !views2d_disjoint(x, ssx, residual, ssr, T, C)) return DTROT_ERR_ALIAS;
    if (!views2d_disjoint(out, sso, x, ssx, T, C)) return DTROT_ERR_ALIAS;
    if (!views2d_disjoint(out, sso, residual, ssr, T, C)) return DTROT_ERR_ALIAS;
    if (!row_disjoint(w, C, residual, ssr, T) || !row_disjoint(w, C, out, sso, T))
        return DTROT_ERR_ALIAS;
    if (!device_ok()) return DTROT_ERR_DEVICE;
    RmsParams p;
    p.x = x;
    p.residual = residual;
    p.w = w;
    p.out = out;
    p.sx = ssx;
    p.sr = ssr;
    p.so = sso;
    p.T = T;
    p.C = C;
    p.eps = eps;
    return launch_status(launch_rmsnorm_residual(p, (cudaStream_t)stream));
}
