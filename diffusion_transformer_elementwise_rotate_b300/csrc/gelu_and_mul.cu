// GEGLU with the eager path's activation rounding:
//   out = RN16(up * RN16(RN32(gelu(gate)))),  gelu(x) = x/2 * (1 + erf(x/sqrt 2)).
//
// ERNIE-Image fusion page (sglang PR #34306 analysis), section 3: up *
// F.gelu(gate) made two full passes over the FFN intermediate; the fused op
// does one, reproducing the bf16 rounding of the GELU output.
//
// Design.  gate is bf16, so the rounded activation g(gate) takes one of 65536
// values.  A first kernel tabulates g for every bf16 bit pattern into a
// 128 KB workspace, one entry per thread over the whole GPU; it evaluates its
// entry before waiting for the kernel before it, and only the store waits.
// The streaming kernel is launched as its programmatic dependent: its
// persistent CTAs (one per SM) are scheduled as the table kernel's CTAs exit,
// wait for it in hardware (griddepcontrol.wait), copy the table into shared
// memory and stream gate/up with 128-bit loads: per element one shared-memory
// lookup and one bf16x2 multiply with .rn rounding.  The erf arithmetic (tens of fp32 instructions
// per element, enough to make a direct evaluation ALU-bound on this part) is
// paid 65536 times per call instead of once per element, and the result is
// the exactly rounded GELU.
//
// Table entries: gelu_entry (shared with the GEGLU epilogue of the gate_up
// projection).
#include <atomic>
#include <mutex>

#include "dtrot_internal.cuh"

namespace dtrot {
namespace {

constexpr int kTable = 1 << 16;
constexpr int kThreads = 1024;

__device__ __forceinline__ uint32_t lookup2(const uint16_t* tab, uint32_t g) {
    const uint32_t lo = tab[g & 0xFFFFu];
    const uint32_t hi = tab[g >> 16];
    return lo | (hi << 16);
}

__device__ __forceinline__ uint4 geglu_vec(const uint16_t* tab, uint4 g, uint4 u) {
    uint4 o;
    o.x = bmul2(u.x, lookup2(tab, g.x));
    o.y = bmul2(u.y, lookup2(tab, g.y));
    o.z = bmul2(u.z, lookup2(tab, g.z));
    o.w = bmul2(u.w, lookup2(tab, g.w));
    return o;
}


// One table entry per thread: table[i] = RN16(RN32(gelu(bf16 bits i))).  The
// entry depends on nothing in memory, so it is computed while the previous
// kernel in the stream may still be running; only the store waits for it (it
// may still read this workspace).
__global__ void __launch_bounds__(256) gelu_table_kernel(uint16_t* __restrict__ table) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const uint16_t v = i < kTable ? gelu_entry((uint32_t)i) : (uint16_t)0;
    pdl_wait();
    if (i < kTable) table[i] = v;
}

// Copies the table from the workspace into shared memory (16 bytes per load).
__device__ __forceinline__ void load_table(uint16_t* tab, const uint16_t* __restrict__ gtab) {
    pdl_wait();  // the table kernel (or whatever ran before) has completed
    const uint4* src = reinterpret_cast<const uint4*>(gtab);
    uint4* dst = reinterpret_cast<uint4*>(tab);
    for (int i = threadIdx.x; i < kTable / 8; i += blockDim.x) dst[i] = __ldcg(src + i);
    __syncthreads();
}

// Vector path: F % 8 == 0, strides % 8 == 0, pointers 16-byte aligned.
// Items are (row, 8-column vector) pairs, U per thread per iteration with all
// loads of an iteration issued before its stores (safe for out == gate).
template <int U>
__global__ void __launch_bounds__(kThreads, 1) geglu_vec_kernel(GegluParams p,
                                                                const uint16_t* __restrict__ gtab) {
    extern __shared__ uint16_t tab[];
    load_table(tab, gtab);
    const uint32_t nv = (uint32_t)(p.F >> 3);
    const int64_t items = p.T * (int64_t)nv;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i0 < items;
         i0 += stride * U) {
        uint4 g[U], u[U];
        int64_t row[U];
        uint32_t col[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * stride;
            if (i < items) {
                row[k] = i / nv;
                col[k] = (uint32_t)(i - row[k] * nv) << 3;
                g[k] = *reinterpret_cast<const uint4*>(p.gate + row[k] * p.s_gate + col[k]);
                u[k] = *reinterpret_cast<const uint4*>(p.up + row[k] * p.s_up + col[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * stride;
            if (i < items) {
                *reinterpret_cast<uint4*>(p.out + row[k] * p.s_out + col[k]) =
                    geglu_vec(tab, g[k], u[k]);
            }
        }
    }
}

// Scalar path for any alignment / width.
__global__ void __launch_bounds__(kThreads, 1) geglu_scalar_kernel(GegluParams p,
                                                                   const uint16_t* __restrict__ gtab) {
    extern __shared__ uint16_t tab[];
    load_table(tab, gtab);
    const int64_t items = p.T * p.F;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < items;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / p.F;
        const int64_t c = i - r * p.F;
        const uint32_t g = p.gate[r * p.s_gate + c];
        const uint32_t u = p.up[r * p.s_up + c];
        p.out[r * p.s_out + c] = (uint16_t)bmul2(u, tab[g]);
    }
}

bool aligned(const void* ptr, int bytes) { return ((uintptr_t)ptr % bytes) == 0; }

constexpr int kMaxDev = 64;
// context (current_context_id) for which the dynamic shared memory attribute
// was set, per device and kernel; 0: not yet
std::atomic<uint64_t> g_attr_ctx[kMaxDev][2];

// Activation table owned by the library, for callers that cannot hand in a
// workspace (dtrot_gelu_and_mul_noalloc).  One copy per device that loads the
// library, 128 KB, kept until the process exits.  Host code may not use this
// name as a device address: it is a host-side stand-in, and its device address
// comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint16_t g_noalloc_table[kTable];

// Its device address per device, with the context it was looked up in: a new
// context (cudaDeviceReset, then any CUDA call) loads the library's device
// code again, and the array may then sit at another address.
struct NoallocSlot {
    uint64_t ctx;
    uintptr_t addr;
};
std::mutex g_noalloc_mu;
NoallocSlot g_noalloc[kMaxDev];

}  // namespace

size_t gelu_table_bytes() { return kTable * sizeof(uint16_t); }

cudaError_t noalloc_gelu_table(uint16_t** table, size_t* capacity) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    const uint64_t ctx = current_context_id();
    NoallocSlot& slot = g_noalloc[dev];
    if (ctx == 0 || slot.ctx != ctx || slot.addr == 0) {
        // first use on this device in this context (the device is current):
        // look the address up; this also creates the context if none exists
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_table);
        if (e != cudaSuccess) return e;
        slot.addr = (uintptr_t)ptr;
        slot.ctx = current_context_id();
    }
    *table = reinterpret_cast<uint16_t*>(slot.addr);
    *capacity = sizeof(g_noalloc_table);
    return cudaSuccess;
}

cudaError_t launch_gelu_table(uint16_t* table, cudaStream_t st) {
    return launch_pdl(gelu_table_kernel, dim3(kTable / 256), dim3(256), 0, st, table);
}

cudaError_t launch_gelu_stream(const GegluParams& p, const uint16_t* table,
                               cudaStream_t st) {
    const size_t smem = kTable * sizeof(uint16_t);
    const bool vec = (p.F % 8 == 0) && (p.s_gate % 8 == 0) && (p.s_up % 8 == 0) &&
                     (p.s_out % 8 == 0) && aligned(p.gate, 16) && aligned(p.up, 16) &&
                     aligned(p.out, 16);
    const int sms = num_sms();
    // One CTA per SM (the table takes 128 KB of shared memory); fewer when the
    // tensor is small.
    const int64_t work = vec ? p.T * (p.F / 8) : p.T * p.F;
    int64_t blocks = (work + kThreads - 1) / kThreads;
    if (blocks > sms) blocks = sms;
    if (blocks < 1) blocks = 1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    const int which = vec ? 0 : 1;
    const uint64_t ctx = current_context_id();
    if (ctx == 0 || g_attr_ctx[dev][which].load(std::memory_order_acquire) != ctx) {
        e = vec ? cudaFuncSetAttribute(geglu_vec_kernel<4>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                : cudaFuncSetAttribute(geglu_scalar_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_ctx[dev][which].store(current_context_id(), std::memory_order_release);
    }
    // a programmatic dependent of the table kernel (or of whatever ran before):
    // it waits with griddepcontrol.wait before touching the table
    return vec ? launch_pdl(geglu_vec_kernel<4>, dim3((unsigned)blocks), dim3(kThreads), smem, st,
                            p, table)
               : launch_pdl(geglu_scalar_kernel, dim3((unsigned)blocks), dim3(kThreads), smem, st,
                            p, table);
}

cudaError_t launch_gelu_and_mul(const GegluParams& p, uint16_t* table, cudaStream_t st) {
    cudaError_t e = launch_gelu_table(table, st);
    if (e != cudaSuccess) return e;
    return launch_gelu_stream(p, table, st);
}

}  // namespace dtrot
