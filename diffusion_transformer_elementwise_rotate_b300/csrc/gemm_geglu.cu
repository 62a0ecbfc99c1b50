// GEGLU applied in the epilogue of the MLP's gate_up projection:
//   gate_up = RN16(x W^T)        x (T, C), W (2F, C) bf16, fp32 accumulation
//   out     = RN16(up * RN16(RN32(gelu(gate))))   gate = first F columns
//
// ERNIE-Image fusion page (sglang PR #34306 analysis), section 3: the MLP runs
// gate_up_proj and then the fused GEGLU; the eager path wrote gate_up to HBM
// and made two more passes over it.  Here the activation is applied to the
// projection's accumulators before anything is stored, so gate_up never
// reaches HBM: the call reads x and W and writes out.
//
// Design (tcgen05 tensor cores, persistent CTAs, warp-specialised):
//   - the B operand of a tile is 256 weight rows: gate rows f0..f0+127 and up
//     rows F+f0..F+f0+127, so one fp32 accumulator row in tensor memory holds
//     gate and up of the same 128 output columns;
//   - a ring of shared-memory stages (x and W tiles, 64 columns of K, 128-byte
//     swizzle) filled by TMA (one thread) and consumed by tcgen05.mma (one
//     thread, K 16 per instruction), with mbarriers for "stage full" (TMA
//     transaction bytes) and "stage empty" (tcgen05.commit);
//   - two accumulators in tensor memory, so the epilogue of one tile overlaps
//     the MMAs of the next;
//   - epilogue: each of 4 warps reads its 32 accumulator lanes (rows) with
//     tcgen05.ld, rounds gate and up to bf16 (the projection's output
//     rounding), looks the activation up in a compact 17 KB table in shared
//     memory, multiplies with one bf16x2 .rn multiply, as the standalone GEGLU
//     kernel does, and stores 32 x 32 output blocks through shared memory
//     with TMA;
//   - optionally the rounded gate and up are stored too (a (T, 2F) gate_up
//     tensor, for a backward pass or for checking);
//   - tiles are visited in groups of row tiles so that the x and W tiles a
//     wave of CTAs reads stay in L2.
// Two kernels share this design:
//   gemm_geglu_pair_kernel  CTA pairs (clusters of 2 on the two SMs of a TPC)
//       with cta_group::2 MMAs of M 256 x N 256: each CTA stages 128 rows of x
//       and 128 rows of W (the first CTA the gate rows, the second the up
//       rows), 32 KB per stage, so a pair reads half the W bytes two single
//       CTAs would and six stages fit in shared memory;
//   gemm_geglu_kernel  one CTA per 128-row tile, M 128 x N 256, 48 KB stages,
//       for T <= 128 (a pair tile would be half empty) or when no cluster of
//       two fits.
// Every mbarrier wait is bounded (about a second of %globaltimer): a wait that
// runs out records a code in the workspace's error word and the CTA finishes
// without further waits (single CTAs that start later and see the word set
// exit at once; the pair kernel's clusters all start together).
#include <cuda.h>

#include <atomic>

#include "dtrot_internal.cuh"

namespace dtrot {
namespace {

constexpr int BM = 128;             // output rows per tile
constexpr int BNH = 128;            // output columns per tile (gate or up half)
constexpr int BN = 2 * BNH;         // MMA N: gate and up columns
constexpr int BK = 64;              // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kGroupM = 16;
constexpr uint32_t kATile = BM * BK * 2;   // 16 KB
constexpr uint32_t kBTile = BN * BK * 2;   // 32 KB
constexpr uint32_t kStageBytes = kATile + kBTile;
constexpr uint32_t kAccCols = 256;   // one 128 x 256 fp32 accumulator
// output staging for TMA stores: per epilogue warp two 32 x 32 bf16 blocks
constexpr uint32_t kOutBlock = 32 * 32 * 2;          // 2 KB
constexpr uint32_t kOutStaging = 4 * 2 * kOutBlock;  // 16 KB
constexpr uint32_t kTmemCols = 512;  // two accumulators: MMA and epilogue overlap

// Compact activation table: entries for |x| in [2^-30, 8) (x > 0) and
// [2^-30, 16) (x < 0), i.e. bf16 exponent fields 97..129 and 97..130; every
// other gate value has a closed form (see gelu_lookup).
constexpr int kExpLo = 97;
constexpr int kPosEntries = (129 - kExpLo + 1) * 128;          // 4224
constexpr int kCompact = kPosEntries + (130 - kExpLo + 1) * 128;  // 8576
constexpr uint32_t kTabBytes = kCompact * 2;                   // 17152
constexpr uint32_t kErrOffset = kTabBytes;                     // error word in the workspace
constexpr uint32_t kWorkspaceBytes = 17408;

constexpr uint32_t kErrTimeoutEmpty = 1, kErrTimeoutFull = 2, kErrTimeoutAccum = 4;
constexpr uint32_t kErrTmemMismatch = 8;  // the two CTAs of a pair got different columns
constexpr uint64_t kWaitNs = 1000000000ull;  // bound on any single wait

// CTA pairs: a pair tile is 256 output rows (128 per CTA) x 128 output columns
constexpr int kStagesP = 6;
// pair row tiles per raster group: a wave of 74 clusters covers 16 pair rows x
// ~5 column tiles, and W is re-read from DRAM once per 4096 rows (at the power
// limit the DRAM traffic saved is worth more than the smaller wave footprint
// of groups of 8)
constexpr int kGroupMP = 16;
constexpr uint32_t kAHalf = BM * BK * 2;          // 16 KB: this CTA's 128 rows of x
constexpr uint32_t kBHalf = BNH * BK * 2;         // 16 KB: this CTA's 128 rows of W
constexpr uint32_t kStageBytesP = kAHalf + kBHalf;
constexpr uint32_t kPairTx = 2 * kStageBytesP;    // bytes both CTAs land per stage
constexpr uint16_t kBothCtas = 0x3;               // multicast mask of a pair

struct GemmGegluParams {
    uint16_t* out;
    int64_t s_out;
    uint16_t* gate_up;  // optional (T, 2F) copy of the rounded projection
    int64_t s_gate_up;
    int64_t T, C, F;
    const uint16_t* table;  // compact activation table in the workspace
    uint32_t* err;          // error word in the workspace
    int num_m, num_n;
    // diagnostic: when set, each producer withholds the loads of its last
    // stage use, so the MMA thread's bounded wait for that stage runs out
    int withhold_last_stage;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false (and `code` recorded) when the phase did not complete in
// kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err,
                                          uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitNs) {
            atomicOr(err, code);
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// TMA store of a 32 x 32 block from shared memory (rows >= T and columns >= F
// of the tensor map are not written).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// At most one store group of this thread still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Every store group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (start address and offsets in 16-byte units).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (not used with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = BN, M = BM.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// 32 consecutive fp32 accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_may_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_prerequisite_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- CTA-pair helpers

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of both CTAs: release this CTA's earlier shared-memory writes
// and wait for the peer's.
__device__ __forceinline__ void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// The waiting thread sleeps in hardware until the phase completes or
// kSuspendNs pass (a spinning wait costs issue slots and power, and the pair
// kernel runs at the power limit).
constexpr uint32_t kSuspendNs = 1000000u;
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
// Bounded wait with cluster-scope acquire (the barrier may receive arrivals
// and transaction bytes from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, uint32_t* err,
                                             uint32_t code) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait_cl(bar, parity)) {
        if (global_ns() - t0 > kWaitNs) {
            atomicOr(err, code);
            return false;
        }
    }
    return true;
}
// TMA load into this CTA's shared memory whose transaction bytes complete on
// `bar_cluster`, an mbarrier of this CTA or of its peer.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2 [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}
// Instruction descriptor of the pair MMA: as kIdesc with M = 256.
constexpr uint32_t kIdescPair = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((2 * BM) >> 4) << 24);

// D[256 x 256] (+)= A[256 x 16] B[16 x 256]: A rows 0-127 and B rows (N)
// 0-127 are read from the issuing CTA's shared memory, A rows 128-255 and B
// rows 128-255 from the same addresses in the peer; D rows 0-127 land in the
// issuing CTA's tensor memory, rows 128-255 in the peer's.
__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t a, uint64_t b,
                                              uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(kIdescPair), "r"(acc)
        : "memory");
}
// Arrive once on the mbarrier at `bar`'s offset in both CTAs of the pair when
// the pair MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(kBothCtas)
        : "memory");
}
// The same, on this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// ---------------------------------------------------------------- activation

// g(x) = RN16(RN32(gelu(x))) for the bf16 pattern b, from the compact table or
// a closed form:
//   |x| < 2^-30 (exponent field < 97, zeros and subnormals included):
//       gelu(x) = x/2 + x^2/sqrt(2 pi) + O(x^4) and x/2 is exact in fp32; the
//       x^2 term is below 2^-25 |x/2|, so RN32 gives x/2 and g = RN16(x/2);
//   x >= 8 (and +inf, NaN): gelu(x) = x (1 - erfc(x/sqrt 2)/2) differs from x
//       by less than 2^-49 |x|, so RN32 gives x back;
//   x <= -16: |gelu(x)| < 1e-55 < 2^-150, so RN32 gives -0; -inf gives NaN
//       (-inf * 0) like the formula.
__device__ __forceinline__ uint32_t gelu_lookup(const uint16_t* tab, uint32_t b) {
    // without branches: one table load at a clamped index, then the closed
    // forms by selection (b is a 16-bit pattern; m = |x|'s pattern, whose
    // exponent field compares like m against e << 7)
    const uint32_t m = b & 0x7FFFu;
    const uint32_t neg = b >> 15;
    int idx = (int)m - (kExpLo << 7) + (int)neg * kPosEntries;
    idx = min(max(idx, 0), kCompact - 1);
    uint32_t r = tab[idx];
    const uint32_t half = rn16f(__fmul_rn(__uint_as_float(b << 16), 0.5f));
    r = m < ((uint32_t)kExpLo << 7) ? half : r;
    r = (!neg && m >= (130u << 7)) ? b : r;
    r = (neg && m >= (131u << 7)) ? (m >= (255u << 7) ? 0x7FC0u : 0x8000u) : r;
    return r;
}

__device__ __forceinline__ uint32_t gelu_lookup2(const uint16_t* tab, uint32_t g2) {
    return gelu_lookup(tab, g2 & 0xFFFFu) | (gelu_lookup(tab, g2 >> 16) << 16);
}

// Compact table entry i (see kExpLo): the gelu_entry of its bf16 pattern.
__global__ void __launch_bounds__(256) gelu_compact_table_kernel(uint16_t* __restrict__ table,
                                                                 uint32_t* __restrict__ err) {
    grid_dependents_may_launch();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) *err = 0;
    if (i < kCompact) {
        const uint32_t b = i < kPosEntries ? (uint32_t)(kExpLo << 7) + i
                                           : 0x8000u | ((uint32_t)(kExpLo << 7) + (i - kPosEntries));
        table[i] = gelu_entry(b);
    }
}

// ---------------------------------------------------------------- the GEMM

// Tile t of the grouped order: row tiles advance fastest within a group of
// kGroup, so the CTAs working at the same time share x and W tiles in L2.
template <int kRows, int kGroup>
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int& m0, int& f0) {
    const int in_group = kGroup * num_n;
    const int first_m = (t / in_group) * kGroup;
    const int gm = min(num_m - first_m, kGroup);
    m0 = (first_m + (t % in_group) % gm) * kRows;
    f0 = ((t % in_group) / gm) * BNH;
}

// Epilogue of one warp's 32 accumulator rows (lane = row row0 + lane): gate in
// columns 0..127 of `taddr`, up in 128..255; output columns f0..f0+127.  Each
// 32 x 32 output block goes through one of the warp's two staging buffers in
// shared memory (`stage0`, 2 x 2 KB) and out by TMA store, 64-byte row
// segments instead of 16-byte pieces of 32 rows.  The staging rows use the
// 64-byte swizzle of the output tensor map (16-byte chunk c of row r at
// chunk c ^ ((r >> 1) & 3)), so the 32 lanes' writes hit distinct banks.
// `nstore` counts this warp's stores (it picks the buffer).
__device__ __forceinline__ void epilogue_rows(const GemmGegluParams& p, const uint16_t* tab,
                                              const CUtensorMap* tma_out, uint32_t taddr,
                                              int64_t row0, int f0, uint32_t stage0,
                                              uint32_t& nstore) {
    const int lane = threadIdx.x & 31;
    const int64_t row = row0 + lane;
    const uint32_t sw = (uint32_t)(lane >> 1) & 3u;
#pragma unroll 1
    for (int j = 0; j < BNH / 32; ++j) {
        uint32_t g[32], u[32];
        tmem_ld32(taddr + 32 * j, g);
        tmem_ld32(taddr + BNH + 32 * j, u);
        tmem_wait_ld();
        uint32_t o[16], gb[16], ub[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            gb[q] = rn16x2f(__uint_as_float(g[2 * q]), __uint_as_float(g[2 * q + 1]));
            ub[q] = rn16x2f(__uint_as_float(u[2 * q]), __uint_as_float(u[2 * q + 1]));
            o[q] = bmul2(ub[q], gelu_lookup2(tab, gb[q]));
        }
        if (p.gate_up && row < p.T) {
            uint16_t* gdst = p.gate_up + row * p.s_gate_up + f0 + 32 * j;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (f0 + 32 * j + 8 * q < p.F) {
                    *reinterpret_cast<uint4*>(gdst + 8 * q) =
                        make_uint4(gb[4 * q], gb[4 * q + 1], gb[4 * q + 2], gb[4 * q + 3]);
                    *reinterpret_cast<uint4*>(gdst + p.F + 8 * q) =
                        make_uint4(ub[4 * q], ub[4 * q + 1], ub[4 * q + 2], ub[4 * q + 3]);
                }
            }
        }
        const uint32_t buf = stage0 + (nstore & 1u) * kOutBlock;
        // the store that used this buffer two blocks ago has read it
        if (lane == 0) bulk_wait_read_1();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c)
            st_shared_v4(buf + (uint32_t)lane * 64 + (((uint32_t)c ^ sw) << 4), o[4 * c],
                         o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        fence_async_smem();
        __syncwarp();
        // a block wholly past the last row or column is not stored (partial
        // blocks are clipped by the tensor map)
        if (lane == 0 && row0 < p.T && f0 + 32 * j < p.F) {
            tma_store_2d(tma_out, buf, f0 + 32 * j, (int32_t)row0);
            bulk_commit();
        }
        ++nstore;
    }
}

// Copy the compact activation table from the workspace into shared memory.
__device__ __forceinline__ void load_table(const GemmGegluParams& p, uint16_t* tab) {
    const uint4* src = reinterpret_cast<const uint4*>(p.table);
    uint4* dst = reinterpret_cast<uint4*>(tab);
    for (int i = threadIdx.x; i < (int)(kTabBytes / 16); i += kThreads) dst[i] = __ldcg(src + i);
}

// The producer's last loads must have landed before the CTA exits (on the
// normal path the MMAs consumed them; after an abort they may be in flight).
// `issued` counts the stage uses this thread filled.
template <int kNumStages>
__device__ __forceinline__ void wait_own_loads(uint32_t full0, uint32_t issued, uint32_t* err,
                                               bool cluster_scope) {
    const uint32_t n = issued < (uint32_t)kNumStages ? issued : (uint32_t)kNumStages;
    for (uint32_t i = 0; i < n; ++i) {
        const uint32_t use = issued - 1 - i;
        const uint32_t bar = full0 + 8 * (use % kNumStages);
        const uint32_t ph = (use / kNumStages) & 1u;
        if (cluster_scope ? !mbar_wait_cl(bar, ph, err, kErrTimeoutFull)
                          : !mbar_wait(bar, ph, err, kErrTimeoutFull))
            return;
    }
}

// Persistent CTAs (one per SM) walk tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// Roles: warp 0 lane 0 feeds the stage ring with TMA, running ahead into the
// next tile; warp 1 lane 0 issues the MMAs into one of two accumulators in
// tensor memory; warps 2-5 drain the other accumulator (the epilogue) while
// the next tile's MMAs run.  Barriers: full/empty per stage, and per
// accumulator acc_full (MMA -> epilogue, by tcgen05.commit) and acc_empty
// (epilogue -> MMA, one arrival per epilogue warp).  A wait that runs out of
// time sets `abort` in shared memory and every role leaves its loop.
__global__ void __launch_bounds__(kThreads, 1)
    gemm_geglu_kernel(const __grid_constant__ CUtensorMap tma_x,
                      const __grid_constant__ CUtensorMap tma_w,
                      const __grid_constant__ CUtensorMap tma_out, GemmGegluParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_skip;
    __shared__ volatile uint32_t s_abort;
    // the table kernel (the prerequisite grid) has written the activation table
    // and cleared the error word once this returns
    wait_for_prerequisite_grid();
    // a CTA that starts after an earlier launch ran out of a wait does nothing
    // (decided by one thread, so the whole CTA leaves together)
    if (threadIdx.x == 0) {
        s_skip = *reinterpret_cast<volatile uint32_t*>(p.err);
        s_abort = 0;
    }
    __syncthreads();
    if (s_skip != 0) return;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // swizzled tiles want 1024-byte alignment
    uint8_t* sm = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + kStages * kATile;
    const uint32_t sOut = base + kStages * kStageBytes;  // output staging, 1024-byte aligned
    uint16_t* tab = reinterpret_cast<uint16_t*>(sm + kStages * kStageBytes + kOutStaging);
    uint64_t* bars =
        reinterpret_cast<uint64_t*>(sm + kStages * kStageBytes + kOutStaging + kTabBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * kStages;
    const uint32_t acc_full0 = full0 + 16 * kStages, acc_empty0 = acc_full0 + 16;
    const uint32_t drain = acc_empty0 + 16;  // every MMA of this CTA has completed

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = p.num_m * p.num_n;
    const int nk = (int)((p.C + BK - 1) / BK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full0 + 8 * a, 1);
            mbar_init(acc_empty0 + 8 * a, 4);
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    load_table(p, tab);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // TMA producer; `it` counts stage uses across all tiles of this CTA
            uint32_t it = 0;
            for (int t = blockIdx.x; t < tiles && !s_abort; t += gridDim.x) {
                int m0, f0;
                tile_coords<BM, kGroupM>(t, p.num_m, p.num_n, m0, f0);
                const bool last_tile = t + (int)gridDim.x >= tiles;
                for (int kb = 0; kb < nk; ++kb) {
                    if (p.withhold_last_stage && last_tile && kb == nk - 1) break;
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (it >= (uint32_t)kStages &&
                        !mbar_wait(empty0 + 8 * s, ph ^ 1u, p.err, kErrTimeoutEmpty)) {
                        s_abort = 1;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * s;
                    mbar_expect_tx(fb, kStageBytes);
                    tma_load_2d(sA + s * kATile, &tma_x, kb * BK, m0, fb);
                    tma_load_2d(sB + s * kBTile, &tma_w, kb * BK, f0, fb);
                    tma_load_2d(sB + s * kBTile + BNH * BK * 2, &tma_w, kb * BK,
                                (int32_t)p.F + f0, fb);
                    ++it;
                }
            }
            wait_own_loads<kStages>(full0, it, p.err, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer: 4 instructions of K 16 per stage into accumulator
            // i % 2; the stage is released when they have read it, the
            // accumulator handed to the epilogue after the tile's last stage
            uint32_t it = 0;
            int i = 0;
            for (int t = blockIdx.x; t < tiles && !s_abort; t += gridDim.x, ++i) {
                const int acc = i & 1;
                if (i >= 2 && !mbar_wait(acc_empty0 + 8 * acc, ((i >> 1) & 1) ^ 1, p.err,
                                         kErrTimeoutAccum)) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)acc * kAccCols;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(full0 + 8 * s, ph, p.err, kErrTimeoutFull)) {
                        s_abort = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a = smem_desc(sA + s * kATile);
                    const uint64_t b = smem_desc(sB + s * kBTile);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_bf16(d, a + 2 * k, b + 2 * k, (kb | k) != 0 ? 1u : 0u);
                    mma_commit(empty0 + 8 * s);
                }
                mma_commit(acc_full0 + 8 * acc);  // after this tile's MMAs complete
                if (s_abort) break;
            }
            // tensor memory is freed below only after every MMA issued here
            // has completed (the epilogue may have stopped early on an abort)
            mma_commit(drain);
            mbar_wait(drain, 0, p.err, kErrTimeoutAccum);
        }
        __syncwarp();
    } else {
        // epilogue: warp w reads accumulator lanes 32 * (w % 4) .. + 31
        const int quarter = warp & 3;
        const uint32_t stage0 = sOut + (uint32_t)quarter * 2 * kOutBlock;
        uint32_t nstore = 0;
        int i = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
            const int acc = i & 1;
            const bool ok = !s_abort && mbar_wait(acc_full0 + 8 * acc, (i >> 1) & 1, p.err,
                                                  kErrTimeoutAccum);
            __syncwarp();
            if (!__all_sync(0xffffffffu, ok)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            int m0, f0;
            tile_coords<BM, kGroupM>(t, p.num_m, p.num_n, m0, f0);
            epilogue_rows(p, tab, &tma_out,
                          tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)acc * kAccCols,
                          (int64_t)m0 + quarter * 32, f0, stage0, nstore);
            // this accumulator may be overwritten once all four warps are done
            tc_fence_before();
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                                            acc_empty0 + 8 * acc)
                                        : "memory");
        }
        // the stores have read the staging buffers and written the output
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

// CTA pairs (clusters of 2).  Both CTAs of a cluster walk the same pair tiles
// (cluster c takes tiles c, c + clusters, ...).  Roles as in gemm_geglu_kernel,
// except that:
//   - each CTA's producer loads its own 128 rows of x and 128 rows of W (rank
//     0 the gate rows, rank 1 the up rows) into its own shared memory, and
//     both signal rank 0's full barrier, whose expected byte count (set by
//     rank 0's producer) covers the two CTAs;
//   - only rank 0's MMA thread issues (cta_group::2, M 256 x N 256); its
//     commits arrive on the empty and acc_full barriers of both CTAs;
//   - the epilogue warps of both CTAs arrive on rank 0's acc_empty barrier
//     (8 arrivals per phase);
//   - tensor memory is allocated and freed by one warp of each CTA together;
//   - a cluster barrier after the set-up (the peer signals rank 0's barriers,
//     which must be initialised first) and one before the exit (no CTA leaves
//     while the other may still signal its barriers or read its stages).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_geglu_pair_kernel(const __grid_constant__ CUtensorMap tma_x,
                           const __grid_constant__ CUtensorMap tma_w,
                           const __grid_constant__ CUtensorMap tma_out, GemmGegluParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ volatile uint32_t s_abort;
    // the table kernel (the prerequisite grid) has written the activation table
    // and cleared the error word once this returns
    wait_for_prerequisite_grid();

    const uint32_t rank = cluster_ctarank();
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // the same offset in both CTAs
    uint8_t* sm = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + kStagesP * kAHalf;
    const uint32_t sOut = base + kStagesP * kStageBytesP;  // output staging, 1024-byte aligned
    uint16_t* tab = reinterpret_cast<uint16_t*>(sm + kStagesP * kStageBytesP + kOutStaging);
    uint64_t* bars =
        reinterpret_cast<uint64_t*>(sm + kStagesP * kStageBytesP + kOutStaging + kTabBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStagesP + 5);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * kStagesP;
    const uint32_t acc_full0 = full0 + 16 * kStagesP, acc_empty0 = acc_full0 + 16;
    const uint32_t drain = acc_empty0 + 16;  // every MMA issued by rank 0 has completed

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cluster = (int)(blockIdx.x >> 1), clusters = (int)(gridDim.x >> 1);
    const int tiles = p.num_m * p.num_n;  // num_m counts 256-row pair tiles
    const int nk = (int)((p.C + BK - 1) / BK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesP; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full0 + 8 * a, 1);
            mbar_init(acc_empty0 + 8 * a, 8);
        }
        mbar_init(drain, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    load_table(p, tab);
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (rank == 1 && threadIdx.x == 0) {
        // the pair MMAs write rank 1's rows at rank 0's tensor-memory address
        uint32_t lead;
        asm volatile("ld.shared::cluster.u32 %0, [%1];"
                     : "=r"(lead)
                     : "r"(peer_addr(smem_u32(tmem_slot), 0))
                     : "memory");
        if (lead != tmem) atomicOr(p.err, kErrTmemMismatch);
    }

    if (warp == 0) {
        if (lane == 0) {
            // TMA producer of this CTA's half of every stage
            const uint32_t full_lead0 = peer_addr(full0, 0);
            uint32_t it = 0;
            for (int t = cluster; t < tiles && !s_abort; t += clusters) {
                int m0, f0;
                tile_coords<2 * BM, kGroupMP>(t, p.num_m, p.num_n, m0, f0);
                const int32_t xrow = m0 + (int32_t)rank * BM;
                const int32_t wrow = (rank ? (int32_t)p.F : 0) + f0;
                const bool last_tile = t + clusters >= tiles;
                for (int kb = 0; kb < nk; ++kb) {
                    // both CTAs of the pair withhold the same stage use
                    if (p.withhold_last_stage && last_tile && kb == nk - 1) break;
                    const uint32_t s = it % kStagesP;
                    const uint32_t ph = (it / kStagesP) & 1u;
                    if (it >= (uint32_t)kStagesP &&
                        !mbar_wait_cl(empty0 + 8 * s, ph ^ 1u, p.err, kErrTimeoutEmpty)) {
                        s_abort = 1;
                        break;
                    }
                    if (rank == 0) mbar_expect_tx(full0 + 8 * s, kPairTx);
                    tma_load_2d_pair(sA + s * kAHalf, &tma_x, kb * BK, xrow, full_lead0 + 8 * s);
                    tma_load_2d_pair(sB + s * kBHalf, &tma_w, kb * BK, wrow, full_lead0 + 8 * s);
                    ++it;
                }
            }
            // rank 0's full barriers also count rank 1's bytes
            if (rank == 0) wait_own_loads<kStagesP>(full0, it, p.err, true);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // MMA issuer for the pair: 4 instructions of K 16 per stage into
            // accumulator i % 2 of both CTAs
            uint32_t it = 0;
            int i = 0;
            for (int t = cluster; t < tiles && !s_abort; t += clusters, ++i) {
                const int acc = i & 1;
                if (i >= 2 && !mbar_wait_cl(acc_empty0 + 8 * acc, ((i >> 1) & 1) ^ 1, p.err,
                                            kErrTimeoutAccum)) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)acc * kAccCols;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const uint32_t s = it % kStagesP;
                    const uint32_t ph = (it / kStagesP) & 1u;
                    if (!mbar_wait_cl(full0 + 8 * s, ph, p.err, kErrTimeoutFull)) {
                        s_abort = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a = smem_desc(sA + s * kAHalf);
                    const uint64_t b = smem_desc(sB + s * kBHalf);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_bf16_pair(d, a + 2 * k, b + 2 * k, (kb | k) != 0 ? 1u : 0u);
                    mma_commit_pair(empty0 + 8 * s);
                }
                mma_commit_pair(acc_full0 + 8 * acc);
                if (s_abort) break;
            }
            mma_commit_pair_local(drain);
            mbar_wait(drain, 0, p.err, kErrTimeoutAccum);
        }
        __syncwarp();
    } else {
        // epilogue: warp w reads accumulator lanes 32 * (w % 4) .. + 31, the
        // rows rank * 128 + lane of the pair tile
        const int quarter = warp & 3;
        const uint32_t acc_empty_lead0 = peer_addr(acc_empty0, 0);
        const uint32_t stage0 = sOut + (uint32_t)quarter * 2 * kOutBlock;
        uint32_t nstore = 0;
        int i = 0;
        for (int t = cluster; t < tiles; t += clusters, ++i) {
            const int acc = i & 1;
            const bool ok = !s_abort && mbar_wait_cl(acc_full0 + 8 * acc, (i >> 1) & 1, p.err,
                                                     kErrTimeoutAccum);
            __syncwarp();
            if (!__all_sync(0xffffffffu, ok)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            int m0, f0;
            tile_coords<2 * BM, kGroupMP>(t, p.num_m, p.num_n, m0, f0);
            epilogue_rows(p, tab, &tma_out,
                          tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)acc * kAccCols,
                          (int64_t)m0 + (int64_t)rank * BM + quarter * 32, f0, stage0, nstore);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acc_empty_lead0 + 8 * acc);
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kOutStaging + kTabBytes +
                              (2 * kStages + 5) * 8 + 16;
constexpr size_t kSmemBytesP = 1024 + (size_t)kStagesP * kStageBytesP + kOutStaging + kTabBytes +
                               (2 * kStagesP + 5) * 8 + 16;
static_assert(kSmemBytes <= 232448 && kSmemBytesP <= 232448, "shared memory per CTA");

constexpr int kMaxDev = 64;
// context (current_context_id) for which the shared memory attributes were set
std::atomic<uint64_t> g_smem_attr_ctx[kMaxDev];
// per device: co-resident clusters of the pair kernel + 1 (0: not asked yet)
std::atomic<int> g_pair_clusters[kMaxDev];

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static std::atomic<EncodeTiled> fn{nullptr};
    EncodeTiled f = fn.load(std::memory_order_acquire);
    if (!f) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !ptr)
            return nullptr;
        f = reinterpret_cast<EncodeTiled>(ptr);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

// 2-D bf16 tensor map over a (rows, cols) row-major matrix, boxes of 128 rows
// x 64 columns, 128-byte swizzle, zero fill outside the matrix.
bool make_map(CUtensorMap* m, const uint16_t* ptr, int64_t rows, int64_t cols) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {BK, 128};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(ptr), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// The output (rows, cols) with row stride `stride` elements, 32 x 32 boxes,
// 64-byte swizzle (the staging layout of epilogue_rows).
bool make_out_map(CUtensorMap* m, uint16_t* ptr, int64_t rows, int64_t cols, int64_t stride) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Clusters of two pair-kernel CTAs that fit on the device at once (0: none).
cudaError_t pair_clusters(int dev, int* out) {
    int c = g_pair_clusters[dev].load(std::memory_order_acquire);
    if (c == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytesP;
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&n, gemm_geglu_pair_kernel, &cfg);
        if (e != cudaSuccess) return e;
        c = (n > 0 ? n : 0) + 1;
        g_pair_clusters[dev].store(c, std::memory_order_release);
    }
    *out = c - 1;
    return cudaSuccess;
}

}  // namespace

size_t gemm_geglu_workspace_bytes() { return kWorkspaceBytes; }
size_t gemm_geglu_error_offset() { return kErrOffset; }

cudaError_t launch_gemm_geglu(const GemmGegluArgs& a, cudaStream_t st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    const uint64_t ctx = current_context_id();
    if (ctx == 0 || g_smem_attr_ctx[dev].load(std::memory_order_acquire) != ctx) {
        e = cudaFuncSetAttribute(gemm_geglu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm_geglu_pair_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesP);
        if (e != cudaSuccess) return e;
        g_smem_attr_ctx[dev].store(current_context_id(), std::memory_order_release);
    }
    CUtensorMap mx, mw, mo;
    if (!make_map(&mx, a.x, a.T, a.C) || !make_map(&mw, a.w, 2 * a.F, a.C) ||
        !make_out_map(&mo, a.out, a.T, a.F, a.s_out))
        return cudaErrorInvalidValue;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    uint16_t* table = reinterpret_cast<uint16_t*>(ws);
    uint32_t* err = reinterpret_cast<uint32_t*>(ws + kErrOffset);
    gelu_compact_table_kernel<<<(kCompact + 255) / 256, 256, 0, st>>>(table, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    GemmGegluParams p;
    p.out = a.out;
    p.s_out = a.s_out;
    p.gate_up = a.gate_up;
    p.s_gate_up = a.s_gate_up;
    p.T = a.T;
    p.C = a.C;
    p.F = a.F;
    p.table = table;
    p.err = err;
    p.num_n = (int)((a.F + BNH - 1) / BNH);
    p.withhold_last_stage = a.withhold_last_stage;

    // CTA pairs unless a pair tile would be half empty or no cluster fits
    int clusters = 0;
    if (a.T > BM) {
        e = pair_clusters(dev, &clusters);
        if (e != cudaSuccess) return e;
    }
    const bool pair = clusters > 0;
    int64_t grid;
    if (pair) {
        p.num_m = (int)((a.T + 2 * BM - 1) / (2 * BM));
        const int64_t tiles = (int64_t)p.num_m * p.num_n;
        grid = 2 * (tiles < clusters ? tiles : (int64_t)clusters);
    } else {
        p.num_m = (int)((a.T + BM - 1) / BM);
        const int64_t tiles = (int64_t)p.num_m * p.num_n;
        grid = num_sms();  // persistent: one CTA per SM (the stage ring fills its smem)
        if (grid > tiles) grid = tiles;
    }

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = pair ? kSmemBytesP : kSmemBytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = pair ? cudaLaunchKernelEx(&cfg, gemm_geglu_pair_kernel, mx, mw, mo, p)
             : cudaLaunchKernelEx(&cfg, gemm_geglu_kernel, mx, mw, mo, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dtrot
