/*
 * dtrot.h — C ABI of the B300 (sm_103a) elementwise hot path of a
 * diffusion-transformer block: rotary cos/sin tables, rotate-half RoPE,
 * GEGLU with activation rounding, and RMSNorm fused with the residual add.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - bf16 tensors are passed as `uint16_t*` holding bfloat16 bit patterns;
 *    fp32 tensors as `float*`.  All data pointers are DEVICE pointers
 *    (cudaMalloc, a caching allocator, or managed memory) on the device that is
 *    current when the call is made.
 *  - Sizes and strides are int64_t counts of ELEMENTS (not bytes).  The last
 *    dimension of every tensor is contiguous (stride 1).
 *  - `stream` is a cudaStream_t passed as `void*`; NULL means the legacy
 *    default stream.  Work is enqueued on it and the call returns without
 *    synchronising.  The library allocates nothing, frees nothing and makes no
 *    host-device synchronisation, so the compute calls may be captured in a
 *    CUDA graph (dtrot_gelu_and_mul_noalloc aside: see its notes below).
 *    dtrot_gemm_gelu_and_mul_error is the one call that copies to host
 *    memory, and it waits for the copy when that memory is pageable.
 *  - Each kernel is launched as a programmatic dependent of the work before it
 *    in the stream (so its launch overlaps the end of that work) and waits for
 *    that work to complete before it reads or writes any memory: the memory
 *    effects of the calls keep plain stream order.
 *  - The caller owns every buffer.  Outputs are fully overwritten; inputs are
 *    only read, except `residual` of dtrot_rmsnorm_residual, which is updated.
 *  - Any alignment is accepted.  Pointers and strides that are multiples of
 *    8 elements (16 bytes) take 128-bit vector paths; others take narrower
 *    vector or scalar paths with identical results.
 *  - A call with a zero-sized dimension does nothing and returns DTROT_OK
 *    (pointers may then be NULL).
 *  - Arguments are validated on the host before anything is launched.  An
 *    invalid call launches nothing and returns its status; a launch failure is
 *    reported as DTROT_ERR_LAUNCH from cudaGetLastError().  No device-side
 *    assert or trap is used.
 *
 * Rounding: RN16 is round-to-nearest-even to bfloat16 (8 significant bits,
 * the fp32 exponent range, subnormals kept); RN32 likewise to fp32.
 *
 * Source pages (cited by title and section):
 *  [P4] "[sglang] ERNIE-Image ... RoPE and GELU-mul fusion and RoPE cos/sin
 *       hoisting" (analysis of sglang PR #34306), sections 1-3.
 *  [P5] "SP: splitting activations alongside TP" (sequence-parallelism post),
 *       section on per-token normalisation and residual add, and the Pre-Norm
 *       layer figure.
 */
#ifndef DTROT_H
#define DTROT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dtrot_status {
    DTROT_OK = 0,
    DTROT_ERR_NULL = 1,   /* a required pointer is NULL */
    DTROT_ERR_SHAPE = 2,  /* a size is negative, or an element count overflows */
    DTROT_ERR_ROTDIM = 3, /* rot_dim is odd, zero, or larger than D */
    DTROT_ERR_STRIDE = 4, /* a stride is not positive, or rows/heads of an output overlap */
    DTROT_ERR_ALIAS = 5,  /* an output overlaps an input in a way the call does not allow */
    DTROT_ERR_LAUNCH = 6, /* the CUDA launch failed (see cudaGetLastError) */
    DTROT_ERR_DEVICE = 7, /* no current CUDA device, or it is not sm_103 */
    DTROT_ERR_VALUE = 8,  /* a scalar argument is out of range (eps) */
    DTROT_ERR_WORKSPACE = 9, /* a workspace is smaller than required or not 16-byte aligned */
    DTROT_ERR_ALIGN = 10   /* a pointer, stride or size misses an op's alignment requirement */
} dtrot_status;

/* Human-readable name of a status code (static storage, never NULL). */
const char* dtrot_status_str(dtrot_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int dtrot_version(void);

/*
 * Rotary cos/sin tables, computed once per forward.            [P4] section 1
 *
 *   cos_out[b*S + s, j] = RN16(RN32(cos(freqs[s, b, 0, j])))
 *   sin_out[b*S + s, j] = RN16(RN32(sin(freqs[s, b, 0, j])))
 *
 * i.e. the (S, B, 1, R) -> (B, S, 1, R) permute, cos/sin in fp32 and the cast
 * to bf16, reshaped to (B*S, R) rows, with the fp32 cos/sin taken as correctly
 * rounded.
 *   freqs    fp32, (S, B, 1, R) contiguous, read only.
 *   cos_out, sin_out  bf16, (B*S, R) contiguous, written.  They must not
 *            overlap each other or freqs (DTROT_ERR_ALIAS).
 */
dtrot_status dtrot_rope_cos_sin_precompute(const float* freqs, int64_t S, int64_t B,
                                           int64_t R, uint16_t* cos_out,
                                           uint16_t* sin_out, void* stream);

/*
 * Rotate-half RoPE over the leading rot_dim columns of x.      [P4] section 2
 *
 * With h = rot_dim / 2 and c, s = row b*S + s of cos/sin (shared by all H
 * heads of that token), for every (b, s, head):
 *   j <  h:          out[j] = RN16(RN16(x[j]*c[j]) + RN16(-x[j+h]*s[j]))
 *   h <= j < rot_dim: out[j] = RN16(RN16(x[j]*c[j]) + RN16( x[j-h]*s[j]))
 *   j >= rot_dim:    out[j] = x[j]        (tail columns pass through)
 * which is the eager chunk / neg / cat / mul / add chain with its per-op bf16
 * rounding, round(round(x1*cos1) + round(-x2*sin1)).
 *   x        bf16, (B, S, H, D) with element strides (sx_b, sx_s, sx_h) and
 *            the D axis contiguous, read only.
 *   cos, sin bf16, (B*S, rot_dim) contiguous (from the call above).
 *   rot_dim  even, 0 < rot_dim <= D (else DTROT_ERR_ROTDIM).
 *   out      bf16, (B, S, H, D) with strides (so_b, so_s, so_h), written.
 *            out == x with identical strides (in place) is allowed; any other
 *            overlap with x, cos or sin is DTROT_ERR_ALIAS.  Distinct output
 *            rows must not overlap (DTROT_ERR_STRIDE).  In place, the tail
 *            columns are left untouched (they already hold x).
 */
dtrot_status dtrot_rope_rotate_half(const uint16_t* x, int64_t B, int64_t S, int64_t H,
                                    int64_t D, int64_t sx_b, int64_t sx_s, int64_t sx_h,
                                    const uint16_t* cos, const uint16_t* sin,
                                    int64_t rot_dim, uint16_t* out, int64_t so_b,
                                    int64_t so_s, int64_t so_h, void* stream);

/*
 * Rotate-half RoPE on q and k in one launch, in place.   [P4] sections 1-2
 *
 * Applies the rotation of dtrot_rope_rotate_half to every head row of q and of
 * k, overwriting them; tail columns [rot_dim, D) are not touched.  The cos/sin
 * row of token (b, s) comes either from the tables (cos, sin, as written by
 * dtrot_rope_cos_sin_precompute) or, when `freqs` is given instead, is
 * evaluated from the angles inside the kernel with the same result as the
 * table kernel (bit for bit) and is never stored.
 *   q         bf16, (B, S, Hq, D), element strides (sq_b, sq_s, sq_h), D
 *             contiguous.  May be NULL when Hq == 0.
 *   k         bf16, (B, S, Hk, D), strides (sk_b, sk_s, sk_h).  May be NULL
 *             when Hk == 0.  q and k must not share elements: either their
 *             byte ranges are disjoint, or they are the two head ranges of one
 *             (B, S, Hq + Hk, D) view (equal strides, the second starting
 *             where the first one's heads end, as the q and k parts of a fused
 *             QKV buffer are); else DTROT_ERR_ALIAS.  Each must have
 *             non-overlapping rows (DTROT_ERR_STRIDE).
 *   cos, sin  bf16, (B*S, rot_dim) contiguous, or both NULL when freqs is given.
 *   freqs     fp32, (S, B, 1, rot_dim) contiguous, or NULL when tables are
 *             given.  Giving both is DTROT_ERR_VALUE; neither, DTROT_ERR_NULL.
 *             Tables or angles must not overlap q or k (DTROT_ERR_ALIAS).
 *   rot_dim   even, 0 < rot_dim <= D (else DTROT_ERR_ROTDIM).
 */
dtrot_status dtrot_rope_rotate_half_qk(uint16_t* q, int64_t Hq, int64_t sq_b, int64_t sq_s,
                                       int64_t sq_h, uint16_t* k, int64_t Hk, int64_t sk_b,
                                       int64_t sk_s, int64_t sk_h, int64_t B, int64_t S,
                                       int64_t D, const uint16_t* cos, const uint16_t* sin,
                                       const float* freqs, int64_t rot_dim, void* stream);

/*
 * Rotate-half RoPE on q and k in one launch, into separate outputs.
 *                                                        [P4] sections 1-2
 *
 * The out-of-place form of dtrot_rope_rotate_half_qk: q_out receives the
 * rotation of q and k_out that of k, tail columns [rot_dim, D) copied, so
 * each output equals what dtrot_rope_rotate_half writes for its input, bit
 * for bit.  One launch for both instead of one per tensor saves a kernel
 * boundary per layer.
 *   q, k        bf16, (B, S, Hq, D) and (B, S, Hk, D), element strides
 *               (sq_*), (sk_*), D contiguous, read only.  q may be NULL when
 *               Hq == 0, k when Hk == 0.  They may overlap each other.
 *   cos, sin, freqs, rot_dim   as for dtrot_rope_rotate_half_qk.
 *   q_out       bf16, (B, S, Hq, D), strides (soq_*), written; k_out
 *               likewise (sok_*).  Each must have non-overlapping rows
 *               (DTROT_ERR_STRIDE); the two must not share elements (their
 *               byte ranges disjoint, or the two head ranges of one
 *               (B, S, Hq + Hk, D) view); neither may overlap q, k, the
 *               tables or the angles (DTROT_ERR_ALIAS).  For in place, use
 *               dtrot_rope_rotate_half_qk.
 */
dtrot_status dtrot_rope_rotate_half_qk_out(
    const uint16_t* q, int64_t Hq, int64_t sq_b, int64_t sq_s, int64_t sq_h, const uint16_t* k,
    int64_t Hk, int64_t sk_b, int64_t sk_s, int64_t sk_h, int64_t B, int64_t S, int64_t D,
    const uint16_t* cos, const uint16_t* sin, const float* freqs, int64_t rot_dim,
    uint16_t* q_out, int64_t soq_b, int64_t soq_s, int64_t soq_h, uint16_t* k_out,
    int64_t sok_b, int64_t sok_s, int64_t sok_h, void* stream);

/*
 * Bytes of device workspace dtrot_gelu_and_mul needs (its activation table:
 * 65536 bf16 entries, 131072 bytes).  Constant for a given library version.
 */
int64_t dtrot_gelu_and_mul_workspace_bytes(void);

/*
 * GEGLU with the eager path's activation rounding.             [P4] section 3
 *
 *   out[t, f] = RN16(up[t, f] * RN16(RN32(gelu(gate[t, f]))))
 *   gelu(x)   = x * 1/2 * (1 + erf(x / sqrt 2))    (exact, erf-based GELU)
 *
 * gelu(-inf) follows IEEE evaluation of the formula (-inf * 0 = NaN).
 *   gate, up  bf16, (T, F), row strides s_gate, s_up >= F (elements), read
 *             only.  They may be the two halves of one (T, 2F) buffer
 *             (gate = columns [0, F), up = columns [F, 2F), strides 2F).
 *   out       bf16, (T, F), row stride s_out >= F, written.  out == gate with
 *             s_out == s_gate (in place) is allowed; any other element overlap
 *             with gate or up is DTROT_ERR_ALIAS.
 *   workspace device memory owned by the caller, at least
 *             dtrot_gelu_and_mul_workspace_bytes() bytes (workspace_bytes says
 *             how many), 16-byte aligned (else DTROT_ERR_WORKSPACE), not
 *             overlapping gate, up or out (else DTROT_ERR_ALIAS).  Its contents
 *             on entry are ignored; the call fills it with the activation table
 *             (two kernels on `stream`: the table, then the streaming kernel as
 *             its programmatic dependent).  Calls that may run at the same time
 *             on the GPU must use different workspaces.
 */
dtrot_status dtrot_gelu_and_mul(const uint16_t* gate, int64_t s_gate, const uint16_t* up,
                                int64_t s_up, uint16_t* out, int64_t s_out, int64_t T,
                                int64_t F, void* workspace, int64_t workspace_bytes,
                                void* stream);

/*
 * GEGLU with an activation table built once and kept.        [P4] sections 1, 3
 *
 * The activation table of dtrot_gelu_and_mul depends on nothing but the
 * function (one entry per bf16 gate value), so a caller that runs GEGLU many
 * times (every layer of every step) can build it once, as the ERNIE-Image page
 * hoists the cos/sin rows out of the per-layer path, and skip the table launch
 * on every call.
 *
 * dtrot_gelu_table_build fills `table` (at least
 * dtrot_gelu_and_mul_workspace_bytes() bytes, 16-byte aligned, else
 * DTROT_ERR_WORKSPACE) with the table, one kernel on `stream`.
 *
 * dtrot_gelu_and_mul_with_table computes exactly what dtrot_gelu_and_mul
 * computes, with the same arguments, layouts and errors, except that `table`
 * must hold a table written by dtrot_gelu_table_build and is only read: work
 * on other streams must be ordered after the build, the caller must not
 * modify the table, and out must not overlap it (DTROT_ERR_ALIAS).
 */
dtrot_status dtrot_gelu_table_build(void* table, int64_t table_bytes, void* stream);
dtrot_status dtrot_gelu_and_mul_with_table(const uint16_t* gate, int64_t s_gate,
                                           const uint16_t* up, int64_t s_up, uint16_t* out,
                                           int64_t s_out, int64_t T, int64_t F,
                                           const void* table, int64_t table_bytes,
                                           void* stream);

/*
 * Bytes of device workspace dtrot_gemm_gelu_and_mul needs (17408).
 */
int64_t dtrot_gemm_gelu_and_mul_workspace_bytes(void);

/*
 * GEGLU applied in the epilogue of the MLP's gate_up projection.   [P4] section 3
 *
 *   gate_up[t, n] = RN16(sum_c x[t, c] * w[n, c])      (the projection's bf16 output)
 *   out[t, f]     = RN16(gate_up[t, F + f] * RN16(RN32(gelu(gate_up[t, f]))))
 *
 * i.e. gate_up_proj followed by gelu_and_mul, without gate_up ever being
 * stored.  The sums are accumulated in fp32 on the tensor cores, in an order
 * this library does not specify, so gate_up may differ from the rounding of
 * the exact sum where that sum lies within the fp32 accumulation error of a
 * bf16 rounding boundary; inputs whose partial sums are all exact in fp32
 * give the exact result.
 *   x         bf16, (T, C) contiguous, read only.
 *   w         bf16, (2F, C) contiguous (an nn.Linear weight: rows [0, F) make
 *             gate, rows [F, 2F) make up), read only.
 *   out       bf16, (T, F), row stride s_out >= F, written; must not overlap
 *             x, w or the workspace (DTROT_ERR_ALIAS).
 *   gate_up   optional (NULL to skip): bf16, (T, 2F), row stride s_gate_up >=
 *             2F, receives the rounded projection (gate columns [0, F), up
 *             columns [F, 2F)), e.g. for a backward pass; must not overlap the
 *             other buffers (DTROT_ERR_ALIAS).
 *   Alignment: x, w, out (and gate_up) 16-byte aligned, C, F, s_out (and
 *   s_gate_up) multiples of 8 (else DTROT_ERR_ALIGN).  C must be > 0 and T, 2F < 2^31 (DTROT_ERR_SHAPE).
 *   workspace at least dtrot_gemm_gelu_and_mul_workspace_bytes() bytes,
 *             16-byte aligned (else DTROT_ERR_WORKSPACE), owned by the caller,
 *             contents on entry ignored: the call writes its activation table
 *             there (bytes [0, 17152)) and an error word (bytes [17152, 17156),
 *             zero unless a wait inside the kernel ran out of time (bits 1, 2,
 *             4) or the two CTAs of a pair were given different tensor-memory
 *             columns (bit 8); either would mean the GPU misbehaved, and the
 *             output is then not valid).  Calls that may run at the same time
 *             on the GPU must use different workspaces.
 * Two kernels are enqueued on `stream`: the activation table, then the GEMM
 * as its programmatic dependent.  For T > 128 the GEMM runs on pairs of CTAs
 * (clusters of two, tcgen05 cta_group::2 MMAs on 256-row tiles); for smaller T
 * on single CTAs.  Needs an sm_103 GPU (tcgen05 tensor cores).
 */
dtrot_status dtrot_gemm_gelu_and_mul(const uint16_t* x, int64_t T, int64_t C, const uint16_t* w,
                                     int64_t F, uint16_t* out, int64_t s_out, uint16_t* gate_up,
                                     int64_t s_gate_up, void* workspace, int64_t workspace_bytes,
                                     void* stream);

/*
 * The error word of a dtrot_gemm_gelu_and_mul call.     [P4] "why this is good",
 *                                                         item 2 (a fused path
 *                                                         whose failure is
 *                                                         detected, not silent)
 *
 * Enqueues on `stream` one copy of the 4-byte error word from `workspace`
 * (the workspace of an earlier call on the same stream) into *host_word.  The
 * word is there once the stream has reached the copy (cudaStreamSynchronize;
 * with pageable host memory the copy has completed when this returns).  0
 * means every wait of that call completed and the output is valid; otherwise
 * bit 1, 2 or 4 says a wait for a free stage, a loaded stage or an
 * accumulator ran out of time (about a second each, after which the kernel
 * stops waiting, drains what it issued, frees its tensor memory and returns),
 * and bit 8 that the two CTAs of a pair were given different tensor-memory
 * columns; the output of that call is then not valid.  Each call clears the
 * word before its GEMM starts, so it reports the last call on the workspace.
 *   workspace  as passed to dtrot_gemm_gelu_and_mul (NULL: DTROT_ERR_NULL; not
 *              16-byte aligned: DTROT_ERR_WORKSPACE).
 *   host_word  host memory, written (NULL: DTROT_ERR_NULL).
 * A failed copy returns DTROT_ERR_LAUNCH.
 */
dtrot_status dtrot_gemm_gelu_and_mul_error(const void* workspace, uint32_t* host_word,
                                           void* stream);

/*
 * Diagnostic run of dtrot_gemm_gelu_and_mul: the same arguments, validation
 * and launch, except that the TMA producer of every CTA (of both CTAs of a
 * pair) withholds the loads of its last pipeline stage, so the MMA thread's
 * bounded wait for that stage runs out after about a second.  The kernel
 * then records bit 2 in the error word, drains what it issued, frees its
 * tensor memory and returns; the output is not valid.  It exists to check,
 * on a real GPU, that a stalled pipeline is reported through
 * dtrot_gemm_gelu_and_mul_error instead of hanging the device; nothing on
 * the hot path calls it.
 */
dtrot_status dtrot_gemm_gelu_and_mul_withhold_last_stage(
    const uint16_t* x, int64_t T, int64_t C, const uint16_t* w, int64_t F, uint16_t* out,
    int64_t s_out, uint16_t* gate_up, int64_t s_gate_up, void* workspace,
    int64_t workspace_bytes, void* stream);

/*
 * GEGLU that allocates nothing and needs no workspace.  The paper has no
 * counterpart to this entry point; it is an addition of this library.
 *
 * Same arguments, result and error codes as dtrot_gelu_and_mul, without the
 * workspace (every argument is checked before the device is queried, so an
 * invalid call returns the same status from both).  For callers that cannot
 * obtain device memory of their own: for example code embedded in a host
 * framework that plans every device allocation ahead and hands the code only
 * its input and output tensors (an extra cudaMalloc would break the
 * framework's memory budget or is not permitted there), or a plain C caller
 * that has no allocator to draw from.  The 128 KB activation table lives in a
 * static device array inside this library instead; every GPU that loads the
 * library holds one such array until the process exits.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress, with the device current) and caches it with the
 *     device's current context; make that first call before any stream
 *     capture on the device.  After cudaDeviceReset the device gets a new
 *     context, in which the array may lie elsewhere: the next call sees the
 *     new context and looks the address up again (so that call, too, should
 *     come before any stream capture).
 *   - The table's size does not depend on T or F, so no valid size is too big
 *     for the array; if a library build's table ever exceeded the array, every
 *     call would return DTROT_ERR_WORKSPACE.  T and F are limited as for
 *     dtrot_gelu_and_mul (overflow: DTROT_ERR_SHAPE).
 *   - All calls on a device share the one array and each call rewrites it in
 *     full before reading it (nothing in it needs to start at zero).  Calls
 *     that overlap on the GPU (different streams with no ordering between
 *     them) race on it and may read a half-written table: order them, or use
 *     dtrot_gelu_and_mul with one workspace per stream.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
dtrot_status dtrot_gelu_and_mul_noalloc(const uint16_t* gate, int64_t s_gate, const uint16_t* up,
                                        int64_t s_up, uint16_t* out, int64_t s_out, int64_t T,
                                        int64_t F, void* stream);

/*
 * Token-wise RMSNorm fused with the residual add (Pre-Norm).   [P5]
 *
 * For every token row t:
 *   h[c]          = RN16(x[c] + residual[c])             (new residual stream)
 *   residual[c]  := h[c]
 *   out[c]        = RN16(h[c] * (mean_c(h^2) + eps)^(-1/2) * w[c])
 * Each row uses only its own features, so any subset of rows gives the same
 * values as the corresponding rows of the whole tensor.
 *   x         bf16, (T, C), row stride sx >= C, read only.
 *   residual  bf16, (T, C), row stride sr >= C, read and overwritten with h.
 *             x == residual with sx == sr is allowed (h = RN16(2x)); any other
 *             overlap of x and residual is DTROT_ERR_ALIAS.
 *   w         bf16, (C), read only; must not overlap residual or out.
 *   eps       finite and >= 0 (else DTROT_ERR_VALUE); added inside the root.
 *   out       bf16, (T, C), row stride so >= C, written; must not overlap x,
 *             residual or w.
 */
dtrot_status dtrot_rmsnorm_residual(const uint16_t* x, int64_t sx, uint16_t* residual,
                                    int64_t sr, const uint16_t* w, float eps,
                                    uint16_t* out, int64_t so, int64_t T, int64_t C,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DTROT_H */
