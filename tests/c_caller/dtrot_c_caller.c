/*
 * A plain C caller of libdtrot: device buffers from the CUDA runtime, the ops
 * called through dtrot.h alone.  Reads its inputs from raw files written by
 * the test (little-endian bf16 bit patterns, fp32 angles) and writes the
 * outputs next to them; the test compares them with the oracle.
 *
 *   dtrot_c_caller DIR B S H D R T F C
 *
 * DIR holds freqs.f32 (S,B,1,R), x.bf16 (B,S,H,D), gate_up.bf16 (T,2F),
 * hx.bf16 and hr.bf16 (T,C), hw.bf16 (C).  Written: cos.bf16, sin.bf16,
 * rope.bf16, geglu.bf16, geglu_noalloc.bf16, residual.bf16, norm.bf16.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "dtrot.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) { fprintf(stderr, "cannot open %s\n", path); exit(2); }
    void* p = malloc(bytes ? bytes : 1);
    if (fread(p, 1, bytes, f) != bytes) { fprintf(stderr, "short read %s\n", path); exit(2); }
    fclose(f);
    return p;
}

static void write_file(const char* dir, const char* name, const void* p, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "wb");
    if (!f || fwrite(p, 1, bytes, f) != bytes) { fprintf(stderr, "cannot write %s\n", path); exit(2); }
    fclose(f);
}

#define CUDA(call)                                                              \
    do {                                                                        \
        cudaError_t e_ = (call);                                                \
        if (e_ != cudaSuccess) {                                                \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));         \
            exit(3);                                                            \
        }                                                                       \
    } while (0)

#define DTROT(call)                                                             \
    do {                                                                        \
        dtrot_status s_ = (call);                                               \
        if (s_ != DTROT_OK) {                                                   \
            fprintf(stderr, "%s: %s\n", #call, dtrot_status_str(s_));           \
            exit(4);                                                            \
        }                                                                       \
    } while (0)

static void* to_device(const void* h, size_t bytes) {
    void* d = NULL;
    CUDA(cudaMalloc(&d, bytes ? bytes : 16));
    CUDA(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice));
    return d;
}

static void from_device(const char* dir, const char* name, const void* d, size_t bytes) {
    void* h = malloc(bytes ? bytes : 1);
    CUDA(cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost));
    write_file(dir, name, h, bytes);
    free(h);
}

int main(int argc, char** argv) {
    if (argc != 10) {
        fprintf(stderr, "usage: %s DIR B S H D R T F C\n", argv[0]);
        return 1;
    }
    const char* dir = argv[1];
    const int64_t B = atoll(argv[2]), S = atoll(argv[3]), H = atoll(argv[4]), D = atoll(argv[5]);
    const int64_t R = atoll(argv[6]), T = atoll(argv[7]), F = atoll(argv[8]), C = atoll(argv[9]);
    const size_t nf = (size_t)(S * B * R), nx = (size_t)(B * S * H * D), nt = (size_t)(B * S * R);
    const size_t ng = (size_t)(T * 2 * F), no = (size_t)(T * F), nn = (size_t)(T * C);

    float* freqs = (float*)to_device(read_file(dir, "freqs.f32", nf * 4), nf * 4);
    uint16_t* x = (uint16_t*)to_device(read_file(dir, "x.bf16", nx * 2), nx * 2);
    uint16_t* gu = (uint16_t*)to_device(read_file(dir, "gate_up.bf16", ng * 2), ng * 2);
    uint16_t* hx = (uint16_t*)to_device(read_file(dir, "hx.bf16", nn * 2), nn * 2);
    uint16_t* hr = (uint16_t*)to_device(read_file(dir, "hr.bf16", nn * 2), nn * 2);
    uint16_t* hw = (uint16_t*)to_device(read_file(dir, "hw.bf16", (size_t)C * 2), (size_t)C * 2);
    uint16_t *cs, *sn, *out, *qo, *ko, *ff, *ff2, *y;
    void* ws;
    const int64_t wsb = dtrot_gelu_and_mul_workspace_bytes();
    CUDA(cudaMalloc((void**)&cs, nt * 2));
    CUDA(cudaMalloc((void**)&sn, nt * 2));
    CUDA(cudaMalloc((void**)&out, nx * 2));
    CUDA(cudaMalloc((void**)&qo, nx * 2));
    CUDA(cudaMalloc((void**)&ko, nx * 2));
    CUDA(cudaMalloc((void**)&ff, no * 2));
    CUDA(cudaMalloc((void**)&ff2, no * 2));
    CUDA(cudaMalloc((void**)&y, nn * 2));
    CUDA(cudaMalloc(&ws, (size_t)wsb));

    /* the default stream (NULL); contiguous layouts */
    DTROT(dtrot_rope_cos_sin_precompute(freqs, S, B, R, cs, sn, NULL));
    DTROT(dtrot_rope_rotate_half(x, B, S, H, D, S * H * D, H * D, D, cs, sn, R, out, S * H * D,
                                 H * D, D, NULL));
    /* q and k in one out-of-place launch; both read x (inputs may overlap) */
    DTROT(dtrot_rope_rotate_half_qk_out(x, H, S * H * D, H * D, D, x, H, S * H * D, H * D, D, B,
                                        S, D, cs, sn, NULL, R, qo, S * H * D, H * D, D, ko,
                                        S * H * D, H * D, D, NULL));
    DTROT(dtrot_gelu_and_mul(gu, 2 * F, gu + F, 2 * F, ff, F, T, F, ws, wsb, NULL));
    DTROT(dtrot_gelu_and_mul_noalloc(gu, 2 * F, gu + F, 2 * F, ff2, F, T, F, NULL));
    DTROT(dtrot_rmsnorm_residual(hx, C, hr, C, hw, 1e-6f, y, C, T, C, NULL));
    /* an invalid call returns its status and launches nothing */
    if (dtrot_rope_rotate_half(x, B, S, H, D, S * H * D, H * D, D, cs, sn, R + 1, out,
                               S * H * D, H * D, D, NULL) != DTROT_ERR_ROTDIM) {
        fprintf(stderr, "odd rot_dim was not rejected\n");
        return 5;
    }
    CUDA(cudaDeviceSynchronize());

    from_device(dir, "cos.bf16", cs, nt * 2);
    from_device(dir, "sin.bf16", sn, nt * 2);
    from_device(dir, "rope.bf16", out, nx * 2);
    from_device(dir, "rope_qk_q.bf16", qo, nx * 2);
    from_device(dir, "rope_qk_k.bf16", ko, nx * 2);
    from_device(dir, "geglu.bf16", ff, no * 2);
    from_device(dir, "geglu_noalloc.bf16", ff2, no * 2);
    from_device(dir, "residual.bf16", hr, nn * 2);
    from_device(dir, "norm.bf16", y, nn * 2);
    printf("dtrot_c_caller ok (library version %d)\n", dtrot_version());
    return 0;
}
