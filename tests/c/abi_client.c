/*
 * abi_client.c -- a plain C11 caller of the library's C ABI (test helper).
 *
 *   abi_client args            host-side argument checks only (no GPU needed)
 *   abi_client run DIR N R H   on the current GPU: reads DIR/{x,b1,b2}.f32 (N
 *                              floats each) and DIR/{lx,lr}.f32 (R*H floats),
 *                              DIR/{lw,lb}.f32 (H floats); runs
 *                              fused_add_relu_scale and
 *                              fused_residual_layernorm_gelu through cudaMalloc'd
 *                              buffers; writes DIR/y.f32 and DIR/lout.f32.
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "memory_bound.h"

#define CHECK(cond)                                                       \
    do {                                                                  \
        if (!(cond)) {                                                    \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
            return 1;                                                     \
        }                                                                 \
    } while (0)

static int args_mode(void)
{
    char *A = (char *)0x10000000, *B = (char *)0x20000000, *C = (char *)0x30000000,
         *D = (char *)0x40000000, *E = (char *)0x50000000;
    CHECK(mb_abi_version() == MB_ABI_VERSION);
    CHECK(strlen(mb_status_string(MB_ERR_OVERLAP)) > 0);
    CHECK(fused_add_relu_scale(A, B, C, D, 0, 0.5f, MB_F32, 0) == MB_OK);
    CHECK(fused_add_relu_scale(NULL, B, C, D, 8, 0.5f, MB_F32, 0) == MB_ERR_NULL);
    CHECK(fused_add_relu_scale(A, B, C, A + 4, 8, 0.5f, MB_F32, 0) == MB_ERR_OVERLAP);
    CHECK(fused_add_relu_scale(A + 1, B, C, D, 8, 0.5f, MB_BF16, 0) == MB_ERR_ALIGN);
    CHECK(fused_residual_layernorm_gelu(A, B, C, D, E, 4, MB_MAX_COLS + 1, 1e-5f, MB_F32, 0) ==
          MB_ERR_SHAPE);
    CHECK(fused_residual_layernorm_gelu(A, B, C, D, E, 4, 64, -1.0f, MB_F32, 0) == MB_ERR_VALUE);
    CHECK(fused_layernorm_act(A, NULL, C, D, E, NULL, 4, 64, 1e-5f, (mb_activation)7, MB_F32, 0) ==
          MB_ERR_VALUE);
    CHECK(fused_row_softmax(A, A, 4, 64, MB_F32, 0) == MB_ERR_OVERLAP);
    CHECK(fused_layernorm_act_ex(A, B, C, D, E, NULL, NULL, NULL, 4, 64, 1e-5f, MB_ACT_RELU,
                                 1.0f, 7u, 0u, MB_F32, 0) == MB_ERR_VALUE);
    CHECK(fused_layernorm_act_ex(A, B, C, D, E, NULL, (float *)(A + 8), NULL, 4, 64, 1e-5f,
                                 MB_ACT_RELU, 0.1f, 7u, 0u, MB_F32, 0) == MB_ERR_OVERLAP);
    CHECK(fused_add_relu_scale_bcast(A, B, C, D, 4, 64, 2, 1, 0.5f, MB_F32, 0) == MB_ERR_VALUE);
    CHECK(fused_add_relu_scale_bcast(A, B, C, A + 16, 4, 64, 1, 1, 0.5f, MB_F32, 0) ==
          MB_ERR_OVERLAP);
    CHECK(mb_set_row_path(MB_ROW_AUTO, 0, 0, 0) == MB_OK);
    printf("args ok\n");
    return 0;
}

static float *read_f32(const char *dir, const char *name, size_t n)
{
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    float *p = (float *)malloc(n * sizeof(float));
    size_t got = p ? fread(p, sizeof(float), n, f) : 0;
    fclose(f);
    if (got != n) { free(p); return NULL; }
    return p;
}

static int write_f32(const char *dir, const char *name, const float *p, size_t n)
{
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f) return 1;
    size_t put = fwrite(p, sizeof(float), n, f);
    fclose(f);
    return put != n;
}

static void *to_device(const float *h, size_t n)
{
    void *d = NULL;
    if (cudaMalloc(&d, n * sizeof(float)) != cudaSuccess) return NULL;
    if (cudaMemcpy(d, h, n * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
    return d;
}

static int run_mode(const char *dir, size_t n, size_t rows, size_t hidden)
{
    float *x = read_f32(dir, "x.f32", n), *b1 = read_f32(dir, "b1.f32", n),
          *b2 = read_f32(dir, "b2.f32", n);
    float *lx = read_f32(dir, "lx.f32", rows * hidden), *lr = read_f32(dir, "lr.f32", rows * hidden),
          *lw = read_f32(dir, "lw.f32", hidden), *lb = read_f32(dir, "lb.f32", hidden);
    CHECK(x && b1 && b2 && lx && lr && lw && lb);
    void *dx = to_device(x, n), *db1 = to_device(b1, n), *db2 = to_device(b2, n), *dy = NULL;
    void *dlx = to_device(lx, rows * hidden), *dlr = to_device(lr, rows * hidden),
         *dlw = to_device(lw, hidden), *dlb = to_device(lb, hidden), *dlo = NULL;
    CHECK(dx && db1 && db2 && dlx && dlr && dlw && dlb);
    CHECK(cudaMalloc(&dy, n * sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc(&dlo, rows * hidden * sizeof(float)) == cudaSuccess);
    cudaStream_t s;
    CHECK(cudaStreamCreate(&s) == cudaSuccess);
    mb_status st = fused_add_relu_scale(dx, db1, db2, dy, (int64_t)n, 0.5f, MB_F32, s);
    if (st != MB_OK) { fprintf(stderr, "%s\n", mb_status_string(st)); return 1; }
    st = fused_residual_layernorm_gelu(dlx, dlr, dlw, dlb, dlo, (int64_t)rows, (int64_t)hidden,
                                       1e-5f, MB_F32, s);
    if (st != MB_OK) { fprintf(stderr, "%s\n", mb_status_string(st)); return 1; }
    CHECK(cudaStreamSynchronize(s) == cudaSuccess);
    uint32_t flags = 0;
    CHECK(mb_device_error(&flags) == MB_OK && flags == 0);
    float *y = (float *)malloc(n * sizeof(float)), *lo = (float *)malloc(rows * hidden * sizeof(float));
    CHECK(y && lo);
    CHECK(cudaMemcpy(y, dy, n * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(lo, dlo, rows * hidden * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(write_f32(dir, "y.f32", y, n) == 0);
    CHECK(write_f32(dir, "lout.f32", lo, rows * hidden) == 0);
    printf("run ok\n");
    return 0;
}

int main(int argc, char **argv)
{
    if (argc >= 2 && strcmp(argv[1], "args") == 0) return args_mode();
    if (argc >= 6 && strcmp(argv[1], "run") == 0)
        return run_mode(argv[2], (size_t)atoll(argv[3]), (size_t)atoll(argv[4]),
                        (size_t)atoll(argv[5]));
    fprintf(stderr, "usage: abi_client args | run DIR N ROWS HIDDEN\n");
    return 2;
}
