/*
 * A plain C (C11) client of the library's C ABI.  It reads x, w and b (raw little-endian
 * fp32 files), runs fc_conv3x3_act_pool (erf-GELU, padding 0, NCHW) on the current
 * CUDA device and writes y [N][Cout] as raw fp32.  It needs nothing but include/fc.h,
 * the shared library and the CUDA runtime: no C++, no torch.
 *
 *   c_abi_client N Cin H W Cout x.bin w.bin b.bin y.bin
 *
 * Exit status: 0 on success, 2 for usage or file errors, 3 for CUDA runtime errors,
 * 10 + fc_status for a library error.
 */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "fc.h"

static void* read_all(const char* path, size_t bytes)
{
    FILE* f = fopen(path, "rb");
    void* p = malloc(bytes > 0 ? bytes : 1);
    size_t got = 0;
    if (f != NULL && p != NULL) got = fread(p, 1, bytes, f);
    if (f != NULL) fclose(f);
    if (p == NULL || got != bytes) {
        free(p);
        return NULL;
    }
    return p;
}

int main(int argc, char** argv)
{
    if (argc != 10) {
        fprintf(stderr, "usage: %s N Cin H W Cout x.bin w.bin b.bin y.bin\n", argv[0]);
        return 2;
    }
    const int N = atoi(argv[1]), Cin = atoi(argv[2]), H = atoi(argv[3]), W = atoi(argv[4]), Cout = atoi(argv[5]);
    if (N < 1 || Cin < 1 || H < 1 || W < 1 || Cout < 1) return 2;
    const size_t nx = (size_t)N * Cin * H * W, nw = (size_t)Cout * Cin * 9, nb = (size_t)Cout, ny = (size_t)N * Cout;
    float* hx = (float*)read_all(argv[6], nx * sizeof(float));
    float* hw = (float*)read_all(argv[7], nw * sizeof(float));
    float* hb = (float*)read_all(argv[8], nb * sizeof(float));
    float* hy = (float*)malloc(ny * sizeof(float));
    if (hx == NULL || hw == NULL || hb == NULL || hy == NULL) return 2;

    float *dx = NULL, *dw = NULL, *db = NULL, *dy = NULL;
    void* ws = NULL;
    const size_t ws_bytes = fc_workspace_bytes(FC_OP_CONV3X3_ACT_POOL, N, Cin, H, W, Cout, FC_F32);
    if (cudaMalloc((void**)&dx, nx * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void**)&dw, nw * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void**)&db, nb * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void**)&dy, ny * sizeof(float)) != cudaSuccess ||
        (ws_bytes > 0 && cudaMalloc(&ws, ws_bytes) != cudaSuccess))
        return 3;
    if (cudaMemcpy(dx, hx, nx * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(dw, hw, nw * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(db, hb, nb * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess)
        return 3;

    fc_status st = fc_conv3x3_act_pool(dx, dw, db, dy, N, Cin, H, W, Cout, FC_F32, FC_ACT_GELU_ERF, ws, ws_bytes,
                                       (fc_stream_t)0);
    if (st != FC_OK) {
        fprintf(stderr, "fc_conv3x3_act_pool: %s\n", fc_status_string(st));
        return 10 + (int)st;
    }
    st = fc_device_status(1);   /* synchronizes; a kernel's bounded wait that ran out shows here */
    if (st != FC_OK) {
        fprintf(stderr, "device status: %s\n", fc_status_string(st));
        return 10 + (int)st;
    }
    if (cudaMemcpy(hy, dy, ny * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess) return 3;

    FILE* f = fopen(argv[9], "wb");
    if (f == NULL || fwrite(hy, sizeof(float), ny, f) != ny) return 2;
    fclose(f);
    printf("fc_version %d: y[0][0] = %.7g\n", fc_version(), (double)hy[0]);
    cudaFree(dx);
    cudaFree(dw);
    cudaFree(db);
    cudaFree(dy);
    cudaFree(ws);
    free(hx);
    free(hw);
    free(hb);
    free(hy);
    return 0;
}
