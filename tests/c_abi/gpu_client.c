/* A plain C client of the W8A8 linear on the GPU: CUDA runtime and the
 * library's header only, no Python.  Reads X [M][K], W [N][K] and bias [N]
 * as bf16 bit patterns from a file, runs w8a8_quantize_weight,
 * w8a8_pack_weight and w8a8_linear on the current device, and writes Y [M][N]
 * (bf16 bits) to a second file.  Usage: gpu_client in.bin out.bin
 * (in.bin: int64 M, K, N, then the three arrays). */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "w8a8.h"

#define CHECK_CUDA(x) do { if ((x) != cudaSuccess) { fprintf(stderr, "CUDA error at line %d\n", __LINE__); return 2; } } while (0)
#define CHECK_W8A8(x) do { w8a8_status st_ = (x); if (st_ != W8A8_OK) { fprintf(stderr, "%s: %s\n", #x, w8a8_status_str(st_)); return 3; } } while (0)

int main(int argc, char** argv)
{
    if (argc != 3) return 1;
    FILE* f = fopen(argv[1], "rb");
    if (!f) return 1;
    int64_t dims[3];
    if (fread(dims, sizeof dims, 1, f) != 1) return 1;
    const int64_t M = dims[0], K = dims[1], N = dims[2];
    uint16_t* hX = malloc((size_t)(M * K) * 2);
    uint16_t* hW = malloc((size_t)(N * K) * 2);
    uint16_t* hb = malloc((size_t)N * 2);
    uint16_t* hY = malloc((size_t)(M * N) * 2);
    if (!hX || !hW || !hb || !hY) return 1;
    if (fread(hX, 2, (size_t)(M * K), f) != (size_t)(M * K) || fread(hW, 2, (size_t)(N * K), f) != (size_t)(N * K) ||
        fread(hb, 2, (size_t)N, f) != (size_t)N)
        return 1;
    fclose(f);

    void *X, *W, *b, *Y, *ws;
    int8_t* Wq;
    float* sw;
    uint16_t* Wp;
    const size_t ws_bytes = w8a8_linear_workspace_bytes(M, N, K);
    CHECK_CUDA(cudaMalloc(&X, (size_t)(M * K) * 2));
    CHECK_CUDA(cudaMalloc(&W, (size_t)(N * K) * 2));
    CHECK_CUDA(cudaMalloc(&b, (size_t)N * 2));
    CHECK_CUDA(cudaMalloc(&Y, (size_t)(M * N) * 2));
    CHECK_CUDA(cudaMalloc((void**)&Wq, (size_t)(N * K)));
    CHECK_CUDA(cudaMalloc((void**)&sw, (size_t)N * 4));
    CHECK_CUDA(cudaMalloc((void**)&Wp, (size_t)(N * K) * 2));
    CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
    CHECK_CUDA(cudaMemcpy(X, hX, (size_t)(M * K) * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(W, hW, (size_t)(N * K) * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(b, hb, (size_t)N * 2, cudaMemcpyHostToDevice));

    CHECK_W8A8(w8a8_quantize_weight(W, W8A8_BF16, N, K, Wq, sw, NULL));
    CHECK_W8A8(w8a8_pack_weight(Wq, N, K, Wp, NULL));
    CHECK_W8A8(w8a8_linear(X, W8A8_BF16, M, K, Wp, sw, N, b, W8A8_BF16, (uint16_t*)Y, ws, ws_bytes, NULL));
    uint32_t bits = 0;
    CHECK_W8A8(w8a8_read_status(ws, NULL, &bits));
    CHECK_CUDA(cudaMemcpy(hY, Y, (size_t)(M * N) * 2, cudaMemcpyDeviceToHost));

    FILE* g = fopen(argv[2], "wb");
    if (!g || fwrite(hY, 2, (size_t)(M * N), g) != (size_t)(M * N)) return 1;
    fclose(g);
    cudaFree(X); cudaFree(W); cudaFree(b); cudaFree(Y); cudaFree(Wq); cudaFree(sw); cudaFree(Wp); cudaFree(ws);
    free(hX); free(hW); free(hb); free(hY);
    return 0;
}
