/* Y[M, N] (bf16) = X[M, K] . W[N, K]^T with both operands quantised on the
 * device through the C ABI.  x, w: device bf16 buffers; y: device bf16 [M, N].
 * Link with -Lnvfp4_precision_02_b300 -lnvfp4 and the CUDA runtime. */
#include <cuda_runtime.h>
#include "nvfp4.h"

int fprop(const void *x, const void *w, void *y, int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    nvfp4_tensor qx = {0}, qw = {0};
    qx.rows = M; qx.cols = K;
    qw.rows = N; qw.cols = K;
    cudaMalloc(&qx.codes, (size_t)M * K / 2);
    cudaMalloc((void **)&qx.sf, nvfp4_sf_bytes(M, K));
    cudaMalloc((void **)&qx.amax, sizeof(float));
    cudaMalloc(&qw.codes, (size_t)N * K / 2);
    cudaMalloc((void **)&qw.sf, nvfp4_sf_bytes(N, K));
    cudaMalloc((void **)&qw.amax, sizeof(float));
    nvfp4_status st = nvfp4_quantize_1d(x, M, K, K, NVFP4_ROUND_RNE, 0, NULL, &qx, s);
    if (st == NVFP4_OK) st = nvfp4_quantize_2d(w, 1, N, K, K, NULL, &qw, NULL, NULL, s);
    if (st == NVFP4_OK) st = nvfp4_gemm(&qx, &qw, y, N, NVFP4_OUT_BF16, NULL, s);
    cudaStreamSynchronize(s);
    cudaFree(qx.codes); cudaFree(qx.sf); cudaFree(qx.amax);
    cudaFree(qw.codes); cudaFree(qw.sf); cudaFree(qw.amax);
    return st == NVFP4_OK ? 0 : (int)st;
}
