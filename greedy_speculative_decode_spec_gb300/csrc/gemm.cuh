// gemm.cuh -- internal entry of the skinny GEMM shared by the LM head and the MTP fc.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

namespace spec {

// out[m][n] = bf16( sum_k A[m][k] * W[n][k] ), fp32 accumulation; A bf16 [M][K],
// W bf16 [N][K], out bf16 [M][N]. Workspace of gemm_store_ws_bytes(M, N, K) bytes.
size_t gemm_store_ws_bytes(int M, int N, int K);
int gemm_store_bf16(const void *A, const void *W, int M, int N, int K, void *out, void *ws, size_t ws_bytes,
                    cudaStream_t s);

}  // namespace spec
