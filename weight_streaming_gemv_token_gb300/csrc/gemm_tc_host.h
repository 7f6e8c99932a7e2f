// Host interface of the tensor-core projection GEMM (gemm_tc.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "common.h"

namespace wsg {

// Tensor map (128 bytes at `out`, 64-byte aligned) of a bfloat16 operand
// [rows][K], row-major, in the GEMM's 128-row x 64-column swizzled tiles.
dec_status encode_gemm_operand(void* out, const void* base, long long rows, int K, std::string* err);

// C[:, col0 + n] (=, or += with accumulate) sum_k A[m][k] W[n][k] for
// m < M, n < N; maps from encode_gemm_operand (their contents are copied
// into the launch). With mapA2 (not NULL) the activation operand is the sum
// of two bfloat16 matrices A + A2 (value and remainder), both multiplied into
// the same accumulator. Asynchronous on st.
dec_status launch_gemm_bf16(const void* mapA, const void* mapA2, const void* mapB, float* C, int ldc, int col0, int M,
                            int N, int K, bool accumulate, uint32_t* err, cudaStream_t st, std::string* where);

}  // namespace wsg
