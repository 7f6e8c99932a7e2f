// Host interface of the tensor-core projection GEMM (gemm_tc.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "common.h"

namespace wsg {

// Width in N of one output tile: the boundaries between weights that share a
// launch must be multiples of it.
constexpr int kGemmTileN = 128;

// Tensor map (128 bytes at `out`, 64-byte aligned) of a bfloat16 operand
// [rows][K], row-major, in the GEMM's 128-row x 64-column swizzled tiles.
dec_status encode_gemm_operand(void* out, const void* base, long long rows, int K, std::string* err);

// C[:, col0 + n] (=, or += with accumulate) sum_k A[m][k] W[n][k] for
// m < M, n < N; maps from encode_gemm_operand (their contents are copied
// into the launch). W is nmaps (1 to 3) weight matrices side by side: rows
// [0, nb[0]) of W are mapsB[0], [nb[0], nb[1]) mapsB[1], the rest mapsB[2],
// each boundary a multiple of 128 inside N (nb unused when nmaps == 1). With
// mapA2 (not NULL) the activation operand is the sum of two bfloat16 matrices
// A + A2 (value and remainder), both multiplied into the same accumulator.
// Asynchronous on st.
dec_status launch_gemm_bf16(const void* mapA, const void* mapA2, const void* const* mapsB, const int* nb, int nmaps,
                            float* C, int ldc, int col0, int M, int N, int K, bool accumulate, uint32_t* err,
                            cudaStream_t st, std::string* where);

}  // namespace wsg
