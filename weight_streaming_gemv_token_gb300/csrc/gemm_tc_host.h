// Host interface of the tensor-core projection GEMM (gemm_tc.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "common.h"

namespace wsg {

// Widest output tile in N: boundaries between weights that share a launch
// on multiples of it suit both tile widths (128 and 64).
constexpr int kGemmTileN = 128;

// Tile width in N for an M x N product on `sms` SMs: 64 when 128-column
// tiles would leave SMs idle, else 128.
int gemm_tile_n(int M, int N, int sms);

// Tensor map (128 bytes at `out`, 64-byte aligned) of a bfloat16 operand
// [rows][K], row-major, in box_rows x 64-column swizzled tiles (activations:
// 128 rows; weights: the tile width in N, 128 or 64).
dec_status encode_gemm_operand(void* out, const void* base, long long rows, int K, int box_rows, std::string* err);

// C[:, col0 + n] (=, or += with accumulate) sum_k A[m][k] W[n][k] for
// m < M, n < N; maps from encode_gemm_operand (their contents are copied
// into the launch). W is nmaps (1 to 3) weight matrices side by side: rows
// [0, nb[0]) of W are mapsB[0], [nb[0], nb[1]) mapsB[1], the rest mapsB[2],
// each boundary a multiple of bn inside N (nb unused when nmaps == 1). bn is
// the tile width in N (64 or 128); the weight maps' boxes are bn rows. With
// mapA2 (not NULL) the activation operand is the sum of two bfloat16 matrices
// A + A2 (value and remainder), both multiplied into the same accumulator.
// Asynchronous on st.
dec_status launch_gemm_bf16(const void* mapA, const void* mapA2, const void* const* mapsB, const int* nb, int nmaps,
                            int bn, float* C, int ldc, int col0, int M, int N, int K, bool accumulate, uint32_t* err,
                            cudaStream_t st, std::string* where);

// Gate/up product of the chunk rows with SwiGLU fused: act / act2 [M][ld_act]
// (bfloat16 value and remainder) = silu(A . Wg^T) * (A . Wu^T), A = A + A2
// from mapA / mapA2, the gate and up weights [I][K] in 64-row boxes. The
// gate/up product itself is not written. Asynchronous on st.
dec_status launch_gemm_swiglu(const void* mapA, const void* mapA2, const void* mapGate64, const void* mapUp64,
                              uint16_t* act, uint16_t* act2, int ld_act, int M, int I, int K, uint32_t* err,
                              cudaStream_t st, std::string* where);

}  // namespace wsg
