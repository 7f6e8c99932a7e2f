// Host interface of the tensor-core projection GEMM (gemm_tc.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "common.h"

namespace wsg {

// Boundaries between weights that share a launch are multiples of this
// (they suit 64- and 128-column tiles; 256-column tiles are used only where
// the boundaries are multiples of 256 too).
constexpr int kGemmTileN = 128;

// Tile width in N (256, 128 or 64) for an M x N x K product on `sms` SMs,
// one CTA per SM: among the widths that divide `align` (0: any), the one with
// the fewest operand bytes streamed by the busiest SM (waves of tiles x bytes
// per tile, plus a fixed cost per tile); split_a: the activation operand is a
// value + remainder pair.
int gemm_plan(int M, int N, int K, int sms, int align, bool split_a);

// Tensor map (128 bytes at `out`, 64-byte aligned) of a bfloat16 operand
// [rows][K], row-major, in box_rows x 64-column swizzled tiles (activations:
// 128 rows; weights: the tile width in N, or half of it for the gate/up
// pairs).
dec_status encode_gemm_operand(void* out, const void* base, long long rows, int K, int box_rows, std::string* err);

// C[:, col0 + n] (=, or += with accumulate) sum_k A[m][k] W[n][k] for
// m < M, n < N; maps from encode_gemm_operand (their contents are copied
// into the launch). W is nmaps (1 to 3) weight matrices side by side: rows
// [0, nb[0]) of W are mapsB[0], [nb[0], nb[1]) mapsB[1], the rest mapsB[2],
// each boundary a multiple of bn inside N (nb unused when nmaps == 1). bn is
// the tile width in N (64, 128 or 256); the weight maps' boxes are bn rows.
// With mapA2 (not NULL) the activation operand is the sum of two bfloat16
// matrices A + A2 (value and remainder), both multiplied into the same
// accumulator. Asynchronous on st.
dec_status launch_gemm_bf16(const void* mapA, const void* mapA2, const void* const* mapsB, const int* nb, int nmaps,
                            int bn, float* C, int ldc, int col0, int M, int N, int K, bool accumulate, uint32_t* err,
                            cudaStream_t st, std::string* where);

// Gate/up product of the chunk rows with SwiGLU fused: act / act2 [M][ld_act]
// (bfloat16 value and remainder) = silu(A . Wg^T) * (A . Wu^T), A = A + A2
// from mapA / mapA2, the gate and up weights [I][K] in bn/2-row boxes (bn 128
// or 256: a tile pairs bn/2 gate and bn/2 up outputs). The gate/up product
// itself is not written. Asynchronous on st.
dec_status launch_gemm_swiglu(const void* mapA, const void* mapA2, const void* mapGate, const void* mapUp, int bn,
                              uint16_t* act, uint16_t* act2, int ld_act, int M, int I, int K, uint32_t* err,
                              cudaStream_t st, std::string* where);

}  // namespace wsg
