// Host side of the tensor-core projection GEMM (gemm_tc.cuh): launch helper
// used by the chunked prefill, and the standalone gemm_bf16 entry point.
#include <cuda.h>

#include "common.h"
#include "gemm_tc.cuh"
#include "gemm_tc_host.h"

namespace wsg {

static_assert(kGemmTileN == kTcBN, "the host's tile width is the kernel's widest");

template <int BN>
dec_status set_smem_once(int dev, std::string* where) {
  static bool ready[64] = {};
  if (ready[dev]) return DEC_OK;
  WSG_CUDA_TRY(where, cudaFuncSetAttribute(gemm_bf16_tc_kernel<TC_STORE, false, BN>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(tc_smem_bytes<false, BN>())));
  WSG_CUDA_TRY(where, cudaFuncSetAttribute(gemm_bf16_tc_kernel<TC_ADD, false, BN>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(tc_smem_bytes<false, BN>())));
  WSG_CUDA_TRY(where, cudaFuncSetAttribute(gemm_bf16_tc_kernel<TC_STORE, true, BN>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(tc_smem_bytes<true, BN>())));
  WSG_CUDA_TRY(where, cudaFuncSetAttribute(gemm_bf16_tc_kernel<TC_ADD, true, BN>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(tc_smem_bytes<true, BN>())));
  if constexpr (BN == 128)
    WSG_CUDA_TRY(where, cudaFuncSetAttribute(gemm_bf16_tc_kernel<TC_SWIGLU, true, BN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(tc_smem_bytes<true, BN>())));
  ready[dev] = true;
  return DEC_OK;
}

template <int BN>
void launch_tc(bool split, bool accumulate, dim3 grid, const CUtensorMap& ma, const CUtensorMap& ma2,
               const CUtensorMap& mb0, const CUtensorMap& mb1, const CUtensorMap& mb2, const TcArgs& a,
               cudaStream_t st) {
  if (split) {
    if (accumulate)
      gemm_bf16_tc_kernel<TC_ADD, true, BN><<<grid, kTcThreads, tc_smem_bytes<true, BN>(), st>>>(ma, ma2, mb0, mb1, mb2, a);
    else
      gemm_bf16_tc_kernel<TC_STORE, true, BN><<<grid, kTcThreads, tc_smem_bytes<true, BN>(), st>>>(ma, ma2, mb0, mb1, mb2,
                                                                                                    a);
  } else {
    if (accumulate)
      gemm_bf16_tc_kernel<TC_ADD, false, BN><<<grid, kTcThreads, tc_smem_bytes<false, BN>(), st>>>(ma, ma2, mb0, mb1, mb2,
                                                                                                    a);
    else
      gemm_bf16_tc_kernel<TC_STORE, false, BN><<<grid, kTcThreads, tc_smem_bytes<false, BN>(), st>>>(ma, ma2, mb0, mb1,
                                                                                                      mb2, a);
  }
}

dec_status launch_gemm_swiglu(const void* mapA, const void* mapA2, const void* mapGate64, const void* mapUp64,
                              uint16_t* act, uint16_t* act2, int ld_act, int M, int I, int K, uint32_t* err,
                              cudaStream_t st, std::string* where) {
  DeviceInfo di;
  dec_status s = device_info(&di, where);
  if (s != DEC_OK) return s;
  if ((s = set_smem_once<128>(di.device, where)) != DEC_OK) return s;
  TcArgs a;
  a.C = nullptr;
  a.ldc = 0;
  a.col0 = 0;
  a.M = M;
  a.N = 2 * I;
  a.K = K;
  a.nb1 = a.nb2 = 2 * I;
  a.act = act;
  a.act2 = act2;
  a.ld_act = ld_act;
  a.err = err;
  // 64 outputs (128 accumulator columns) per tile; persistent, one CTA per SM
  const long long tiles = static_cast<long long>((I + 63) / 64) * ((M + kTcBM - 1) / kTcBM);
  const dim3 grid(static_cast<unsigned>(tiles < di.sms ? tiles : di.sms));
  const CUtensorMap& ma = *static_cast<const CUtensorMap*>(mapA);
  const CUtensorMap& ma2 = *static_cast<const CUtensorMap*>(mapA2);
  const CUtensorMap& mg = *static_cast<const CUtensorMap*>(mapGate64);
  const CUtensorMap& mu = *static_cast<const CUtensorMap*>(mapUp64);
  gemm_bf16_tc_kernel<TC_SWIGLU, true, 128><<<grid, kTcThreads, tc_smem_bytes<true, 128>(), st>>>(ma, ma2, mg, mu, mg,
                                                                                                   a);
  WSG_CUDA_TRY(where, cudaGetLastError());
  return DEC_OK;
}

int gemm_tile_n(int M, int N, int sms) {
  const long long tiles = static_cast<long long>((N + kTcBN - 1) / kTcBN) * ((M + kTcBM - 1) / kTcBM);
  return tiles < sms ? 64 : 128;
}

dec_status launch_gemm_bf16(const void* mapA, const void* mapA2, const void* const* mapsB, const int* nb, int nmaps,
                            int bn, float* C, int ldc, int col0, int M, int N, int K, bool accumulate, uint32_t* err,
                            cudaStream_t st, std::string* where) {
  if (bn != 64 && bn != 128) return fail(where, DEC_EINVAL, "gemm: tile width %d", bn);
  if (nmaps < 1 || nmaps > 3) return fail(where, DEC_EINVAL, "gemm: %d weight maps", nmaps);
  for (int i = 1; i < nmaps; ++i)
    if (nb[i - 1] % bn || nb[i - 1] <= 0 || nb[i - 1] >= N || (i > 1 && nb[i - 1] <= nb[i - 2]))
      return fail(where, DEC_EINVAL, "gemm: weight boundary %d is not a tile boundary inside N", nb[i - 1]);
  DeviceInfo di;
  dec_status s = device_info(&di, where);
  if (s != DEC_OK) return s;
  if ((s = bn == 64 ? set_smem_once<64>(di.device, where) : set_smem_once<128>(di.device, where)) != DEC_OK) return s;
  TcArgs a;
  a.C = C;
  a.ldc = ldc;
  a.col0 = col0;
  a.M = M;
  a.N = N;
  a.K = K;
  a.nb1 = nmaps > 1 ? nb[0] : N;
  a.nb2 = nmaps > 2 ? nb[1] : N;
  a.err = err;
  // persistent: one CTA per SM (fewer when there are fewer tiles)
  const long long tiles = static_cast<long long>((N + bn - 1) / bn) * ((M + kTcBM - 1) / kTcBM);
  const dim3 grid(static_cast<unsigned>(tiles < di.sms ? tiles : di.sms));
  const CUtensorMap& ma = *static_cast<const CUtensorMap*>(mapA);
  const CUtensorMap& ma2 = *static_cast<const CUtensorMap*>(mapA2 ? mapA2 : mapA);
  const CUtensorMap& mb0 = *static_cast<const CUtensorMap*>(mapsB[0]);
  const CUtensorMap& mb1 = *static_cast<const CUtensorMap*>(mapsB[nmaps > 1 ? 1 : 0]);
  const CUtensorMap& mb2 = *static_cast<const CUtensorMap*>(mapsB[nmaps > 2 ? 2 : 0]);
  if (bn == 64)
    launch_tc<64>(mapA2 != nullptr, accumulate, grid, ma, ma2, mb0, mb1, mb2, a, st);
  else
    launch_tc<128>(mapA2 != nullptr, accumulate, grid, ma, ma2, mb0, mb1, mb2, a, st);
  WSG_CUDA_TRY(where, cudaGetLastError());
  return DEC_OK;
}

dec_status encode_gemm_operand(void* out, const void* base, long long rows, int K, int box_rows, std::string* err) {
  return encode_map_2d(out, base, rows, K, 2, kTcBK, box_rows, true, err);
}

}  // namespace wsg

using namespace wsg;

extern "C" dec_status gemm_bf16(const uint16_t* d_A, const uint16_t* d_W, float* d_C, int32_t M, int32_t N, int32_t K,
                                int32_t ldc, int32_t accumulate, void* stream) {
  if (!d_A || !d_W || !d_C) return fail(nullptr, DEC_EINVAL, "gemm_bf16: NULL pointer");
  if (M < 1 || N < 1 || K < 1) return fail(nullptr, DEC_EINVAL, "gemm_bf16: M, N, K must be >= 1");
  if (K % 8) return fail(nullptr, DEC_EINVAL, "gemm_bf16: K must be a multiple of 8 (16-byte rows)");
  if (ldc < N) return fail(nullptr, DEC_EINVAL, "gemm_bf16: ldc %d < N %d", ldc, N);
  if (!aligned16(d_A) || !aligned16(d_W)) return fail(nullptr, DEC_EINVAL, "gemm_bf16: A and W must be 16-byte aligned");
  DeviceInfo di;
  dec_status s = device_info(&di, nullptr);
  if (s != DEC_OK) return s;
  alignas(64) unsigned char ma[128], mb[128];
  const int bn = gemm_tile_n(M, N, di.sms);
  if ((s = encode_gemm_operand(ma, d_A, M, K, kTcBM, nullptr)) != DEC_OK) return s;
  if ((s = encode_gemm_operand(mb, d_W, N, K, bn, nullptr)) != DEC_OK) return s;
  const void* mbs[1] = {mb};
  return launch_gemm_bf16(ma, nullptr, mbs, nullptr, 1, bn, d_C, ldc, 0, M, N, K, accumulate != 0,
                          di.err, static_cast<cudaStream_t>(stream), nullptr);
}
