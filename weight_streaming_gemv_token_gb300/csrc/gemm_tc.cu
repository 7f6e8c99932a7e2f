// Host side of the tensor-core projection GEMM (gemm_tc.cuh): launch helper
// used by the chunked prefill, and the standalone gemm_bf16 entry point.
#include <cuda.h>

#include "common.h"
#include "gemm_tc.cuh"
#include "gemm_tc_host.h"

namespace wsg {

static_assert(kTcBN % kGemmTileN == 0, "the weight boundaries suit the narrower tiles");

template <int EPI, bool SPLIT, int BN>
dec_status lift_smem(std::string* where) {
  WSG_CUDA_TRY(where, cudaFuncSetAttribute(gemm_bf16_tc_kernel<EPI, SPLIT, BN>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(tc_smem_bytes<SPLIT, BN>())));
  return DEC_OK;
}

template <int BN>
dec_status set_smem_once(int dev, std::string* where) {
  static bool ready[64] = {};
  if (ready[dev]) return DEC_OK;
  dec_status s;
  if ((s = lift_smem<TC_STORE, false, BN>(where)) != DEC_OK) return s;
  if ((s = lift_smem<TC_ADD, false, BN>(where)) != DEC_OK) return s;
  if ((s = lift_smem<TC_STORE, true, BN>(where)) != DEC_OK) return s;
  if ((s = lift_smem<TC_ADD, true, BN>(where)) != DEC_OK) return s;
  if constexpr (BN >= 128)
    if ((s = lift_smem<TC_SWIGLU, true, BN>(where)) != DEC_OK) return s;
  ready[dev] = true;
  return DEC_OK;
}

dec_status set_smem_all(int dev, std::string* where) {
  dec_status s;
  if ((s = set_smem_once<64>(dev, where)) != DEC_OK) return s;
  if ((s = set_smem_once<128>(dev, where)) != DEC_OK) return s;
  return set_smem_once<256>(dev, where);
}

// A launch may begin (set-up, weight tiles) while the previous kernel of the
// stream finishes: the kernel waits for it before its activation reads and C.
template <int EPI, bool SPLIT, int BN>
cudaError_t launch_one(dim3 grid, const CUtensorMap& ma, const CUtensorMap& ma2, const CUtensorMap& mb0,
                       const CUtensorMap& mb1, const CUtensorMap& mb2, const TcArgs& a, cudaStream_t st) {
  return launch_k(gemm_bf16_tc_kernel<EPI, SPLIT, BN>, grid, dim3(kTcThreads), tc_smem_bytes<SPLIT, BN>(), st, true,
                  ma, ma2, mb0, mb1, mb2, a);
}

template <int BN>
cudaError_t launch_tc(bool split, bool accumulate, dim3 grid, const CUtensorMap& ma, const CUtensorMap& ma2,
                      const CUtensorMap& mb0, const CUtensorMap& mb1, const CUtensorMap& mb2, const TcArgs& a,
                      cudaStream_t st) {
  if (split)
    return accumulate ? launch_one<TC_ADD, true, BN>(grid, ma, ma2, mb0, mb1, mb2, a, st)
                      : launch_one<TC_STORE, true, BN>(grid, ma, ma2, mb0, mb1, mb2, a, st);
  return accumulate ? launch_one<TC_ADD, false, BN>(grid, ma, ma2, mb0, mb1, mb2, a, st)
                    : launch_one<TC_STORE, false, BN>(grid, ma, ma2, mb0, mb1, mb2, a, st);
}

dec_status launch_gemm_swiglu(const void* mapA, const void* mapA2, const void* mapGate, const void* mapUp, int bn,
                              uint16_t* act, uint16_t* act2, int ld_act, int M, int I, int K, uint32_t* err,
                              cudaStream_t st, std::string* where) {
  if (bn != 128 && bn != 256) return fail(where, DEC_EINVAL, "gemm_swiglu: tile width %d", bn);
  DeviceInfo di;
  dec_status s = device_info(&di, where);
  if (s != DEC_OK) return s;
  if ((s = set_smem_all(di.device, where)) != DEC_OK) return s;
  TcArgs a{};
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
  // bn/2 outputs (bn accumulator columns) per tile; persistent, one CTA per SM
  const long long tiles = static_cast<long long>((I + bn / 2 - 1) / (bn / 2)) * ((M + kTcBM - 1) / kTcBM);
  const dim3 grid(static_cast<unsigned>(tiles < di.sms ? tiles : di.sms));
  const CUtensorMap& ma = *static_cast<const CUtensorMap*>(mapA);
  const CUtensorMap& ma2 = *static_cast<const CUtensorMap*>(mapA2);
  const CUtensorMap& mg = *static_cast<const CUtensorMap*>(mapGate);
  const CUtensorMap& mu = *static_cast<const CUtensorMap*>(mapUp);
  const cudaError_t e = bn == 256 ? launch_one<TC_SWIGLU, true, 256>(grid, ma, ma2, mg, mu, mg, a, st)
                                  : launch_one<TC_SWIGLU, true, 128>(grid, ma, ma2, mg, mu, mg, a, st);
  WSG_CUDA_TRY(where, e);
  return DEC_OK;
}

int gemm_plan(int M, int N, int K, int sms, int align, bool split_a) {
  const int KB = (K + kTcBK - 1) / kTcBK;
  const long long mt = (M + kTcBM - 1) / kTcBM;
  int best = 128;
  double best_cost = -1.0;
  for (int bn : {256, 128, 64}) {
    if (align > 0 && align % bn) continue;
    const long long tiles = mt * ((N + bn - 1) / bn);
    const long long waves = (tiles + sms - 1) / sms;
    // bytes per tile: A (1 or 2 bfloat16 parts) and W rows over every K
    // block, plus a fixed cost (pipeline fill, epilogue) of ~64 KB; a ring of
    // three stages (the widest tiles with a value + remainder operand) hides
    // less load latency than four: measured ~1.2x per byte
    const double tile = (static_cast<double>(kTcBM) * (split_a ? 2 : 1) + bn) * kTcBK * 2.0 * KB + 65536.0;
    const bool three = split_a ? tc_stages<true, 256>() == 3 && bn == 256 : tc_stages<false, 256>() == 3 && bn == 256;
    const double cost = static_cast<double>(waves) * tile * (three ? 1.2 : 1.0);
    if (best_cost < 0.0 || cost < best_cost * 0.999) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

dec_status launch_gemm_bf16(const void* mapA, const void* mapA2, const void* const* mapsB, const int* nb, int nmaps,
                            int bn, float* C, int ldc, int col0, int M, int N, int K, bool accumulate, uint32_t* err,
                            cudaStream_t st, std::string* where) {
  if (bn != 64 && bn != 128 && bn != 256) return fail(where, DEC_EINVAL, "gemm: tile width %d", bn);
  if (nmaps < 1 || nmaps > 3) return fail(where, DEC_EINVAL, "gemm: %d weight maps", nmaps);
  for (int i = 1; i < nmaps; ++i)
    if (nb[i - 1] % bn || nb[i - 1] <= 0 || nb[i - 1] >= N || (i > 1 && nb[i - 1] <= nb[i - 2]))
      return fail(where, DEC_EINVAL, "gemm: weight boundary %d is not a tile boundary inside N", nb[i - 1]);
  DeviceInfo di;
  dec_status s = device_info(&di, where);
  if (s != DEC_OK) return s;
  if ((s = set_smem_all(di.device, where)) != DEC_OK) return s;
  TcArgs a{};
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
  const bool sa = mapA2 != nullptr;
  const cudaError_t e = bn == 64    ? launch_tc<64>(sa, accumulate, grid, ma, ma2, mb0, mb1, mb2, a, st)
                        : bn == 128 ? launch_tc<128>(sa, accumulate, grid, ma, ma2, mb0, mb1, mb2, a, st)
                                    : launch_tc<256>(sa, accumulate, grid, ma, ma2, mb0, mb1, mb2, a, st);
  WSG_CUDA_TRY(where, e);
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
  const int bn = gemm_plan(M, N, K, di.sms, 0, false);
  if ((s = encode_gemm_operand(ma, d_A, M, K, kTcBM, nullptr)) != DEC_OK) return s;
  if ((s = encode_gemm_operand(mb, d_W, N, K, bn, nullptr)) != DEC_OK) return s;
  const void* mbs[1] = {mb};
  return launch_gemm_bf16(ma, nullptr, mbs, nullptr, 1, bn, d_C, ldc, 0, M, N, K, accumulate != 0, di.err,
                          static_cast<cudaStream_t>(stream), nullptr);
}
