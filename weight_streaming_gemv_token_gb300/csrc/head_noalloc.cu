// greedy_head_noalloc: the greedy head (final RMSNorm, tied vocabulary GEMV,
// lowest-ID argmax) for callers that cannot allocate device memory: code
// running inside a host framework that owns every device allocation, or a
// latency-critical path that must not call cudaMalloc (which can synchronise
// the device) in the middle of a generation loop.
//
// It runs the same kernel as the staged engine's head (gemv_stream_kernel with
// the RMSNorm prologue and the logits + two-pass argmax epilogue). That kernel
// needs scratch for the per-CTA argmax partials, the last-CTA counter and a
// position word; here the scratch is a file-scope device array instead of a
// caller-provided workspace.
#include <mutex>

#include "common.h"
#include "gemv_stream.cuh"

namespace wsg {
namespace {

constexpr int kNW = 8, kNSMAX = 8, kRING = 12288, kSEGMAX = 4096;

// Scratch layout: argmax partial values [kMaxCtas] float, partial indices
// [kMaxCtas] int32, then counter, position word and two token slots. Device
// errors go to the context-free error word (gemv_device_errors).
constexpr int kMaxCtas = 1024;
constexpr size_t kOffIdx = sizeof(float) * kMaxCtas;
constexpr size_t kOffCounter = kOffIdx + sizeof(int32_t) * kMaxCtas;
constexpr size_t kOffCtrl = kOffCounter + 4;
constexpr size_t kOffTok = kOffCtrl + 4;
constexpr size_t kScratchBytes = ((kOffTok + 8) + 255) / 256 * 256;  // 8448 bytes per device

static __device__ __align__(256) unsigned char g_head_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  unsigned char* scratch = nullptr;  // device address of g_head_scratch
  size_t smem_limit[2] = {0, 0};     // dynamic shared memory lifted for the float32 / bfloat16 kernel
  bool ready = false;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

}  // namespace
}  // namespace wsg

using namespace wsg;

extern "C" dec_status greedy_head_noalloc(int32_t wdtype, const void* d_embed, const float* d_h, const float* d_gain,
                                          float eps, int32_t vocab, int32_t hidden, float* d_logits,
                                          int32_t* d_token, void* stream) {
  if (wdtype != DEC_F32 && wdtype != DEC_BF16)
    return fail(nullptr, DEC_EINVAL, "greedy_head_noalloc: wdtype %d", wdtype);
  if (vocab < 1 || hidden < 1) return fail(nullptr, DEC_EINVAL, "greedy_head_noalloc: vocab and hidden must be >= 1");
  if (!d_embed || !d_h || !d_gain || !d_token) return fail(nullptr, DEC_EINVAL, "greedy_head_noalloc: NULL pointer");
  const int elem = wdtype == DEC_F32 ? 4 : 2;
  const long long row_bytes = static_cast<long long>(hidden) * elem;
  if (row_bytes % 16 || !aligned16(d_embed))
    return fail(nullptr, DEC_EINVAL,
                "greedy_head_noalloc: embedding must be 16-byte aligned with rows a multiple of 16 bytes");
  DeviceInfo di;
  dec_status st = device_info(&di, nullptr);
  if (st != DEC_OK) return st;

  // One-time set-up per device (on the first call with that device current),
  // under a lock so that first calls from several host threads are safe: the
  // scratch's device address and the kernels' shared-memory limits.
  if (di.device < 0 || di.device >= kMaxDevices)
    return fail(nullptr, DEC_EDEVICE, "greedy_head_noalloc: device ordinal %d out of range", di.device);
  using KernT = void (*)(GemvArgs);
  const KernT kerns[2] = {gemv_stream_kernel<float, float, PRO_NORM, EPI_ARGMAX, kNW, kNSMAX, kRING>,
                          gemv_stream_kernel<uint16_t, float, PRO_NORM, EPI_ARGMAX, kNW, kNSMAX, kRING>};
  const int ki = wdtype == DEC_F32 ? 0 : 1;
  DeviceSetup ds;
  {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup& slot = g_setup[di.device];
    if (!slot.ready) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_head_scratch);
      if (e != cudaSuccess)
        return fail(nullptr, DEC_ECUDA, "greedy_head_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      // dynamic limit = device maximum minus the kernel's static shared memory
      size_t lim[2];
      for (int k = 0; k < 2; ++k) {
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, kerns[k]);
        lim[k] = di.smem_optin - fa.sharedSizeBytes;
        if (e == cudaSuccess)
          e = cudaFuncSetAttribute(kerns[k], cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(lim[k]));
        if (e != cudaSuccess)
          return fail(nullptr, DEC_ECUDA, "greedy_head_noalloc: kernel set-up failed: %s", cudaGetErrorString(e));
      }
      slot.scratch = static_cast<unsigned char*>(p);
      slot.smem_limit[0] = lim[0];
      slot.smem_limit[1] = lim[1];
      slot.ready = true;
    }
    ds = slot;
  }
  const KernT kern = kerns[ki];

  // Launch shape (same plan as the decoder's head).
  int spr = static_cast<int>((row_bytes + kSEGMAX - 1) / kSEGMAX);
  const int seg = static_cast<int>(((row_bytes + spr - 1) / spr + 15) / 16 * 16);
  spr = static_cast<int>((row_bytes + seg - 1) / seg);
  int grid = vocab < di.sms ? vocab : di.sms;
  int max_rows = (vocab + grid - 1) / grid;
  while (static_cast<size_t>(max_rows) * spr * 4 > 64 * 1024 && grid * 2 <= kMaxCtas) {
    grid *= 2;
    max_rows = (vocab + grid - 1) / grid;
  }
  if (grid > kMaxCtas || static_cast<size_t>(max_rows) * spr * 4 > 64 * 1024)
    return fail(nullptr, DEC_EINVAL, "greedy_head_noalloc: vocab %d x hidden %d needs more than %d CTAs of scratch",
                vocab, hidden, kMaxCtas);
  const size_t smem = gemv_smem_bytes(gemv_ring_bytes<kNW, kNSMAX, kRING>(), hidden, max_rows, spr);
  if (smem > ds.smem_limit[ki])
    return fail(nullptr, DEC_EINVAL, "greedy_head_noalloc: hidden %d needs %zu B of shared memory (max %zu)", hidden,
                smem, ds.smem_limit[ki]);

  GemvArgs a = {};
  a.w.base[0] = a.w.base[1] = a.w.base[2] = static_cast<const char*>(d_embed);
  a.w.split1 = a.w.split2 = vocab;
  a.out = vocab;
  a.in = hidden;
  a.row_bytes = static_cast<int>(row_bytes);
  a.seg_bytes = seg;
  a.segs_per_row = spr;
  a.row_unit = 1;
  a.x = d_h;
  a.norm_g = d_gain;
  a.eps = eps;
  a.vocab = vocab;
  a.y = d_logits;
  a.part_val = reinterpret_cast<float*>(ds.scratch);
  a.part_idx = reinterpret_cast<int32_t*>(ds.scratch + kOffIdx);
  a.counter = reinterpret_cast<uint32_t*>(ds.scratch + kOffCounter);
  a.ctrl = reinterpret_cast<int32_t*>(ds.scratch + kOffCtrl);
  a.err = di.err;
  a.tok_w = reinterpret_cast<int32_t*>(ds.scratch + kOffTok);
  a.l2_prefetch = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The kernel reads the position word (must be 0) and counts finished CTAs
  // from 0; the previous call leaves the position at 1, so clear both.
  WSG_CUDA_TRY(nullptr, cudaMemsetAsync(ds.scratch + kOffCounter, 0, 8, s));
  WSG_CUDA_TRY(nullptr, launch_k(kern, dim3(grid), dim3(kNW * 32), smem, s, false, a));
  // Position 0 writes the token to slot 1.
  WSG_CUDA_TRY(nullptr, cudaMemcpyAsync(d_token, ds.scratch + kOffTok + 4, 4, cudaMemcpyDeviceToDevice, s));
  return DEC_OK;
}
