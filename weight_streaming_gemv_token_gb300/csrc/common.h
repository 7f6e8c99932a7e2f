// Host-side helpers shared by the library's translation units: error
// strings, device checks and kernel launch with programmatic dependent launch.
#pragma once
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <string>
#include <utility>

#include "../../include/wsg.h"

namespace wsg {

// Last error of context-free calls, per thread.
std::string& thread_error();

inline dec_status fail(std::string* where, dec_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (where) *where = buf;
  thread_error() = buf;
  return st;
}

#define WSG_CUDA_TRY(where, call)                                                                          \
  do {                                                                                                     \
    cudaError_t e_ = (call);                                                                               \
    if (e_ != cudaSuccess)                                                                                 \
      return ::wsg::fail((where), DEC_ECUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, \
                         __LINE__);                                                                        \
  } while (0)

struct DeviceInfo {
  int device = -1;
  int sms = 0;
  int major = 0, minor = 0;
  size_t smem_optin = 0;
  size_t smem_per_sm = 0;
  uint32_t* err = nullptr;  // device error word of the context-free entry points on this device
};

// Properties of the current device (cached per device; thread-safe), with
// the device address of the context-free error word.
dec_status device_info(DeviceInfo* out, std::string* err);

// Launch `kern` with an optional programmatic-dependent-launch edge to the
// previous work on `st`.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raise a kernel's dynamic shared memory limit (idempotent per device).
template <typename K>
cudaError_t allow_smem(K kern, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tiled TMA descriptor (CUtensorMap, 128 bytes, opaque here) of a row-major
// [rows][cols] matrix of `elem`-byte elements (2: bfloat16, 4: float32) with
// boxes of box_rows x box_cols; swizzle128 selects the 128-byte swizzle
// (box_cols * elem must then be 128). Elements outside the matrix read as 0.
dec_status encode_map_2d(void* out, const void* base, long long rows, long long cols, int elem, int box_cols,
                         int box_rows, bool swizzle128, std::string* err);

}  // namespace wsg
