// Persistent decode kernel instances for f32 weights (split from the runtime
// so the instances compile in parallel).
#include "megakernel.cuh"

namespace wsg {

void* mk_kernel_f32(bool kv_bf16, bool group_le2) {
  if (kv_bf16)
    return group_le2 ? reinterpret_cast<void*>(decode_megakernel<float, uint16_t, 2>)
                     : reinterpret_cast<void*>(decode_megakernel<float, uint16_t, 8>);
  return group_le2 ? reinterpret_cast<void*>(decode_megakernel<float, float, 2>)
                   : reinterpret_cast<void*>(decode_megakernel<float, float, 8>);
}

}  // namespace wsg
