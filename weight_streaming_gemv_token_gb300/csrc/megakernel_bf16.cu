// Persistent decode kernel instances for bf16 weights (split from the runtime
// so the instances compile in parallel).
#include "megakernel.cuh"

namespace wsg {

void* mk_kernel_bf16(bool kv_bf16, bool group_le2) {
  if (kv_bf16)
    return group_le2 ? reinterpret_cast<void*>(decode_megakernel<uint16_t, uint16_t, 2>)
                     : reinterpret_cast<void*>(decode_megakernel<uint16_t, uint16_t, 8>);
  return group_le2 ? reinterpret_cast<void*>(decode_megakernel<uint16_t, float, 2>)
                   : reinterpret_cast<void*>(decode_megakernel<uint16_t, float, 8>);
}

}  // namespace wsg
