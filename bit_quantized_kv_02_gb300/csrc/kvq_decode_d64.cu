// kvq_decode_d64.cu — decode kernel instances for head_dim 64.
#include "kvq_decode.cuh"

namespace kvq {

void* decode_kernel_ptr_d64(bool r8, int vaxis) {
  if (!r8) return vaxis ? reinterpret_cast<void*>(&decode_kernel<64, false, 1>)
                        : reinterpret_cast<void*>(&decode_kernel<64, false, 0>);
  return vaxis ? reinterpret_cast<void*>(&decode_kernel<64, true, 1>)
               : reinterpret_cast<void*>(&decode_kernel<64, true, 0>);
}

}  // namespace kvq
