// kvq_decode_d256.cu — generic (runtime-format) decode kernel instances for head_dim 256.
#include "kvq_decode.cuh"

namespace kvq {

void* decode_kernel_ptr_d256(bool r8, int vaxis) {
  if (!r8) return vaxis ? reinterpret_cast<void*>(&decode_kernel<256, false, 1, DynCfg>)
                        : reinterpret_cast<void*>(&decode_kernel<256, false, 0, DynCfg>);
  return vaxis ? reinterpret_cast<void*>(&decode_kernel<256, true, 1, DynCfg>)
               : reinterpret_cast<void*>(&decode_kernel<256, true, 0, DynCfg>);
}

}  // namespace kvq
