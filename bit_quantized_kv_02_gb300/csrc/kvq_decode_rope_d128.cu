// kvq_decode_rope_d128.cu — decode kernel instances for head_dim 128 with the rotary
// embedding of pre-RoPE keys (runtime formats).
#include "kvq_decode.cuh"

namespace kvq {

void* decode_kernel_ptr_rope_d128(bool r8, int vaxis) {
  if (!r8) return vaxis ? reinterpret_cast<void*>(&decode_kernel<128, false, 1, DynCfg, false, true>)
                        : reinterpret_cast<void*>(&decode_kernel<128, false, 0, DynCfg, false, true>);
  return vaxis ? reinterpret_cast<void*>(&decode_kernel<128, true, 1, DynCfg, false, true>)
               : reinterpret_cast<void*>(&decode_kernel<128, true, 0, DynCfg, false, true>);
}

}  // namespace kvq
