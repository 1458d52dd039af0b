// kvq_decode_fused.cu — the compile-time specialisations of the decode kernel
// with the append of the new token fused in (kvq_append_decode_attn).  Other
// formats run the append kernel and the decode kernel back to back.
#include "kvq_decode_table.cuh"

namespace kvq {

void* decode_kernel_fused(const kvq_cache* C) { return lookup_specialised<true>(C); }

}  // namespace kvq
