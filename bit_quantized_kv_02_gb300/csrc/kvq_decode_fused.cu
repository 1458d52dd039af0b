// kvq_decode_fused.cu — the compile-time specialisations of the decode kernel
// with the append of the new token fused in (kvq_append_decode_attn), part 0
// of the table (part 1: kvq_decode_fused2.cu).  Other formats run the append
// kernel and the decode kernel back to back.
#include "kvq_decode_table.cuh"

namespace kvq {

void* decode_kernel_fused(const kvq_cache* C, int* nw) {
  void* fn = lookup_specialised<true, 0>(C, nw);
  return fn ? fn : decode_kernel_fused_part1(C, nw);
}

}  // namespace kvq
