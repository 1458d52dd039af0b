// kvq_decode_fast.cu — the plain compile-time specialisations of the decode
// kernel, part 0 of the table (part 1: kvq_decode_fast2.cu).  Any other
// format runs the generic kernel.
#include "kvq_decode_table.cuh"

namespace kvq {

void* decode_kernel_fast(const kvq_cache* C, int* nw) {
  void* fn = lookup_specialised<false, 0>(C, nw);
  return fn ? fn : decode_kernel_fast_part1(C, nw);
}

}  // namespace kvq
