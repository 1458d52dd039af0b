// kvq_decode_fused2.cu — the fused-append specialisations of the decode
// kernel, part 1 of the table.
#include "kvq_decode_table.cuh"

namespace kvq {

void* decode_kernel_fused_part1(const kvq_cache* C, int* nw) { return lookup_specialised<true, 1>(C, nw); }

}  // namespace kvq
