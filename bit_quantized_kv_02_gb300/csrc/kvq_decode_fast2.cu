// kvq_decode_fast2.cu — the plain compile-time specialisations of the decode
// kernel, part 1 of the table.
#include "kvq_decode_table.cuh"

namespace kvq {

void* decode_kernel_fast_part1(const kvq_cache* C, int* nw) { return lookup_specialised<false, 1>(C, nw); }

void* decode_kernel_rope_fast(const kvq_cache* C) { return lookup_specialised_rope(C); }

}  // namespace kvq
