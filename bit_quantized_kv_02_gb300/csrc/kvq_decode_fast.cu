// kvq_decode_fast.cu — the plain compile-time specialisations of the decode
// kernel.  Any other format runs the generic kernel.
#include "kvq_decode_table.cuh"

namespace kvq {

void* decode_kernel_fast(const kvq_cache* C) { return lookup_specialised<false>(C); }

}  // namespace kvq
