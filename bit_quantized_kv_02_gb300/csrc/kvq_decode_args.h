// kvq_decode_args.h — launch arguments of the decode kernel (host + device).
#pragma once

#include "kvq_internal.h"

namespace kvq {

// ------------------------------------------------------------ arguments ----

struct DecodeArgs {
  TensorLayout K, V;
  int layer, B, H, rep, tcap, ntiles;
  const char* base;
  const int32_t* lens;      // [B] of this layer
  const uint32_t* smax_v;   // [B][H] largest value step of this layer (float bits)
  const void* q;
  int q_f32;
  float scale_log2;         // softmax scale * log2(e)
  int S, Sw;                // tokens per CTA / per warp
  int max_chunks;
  float* work;              // [B][H*rep][max_chunks][D+2]
  uint32_t* tickets;        // [B][H]
  float* out;               // [B][H*rep][D]
  int* err;
  // shared-memory plan (bytes)
  int nstages, stage_bytes;
  int st_kc, st_km, st_vc, st_vm;  // offsets inside a stage
  int kc_bytes, vc_bytes;          // packed tile bytes
  int km_tile_bytes, vm_tile_bytes;  // per-token metadata bytes per tile
  int km_group_bytes, vm_group_bytes;  // per-channel metadata bytes per group
  int warp_bytes;           // per-warp region: B operand area + stages + barriers
  int barea_bytes;
  int head_bytes;           // CTA head region (q, group sums)
};


// per-head-dim kernel entry points (one translation unit each, compiled in parallel)
void* decode_kernel_ptr_d64(bool r8, int vaxis);
void* decode_kernel_ptr_d128(bool r8, int vaxis);
void* decode_kernel_ptr_d256(bool r8, int vaxis);

}  // namespace kvq
