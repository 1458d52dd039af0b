// kvq_decode_table.cuh — the compile-time specialisations of the decode
// kernel (cache formats of the benchmarked workloads: fp16 metadata, no
// whole-vector groups) and their lookup.  kvq_decode_fast.cu instantiates
// the plain kernels, kvq_decode_fused.cu the ones with the append fused in
// (two translation units, compiled in parallel).
#pragma once

#include "kvq_decode.cuh"

namespace kvq {

struct FastEntry {
  int D, rep, kb, kax, kg, ksym, vb, vax, vg, vsym;
  void* fn;
};

template <bool FUSED, int D, int REP, int KB, int KAX, int KG, int KSYM, int VB, int VAX, int VG, int VSYM>
FastEntry fast_entry() {
  using C = StatCfg<D, REP, KB, KAX, KG, KSYM, VB, VAX, VG, VSYM>;
  return {D, REP, KB, KAX, KG, KSYM, VB, VAX, VG, VSYM,
          reinterpret_cast<void*>(&decode_kernel<D, REP == 8, VAX, C, FUSED>)};
}

template <bool FUSED>
void* lookup_specialised(const kvq_cache* C) {
  // D, rep, K bits/axis/group/sym, V bits/axis/group/sym (axis 0 per token, 1 per channel)
  static const FastEntry table[] = {
      fast_entry<FUSED, 64, 1, 4, 1, 32, 0, 4, 0, 32, 0>(),    // 4-bit, keys per channel / values per token, G=32
      fast_entry<FUSED, 64, 1, 6, 0, 64, 0, 4, 0, 64, 0>(),    // K6/V4 per-head 64-channel groups
      fast_entry<FUSED, 128, 1, 2, 1, 32, 0, 2, 0, 32, 0>(),   // 2-bit MHA, head_dim 128, G=32
      fast_entry<FUSED, 128, 4, 2, 1, 64, 0, 2, 0, 64, 0>(),   // 2-bit GQA 4:1, G=64
      fast_entry<FUSED, 256, 8, 4, 0, 32, 0, 8, 0, 32, 0>(),   // K4/V8 GQA 8:1, 32-channel groups
      fast_entry<FUSED, 256, 8, 4, 1, 32, 0, 8, 0, 32, 0>(),   // same with keys per channel
      fast_entry<FUSED, 256, 8, 6, 0, 32, 1, 6, 0, 32, 1>(),   // symmetric 6-bit
  };
  const kvq_config& c = C->cfg;
  if (c.meta_dtype != KVQ_F16 || C->k.whole || C->v.whole) return nullptr;
  const int rep = c.q_heads / c.kv_heads;
  for (const FastEntry& e : table) {
    if (e.D == c.head_dim && e.rep == rep && e.kb == c.k.bits && e.kax == c.k.axis && e.kg == c.k.group &&
        e.ksym == c.k.mode && e.vb == c.v.bits && e.vax == c.v.axis && e.vg == c.v.group && e.vsym == c.v.mode)
      return e.fn;
  }
  return nullptr;
}

}  // namespace kvq
