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
  int nw;  // warps per CTA
};

template <bool FUSED, int D, int REP, int KB, int KAX, int KG, int KSYM, int VB, int VAX, int VG, int VSYM,
          int NW = kWarps>
FastEntry fast_entry() {
  using C = StatCfg<D, REP, KB, KAX, KG, KSYM, VB, VAX, VG, VSYM>;
  return {D, REP, KB, KAX, KG, KSYM, VB, VAX, VG, VSYM,
          reinterpret_cast<void*>(&decode_kernel<D, REP == 8, VAX, C, FUSED, false, NW>), NW};
}

// The table is split in two parts, instantiated in separate translation units
// (compiled in parallel): part 0 the benchmark workloads' default formats, part
// 1 the other axis combinations of the Llama-2-13B shape and the symmetric
// wide-GQA format with keys per channel.
template <bool FUSED, int PART>
void* lookup_specialised(const kvq_cache* C, int* nw) {
  // D, rep, K bits/axis/group/sym, V bits/axis/group/sym (axis 0 per token, 1 per channel)
  const FastEntry* table = nullptr;
  int count = 0;
  if constexpr (PART == 0) {
  static const FastEntry table0[] = {
      fast_entry<FUSED, 64, 1, 4, 1, 32, 0, 4, 0, 32, 0>(),    // 4-bit, keys per channel / values per token, G=32
      fast_entry<FUSED, 64, 1, 6, 0, 64, 0, 4, 0, 64, 0>(),    // K6/V4 per-head 64-channel groups
      fast_entry<FUSED, 128, 1, 2, 1, 32, 0, 2, 0, 32, 0>(),   // 2-bit MHA, head_dim 128, G=32
      fast_entry<FUSED, 128, 1, 2, 1, 32, 0, 2, 0, 32, 0, 1>(),  // the same in one-warp CTAs
      fast_entry<FUSED, 128, 4, 2, 1, 64, 0, 2, 0, 64, 0>(),   // 2-bit GQA 4:1, G=64
      fast_entry<FUSED, 256, 8, 4, 0, 32, 0, 8, 0, 32, 0>(),   // K4/V8 GQA 8:1, 32-channel groups
      fast_entry<FUSED, 256, 8, 4, 1, 32, 0, 8, 0, 32, 0>(),   // same with keys per channel
      fast_entry<FUSED, 256, 8, 6, 0, 32, 1, 6, 0, 32, 1>(),   // symmetric 6-bit
  };
  table = table0;
  count = (int)(sizeof(table0) / sizeof(table0[0]));
  } else {
  static const FastEntry table1[] = {
      fast_entry<FUSED, 128, 1, 2, 0, 32, 0, 2, 0, 32, 0>(),   // 2-bit MHA, keys and values per token
      fast_entry<FUSED, 128, 1, 2, 1, 32, 0, 2, 1, 32, 0>(),   // keys and values per channel
      fast_entry<FUSED, 128, 1, 2, 0, 32, 0, 2, 1, 32, 0>(),   // keys per token, values per channel
      fast_entry<FUSED, 256, 8, 6, 1, 32, 1, 6, 0, 32, 1>(),   // symmetric 6-bit, keys per channel
  };
  table = table1;
  count = (int)(sizeof(table1) / sizeof(table1[0]));
  }
  const kvq_config& c = C->cfg;
  if (c.meta_dtype != KVQ_F16 || C->k.whole || C->v.whole) return nullptr;
  const int rep = c.q_heads / c.kv_heads;
  // one-warp CTAs where the format has them and the cache asks for them
  for (int want : {C->one_warp ? 1 : kWarps, kWarps}) {
    for (int i = 0; i < count; ++i) {
      const FastEntry& e = table[i];
      if (e.nw == want && e.D == c.head_dim && e.rep == rep && e.kb == c.k.bits && e.kax == c.k.axis &&
          e.kg == c.k.group && e.ksym == c.k.mode && e.vb == c.v.bits && e.vax == c.v.axis && e.vg == c.v.group &&
          e.vsym == c.v.mode) {
        if (nw) *nw = e.nw;
        return e.fn;
      }
    }
  }
  return nullptr;
}

// Compile-time specialisations of the rotary (pre-RoPE key) decode kernel.
inline void* lookup_specialised_rope(const kvq_cache* C) {
  static const FastEntry table[] = {
      // 2-bit MHA, head_dim 128, keys per channel / values per token, G=32
      {128, 1, 2, 1, 32, 0, 2, 0, 32, 0,
       reinterpret_cast<void*>(&decode_kernel<128, false, 0, StatCfg<128, 1, 2, 1, 32, 0, 2, 0, 32, 0, 1>, false, true>),
       kWarps},
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
