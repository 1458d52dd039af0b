// kvq_decode_args.h — launch arguments of the decode kernel (host + device).
#pragma once

#include "kvq_internal.h"

namespace kvq {

// One tensor (keys or values) of the decoded layer, resolved on the host so
// the kernel's hot loop only does shifts, masks and adds.
struct DecTensor {
  const char* codes;    // packed tiles of the layer: [B][H][ntiles][tile_bytes]
  const char* meta;     // metadata of the layer
  const __half* tail;   // fp16 tail of the layer (per-channel axis): [B][H][G][D]
  int bits, sym, meta_f32, axis, whole;
  int lg_group;         // log2 of the group size (tokens per-channel, channels per-token); 0 when whole
  int group;            // group size (per-channel: tokens)
  int gpt;              // per-token axis: groups per head row (1 when whole)
  int meta_bytes;       // bytes of one stored entry
  int tile_bytes;       // packed bytes of one 16-token tile
  int mtile_bytes;      // per-token: metadata bytes per tile; per-channel: per group
  int window;           // full-precision window of the newest tokens (0: none)
  int ring;             // fp16 rows per (sequence, head): token t at row t % ring
};

// Arguments of the quantizer kernels for one layer-tensor.
struct QuantArgs {
  TensorLayout L;
  int is_value;
  int layer, B, H, D, tcap, ntiles;
  const void* x;  // [B][t_stride][H][D]
  int x_f32;
  long t_stride;
  const int32_t* lens;  // device lens of this layer
  char* base;           // cache buffer
  uint32_t* smax;       // [B][H] for this tensor and layer
};

// Append of one token per (sequence, kv head) to both tensors of a layer.
struct AppendArgs {
  QuantArgs k, v;       // x points at [B][H][D] new tokens (t_stride unused)
  int32_t* lens;        // device lens of the layer
  int32_t* head_lens;   // [B][H] per-head length counters of the layer
  int warp_smem;        // per-warp scratch bytes for the per-token path
};

struct DecodeArgs {
  DecTensor K, V;
  int B, H, rep, tcap, ntiles;
  const int32_t* lens;      // [B] of this layer
  const uint32_t* smax_k;   // [B][H] largest key step of this layer (float bits)
  const uint32_t* smax_v;   // [B][H] largest value step of this layer (float bits)
  const void* q;
  int q_f32;
  float scale_log2;         // softmax scale * log2(e)
  int S, Sw;                // work per CTA / per warp (tokens, fp16-row tokens counted fw times)
  int fw;                   // work of a token still in fp16 rows (1: every token counts once)
  int max_chunks;
  float* work;              // [B][H*rep][max_chunks][D+4] chunk partials
  float* gwork;             // [B][H*rep][max_groups][D+4] group partials
  int max_groups;           // ceil(max_chunks / kCombineGroup)
  int csize;                // > 0: the grid's x dimension forms clusters of csize CTAs (all splits of one
                            // sequence and head) that merge through distributed shared memory
  int gath_off;             // cluster launch: byte offset of [csize][rep][D+2] split partials, gathered in
                            // the cluster's first CTA (after the per-warp regions)
  uint32_t* tickets;        // [B][H][1 + max_groups]: head ticket, then one per chunk group
  float* out;               // [B][H*rep][D]
  int* err;
  // shared-memory plan (bytes)
  int lg_nstages, stage_bytes;
  int st_kc, st_km, st_vc, st_vm;  // offsets inside a stage
  int warp_bytes;           // per-warp region: B operand + canonical metadata + stages
  int barea_bytes;
  int canon_k, canon_v;     // canonical (step, zero') entries per warp for per-token keys / values
  int stage_off;            // offset of the stage ring inside the per-warp region
  int head_bytes;           // CTA head region (q, group sums)
  int stage_f16;            // fp16 rows (window, unsealed groups) are staged through the ring too
  double rope_l2b;          // log2 of the rotary embedding's base (the kernel's ROPE instantiation)
  int rope_off;             // byte offset of the rotary tables inside the CTA head region
  // fused append (the kernel's FUSED instantiation, kvq_append_decode_attn):
  // the warp whose range holds the new token appends it first; lengths come
  // from ap.head_lens (old length + 1) and the last CTA of each (sequence,
  // head) to count itself in `arrive` advances them
  uint32_t* arrive;         // [B][H] arrival counters (zero between launches)
  AppendArgs ap;
};

// Scratch bytes one warp needs for the fused append: a per-channel seal's
// (3*D floats of group parameters + 16 rows of D halves), or with a
// full-precision window the seal of a per-token block (16 rows of D halves +
// 3 floats per (token, group), at most 12*D bytes for groups of 16); per-token
// tensors without a window need none.
__host__ __device__ constexpr int fused_append_scratch(int D, int k_axis, int v_axis, int window = 0) {
  return (k_axis == 1 || v_axis == 1 || window) ? 44 * D : 0;
}

// Host: the append arguments of a layer (kvq_quant.cu).
AppendArgs make_append_args(const kvq_cache* C, int layer, const void* k, const void* v, int x_f32);

// Shared-memory plan of the decode kernel; one constexpr function serves the
// host planner and the compile-time specialisations, so both always agree.
struct DecLayout {
  int kc_bytes, vc_bytes, km_bytes, vm_bytes;  // packed tile / metadata bytes per stage
  int st_kc, st_km, st_vc, st_vm;              // offsets inside a stage
  int stage_bytes, lg_ns;                      // stage size, log2 of the stage count
  int barea_bytes, canon_k, canon_v, stage_off, warp_bytes, head_bytes;
  int rope_off;                                // rotary tables inside the head region (rope layouts)
};

// Rotary tables of a decode CTA (floats2): the pair frequencies theta_i as
// (hi, lo) [D/2], the in-tile turns (cos, sin)(u * theta_i) [16][D/2 + 4]
// (rows padded against bank conflicts), and each warp's per-tile bases [4][D/2].
__host__ __device__ constexpr int rope_row(int D) { return D / 2 + 4; }
__host__ __device__ constexpr int rope_bytes(int D) { return (D / 2 + 16 * rope_row(D) + 4 * (D / 2)) * 8; }

__host__ __device__ constexpr int dl_round(int x, int m) { return (x + m - 1) / m * m; }
__host__ __device__ constexpr int dl_max(int x, int y) { return x > y ? x : y; }

// f16: stage slots also hold a 16-token tile of fp16 rows (32 * D bytes per tensor)
__host__ __device__ constexpr DecLayout dec_layout(int D, int rep, int kbits, int kaxis, int kwhole, int kgpt,
                                                   int kmb, int vbits, int vaxis, int vwhole, int vgpt, int vmb,
                                                   int f16 = 0, int rope = 0) {
  DecLayout L{};
  L.kc_bytes = D * kbits * 2;
  L.vc_bytes = D * vbits * 2;
  const int kslot = f16 ? dl_max(L.kc_bytes, 32 * D) : L.kc_bytes;
  const int vslot = f16 ? dl_max(L.vc_bytes, 32 * D) : L.vc_bytes;
  L.km_bytes = kaxis == 0 ? 16 * (kwhole ? 1 : kgpt) * kmb : D * kmb;
  L.vm_bytes = vaxis == 0 ? 16 * (vwhole ? 1 : vgpt) * vmb : D * vmb;
  L.st_kc = 0;
  L.st_km = dl_round(L.st_kc + kslot, 16);
  L.st_vc = dl_round(L.st_km + L.km_bytes, 16);
  L.st_vm = dl_round(L.st_vc + vslot, 16);
  L.stage_bytes = dl_round(L.st_vm + L.vm_bytes, 128);
  L.lg_ns = L.stage_bytes <= 4096 ? 2 : 1;
  L.barea_bytes = (D / 16) * 32 * 8 * (rep == 8 ? 2 : 1);
  // keys are read from the stage, except by the rotary kernel, which keeps their (step, zero') entries
  L.canon_k = rope ? (kaxis == 0 ? 16 * (kwhole ? 1 : kgpt) : D) : 0;  // only the rotary kernel canonicalises keys
  L.canon_v = vaxis == 0 ? 0 : D;  // per-token values are read from the stage
  L.stage_off = dl_round(L.barea_bytes + (L.canon_k + L.canon_v) * 8 + 32, 128);
  L.warp_bytes = dl_round(L.stage_off + (L.stage_bytes << L.lg_ns), 128);
  const int merge_bytes = 4 * rep * (D + 2) * 4;
  if (L.warp_bytes * 4 < merge_bytes) L.warp_bytes = dl_round((merge_bytes + 3) / 4, 128);
  L.rope_off = dl_round((rep * D + (kaxis == 0 ? kgpt * rep : 0)) * 4, 16);
  L.head_bytes = dl_round(L.rope_off + (rope ? rope_bytes(D) : 0), 128);
  return L;
}

// per-head-dim kernel entry points (one translation unit each, compiled in parallel)
void* decode_kernel_ptr_d64(bool r8, int vaxis);
void* decode_kernel_ptr_d128(bool r8, int vaxis);
void* decode_kernel_ptr_d256(bool r8, int vaxis);
// the same with the rotary embedding of the keys (pre-RoPE caches)
void* decode_kernel_ptr_rope_d64(bool r8, int vaxis);
void* decode_kernel_ptr_rope_d128(bool r8, int vaxis);
void* decode_kernel_ptr_rope_d256(bool r8, int vaxis);

// the second part of the compile-time specialisation table (plain and fused;
// decode_kernel_fast / decode_kernel_fused search both parts)
void* decode_kernel_fast_part1(const kvq_cache* C, int* nw);
void* decode_kernel_fused_part1(const kvq_cache* C, int* nw);
// compile-time specialisation of the rotary decode kernel for this cache, or null
void* decode_kernel_rope_fast(const kvq_cache* C);

}  // namespace kvq
