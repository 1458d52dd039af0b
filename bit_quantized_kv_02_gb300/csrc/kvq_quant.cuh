// kvq_quant.cuh — device helpers of the quantizer shared by the prefill,
// append and export kernels and by the decode kernel's fused append: group
// statistics, tile-word packing, cache addressing, the per-warp append of one
// token and the per-warp seal of a per-channel group.
//
// The arithmetic follows "O Seu Cache KV Nao Tem um Problema de Bits. Tem um
// Problema de Geometria", section "O Que o Erro de Quantizacao E Realmente
// Feito" (zero = group minimum, step = range/(2^B-1), round to nearest), with
// per-channel groups sealed once G tokens exist (section "O Imposto dos
// Sistemas e Por Que Nao E um Detalhe").
#pragma once

#include "kvq_decode_args.h"

namespace kvq {

// ------------------------------------------------------- group statistics --

// Warp-cooperative min / max / absmax over count values base[i*stride].
__device__ __forceinline__ void warp_stats(const float* base, int count, int stride, float* mn, float* mx,
                                           float* am) {
  float a = INFINITY, b = -INFINITY, c = 0.0f;
  for (int i = threadIdx.x & 31; i < count; i += 32) {
    float v = base[(long)i * stride];
    a = fminf(a, v);
    b = fmaxf(b, v);
    c = fmaxf(c, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
    c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, o));
  }
  *mn = a;
  *mx = b;
  *am = c;
}

__device__ __forceinline__ float load_in(const void* p, long idx, int f32) {
  return f32 ? reinterpret_cast<const float*>(p)[idx] : __half2float(reinterpret_cast<const __half*>(p)[idx]);
}

// Inverse of elem_pos: which (token, channel) of the tile a (lane, pair, half) holds.
__device__ __forceinline__ void elem_of(int is_value, int lane, int pi, int e, int* t, int* c) {
  int j = pi >> 2, r = pi & 3, rh = r & 1, kh = r >> 1;
  int g = lane >> 2, tig = lane & 3;
  int R = g + 8 * rh, kk = 2 * tig + 8 * kh + e;
  if (is_value) {
    *t = kk;
    *c = 16 * j + R;
  } else {
    *t = R;
    *c = 16 * j + kk;
  }
}

// Value of tile word `wi` (0 .. D*bits/2-1) with the code of (token t,
// channel c) given by code(t, c) (t < 16).
template <class CodeF>
__device__ __forceinline__ uint32_t build_word_f(int D, const Planes& pl, int is_value, int wi, CodeF code) {
  // which plane
  int p = 0;
  for (int q = 1; q < pl.n; ++q)
    if (wi >= D * pl.off[q] / 2) p = q;
  int w = pl.w[p];
  int W = D * w / 64, P = 16 / w;
  int rel = wi - D * pl.off[p] / 2;
  int lane = rel / W, i = rel % W;
  uint32_t word = 0, mask = (1u << w) - 1u;
  for (int k = 0; k < P; ++k) {
    for (int e = 0; e < 2; ++e) {
      int t, c;
      elem_of(is_value, lane, i * P + k, e, &t, &c);
      word |= (((uint32_t)code(t, c) >> pl.off[p]) & mask) << (k * w + 16 * e);
    }
  }
  return word;
}

// Value of tile word `wi` built from codes[t*D + c] (t < 16).
__device__ __forceinline__ uint32_t build_word(const uint8_t* codes, int D, const Planes& pl, int is_value, int wi) {
  return build_word_f(D, pl, is_value, wi, [&](int t, int c) { return (uint32_t)codes[t * D + c]; });
}

// Write the tile words of one 16-token tile (codes in shared memory, [16][D]).
__device__ inline void store_tile(uint32_t* dst, const uint8_t* codes, int D, const TensorLayout& L, int is_value) {
  int nw = L.tile_words;  // multiple of 32 (D*bits/2, D >= 64)
  for (int q = threadIdx.x; q < nw / 4; q += blockDim.x) {
    uint4 v;
    v.x = build_word(codes, D, L.planes, is_value, 4 * q + 0);
    v.y = build_word(codes, D, L.planes, is_value, 4 * q + 1);
    v.z = build_word(codes, D, L.planes, is_value, 4 * q + 2);
    v.w = build_word(codes, D, L.planes, is_value, 4 * q + 3);
    reinterpret_cast<uint4*>(dst)[q] = v;
  }
}

__device__ __forceinline__ void atomic_max_pos(uint32_t* addr, float v) {
  // non-negative floats order like their bit patterns
  if (v > 0.0f) atomicMax(addr, __float_as_uint(v));
}

__device__ __forceinline__ uint32_t* codes_ptr(const QuantArgs& a, int b, int h, int tile) {
  return reinterpret_cast<uint32_t*>(a.base + a.L.codes_off + a.layer * a.L.codes_layer) +
         ((((long)b * a.H + h) * a.ntiles + tile) * a.L.tile_words);
}
__device__ __forceinline__ char* meta_ptr(const QuantArgs& a) {
  return a.base + a.L.meta_off + a.layer * a.L.meta_layer;
}
__device__ __forceinline__ long bh_of(const QuantArgs& a, int b, int h) { return (long)b * a.H + h; }
// fp16 rows of (b, h): ring of L.ring rows, token t at row t % ring
__device__ __forceinline__ __half* tail_ptr(const QuantArgs& a, int b, int h) {
  return reinterpret_cast<__half*>(a.base + a.L.tail_off + a.layer * a.L.tail_layer) +
         (((long)b * a.H + h) * a.L.ring) * a.D;
}
__device__ __forceinline__ __half* tail_row(const QuantArgs& a, int b, int h, long t) {
  // token indices stay far below 2^31: a 32-bit remainder
  return tail_ptr(a, b, h) + (long)((int)t % a.L.ring) * a.D;
}

// One warp appends the new token of (b, h) (old length n) to one tensor: a
// per-token tensor quantizes the token row now and merges its codes into the
// tile words that hold that row; a per-channel tensor stores it in the fp16
// tail and reports (returns true) when the tail just filled up, so that the
// caller seals the group.  xs / cs: per-warp shared scratch; *step_max (if
// given) receives the largest step the token's groups got (0 for a row that
// is only stored); pre (if given): the row already loaded into shared memory
// as floats (no whole-vector groups, no window), so xs is not used.
__device__ inline bool append_warp(const QuantArgs& a, int b, int h, int n, float* xs, uint8_t* cs, float* zs,
                                   float* ss, float* step_max = nullptr, const float* pre = nullptr) {
  const int lane = threadIdx.x & 31;
  const int D = a.D;
  const long xs_t = (long)a.H * D;
  const int R = a.L.window;
  if (a.L.axis == 1) {
    // fp16 row; a group seals once all its tokens are older than the window
    const int G = a.L.group;
    __half* row = tail_row(a, b, h, n);
    for (int c = lane; c < D; c += 32)
      row[c] = __float2half_rn(pre ? pre[c] : load_in(a.x, (long)b * xs_t + (long)h * D + c, a.x_f32));
    if (step_max) *step_max = 0.0f;
    const int old = n + 1 - R;
    return old >= G && old % G == 0;
  }
  const int whole = a.L.whole;
  const int nh = whole ? a.H : 1;
  const int rowlen = nh * D;
  if (R) {
    // per-token tensor with a window: fp16 row now, its 16-token block is
    // quantized once all of it is older than the window
    for (int c = lane; c < rowlen; c += 32)
      tail_row(a, b, h + c / D, n)[c % D] = __float2half_rn(load_in(a.x, (long)b * xs_t + (long)h * D + c, a.x_f32));
    if (step_max) *step_max = 0.0f;
    const int old = n + 1 - R;
    return old >= kTile && old % kTile == 0;
  }
  const int G = whole ? rowlen : a.L.group;
  const int gpr = rowlen / G;
  if (!pre) {
    for (int c = lane; c < rowlen; c += 32) xs[c] = load_in(a.x, (long)b * xs_t + (long)h * D + c, a.x_f32);
    __syncwarp();
  }
  const float* xr = pre ? pre : xs;
  char* meta = meta_ptr(a);
  float smax_local = 0.0f;
  for (int j = 0; j < gpr; ++j) {
    float mn, mx, am;
    warp_stats(xr + j * G, G, 1, &mn, &mx, &am);
    float z, s;
    group_params(mn, mx, am, a.L.bits, a.L.sym, a.L.meta_f32, &z, &s);
    smax_local = fmaxf(smax_local, s);
    if (lane == 0) {
      zs[j] = z;
      ss[j] = s;
      const long mi = whole ? ((long)b * a.tcap + n) : ((((long)b * a.H + h) * a.tcap + n) * gpr + j);
      store_meta(meta, mi, a.L.meta_f32, a.L.sym, z, s);
    }
  }
  __syncwarp();
  for (int c = lane; c < rowlen; c += 32) cs[c] = (uint8_t)quant_code(xr[c], zs[c / G], ss[c / G], a.L.bits, a.L.sym);
  __syncwarp();
  // merge into the tile words that hold token row trow
  const int trow = n & 15, tile = n >> 4;
  const Planes& pl = a.L.planes;
  if (trow == 0) {
    // a tile's first token clears the whole tile (a shorter re-prefill can leave
    // older codes behind), so that later tokens only OR their bits in
    for (int hh = 0; hh < nh; ++hh) {
      uint4* dst = reinterpret_cast<uint4*>(codes_ptr(a, b, h + hh, tile));
      for (int q = lane; q < a.L.tile_words / 4; q += 32) dst[q] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
  }
  // each lane ORs the bits of its channels' codes into the words that hold
  // them (the token row's bits are zero: the tile was cleared at its first
  // token), fire-and-forget with no read of the old words
  for (int i = lane; i < rowlen; i += 32) {
    const int hh = i / D, c = i - hh * D;
    const uint32_t code = cs[i];
    const FragPos f = elem_pos(a.is_value, trow, c);
    uint32_t* dst = codes_ptr(a, b, h + hh, tile);
    for (int p = 0; p < pl.n; ++p) {
      const int w = pl.w[p], lw = w == 1 ? 0 : (w == 2 ? 1 : (w == 4 ? 2 : 3));
      const int word = D * pl.off[p] / 2 + f.lane * (D >> (6 - lw)) + (f.pi >> (4 - lw));
      const int bit = ((f.pi & ((16 >> lw) - 1)) << lw) + 16 * f.e;
      const uint32_t v = ((code >> pl.off[p]) & ((1u << w) - 1u)) << bit;
      if (v) atomicOr(dst + word, v);
    }
  }
  if (lane == 0 && smax_local > 0.0f)
    for (int hh = 0; hh < nh; ++hh) atomic_max_pos(a.smax + (long)b * a.H + h + hh, smax_local);
  if (step_max) *step_max = smax_local;
  return false;
}

// One warp seals per-channel group g of (b, h) from its G fp16 rows: the
// same statistics, metadata and tile words as the CTA-wide seal (min, max
// and absmax are exact in any order; each code is quant_code of the same
// value).  Lane l owns the CPL = D/32 adjacent channels [l*CPL, l*CPL+CPL)
// and reads its slice of four rows per step with vector loads; codes are
// packed tile by tile from 16 rows staged in scratch.  scratch: 3*D floats
// of group parameters (zero, step, step reciprocal) + 16*D halves (44*D
// bytes, 16-byte aligned).  Returns the group's largest step.
template <int CPL>
__device__ inline float seal_channel_warp(const QuantArgs& a, int b, int h, int g, unsigned char* scratch) {
  const int lane = threadIdx.x & 31;
  const int G = a.L.group, D = CPL * 32;
  float* zs = reinterpret_cast<float*>(scratch);
  float* ss = zs + D;
  float* rs = ss + D;                                // step reciprocals
  __half* rows = reinterpret_cast<__half*>(rs + D);  // [16][D]
  char* meta = meta_ptr(a);
  // ring row of the group's first token; the G rows follow it, wrapping once
  const __half* ring0 = tail_ptr(a, b, h) + lane * CPL;
  const int ring = a.L.ring;
  int r = (g * G) % ring;
  float mn[CPL], mx[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    mn[i] = INFINITY;
    mx[i] = -INFINITY;
  }
  for (int t = 0; t < G; t += 4) {  // G is a multiple of 16
    __half2 v[4][CPL / 2];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __half2* src = reinterpret_cast<const __half2*>(ring0 + (long)r * D);
#pragma unroll
      for (int i = 0; i < CPL / 2; ++i) v[u][i] = src[i];
      r = r + 1 == ring ? 0 : r + 1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int i = 0; i < CPL / 2; ++i) {
        const float2 f = __half22float2(v[u][i]);
        mn[2 * i] = fminf(mn[2 * i], f.x);
        mx[2 * i] = fmaxf(mx[2 * i], f.x);
        mn[2 * i + 1] = fminf(mn[2 * i + 1], f.y);
        mx[2 * i + 1] = fmaxf(mx[2 * i + 1], f.y);
      }
  }
  float smax_local = 0.0f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = lane * CPL + i;
    float z, s;
    group_params(mn[i], mx[i], fmaxf(fabsf(mn[i]), fabsf(mx[i])), a.L.bits, a.L.sym, a.L.meta_f32, &z, &s);
    zs[c] = z;
    ss[c] = s;
    rs[c] = __frcp_rn(s);
    store_meta(meta, (((long)b * a.H + h) * (a.tcap / G) + g) * D + c, a.L.meta_f32, a.L.sym, z, s);
    smax_local = fmaxf(smax_local, s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) smax_local = fmaxf(smax_local, __shfl_xor_sync(0xffffffffu, smax_local, o));
  for (int tt = 0; tt < G / kTile; ++tt) {
    const long t0 = (long)g * G + tt * kTile;
    __syncwarp();  // group parameters written / previous tile's rows consumed
    for (int i = lane; i < kTile * D / 8; i += 32) {
      const int r = i / (D / 8), c8 = i - r * (D / 8);
      reinterpret_cast<uint4*>(rows)[i] = reinterpret_cast<const uint4*>(tail_row(a, b, h, t0 + r))[c8];
    }
    __syncwarp();
    auto code = [&](int t, int c) {
      return (uint32_t)quant_code_r(__half2float(rows[t * D + c]), zs[c], ss[c], rs[c], a.L.bits, a.L.sym);
    };
    uint4* dst = reinterpret_cast<uint4*>(codes_ptr(a, b, h, (int)(t0 / kTile)));
    for (int q = lane; q < a.L.tile_words / 4; q += 32) {
      uint4 v;
      v.x = build_word_f(D, a.L.planes, a.is_value, 4 * q + 0, code);
      v.y = build_word_f(D, a.L.planes, a.is_value, 4 * q + 1, code);
      v.z = build_word_f(D, a.L.planes, a.is_value, 4 * q + 2, code);
      v.w = build_word_f(D, a.L.planes, a.is_value, 4 * q + 3, code);
      dst[q] = v;
    }
  }
  if (lane == 0) atomic_max_pos(a.smax + (long)b * a.H + h, smax_local);
  return smax_local;
}

// One warp quantizes per-token block `tile` (tokens 16*tile .. 16*tile+15) of
// (b, h) from its fp16 rows, once all of it is older than the window: the same
// statistics, parameters, metadata and tile words as the CTA-wide
// quant_token_tile (min and max are exact in any order, the largest magnitude
// is at an end of the range, and quant_code_r gives quant_code's integer).  No
// whole-vector groups.  scratch: 16 rows of D halves + 3 * 16 * (D / G) floats
// (token_block_scratch bytes, 16-byte aligned).  Returns the block's largest step.
template <int CPL>
__device__ inline float seal_token_block_warp(const QuantArgs& a, int b, int h, int tile, unsigned char* scratch) {
  const int lane = threadIdx.x & 31;
  constexpr int D = CPL * 32;
  const int G = a.L.group, gpr = D / G;
  __half* rows = reinterpret_cast<__half*>(scratch);       // [16][D]
  float* zs = reinterpret_cast<float*>(rows + kTile * D);  // [16 * gpr] per (token, group)
  float* ss = zs + kTile * gpr;
  float* rs = ss + kTile * gpr;                            // step reciprocals
  for (int i = lane; i < kTile * D / 8; i += 32) {
    const int r = i / (D / 8), c8 = i - r * (D / 8);
    reinterpret_cast<uint4*>(rows)[i] = reinterpret_cast<const uint4*>(tail_row(a, b, h, (long)tile * kTile + r))[c8];
  }
  __syncwarp();
  char* meta = meta_ptr(a);
  float smax_local = 0.0f;
  for (int gi = lane; gi < kTile * gpr; gi += 32) {  // one (token, group) per lane at a time
    const int tt = gi / gpr, j = gi - tt * gpr;
    const __half2* src = reinterpret_cast<const __half2*>(rows + tt * D + j * G);
    float mn = INFINITY, mx = -INFINITY;
    for (int c = 0; c < G / 2; ++c) {
      const float2 f = __half22float2(src[c]);
      mn = fminf(mn, fminf(f.x, f.y));
      mx = fmaxf(mx, fmaxf(f.x, f.y));
    }
    float z, st;
    group_params(mn, mx, fmaxf(fabsf(mn), fabsf(mx)), a.L.bits, a.L.sym, a.L.meta_f32, &z, &st);
    zs[gi] = z;
    ss[gi] = st;
    rs[gi] = __frcp_rn(st);
    store_meta(meta, (((long)b * a.H + h) * a.tcap + (long)tile * kTile + tt) * gpr + j, a.L.meta_f32, a.L.sym, z,
               st);
    smax_local = fmaxf(smax_local, st);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) smax_local = fmaxf(smax_local, __shfl_xor_sync(0xffffffffu, smax_local, o));
  __syncwarp();  // group parameters written
  auto code = [&](int t, int c) {
    const int gi = t * gpr + c / G;
    return (uint32_t)quant_code_r(__half2float(rows[t * D + c]), zs[gi], ss[gi], rs[gi], a.L.bits, a.L.sym);
  };
  uint4* dst = reinterpret_cast<uint4*>(codes_ptr(a, b, h, tile));
  for (int q = lane; q < a.L.tile_words / 4; q += 32) {
    uint4 v;
    v.x = build_word_f(D, a.L.planes, a.is_value, 4 * q + 0, code);
    v.y = build_word_f(D, a.L.planes, a.is_value, 4 * q + 1, code);
    v.z = build_word_f(D, a.L.planes, a.is_value, 4 * q + 2, code);
    v.w = build_word_f(D, a.L.planes, a.is_value, 4 * q + 3, code);
    dst[q] = v;
  }
  if (lane == 0 && smax_local > 0.0f) atomic_max_pos(a.smax + (long)b * a.H + h, smax_local);
  return smax_local;
}

// Per-token quantization of token n of (b, h) by one warp with lane l owning
// the CPL = D/32 channels [l*CPL, l*CPL + CPL) (values in x): every group is
// reduced at once over its G/CPL lanes, so the work is a few dependent steps
// instead of one warp-wide reduction per group.  Same statistics, parameters,
// metadata and codes as append_warp (min, max and absmax do not depend on the
// order of reduction).  No whole-vector groups, no window.  Returns the
// largest step written.
template <int CPL>
__device__ __forceinline__ float append_token_lanes(const QuantArgs& a, int b, int h, int n, const float* x) {
  const int lane = threadIdx.x & 31;
  const int D = CPL * 32, G = a.L.group, lpg = G / CPL;  // lanes per group (a power of two, <= 32)
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int i = 1; i < CPL; ++i) {
    mn = fminf(mn, x[i]);
    mx = fmaxf(mx, x[i]);
  }
  for (int o = lpg >> 1; o > 0; o >>= 1) {  // stays inside the aligned group of lpg lanes
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const float am = fmaxf(fabsf(mn), fabsf(mx));  // the largest magnitude is at an end of the range
  float z, s;
  group_params(mn, mx, am, a.L.bits, a.L.sym, a.L.meta_f32, &z, &s);
  const int gpr = D / G;
  if ((lane & (lpg - 1)) == 0)
    store_meta(meta_ptr(a), (((long)b * a.H + h) * a.tcap + n) * gpr + lane / lpg, a.L.meta_f32, a.L.sym, z, s);
  uint32_t code[CPL];
  const float rcp = __frcp_rn(s);
#pragma unroll
  for (int i = 0; i < CPL; ++i) code[i] = (uint32_t)quant_code_r(x[i], z, s, rcp, a.L.bits, a.L.sym);
  const int trow = n & 15, tile = n >> 4;
  uint32_t* dst = codes_ptr(a, b, h, tile);
  if (trow == 0) {
    // a tile's first token clears the tile (a shorter re-prefill can leave
    // older codes behind); later tokens only OR their bits in
    for (int q = lane; q < a.L.tile_words / 4; q += 32) reinterpret_cast<uint4*>(dst)[q] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
  }
  const Planes& pl = a.L.planes;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const FragPos f = elem_pos(a.is_value, trow, lane * CPL + i);
    for (int p = 0; p < pl.n; ++p) {
      const int w = pl.w[p], lw = w == 1 ? 0 : (w == 2 ? 1 : (w == 4 ? 2 : 3));
      const int word = D * pl.off[p] / 2 + f.lane * (D >> (6 - lw)) + (f.pi >> (4 - lw));
      const int bit = ((f.pi & ((16 >> lw) - 1)) << lw) + 16 * f.e;
      const uint32_t v = ((code[i] >> pl.off[p]) & ((1u << w) - 1u)) << bit;
      if (v) atomicOr(dst + word, v);
    }
  }
  // every lane of a group holds its step: the largest over the groups needs
  // only the rounds across groups
  for (int o = 16; o >= lpg; o >>= 1) s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, o));
  if (lane == 0) atomic_max_pos(a.smax + (long)b * a.H + h, s);
  return s;
}

// Lane l's CPL consecutive values of a [..][D] row of fp16 or fp32 inputs.
template <int CPL>
__device__ __forceinline__ void load_lane_row(const void* x, long off, int f32, float* v) {
  if (f32) {
    const float* p = reinterpret_cast<const float*>(x) + off;
#pragma unroll
    for (int i = 0; i < CPL; i += 2) {
      const float2 u = *reinterpret_cast<const float2*>(p + i);
      v[i] = u.x;
      v[i + 1] = u.y;
    }
  } else {
    const __half2* p = reinterpret_cast<const __half2*>(reinterpret_cast<const __half*>(x) + off);
#pragma unroll
    for (int i = 0; i < CPL; i += 2) {
      const float2 u = __half22float2(p[i / 2]);
      v[i] = u.x;
      v[i + 1] = u.y;
    }
  }
}

// Append of token n (the old length) of (b, h) by one warp, with the same
// effect on the cache as the append kernel: per-token rows are quantized and
// merged into their tile, per-channel rows go to the fp16 tail and a filled
// group is sealed; a tensor with a full-precision window only stores the fp16
// row (the block or group that leaves the window is sealed by the decode warp
// whose range holds it).  No whole-vector groups (each (b, h) then owns
// everything it writes).  Both new rows come straight into registers, lane l
// holding channels [l*D/32, (l+1)*D/32), loaded together.  scratch: the seal's
// (44*D bytes).  *kstep / *vstep: the largest key / value step written (0 when none).
template <int D>
__device__ __forceinline__ void fused_append_body(const AppendArgs& ap, int b, int h, int n, unsigned char* scratch,
                                                  float* kstep, float* vstep) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31;
  const long xo = ((long)b * ap.k.H + h) * D + lane * CPL;
  float xk[CPL], xv[CPL];
  load_lane_row<CPL>(ap.k.x, xo, ap.k.x_f32, xk);
  load_lane_row<CPL>(ap.v.x, xo, ap.v.x_f32, xv);
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const QuantArgs& q = t ? ap.v : ap.k;
    const float* x = t ? xv : xk;
    float st = 0.0f;
    if (q.L.axis == 1 || q.L.window) {
      __half2* row = reinterpret_cast<__half2*>(tail_row(q, b, h, n) + lane * CPL);
#pragma unroll
      for (int i = 0; i < CPL; i += 2) row[i / 2] = __halves2half2(__float2half_rn(x[i]), __float2half_rn(x[i + 1]));
      if (!q.L.window && ((n + 1) & (q.L.group - 1)) == 0) {
        __syncwarp();  // the new row is in the tail
        st = seal_channel_warp<CPL>(q, b, h, (n + 1) / q.L.group - 1, scratch);
      }
    } else {
      st = append_token_lanes<CPL>(q, b, h, n, x);
    }
    __syncwarp();  // scratch free for the next tensor
    if (t) *vstep = st;
    else *kstep = st;
  }
}

// The append as the decode kernel calls it.  head_dim 64 kernels have
// registers to spare and take it inline (measured faster); the 128 / 256 ones
// are at their register cap, where inlining it slowed every warp's tile loop
// (about 4 % on a Llama-2-13B-shaped batch), so they call it out of line.
template <int D>
static __device__ __noinline__ void fused_append_call(const AppendArgs& ap, int b, int h, int n,
                                                      unsigned char* scratch, float* kstep, float* vstep) {
  fused_append_body<D>(ap, b, h, n, scratch, kstep, vstep);
}

// Seal, inside a fused append + decode launch, the block (per-token tensor:
// the 16 tokens from t0) or group (per-channel tensor) of (b, h) that leaves
// the full-precision window, from its fp16 rows; returns its largest step.
// Out of line: it runs once per 16 or G steps of a sequence.
template <int D>
static __device__ __noinline__ float seal_window_block(const QuantArgs& q, int b, int h, int t0,
                                                       unsigned char* scratch) {
  const float st = q.L.axis == 1 ? seal_channel_warp<D / 32>(q, b, h, t0 / q.L.group, scratch)
                                 : seal_token_block_warp<D / 32>(q, b, h, t0 / kTile, scratch);
  __syncwarp();  // scratch free for the next tensor
  return st;
}

template <int D>
__device__ __forceinline__ void fused_append(const AppendArgs& ap, int b, int h, int n, unsigned char* scratch,
                                             float* kstep, float* vstep) {
  if constexpr (D == 64) fused_append_body<D>(ap, b, h, n, scratch, kstep, vstep);
  else fused_append_call<D>(ap, b, h, n, scratch, kstep, vstep);
}

}  // namespace kvq
