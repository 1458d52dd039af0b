// kvq_quant.cu — quantize-and-pack kernels of libkvq: prefill, append with
// group sealing, and the canonical export used for inspection.
//
// The quantizer follows "O Seu Cache KV Nao Tem um Problema de Bits. Tem um
// Problema de Geometria", section "O Que o Erro de Quantizacao E Realmente
// Feito" (zero = group minimum, step = range/(2^B-1), round to nearest) and the
// symmetric form of "Kuantisasi KV Cache untuk Mengurangi Memory Inferensi Long
// Context", section "Scale menentukan sistem koordinat kuantisasi".  Grouping
// axes follow sections "Chaves..." (keys per channel along tokens) and
// "Valores..." (values per token along channels); per-channel groups are only
// sealed once G tokens exist, the newer tokens stay in an fp16 tail (section
// "O Imposto dos Sistemas e Por Que Nao E um Detalhe").
//
// Group statistics are warp-shuffle min/max/absmax reductions; codes are
// assembled into the fragment-ordered tile words of kvq_common.cuh and written
// with 128-bit stores where a thread owns four consecutive words.
#include <algorithm>

#include "kvq_decode.cuh"
#include "kvq_internal.h"

namespace kvq {

// --------------------------------------------------------------- prefill ---

// Quantize a per-channel group block: G tokens x D channels of head h held in
// shared memory as floats; writes the D metadata entries of group g and the
// G/16 tiles.  All threads of the block participate.
__device__ void quant_channel_block(const QuantArgs& a, int b, int h, int g, const float* xs, uint8_t* cs,
                                    float* zs, float* ss) {
  const int G = a.L.group, D = a.D;
  char* meta = meta_ptr(a);
  float smax_local = 0.0f;
  // one thread per channel, reading the column in token order (consecutive
  // threads, consecutive banks); min, max and absmax are exact in any order
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float mn = INFINITY, mx = -INFINITY, am = 0.0f;
    for (int t = 0; t < G; ++t) {
      const float v = xs[t * D + c];
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
      am = fmaxf(am, fabsf(v));
    }
    float z, s;
    group_params(mn, mx, am, a.L.bits, a.L.sym, a.L.meta_f32, &z, &s);
    zs[c] = z;
    ss[c] = s;
    store_meta(meta, (((long)b * a.H + h) * (a.tcap / G) + g) * D + c, a.L.meta_f32, a.L.sym, z, s);
    smax_local = fmaxf(smax_local, s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) smax_local = fmaxf(smax_local, __shfl_xor_sync(0xffffffffu, smax_local, o));
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    int c = i % D;
    cs[i] = (uint8_t)quant_code(xs[i], zs[c], ss[c], a.L.bits, a.L.sym);
  }
  __syncthreads();
  for (int tt = 0; tt < G / kTile; ++tt)
    store_tile(codes_ptr(a, b, h, (g * G) / kTile + tt), cs + tt * kTile * D, D, a.L, a.is_value);
  if ((threadIdx.x & 31) == 0) atomic_max_pos(a.smax + (long)b * a.H + h, smax_local);
}

// Per-channel tensors: one CTA per (group, head, sequence).  The CTA of the
// first unsealed group also writes the fp16 tail.
__global__ void prefill_channel_kernel(QuantArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int G = a.L.group, D = a.D;
  const int n = a.lens[b];
  const int ns = (int)sealed_tokens(a.L, n);
  const int ng = ns / G;
  if (g > ng || (g == ng && ns == n)) return;
  const long xs_t = (long)a.H * D;
  const char* xb = reinterpret_cast<const char*>(a.x);
  if (g == ng) {  // unsealed tokens [ns, n) rounded to nearest fp16, into the fp16 rows
    int cnt = (n - ns) * D;
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
      int tt = i / D, c = i % D;
      long src = ((long)b * a.t_stride + ns + tt) * xs_t + (long)h * D + c;
      tail_row(a, b, h, ns + tt)[c] = __float2half_rn(load_in(xb, src, a.x_f32));
    }
    return;
  }
  float* xs = reinterpret_cast<float*>(smem);
  uint8_t* cs = reinterpret_cast<uint8_t*>(xs + G * D);
  float* zs = reinterpret_cast<float*>(cs + G * D);
  float* ss = zs + D;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    int tt = i / D, c = i % D;
    long src = ((long)b * a.t_stride + (long)g * G + tt) * xs_t + (long)h * D + c;
    // per-channel groups are formed from the fp16 staging precision of the tail
    xs[i] = __half2float(__float2half_rn(load_in(xb, src, a.x_f32)));
  }
  __syncthreads();
  quant_channel_block(a, b, h, g, xs, cs, zs, ss);
}

// Quantize one 16-token tile of a per-token tensor: tokens tile*16 + tt (tt <
// valid) of heads h0 .. h0+nh-1 held in shared memory as floats xs[16][nh*D];
// writes each token's group metadata and the nh packed tiles.  All threads of
// the block participate.
__device__ void quant_token_tile(const QuantArgs& a, int b, int h0, int nh, int tile, int valid, const float* xs,
                                 uint8_t* cs, float* zs, float* ss) {
  const int D = a.D, whole = a.L.whole;
  const int rowlen = nh * D;
  const int G = whole ? rowlen : a.L.group;
  const int gpr = rowlen / G;  // groups per token row in this CTA
  const int warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  char* meta = meta_ptr(a);
  float smax_local = 0.0f;
  for (int gi = warp; gi < kTile * gpr; gi += nwarp) {
    int tt = gi / gpr, j = gi % gpr;
    int t = tile * kTile + tt;
    if (tt >= valid) continue;
    float mn, mx, am;
    warp_stats(xs + tt * rowlen + j * G, G, 1, &mn, &mx, &am);
    float z, s;
    group_params(mn, mx, am, a.L.bits, a.L.sym, a.L.meta_f32, &z, &s);
    if ((threadIdx.x & 31) == 0) {
      zs[gi] = z;
      ss[gi] = s;
      long mi = whole ? ((long)b * a.tcap + t) : ((((long)b * a.H + h0) * a.tcap + t) * gpr + j);
      store_meta(meta, mi, a.L.meta_f32, a.L.sym, z, s);
      smax_local = fmaxf(smax_local, s);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kTile * rowlen; i += blockDim.x) {
    int tt = i / rowlen, c = i % rowlen;
    int hh = c / D, cc = c % D;
    uint8_t code = 0;
    if (tt < valid) code = (uint8_t)quant_code(xs[i], zs[tt * gpr + c / G], ss[tt * gpr + c / G], a.L.bits, a.L.sym);
    cs[(hh * kTile + tt) * D + cc] = code;
  }
  __syncthreads();
  for (int hh = 0; hh < nh; ++hh) store_tile(codes_ptr(a, b, h0 + hh, tile), cs + hh * kTile * D, D, a.L, a.is_value);
  if ((threadIdx.x & 31) == 0 && smax_local > 0.0f)
    for (int hh = 0; hh < nh; ++hh) atomic_max_pos(a.smax + (long)b * a.H + h0 + hh, smax_local);
}

// Per-token tensors: one CTA per (tile, head, sequence); for whole-vector
// groups one CTA per (tile, sequence) covering every head (blockIdx.y == 0).
// With a recent window, tiles older than the window are quantized from the
// inputs rounded to fp16 and the newer tiles go to the fp16 rows.
__global__ void prefill_token_kernel(QuantArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tile = blockIdx.x, b = blockIdx.z;
  const int D = a.D;
  const int n = a.lens[b];
  if (tile * kTile >= n) return;
  const int ns = (int)sealed_tokens(a.L, n);
  const int whole = a.L.whole;
  const int h0 = whole ? 0 : blockIdx.y, nh = whole ? a.H : 1;
  const int rowlen = nh * D;  // channels handled per token
  const int G = whole ? rowlen : a.L.group;
  const int gpr = rowlen / G;
  const long xs_t = (long)a.H * D;
  if (tile * kTile >= ns) {  // fp16 rows (a window's tiles are never partly sealed)
    for (int i = threadIdx.x; i < kTile * rowlen; i += blockDim.x) {
      int tt = i / rowlen, c = i % rowlen;
      int t = tile * kTile + tt;
      if (t >= n) continue;
      tail_row(a, b, h0 + c / D, t)[c % D] =
          __float2half_rn(load_in(a.x, ((long)b * a.t_stride + t) * xs_t + (long)h0 * D + c, a.x_f32));
    }
    return;
  }
  float* xs = reinterpret_cast<float*>(smem);                       // [16][rowlen]
  uint8_t* cs = reinterpret_cast<uint8_t*>(xs + kTile * rowlen);    // [nh][16][D]
  float* zs = reinterpret_cast<float*>(cs + kTile * rowlen);        // [16*gpr]
  float* ss = zs + kTile * gpr;
  for (int i = threadIdx.x; i < kTile * rowlen; i += blockDim.x) {
    int tt = i / rowlen, c = i % rowlen;
    int t = tile * kTile + tt;
    float x = t < n ? load_in(a.x, ((long)b * a.t_stride + t) * xs_t + (long)h0 * D + c, a.x_f32) : 0.0f;
    if (a.L.window) x = __half2float(__float2half_rn(x));  // quantized after a stay in the window
    xs[i] = x;
  }
  __syncthreads();
  quant_token_tile(a, b, h0, nh, tile, min(kTile, n - tile * kTile), xs, cs, zs, ss);
}

// lens[b] and every per-head copy head_lens[b][h] of the layer
__global__ void set_lens_kernel(int32_t* lens, int32_t* head_lens, LensArg la, int B, int H) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < B * H) {
    const int b = i / H;
    head_lens[i] = la.v[b];
    if (i % H == 0) lens[b] = la.v[b];
  }
}

// ---------------------------------------------------------------- append ---


// One CTA of 128 threads per (sequence, kv head): warp 0 appends the key, warp 1
// the value; a per-channel tensor whose tail just filled up is then sealed by
// all four warps.  Each CTA reads and advances only its own per-head length
// counter (no other CTA of the launch touches it), and the head-0 CTA also
// advances the sequence length, which no CTA of the launch reads: no ticket,
// fence or waiting is needed.
__global__ void append_kernel(const __grid_constant__ AppendArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int seal[2];
  const int b = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  int32_t* my_len = a.head_lens + (long)b * gridDim.y + h;
  pdl_wait();
  pdl_trigger();  // the decode that follows may get its CTAs resident now
  const int n = *my_len;
  const QuantArgs& t = warp == 0 ? a.k : a.v;
  bool full = false;
  if (warp < 2 && !(t.L.whole && h != 0)) {
    const int rowlen = (t.L.whole ? t.H : 1) * t.D;
    unsigned char* base = smem + warp * a.warp_smem;
    float* xs = reinterpret_cast<float*>(base);
    float* zs = xs + rowlen;
    float* ss = zs + 16;
    uint8_t* cs = reinterpret_cast<uint8_t*>(ss + 16);
    full = append_warp(t, b, h, n, xs, cs, zs, ss);
  }
  if (warp < 2 && (threadIdx.x & 31) == 0) seal[warp] = full ? 1 : 0;
  __syncthreads();
  for (int w = 0; w < 2; ++w) {
    if (!seal[w]) continue;
    const QuantArgs& q = w == 0 ? a.k : a.v;
    const int D = q.D, old = n + 1 - q.L.window;
    if (q.L.axis == 1) {
      // seal per-channel group g from its fp16 rows
      const int G = q.L.group, g = old / G - 1;
      float* xs = reinterpret_cast<float*>(smem);
      uint8_t* cs = reinterpret_cast<uint8_t*>(xs + G * D);
      float* zs = reinterpret_cast<float*>(cs + G * D);
      float* ss = zs + D;
      const int lgD = 31 - __clz(D);  // D is a power of two
      for (int i = threadIdx.x; i < G * D; i += blockDim.x)
        xs[i] = __half2float(tail_row(q, b, h, (long)g * G + (i >> lgD))[i & (D - 1)]);
      __syncthreads();
      quant_channel_block(q, b, h, g, xs, cs, zs, ss);
    } else {
      // quantize per-token block `tile` from its fp16 rows (all heads for whole-vector groups)
      const int tile = old / kTile - 1;
      const int nh = q.L.whole ? q.H : 1, rowlen = nh * D;
      const int gpr = rowlen / (q.L.whole ? rowlen : q.L.group);
      float* xs = reinterpret_cast<float*>(smem);                     // [16][rowlen]
      uint8_t* cs = reinterpret_cast<uint8_t*>(xs + kTile * rowlen);  // [nh][16][D]
      float* zs = reinterpret_cast<float*>(cs + kTile * rowlen);
      float* ss = zs + kTile * gpr;
      for (int i = threadIdx.x; i < kTile * rowlen; i += blockDim.x) {
        const int tt = i / rowlen, c = i % rowlen;
        xs[i] = __half2float(tail_row(q, b, h + c / D, (long)tile * kTile + tt)[c % D]);
      }
      __syncthreads();
      quant_token_tile(q, b, h, nh, tile, kTile, xs, cs, zs, ss);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *my_len = n + 1;
    if (h == 0) a.lens[b] = n + 1;
  }
}

// ---------------------------------------------------------------- export ---

struct ExportArgs {
  QuantArgs a;
  uint8_t* codes;    // [B][H][tcap][D] or null
  float* meta;       // [groups][2] or null
  uint16_t* tail;    // [B][H][G][D] or null
};

__device__ __forceinline__ int sealed_of(const TensorLayout& L, int n) { return (int)sealed_tokens(L, n); }
// codes: one CTA per (tile, head, sequence)
__global__ void export_codes_kernel(ExportArgs e) {
  const QuantArgs& a = e.a;
  const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z, D = a.D;
  const int ns = sealed_of(a.L, a.lens[b]);
  const uint32_t* src = codes_ptr(a, b, h, tile);
  for (int i = threadIdx.x; i < kTile * D; i += blockDim.x) {
    int tt = i / D, c = i % D, t = tile * kTile + tt;
    uint32_t code = 0;
    if (t < ns) {
      FragPos f = elem_pos(a.is_value, tt, c);
      for (int p = 0; p < a.L.planes.n; ++p) {
        int word, bit;
        plane_word_bit(f, D, a.L.planes.w[p], a.L.planes.off[p], &word, &bit);
        code |= ((src[word] >> bit) & ((1u << a.L.planes.w[p]) - 1u)) << a.L.planes.off[p];
      }
    }
    e.codes[(((long)b * a.H + h) * a.tcap + t) * D + c] = (uint8_t)code;
  }
}

// metadata: one thread per canonical group entry
__global__ void export_meta_kernel(ExportArgs e, long ngroups) {
  const QuantArgs& a = e.a;
  long gi = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gi >= ngroups) return;
  const int D = a.D;
  int b, valid;
  if (a.L.axis == 1) {
    long per_b = (long)a.H * (a.tcap / a.L.group) * D;
    b = (int)(gi / per_b);
    long g = (gi / D) % (a.tcap / a.L.group);
    valid = g < sealed_of(a.L, a.lens[b]) / a.L.group;
  } else if (a.L.whole) {
    b = (int)(gi / a.tcap);
    valid = (gi % a.tcap) < sealed_of(a.L, a.lens[b]);
  } else {
    long per_b = (long)a.H * a.tcap * a.L.gpt;
    b = (int)(gi / per_b);
    long t = (gi / a.L.gpt) % a.tcap;
    valid = t < sealed_of(a.L, a.lens[b]);
  }
  float z = 0.0f, s = 0.0f;
  if (valid) load_meta(meta_ptr(a), gi, a.L.meta_f32, a.L.sym, &z, &s);
  e.meta[2 * gi] = z;
  e.meta[2 * gi + 1] = s;
}

// fp16 rows in token order (row t - sealed): one CTA per (head, sequence)
__global__ void export_tail_kernel(ExportArgs e) {
  const QuantArgs& a = e.a;
  const int h = blockIdx.y, b = blockIdx.z, D = a.D, rows = a.L.ring;
  const int n = a.lens[b], ns = sealed_of(a.L, n);
  for (int i = threadIdx.x; i < rows * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    uint16_t v = ns + r < n ? __half_as_ushort(tail_row(a, b, h, ns + r)[c]) : (uint16_t)0;
    e.tail[(((long)b * a.H + h) * rows) * D + i] = v;
  }
}

// ------------------------------------------------------ materialised path --

// Dequantise one tensor of a layer into fp16 rows out[b][h][t][D] (t < lens[b]):
// x_hat = z + code * s (asymmetric, one fp32 fma), (code - 2^(B-1)) * s
// (symmetric), the stored fp16 value for the tail, then rounded to nearest
// fp16.  This is the "dequantise the cached block into a temporary
// floating-point tensor before attention" design of "Kuantisasi KV Cache untuk
// Mengurangi Memory Inferensi Long Context", section "Kuantisasi dapat
// memindahkan pekerjaan ke decode path", kept as the baseline the fused decode
// is measured against.  One CTA per (tile, head, sequence): each warp turns
// whole 16-channel chunks into exact fp16 codes with the decode path's
// register conversion, applies the group's zero point and step per element
// into a shared tile, and the CTA writes the tile's valid rows with 16-byte
// stores.
template <int D>
__global__ void __launch_bounds__(128) dequant_kernel(QuantArgs a, __half* out, long t_stride) {
  // one 16-token tile per warp, four consecutive tiles per CTA
  __shared__ __align__(16) __half tileo[kWarps][kTile * D];
  const int h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const int tile = blockIdx.x * kWarps + warp;
  const int n = a.lens[b];
  const int t_base = tile * kTile;
  if (t_base >= n) return;
  const int ns = sealed_of(a.L, n);
  __half* to = tileo[warp];
  if (t_base < ns) {
    const uint32_t* src = codes_ptr(a, b, h, tile);
    const char* meta = meta_ptr(a);
    const int bits = a.L.bits;
    const int cg = conv_g(bits), cr = conv_r(bits), cc = conv_c(bits);
    const float off = (float)conv_off(bits), soff = (float)(1 << (bits - 1));
    const int G = a.L.whole ? a.H * D : a.L.group;
    const int lgG = 31 - __clz(G);
    const long bh = (long)b * a.H + h;
    for (int j = 0; j < D / 16; ++j) {
      uint32_t A[4];
      convert_dispatch<D>(bits, src, lane, j, A);
      // the lane's 8 elements share 4 metadata entries: keys (rows = tokens) need
      // channels 2tig, 2tig+1, 2tig+8, 2tig+9 of the chunk (per-channel) or the
      // group of each row token (per-token); values (rows = channels) need
      // tokens 2tig, 2tig+1, 2tig+8, 2tig+9 (per-token) or the two row channels
      float mz[4], ms[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int kk = 2 * tig + (m & 1) + 8 * (m >> 1);  // column of entry m
        long mi;
        if (a.L.axis == 1) {
          // per-channel: entry per column channel (keys) or row channel (values)
          const int c = a.is_value ? 16 * j + g + 8 * (m & 1) : 16 * j + kk;
          mi = (bh * (a.tcap >> lgG) + (t_base >> lgG)) * D + c;
        } else {
          // per-token: entry per column token (values) or row token (keys)
          const long ta = t_base + (a.is_value ? kk : g + 8 * (m & 1));
          const int c = a.is_value ? 16 * j + g : 16 * j + kk;
          mi = a.L.whole ? (long)b * a.tcap + ta : (bh * a.tcap + ta) * a.L.gpt + (c >> lgG);
        }
        load_meta(meta, mi, a.L.meta_f32, a.L.sym, &mz[m], &ms[m]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float unscale = exp2i(-(cg + cr * (r & 1) + cc * (r >> 1)));
        const __half2 hv = *reinterpret_cast<const __half2*>(&A[r]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int R = g + 8 * (r & 1), kk = 2 * tig + 8 * (r >> 1) + e;
          const int t = a.is_value ? kk : R, c = 16 * j + (a.is_value ? R : kk);
          // entry index: the column (e, column half) for per-channel keys and
          // per-token values, the row (row half) otherwise
          const bool by_col = (a.L.axis == 1) != (a.is_value != 0);
          const int m = by_col ? (e + 2 * (r >> 1)) : (r & 1);
          const float code = (e ? __high2float(hv) : __low2float(hv)) * unscale - off;
          const float x = a.L.sym ? (code - soff) * ms[m] : __fmaf_rn(code, ms[m], mz[m]);
          to[t * D + c] = __float2half_rn(x);
        }
      }
    }
  }
  __syncwarp();
  __half* dst = out + ((bh_of(a, b, h)) * t_stride + t_base) * D;
  for (int i = lane; i < kTile * D / 8; i += 32) {
    const int t = (i * 8) / D, c = (i * 8) % D, ta = t_base + t;
    if (ta >= n) continue;
    const uint4 v = ta < ns ? *reinterpret_cast<const uint4*>(to + t * D + c)
                            : *reinterpret_cast<const uint4*>(tail_row(a, b, h, ta) + c);
    *reinterpret_cast<uint4*>(dst + (long)t * D + c) = v;
  }
}

// ------------------------------------------------------------- launchers ---

static QuantArgs make_args(const kvq_cache* C, int is_value, int layer, const void* x, int x_f32, long t_stride) {
  QuantArgs a;
  a.L = is_value ? C->v : C->k;
  a.is_value = is_value;
  a.layer = layer;
  a.B = C->cfg.batch;
  a.H = C->cfg.kv_heads;
  a.D = C->cfg.head_dim;
  a.tcap = C->tcap;
  a.ntiles = C->tcap / kTile;
  a.x = x;
  a.x_f32 = x_f32;
  a.t_stride = t_stride;
  a.lens = C->d_lens + (long)layer * C->cfg.batch;
  a.base = C->base;
  a.smax = C->d_smax + ((long)is_value * C->cfg.layers + layer) * C->cfg.batch * C->cfg.kv_heads;
  return a;
}

static size_t channel_smem(int G, int D) { return (size_t)G * D * 5 + (size_t)D * 8 + 16; }
static size_t token_smem(const kvq_cache* C, const TensorLayout& L);

cudaError_t launch_prefill(kvq_cache* C, int layer, const void* k, const void* v, int x_f32,
                           const int32_t* lens_host, long t_stride, cudaStream_t st, int* launches) {
  const int B = C->cfg.batch, H = C->cfg.kv_heads, D = C->cfg.head_dim;
  LensArg la;
  for (int b = 0; b < B; ++b) la.v[b] = lens_host[b];
  int32_t* dl = C->d_lens + (long)layer * B;
  int32_t* dhl = C->d_head_lens + (long)layer * B * H;
  set_lens_kernel<<<(B * H + 127) / 128, 128, 0, st>>>(dl, dhl, la, B, H);
  ++*launches;
  // the layer's max-step statistics restart with the new contents
  for (int is_v = 0; is_v < 2; ++is_v) {
    uint32_t* sm = C->d_smax + ((long)is_v * C->cfg.layers + layer) * B * H;
    cudaError_t e = cudaMemsetAsync(sm, 0, sizeof(uint32_t) * B * H, st);
    if (e != cudaSuccess) return e;
  }
  int maxn = 0;
  for (int b = 0; b < B; ++b) maxn = lens_host[b] > maxn ? lens_host[b] : maxn;
  for (int is_v = 0; is_v < 2; ++is_v) {
    QuantArgs a = make_args(C, is_v, layer, is_v ? v : k, x_f32, t_stride);
    if (maxn == 0) continue;
    if (prefill_fast_ok(a)) {
      cudaError_t e = launch_prefill_fast(a, maxn, st);
      if (e != cudaSuccess) return e;
    } else if (a.L.axis == 1) {
      size_t sm = channel_smem(a.L.group, D);
      dim3 grid((maxn + a.L.group - 1) / a.L.group + 1, H, B);
      prefill_channel_kernel<<<grid, 256, sm, st>>>(a);
    } else {
      size_t sm = token_smem(C, a.L);
      dim3 grid((maxn + kTile - 1) / kTile, a.L.whole ? 1 : H, B);
      prefill_token_kernel<<<grid, 256, sm, st>>>(a);
    }
    ++*launches;
  }
  return cudaGetLastError();
}

static int append_warp_smem(const kvq_cache* C) {
  const int H = C->cfg.kv_heads, D = C->cfg.head_dim;
  int m = 0;
  const TensorLayout* ls[2] = {&C->k, &C->v};
  for (int i = 0; i < 2; ++i) {
    const int rowlen = (ls[i]->whole ? H : 1) * D;
    m = std::max(m, rowlen * 5 + 128 + 16);
  }
  return (m + 15) / 16 * 16;
}

size_t append_smem(const kvq_cache* C) {
  size_t m = 2 * (size_t)append_warp_smem(C);
  const TensorLayout* ls[2] = {&C->k, &C->v};
  for (int i = 0; i < 2; ++i) {
    if (ls[i]->axis == 1) m = std::max(m, channel_smem(ls[i]->group, C->cfg.head_dim));
    else if (ls[i]->window) m = std::max(m, token_smem(C, *ls[i]));  // per-token block seal
  }
  return m;
}

cudaError_t launch_dequantize(kvq_cache* C, int layer, void* k_out, void* v_out, cudaStream_t st, int* launches) {
  const int B = C->cfg.batch, H = C->cfg.kv_heads;
  int maxn = 0;
  // host mirror raised to the plan hint, as for decode (CTAs past a length exit)
  for (int b = 0; b < B; ++b)
    maxn = std::max(maxn, std::max((int)C->lens[(long)layer * B + b], std::min(C->plan_tokens, C->cfg.max_tokens)));
  if (maxn == 0) return cudaSuccess;
  for (int is_v = 0; is_v < 2; ++is_v) {
    QuantArgs a = make_args(C, is_v, layer, nullptr, 0, 0);
    const dim3 grid((maxn + kTile * kWarps - 1) / (kTile * kWarps), H, B);
    __half* o = static_cast<__half*>(is_v ? v_out : k_out);
    const int D = C->cfg.head_dim;
    if (D == 64) dequant_kernel<64><<<grid, 128, 0, st>>>(a, o, C->tcap);
    else if (D == 128) dequant_kernel<128><<<grid, 128, 0, st>>>(a, o, C->tcap);
    else dequant_kernel<256><<<grid, 128, 0, st>>>(a, o, C->tcap);
    ++*launches;
  }
  return cudaGetLastError();
}

AppendArgs make_append_args(const kvq_cache* C, int layer, const void* k, const void* v, int x_f32) {
  AppendArgs a;
  a.k = make_args(C, 0, layer, k, x_f32, 1);
  a.v = make_args(C, 1, layer, v, x_f32, 1);
  a.lens = C->d_lens + (long)layer * C->cfg.batch;
  a.head_lens = C->d_head_lens + (long)layer * C->cfg.batch * C->cfg.kv_heads;
  a.warp_smem = append_warp_smem(C);
  return a;
}

cudaError_t launch_append(kvq_cache* C, int layer, const void* k, const void* v, int x_f32, cudaStream_t st,
                          int* launches) {
  AppendArgs a = make_append_args(C, layer, k, v, x_f32);
  size_t sm = append_smem(C);
  void* args[] = {&a};
  cudaError_t e = launch_pdl(reinterpret_cast<const void*>(&append_kernel), dim3(C->cfg.batch, C->cfg.kv_heads),
                             dim3(128), sm, st, args);
  if (e != cudaSuccess) return e;
  ++*launches;
  return cudaGetLastError();
}

static size_t token_smem(const kvq_cache* C, const TensorLayout& L) {
  const int rowlen = (L.whole ? C->cfg.kv_heads : 1) * C->cfg.head_dim;
  const int gpr = L.whole ? 1 : C->cfg.head_dim / L.group;
  return (size_t)kTile * rowlen * 5 + (size_t)kTile * gpr * 8 + 16;
}

cudaError_t quant_setup(kvq_cache* C) {
  size_t chan = 0, tok = 0;
  const TensorLayout* ls[2] = {&C->k, &C->v};
  for (int i = 0; i < 2; ++i) {
    if (ls[i]->axis == 1) chan = std::max(chan, channel_smem(ls[i]->group, C->cfg.head_dim));
    else tok = std::max(tok, token_smem(C, *ls[i]));
  }
  cudaError_t e = cudaSuccess;
  if (chan) e = cudaFuncSetAttribute(prefill_channel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chan);
  if (e == cudaSuccess && tok)
    e = cudaFuncSetAttribute(prefill_token_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tok);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)append_smem(C));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(append_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess) e = prefill_fast_setup();
  return e;
}

cudaError_t launch_export(kvq_cache* C, int layer, int is_value, uint8_t* codes, float* meta, uint16_t* tail,
                          cudaStream_t st) {
  ExportArgs e;
  e.a = make_args(C, is_value, layer, nullptr, 0, 0);
  e.codes = codes;
  e.meta = meta;
  e.tail = tail;
  const int B = C->cfg.batch, H = C->cfg.kv_heads;
  if (codes) export_codes_kernel<<<dim3(C->tcap / kTile, H, B), 256, 0, st>>>(e);
  if (meta) {
    long ng = meta_groups(C, e.a.L);
    export_meta_kernel<<<(unsigned)((ng + 255) / 256), 256, 0, st>>>(e, ng);
  }
  if (tail && e.a.L.ring) export_tail_kernel<<<dim3(1, H, B), 256, 0, st>>>(e);
  return cudaGetLastError();
}

}  // namespace kvq
