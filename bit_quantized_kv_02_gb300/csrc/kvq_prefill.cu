// kvq_prefill.cu — the fast prefill quantize-and-pack kernels (fp16 inputs,
// per-channel groups or per-token groups within one head, no full-precision
// window).  Any other layout runs the general kernels of kvq_quant.cu; both
// produce the same cache bit for bit.
//
// The quantizer follows "O Seu Cache KV Nao Tem um Problema de Bits. Tem um
// Problema de Geometria", section "O Que o Erro de Quantizacao E Realmente
// Feito" (zero = group minimum, step = range/(2^B-1), round to nearest) and
// the symmetric form of "Kuantisasi KV Cache untuk Mengurangi Memory Inferensi
// Long Context", section "Scale menentukan sistem koordinat kuantisasi";
// per-channel groups are sealed once G tokens exist and newer tokens stay in
// an fp16 tail ("O Imposto dos Sistemas e Por Que Nao E um Detalhe").
//
// One warp per unit of work: a per-channel group (G tokens x head_dim of one
// (sequence, head)) or a 16-token tile of a per-token tensor.
//   1. the unit's fp16 rows are staged in shared memory with 16-byte cp.async
//      (rows padded by 16 bytes so that ldmatrix below is conflict-free);
//   2. group statistics: per channel, each lane owns head_dim/32 adjacent
//      channels and scans the G rows with fp16x2 min/max; per token, each lane
//      owns up to 32 channels of one row and lanes sharing a group finish the
//      reduction with shuffles.  min / max / absmax are exact in any order;
//   3. each element's code (the step's reciprocal, quant_code_try, for a row
//      or vector of values at once; where any of them lies near a
//      half-integer the same values again with quant_code_fast, which takes
//      the IEEE division there) is written back over its fp16 input as a
//      16-bit integer;
//   4. ldmatrix (.trans for values) delivers every lane the codes of exactly
//      its own fragment positions of each 16-token tile (kvq_common.cuh), so
//      each lane shifts them into its tile words and stores them with 16-byte
//      stores: no exchange between lanes.
#include <algorithm>

#include "kvq_quant.cuh"

namespace kvq {

namespace {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Shared-memory row stride (bytes) of D fp16 / 16-bit values: 16 bytes of
// padding put the eight rows an ldmatrix reads in eight different bank groups.
__host__ __device__ constexpr int row_bytes(int D) { return 2 * D + 16; }

// Pack the 16-bit codes of one 16-token tile (shared memory rows at `tile`,
// stride row_bytes(D), token-major) into this lane's tile words and store
// them.  ldmatrix register r of chunk j holds pair 4j + r of this lane: the
// codes of elements e = 0 (low half) and 1 (high half).
template <int D, int BITS>
__device__ __forceinline__ void pack_store_tile(uint32_t tile, int is_value, uint32_t* dst, int lane) {
  constexpr int NCH = D / 16;
  // this lane's ldmatrix row address: matrix m = lane / 8, row lane % 8
  const int m = lane >> 3, rw = lane & 7;
  const int rh = m & 1, kh = m >> 1;
  // keys: stored rows = fragment rows (tokens 8*rh + rw), columns 16j + 8*kh;
  // values: stored rows = fragment columns (tokens 8*kh + rw), columns 16j + 8*rh
  const int trow = is_value ? 8 * kh + rw : 8 * rh + rw;
  const int coff = is_value ? 8 * rh : 8 * kh;
  const uint32_t base = tile + trow * row_bytes(D) + coff * 2;
  constexpr int NP = np_of(BITS);
  // words of every plane of this lane (plane p: D*w/64 words)
  constexpr int WTOT = D * BITS / 64;
  uint32_t words[WTOT];
#pragma unroll
  for (int i = 0; i < WTOT; ++i) words[i] = 0u;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    uint32_t r[4];
    if (is_value) ldsm_x4_t(base + 32 * j, r);
    else ldsm_x4(base + 32 * j, r);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int pi = 4 * j + q;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const int w = pw_of(BITS, p), off = po_of(BITS, p);
        const int P = 16 / w;
        // first word of plane p among this lane's words
        int wbase = 0;
#pragma unroll
        for (int pp = 0; pp < p; ++pp) wbase += D * pw_of(BITS, pp) / 64;
        const uint32_t mask = ((1u << w) - 1u) * 0x00010001u;
        const uint32_t v = (off ? (r[q] >> off) : r[q]) & mask;
        words[wbase + pi / P] |= v << ((pi % P) * w);
      }
    }
  }
  // plane p's words of this lane sit at D*off_p/2 + lane*W_p
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int w = pw_of(BITS, p), off = po_of(BITS, p);
    const int W = D * w / 64;
    int wbase = 0;
#pragma unroll
    for (int pp = 0; pp < p; ++pp) wbase += D * pw_of(BITS, pp) / 64;
    uint32_t* o = dst + D * off / 2 + lane * W;
    if (W % 4 == 0) {
#pragma unroll
      for (int i = 0; i < W; i += 4)
        *reinterpret_cast<uint4*>(o + i) =
            make_uint4(words[wbase + i], words[wbase + i + 1], words[wbase + i + 2], words[wbase + i + 3]);
    } else if (W % 2 == 0) {
#pragma unroll
      for (int i = 0; i < W; i += 2) *reinterpret_cast<uint2*>(o + i) = make_uint2(words[wbase + i], words[wbase + i + 1]);
    } else {
      o[0] = words[wbase];
    }
  }
}

template <int D>
__device__ __forceinline__ void pack_store_dispatch(int bits, uint32_t tile, int is_value, uint32_t* dst, int lane) {
  switch (bits) {
    case 2: pack_store_tile<D, 2>(tile, is_value, dst, lane); break;
    case 3: pack_store_tile<D, 3>(tile, is_value, dst, lane); break;
    case 4: pack_store_tile<D, 4>(tile, is_value, dst, lane); break;
    case 5: pack_store_tile<D, 5>(tile, is_value, dst, lane); break;
    case 6: pack_store_tile<D, 6>(tile, is_value, dst, lane); break;
    case 7: pack_store_tile<D, 7>(tile, is_value, dst, lane); break;
    default: pack_store_tile<D, 8>(tile, is_value, dst, lane); break;
  }
}

// Stage rows [t0, t0 + nrows) of head h of sequence b (fp16, [B][t_stride][H][D])
// into shared memory at `sm` (row stride row_bytes(D)); rows >= valid are left alone.
template <int D>
__device__ __forceinline__ void stage_rows(const QuantArgs& a, int b, int h, long t0, int nrows, int valid,
                                           uint32_t sm, int lane) {
  constexpr int CH = D * 2 / 16;  // 16-byte pieces per row
  const char* src = reinterpret_cast<const char*>(a.x) + (((long)b * a.t_stride + t0) * a.H + h) * (long)D * 2;
  const long rstride = (long)a.H * D * 2;
  const int n = min(nrows, valid);
  for (int i = lane; i < n * CH; i += 32) {
    const int r = i / CH, c = i - r * CH;
    cp_async16_s(sm + r * row_bytes(D) + c * 16, src + r * rstride + c * 16);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
}

constexpr int kPrefillWarps = 4;

}  // namespace

// Per-channel tensors: warp w of CTA (x, h, b) seals group g = 4x + w of
// (b, h) (G tokens x D channels; shared memory G rows per warp); the warp whose
// g is the first unsealed group copies the unsealed tokens to the fp16 rows.
template <int D>
__global__ void __launch_bounds__(kPrefillWarps * 32) prefill_channel_fast(QuantArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int CPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = blockIdx.x * kPrefillWarps + warp;
  const int G = a.L.group;
  const int n = a.lens[b];
  const int ns = (int)sealed_tokens(a.L, n);
  const int ng = ns / G;
  if (g > ng || (g == ng && ns == n)) return;
  if (g == ng) {  // unsealed tokens [ns, n), rounded to nearest fp16 (exact for fp16 inputs)
    const __half* xb = reinterpret_cast<const __half*>(a.x);
    for (int r = 0; r < n - ns; ++r) {
      const long src = ((long)b * a.t_stride + ns + r) * a.H * D + (long)h * D;
      __half* dst = tail_row(a, b, h, ns + r);
      for (int c = lane * 8; c < D; c += 256)
        *reinterpret_cast<uint4*>(dst + c) = *reinterpret_cast<const uint4*>(xb + src + c);
    }
    return;
  }
  const uint32_t sm = smem_u32(smem) + warp * G * row_bytes(D);
  unsigned char* smp = smem + warp * G * row_bytes(D);
  stage_rows<D>(a, b, h, (long)g * G, G, G, sm, lane);
  // statistics of this lane's CPL channels over the G rows
  __half2 mn[CPL / 2], mx[CPL / 2];
#pragma unroll
  for (int i = 0; i < CPL / 2; ++i) {
    mn[i] = __float2half2_rn(INFINITY);
    mx[i] = __float2half2_rn(-INFINITY);
  }
  for (int t = 0; t < G; ++t) {
    const __half2* row = reinterpret_cast<const __half2*>(smp + t * row_bytes(D)) + lane * (CPL / 2);
#pragma unroll
    for (int i = 0; i < CPL / 2; ++i) {
      const __half2 v = row[i];
      mn[i] = __hmin2(mn[i], v);
      mx[i] = __hmax2(mx[i], v);
    }
  }
  float z[CPL], s[CPL], rc[CPL];
  float smax_local = 0.0f;
  char* meta = meta_ptr(a);
  const long mrow = (((long)b * a.H + h) * (a.tcap / G) + g) * D + lane * CPL;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const float lo = (i & 1) ? __high2float(mn[i / 2]) : __low2float(mn[i / 2]);
    const float hi = (i & 1) ? __high2float(mx[i / 2]) : __low2float(mx[i / 2]);
    group_params(lo, hi, fmaxf(fabsf(lo), fabsf(hi)), a.L.bits, a.L.sym, a.L.meta_f32, &z[i], &s[i]);
    rc[i] = s[i] > 0.0f ? __frcp_rn(s[i]) : 0.0f;
    store_meta(meta, mrow + i, a.L.meta_f32, a.L.sym, z[i], s[i]);
    smax_local = fmaxf(smax_local, s[i]);
  }
  // codes, written over the inputs as 16-bit integers: the reciprocal rule
  // for the lane's CPL values of a row at once, the division-checked rule
  // for the (rare) row where any of them needs it
  bool lane_ok = true;
#pragma unroll
  for (int i = 0; i < CPL; ++i) lane_ok = lane_ok && (rc[i] >= 0x1p-125f || s[i] == 0.0f);
  for (int t = 0; t < G; ++t) {
    uint32_t* row = reinterpret_cast<uint32_t*>(smp + t * row_bytes(D)) + lane * (CPL / 2);
    float2 v[CPL / 2];
    uint32_t w[CPL / 2];
    bool ok = lane_ok;
#pragma unroll
    for (int i = 0; i < CPL / 2; ++i) {
      v[i] = __half22float2(*reinterpret_cast<const __half2*>(row + i));
      const uint32_t c0 = (uint32_t)quant_code_try(v[i].x, z[2 * i], rc[2 * i], a.L.bits, a.L.sym, ok);
      const uint32_t c1 = (uint32_t)quant_code_try(v[i].y, z[2 * i + 1], rc[2 * i + 1], a.L.bits, a.L.sym, ok);
      w[i] = c0 | (c1 << 16);
    }
    if (!ok) {
#pragma unroll
      for (int i = 0; i < CPL / 2; ++i) {
        const uint32_t c0 = (uint32_t)quant_code_fast(v[i].x, z[2 * i], s[2 * i], rc[2 * i], a.L.bits, a.L.sym);
        const uint32_t c1 =
            (uint32_t)quant_code_fast(v[i].y, z[2 * i + 1], s[2 * i + 1], rc[2 * i + 1], a.L.bits, a.L.sym);
        w[i] = c0 | (c1 << 16);
      }
    }
#pragma unroll
    for (int i = 0; i < CPL / 2; ++i) row[i] = w[i];
  }
  __syncwarp();
  for (int tt = 0; tt < G / kTile; ++tt)
    pack_store_dispatch<D>(a.L.bits, sm + tt * kTile * row_bytes(D), a.is_value, codes_ptr(a, b, h, g * G / kTile + tt),
                           lane);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) smax_local = fmaxf(smax_local, __shfl_xor_sync(0xffffffffu, smax_local, o));
  if (lane == 0) atomic_max_pos(a.smax + (long)b * a.H + h, smax_local);
}

// Per-token tensors (groups of G channels within one head): warp w of CTA
// (x, h, b) quantizes tile 4x + w of (b, h).  Lane unit u = (token, part of
// E = min(G, 32) channels); the G/E lanes of a group are adjacent and finish
// its statistics with shuffles.  Tokens past the sequence's end get code 0
// and no metadata.
template <int D>
__global__ void __launch_bounds__(kPrefillWarps * 32) prefill_token_fast(QuantArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int tile = blockIdx.x * kPrefillWarps + warp;
  const int n = a.lens[b];
  if (tile * kTile >= n) return;
  const int valid = min(kTile, n - tile * kTile);
  const int G = a.L.group;
  const int E = G < 32 ? G : 32;       // channels per lane unit
  const int lpg = G / E;               // lanes per group (1, 2, 4 or 8)
  const int upr = D / E;               // units per token row
  const int gpr = D / G;               // groups per token row
  const uint32_t sm = smem_u32(smem) + warp * kTile * row_bytes(D);
  unsigned char* smp = smem + warp * kTile * row_bytes(D);
  stage_rows<D>(a, b, h, (long)tile * kTile, kTile, valid, sm, lane);
  char* meta = meta_ptr(a);
  float smax_local = 0.0f;
  for (int u = lane; u < kTile * upr; u += 32) {  // kTile * upr is a multiple of 32
    const int t = u / upr, part = u - t * upr;
    uint4* src = reinterpret_cast<uint4*>(smp + t * row_bytes(D) + part * E * 2);
    const int nv = E / 8;  // 16-byte vectors of 8 fp16 values
    __half2 lo2 = __float2half2_rn(INFINITY), hi2 = __float2half2_rn(-INFINITY);
    if (t < valid) {
      for (int k = 0; k < nv; ++k) {
        const uint4 v = src[k];
        const __half2* hv = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          lo2 = __hmin2(lo2, hv[i]);
          hi2 = __hmax2(hi2, hv[i]);
        }
      }
    }
    float mn = fminf(__low2float(lo2), __high2float(lo2));
    float mx = fmaxf(__low2float(hi2), __high2float(hi2));
    for (int o = 1; o < lpg; o <<= 1) {  // lanes of one group are adjacent and all active
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (t < valid) {
      float z, s;
      group_params(mn, mx, fmaxf(fabsf(mn), fabsf(mx)), a.L.bits, a.L.sym, a.L.meta_f32, &z, &s);
      const float rc = s > 0.0f ? __frcp_rn(s) : 0.0f;
      const int j = part / lpg;
      if ((part & (lpg - 1)) == 0)
        store_meta(meta, (((long)b * a.H + h) * a.tcap + (long)tile * kTile + t) * gpr + j, a.L.meta_f32, a.L.sym, z,
                   s);
      smax_local = fmaxf(smax_local, s);
      // the reciprocal rule for 8 values at once, the division-checked rule
      // for the (rare) vector where any of them needs it
      const bool gok = rc >= 0x1p-125f || s == 0.0f;
      for (int k = 0; k < nv; ++k) {
        const uint4 v = src[k];
        const uint32_t* x = reinterpret_cast<const uint32_t*>(&v);
        uint4 o;
        uint32_t* w = reinterpret_cast<uint32_t*>(&o);
        bool ok = gok;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&x[i]));
          const uint32_t c0 = (uint32_t)quant_code_try(f.x, z, rc, a.L.bits, a.L.sym, ok);
          const uint32_t c1 = (uint32_t)quant_code_try(f.y, z, rc, a.L.bits, a.L.sym, ok);
          w[i] = c0 | (c1 << 16);
        }
        if (!ok) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&x[i]));
            const uint32_t c0 = (uint32_t)quant_code_fast(f.x, z, s, rc, a.L.bits, a.L.sym);
            const uint32_t c1 = (uint32_t)quant_code_fast(f.y, z, s, rc, a.L.bits, a.L.sym);
            w[i] = c0 | (c1 << 16);
          }
        }
        src[k] = o;
      }
    } else {
      for (int k = 0; k < nv; ++k) src[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __syncwarp();
  pack_store_dispatch<D>(a.L.bits, sm, a.is_value, codes_ptr(a, b, h, tile), lane);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) smax_local = fmaxf(smax_local, __shfl_xor_sync(0xffffffffu, smax_local, o));
  if (lane == 0 && smax_local > 0.0f) atomic_max_pos(a.smax + (long)b * a.H + h, smax_local);
}

// Whether the fast kernels take this layer-tensor: fp16 inputs whose rows start
// on 16-byte boundaries, no full-precision window, per-channel groups or
// per-token groups inside one head.
size_t prefill_fast_smem(const QuantArgs& a) {
  const int rows = a.L.axis == 1 ? a.L.group : kTile;
  return (size_t)kPrefillWarps * rows * row_bytes(a.D);
}

// Whether the fast kernels take this layer-tensor: fp16 inputs whose rows start
// on 16-byte boundaries, no full-precision window, per-channel groups or
// per-token groups inside one head, and the warps' rows fit in shared memory.
bool prefill_fast_ok(const QuantArgs& a) {
  if (a.x_f32 || a.L.window || a.L.whole) return false;
  if ((reinterpret_cast<uintptr_t>(a.x) & 15) != 0) return false;
  if (a.D != 64 && a.D != 128 && a.D != 256) return false;
  return prefill_fast_smem(a) <= 227 * 1024;
}

static const void* fast_fn(int axis, int D) {
  if (axis == 1) {
    if (D == 64) return reinterpret_cast<const void*>(&prefill_channel_fast<64>);
    if (D == 128) return reinterpret_cast<const void*>(&prefill_channel_fast<128>);
    return reinterpret_cast<const void*>(&prefill_channel_fast<256>);
  }
  if (D == 64) return reinterpret_cast<const void*>(&prefill_token_fast<64>);
  if (D == 128) return reinterpret_cast<const void*>(&prefill_token_fast<128>);
  return reinterpret_cast<const void*>(&prefill_token_fast<256>);
}

cudaError_t prefill_fast_setup() {
  // the largest plan: per-channel groups of 128 tokens at head_dim 256
  const size_t most = (size_t)kPrefillWarps * 128 * row_bytes(256);
  for (int axis = 0; axis < 2; ++axis)
    for (int D : {64, 128, 256}) {
      cudaError_t e = cudaFuncSetAttribute(fast_fn(axis, D), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)std::min<size_t>(most, 227 * 1024));
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

cudaError_t launch_prefill_fast(const QuantArgs& a, int maxn, cudaStream_t st) {
  const size_t smem = prefill_fast_smem(a);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  dim3 grid;
  if (a.L.axis == 1) {
    const int groups = (maxn + a.L.group - 1) / a.L.group + 1;  // + the group holding the tail
    grid = dim3((groups + kPrefillWarps - 1) / kPrefillWarps, a.H, a.B);
  } else {
    const int tiles = (maxn + kTile - 1) / kTile;
    grid = dim3((tiles + kPrefillWarps - 1) / kPrefillWarps, a.H, a.B);
  }
  void* args[] = {const_cast<QuantArgs*>(&a)};
  return cudaLaunchKernel(fast_fn(a.L.axis, a.D), grid, dim3(kPrefillWarps * 32), args, smem, st);
}

}  // namespace kvq
