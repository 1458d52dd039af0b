// kvq_common.cuh — shared definitions of the packed KV-cache layout and the
// device helpers used by every kernel of libkvq (sm_103a).
//
// Packed layout.  Each (layer, sequence, kv head) tensor is stored as tiles of
// 16 tokens x head_dim channels.  A B-bit code is split into bit planes whose
// widths are powers of two (2:[2] 3:[2,1] 4:[4] 5:[4,1] 6:[4,2] 7:[4,2,1]
// 8:[8]; plane p holds bits [off_p, off_p + w_p) of the code), so no code
// straddles a 32-bit word and the tile holds exactly 16*D*B bits.  Inside a
// tile, element (token t, channel c) sits where the mma.sync m16n8k16 operand
// fragment of the decode kernel wants it:
//   keys   : fragment row R = t,      column kk = c % 16, chunk j = c / 16
//   values : fragment row R = c % 16, column kk = t,      chunk j = c / 16
//   lane = 4*(R%8) + (kk%8)/2, pair pi = 4*j + (R/8) + 2*(kk/8), element e = kk%2
// so a lane's 32-bit register of two fp16 operands (e = 0 low half, e = 1 high
// half) comes from one "pair".  Plane p stores, per lane, W_p = D*w_p/64 words;
// word i of the lane holds pairs [i*P, (i+1)*P) with P = 16/w_p; pair slot
// k = pi % P has element e at bits [k*w_p + 16*e, k*w_p + 16*e + w_p).  Word
// address inside the tile: D*off_p/2 + lane*W_p + i.  The metadata and lengths
// that describe these codes live beside them in the same device buffer, indexed
// by the same (layer, sequence, head, token/group) coordinates, so a reorder of
// the codes without their scales cannot happen by construction.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

constexpr int kTile = 16;         // tokens per packed tile
constexpr int kWarps = 4;         // warps per decode CTA
constexpr int kMaxBatch = 1024;   // sequences per cache
constexpr int kCombineGroup = 16; // split-K partials merged per combine step
// At most kMaxSplits / kCombineGroup = 64 group partials, so the combine's
// staging (rep * (2 * 64 + 2) floats) always fits the CTA merge area
// (rep * 4 * (D + 2) floats).
constexpr int kMaxSplits = 1024;
constexpr int kMaxCluster = 8;    // splits merged inside one thread-block cluster (portable size)

// split-K workspace: chunk partials + group partials (rows of head_dim + 4
// floats: outputs, m, l, two pad words), and combine tickets
inline int combine_groups(int max_chunks) { return (max_chunks + kCombineGroup - 1) / kCombineGroup; }
inline size_t decode_work_floats(long batch, long q_heads, int head_dim, int max_chunks) {
  return (size_t)batch * q_heads * (max_chunks + combine_groups(max_chunks)) * (head_dim + 4);
}
inline size_t decode_ticket_words(long batch, long kv_heads, int max_chunks) {
  return (size_t)batch * kv_heads * (1 + combine_groups(max_chunks));
}

struct Planes {
  int n;
  int w[3];
  int off[3];
};

__host__ __device__ inline Planes planes_of(int bits) {
  Planes p;
  switch (bits) {
    case 2: p = {1, {2, 0, 0}, {0, 0, 0}}; break;
    case 3: p = {2, {2, 1, 0}, {0, 2, 0}}; break;
    case 4: p = {1, {4, 0, 0}, {0, 0, 0}}; break;
    case 5: p = {2, {4, 1, 0}, {0, 4, 0}}; break;
    case 6: p = {2, {4, 2, 0}, {0, 4, 0}}; break;
    case 7: p = {3, {4, 2, 1}, {0, 4, 6}}; break;
    default: p = {1, {8, 0, 0}, {0, 0, 0}}; break;
  }
  return p;
}

// The same plane split as compile-time functions of the bit width: plane
// count, width of plane p, bit offset of plane p.
__host__ __device__ constexpr int np_of(int b) { return (b == 3 || b == 5 || b == 6) ? 2 : (b == 7 ? 3 : 1); }
__host__ __device__ constexpr int pw_of(int b, int p) {
  return b == 2   ? 2
         : b == 3 ? (p == 0 ? 2 : 1)
         : b == 4 ? 4
         : b == 5 ? (p == 0 ? 4 : 1)
         : b == 6 ? (p == 0 ? 4 : 2)
         : b == 7 ? (p == 0 ? 4 : (p == 1 ? 2 : 1))
                  : 8;
}
__host__ __device__ constexpr int po_of(int b, int p) { return p == 0 ? 0 : pw_of(b, 0) + (p == 2 ? pw_of(b, 1) : 0); }

// Position of one element inside the fragment-ordered tile.
struct FragPos {
  int lane;
  int pi;  // pair index within the lane
  int e;   // 0 = low half, 1 = high half
};

__host__ __device__ inline FragPos frag_pos(int R, int kk, int j) {
  FragPos f;
  int g = R & 7, rh = R >> 3, tig = (kk & 7) >> 1, kh = kk >> 3;
  f.lane = 4 * g + tig;
  f.pi = 4 * j + rh + 2 * kh;
  f.e = kk & 1;
  return f;
}

// is_value: 0 for keys (rows = tokens), 1 for values (rows = channels)
__host__ __device__ inline FragPos elem_pos(int is_value, int t, int c) {
  return is_value ? frag_pos(c & 15, t, c >> 4) : frag_pos(t, c & 15, c >> 4);
}

// Word index inside a tile and bit position of plane p for an element.
__host__ __device__ inline void plane_word_bit(const FragPos& f, int D, int w, int off, int* word, int* bit) {
  int P = 16 / w;
  int W = D * w / 64;
  int i = f.pi / P, k = f.pi % P;
  *word = D * off / 2 + f.lane * W + i;
  *bit = k * w + 16 * f.e;
}

// Layout of one tensor (keys or values) of every layer inside the buffer.
struct TensorLayout {
  int bits, group, axis, sym, whole;  // whole: per-token group spanning all kv heads
  int window;                         // full-precision window of the newest tokens (0: none)
  int ring;                           // fp16 rows per (sequence, head): token t at row t % ring (0: no fp16 rows)
  int meta_f32;
  int meta_bytes;       // bytes per stored group entry
  int gpt;              // per-token axis: groups per head row (D/G), 1 when whole
  int tile_words;       // D*bits/2
  Planes planes;
  size_t codes_off, codes_layer;  // byte offset of layer 0, bytes per layer
  size_t meta_off, meta_layer;
  size_t tail_off, tail_layer;    // per-channel only
};

// Tokens of a length-n sequence held as codes; the rest [sealed, n) are fp16
// rows.  Per-channel: whole groups older than the window; per-token: every
// token (no window) or whole 16-token blocks older than the window.
__host__ __device__ inline long sealed_tokens(int axis, int group, int window, long n) {
  const long old = n - window > 0 ? n - window : 0;
  if (axis == 1) return (old / group) * group;
  return window ? (old / 16) * 16 : n;
}
__host__ __device__ inline long sealed_tokens(const TensorLayout& L, long n) {
  return sealed_tokens(L.axis, L.group, L.window, n);
}

// ------------------------------------------------------------- fp helpers --

__device__ __forceinline__ float h2f(__half h) { return __half2float(h); }

// Stored metadata entry of group `gi` -> (zero, step) as floats.
__device__ __forceinline__ void load_meta(const char* meta, long gi, int meta_f32, int sym, float* z, float* s) {
  if (!meta_f32) {
    if (sym) {
      *s = __half2float(reinterpret_cast<const __half*>(meta)[gi]);
      *z = 0.0f;
    } else {
      __half2 v = reinterpret_cast<const __half2*>(meta)[gi];
      *z = __low2float(v);
      *s = __high2float(v);
    }
  } else {
    if (sym) {
      *s = reinterpret_cast<const float*>(meta)[gi];
      *z = 0.0f;
    } else {
      float2 v = reinterpret_cast<const float2*>(meta)[gi];
      *z = v.x;
      *s = v.y;
    }
  }
}

__device__ __forceinline__ void store_meta(char* meta, long gi, int meta_f32, int sym, float z, float s) {
  if (!meta_f32) {
    if (sym) reinterpret_cast<__half*>(meta)[gi] = __float2half_rn(s);  // s is fp16-exact here
    else reinterpret_cast<__half2*>(meta)[gi] = __halves2half2(__float2half_rn(z), __float2half_rn(s));
  } else {
    if (sym) reinterpret_cast<float*>(meta)[gi] = s;
    else reinterpret_cast<float2*>(meta)[gi] = make_float2(z, s);
  }
}

// The quantizer's parameter rule (see kvq.h): exact statistics in, stored
// (zero, step) out.  IEEE fp32 round-to-nearest operations via intrinsics so
// no contraction or fast-math can change them.
__device__ __forceinline__ void group_params(float mn, float mx, float amax, int bits, int sym, int meta_f32,
                                             float* z, float* s) {
  if (!sym) {
    float levels = (float)((1 << bits) - 1);
    float z32 = __fadd_rn(mn, 0.0f);
    if (meta_f32) {
      *z = z32;
      *s = __fadd_rn(__fdiv_rn(__fsub_rn(mx, z32), levels), 0.0f);
    } else {
      float zh = __half2float(__float2half_rd(z32));
      float s32 = __fadd_rn(__fdiv_rn(__fsub_rn(mx, zh), levels), 0.0f);
      *z = zh;
      *s = __half2float(__float2half_ru(s32));
    }
  } else {
    float qmax = (float)((1 << (bits - 1)) - 1);
    float s32 = __fdiv_rn(amax, qmax);
    *z = 0.0f;
    *s = meta_f32 ? s32 : __half2float(__float2half_ru(s32));
  }
}

// quant_code with the step's reciprocal r = __frcp_rn(s) given: the same code.
// q0 = (x - z) * r differs from the IEEE quotient Q = fl((x - z) / s) by less
// than 2^-13 whenever |Q| <= 512 (two roundings of 2^-24 relative each, plus
// Q's own), so if q0 lies farther than 2^-12 from a half-integer both round to
// the same integer; otherwise (ties included), or for a subnormal r, a huge
// quotient or a NaN, the IEEE division decides.
__device__ __forceinline__ int quant_code_r(float x, float z, float s, float r, int bits, int sym) {
  if (s == 0.0f) return sym ? (1 << (bits - 1)) : 0;
  const float num = sym ? x : __fsub_rn(x, z);
  const float q0 = __fmul_rn(num, r);
  const float aq = fabsf(q0);
  const float fr = aq - floorf(aq);
  float t = (aq <= 512.0f && r >= 0x1p-125f && fabsf(fr - 0.5f) > 0x1p-12f) ? rintf(q0) : rintf(__fdiv_rn(num, s));
  if (!sym) {
    const float levels = (float)((1 << bits) - 1);
    t = fminf(fmaxf(t, 0.0f), levels);
    return (int)t;
  }
  const float qmax = (float)((1 << (bits - 1)) - 1);
  t = fminf(fmaxf(t, -qmax), qmax);
  return (int)t + (1 << (bits - 1));
}

// The same code again, cheaper per element (the prefill kernels): r is the
// step's reciprocal or 0 for a zero step.  q0 = (x - z) * r is rounded to the
// nearest integer, ties to even, by adding and removing 1.5 * 2^23 (exact for
// |q0| < 2^22), and the distance to that integer comes from the same sums; a
// quotient within 2^-12 of a half-integer, beyond 512, or a subnormal
// reciprocal takes the IEEE division, exactly as in quant_code_r.
__device__ __forceinline__ int quant_code_fast(float x, float z, float s, float r, int bits, int sym) {
  const float num = sym ? x : __fsub_rn(x, z);
  const float q0 = __fmul_rn(num, r);
  const float c = __fsub_rn(__fadd_rn(q0, 12582912.0f), 12582912.0f);
  const float e = __fsub_rn(q0, c);
  float t = c;
  if (!(fabsf(q0) <= 512.0f && fabsf(e) < 0.499755859375f && (r >= 0x1p-125f || s == 0.0f)))
    t = rintf(__fdiv_rn(num, s));
  if (s == 0.0f) t = 0.0f;
  int q = (int)t;
  if (!sym) return min(max(q, 0), (1 << bits) - 1);
  const int qmax = (1 << (bits - 1)) - 1;
  return min(max(q, -qmax), qmax) + (1 << (bits - 1));
}

// quant_code_fast without its division branch, for callers that test a
// whole row of codes at once: the code is quant_code_fast's whenever `ok`
// stays true (the quotient at most 512 and not within 2^-12 of a
// half-integer; the caller starts `ok` from the group's test that the
// reciprocal is normal or the step zero, with r = 0 for a zero step), and the
// integer is read from the rounding sum's bits (1.5 * 2^23 + rint(q0) for
// |q0| < 2^22) instead of a float-to-integer conversion.  Where `ok` turned
// false the caller recomputes the row with quant_code_fast.
__device__ __forceinline__ int quant_code_try(float x, float z, float r, int bits, int sym, bool& ok) {
  const float num = sym ? x : __fsub_rn(x, z);
  const float q0 = __fmul_rn(num, r);
  const float m = __fadd_rn(q0, 12582912.0f);
  const float e = __fsub_rn(q0, __fsub_rn(m, 12582912.0f));
  ok = ok && fabsf(q0) <= 512.0f && fabsf(e) < 0.499755859375f;
  const int q = __float_as_int(m) - 0x4B400000;
  if (!sym) return min(max(q, 0), (1 << bits) - 1);
  const int qmax = (1 << (bits - 1)) - 1;
  return min(max(q, -qmax), qmax) + (1 << (bits - 1));
}

__device__ __forceinline__ int quant_code(float x, float z, float s, int bits, int sym) {
  if (s == 0.0f) return sym ? (1 << (bits - 1)) : 0;
  if (!sym) {
    float t = rintf(__fdiv_rn(__fsub_rn(x, z), s));
    float levels = (float)((1 << bits) - 1);
    t = fminf(fmaxf(t, 0.0f), levels);
    return (int)t;
  } else {
    float qmax = (float)((1 << (bits - 1)) - 1);
    float t = rintf(__fdiv_rn(x, s));
    t = fminf(fmaxf(t, -qmax), qmax);
    return (int)t + (1 << (bits - 1));
  }
}

// ------------------------------------------------------------ PTX helpers --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global -> shared copy that bypasses L1 (shared-window
// address); completion is tracked per thread in commit groups
// (cp.async.commit_group / wait_group).  Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16_s(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_dst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel of the stream still runs;
// pdl_wait() returns once that kernel has completed and its writes are
// visible (immediately for an ordinary launch), and pdl_trigger() lets the next
// such kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Split cluster barrier: every thread of every CTA of the cluster arrives once
// and later waits once per phase.  A relaxed arrival orders no memory; the
// wait returns once all threads of the cluster have arrived.
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;\n" ::: "memory"); }

__device__ __forceinline__ void mma_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t x, uint32_t mask, uint32_t orv) {
  uint32_t d;
  // d = (x & mask) | orv
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(d) : "r"(x), "r"(mask), "r"(orv));
  return d;
}

__device__ __forceinline__ uint32_t rotl(uint32_t x, int n) { return __funnelshift_l(x, x, n); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// fp32 -> (hi, lo) fp16 pair with hi + lo = x to ~22 bits (x pre-scaled into fp16 range)
__device__ __forceinline__ void split_hl(float x, __half* hi, __half* lo) {
  __half h = __float2half_rn(x);
  *hi = h;
  *lo = __float2half_rn(x - __half2float(h));
}

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// 2^e as float for |e| < 127
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// scale exponent E so that m * 2^E lies in [2^14, 2^15) (0 when m == 0)
__device__ __forceinline__ int norm_exp(float m) {
  if (!(m > 0.0f)) return 0;
  int e = ((__float_as_int(m) >> 23) & 0xff) - 127;
  if (e < -126) e = -126;
  int E = 14 - e;
  if (E > 100) E = 100;
  return E;
}

}  // namespace kvq
