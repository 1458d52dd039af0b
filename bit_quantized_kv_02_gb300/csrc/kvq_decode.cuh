// kvq_decode.cuh — split-K decode attention over the packed KV cache (sm_103a).
//
// One CTA = one (sequence, kv head, token chunk); 4 warps, each an independent
// flash-decoding pass over a contiguous, group-aligned sub-range, merged at the
// end of the CTA.  The chunks of a (sequence, kv head) then merge their
// partials (log-sum-exp combine): inside one thread-block cluster through
// distributed shared memory when the grid is a single wave of at most 8 chunks
// per head, otherwise in the global workspace behind atomic tickets (the last
// arriving CTA merges; no CTA ever waits for another).
//
// Per 16-token tile a warp:
//   1. waits for its stage: packed codes + metadata copied global -> shared by
//      16-byte cp.async from all 32 lanes (completion tracked per lane in commit
//      groups, a ring of 2 or 4 stages), and turns the stage's metadata into
//      fp32 (step, folded zero) pairs once;
//   2. QK: converts the key codes of each 16-channel chunk to exact fp16
//      operands in registers (one rotate + one LOP3 per code pair and bit
//      plane: the code lands in the top mantissa bits of an fp16 whose
//      exponent makes its value 2^B + code) and runs mma.sync m16n8k16 against
//      the query split into fp16 hi + lo parts (~22-bit operand, fp32
//      accumulation); steps, zero points and the 2^B offset are folded into
//      the query (per-channel keys) or applied to the fp32 accumulators
//      (per-token keys);
//   3. online softmax in base 2 (fp32);
//   4. PV: converts the value codes the same way (fragment rows = channels,
//      columns = tokens) and runs mma.sync against the probabilities, split
//      hi + lo, with the per-token step folded in (per-token values) or applied
//      per channel at group end (per-channel values).
// The unsealed fp16 tail of a per-channel tensor is fed to the same MMAs as
// plain fp16 operands.
//
// The pages describe fusing unpacking and scale application into attention in
// words ("Kuantisasi KV Cache untuk Mengurangi Memory Inferensi Long Context",
// section "Kuantisasi dapat memindahkan pekerjaan ke decode path"); the GPU
// design here is this library's own.
#pragma once

#include <cooperative_groups.h>

#include "kvq_decode_args.h"
#include "kvq_quant.cuh"

namespace kvq {

// Code-to-operand conversion.  Widths 2, 4 and 8 place each code, unshifted
// or after one shift shared by several registers, in the low mantissa bits of
// an fp16 subnormal: the register's value is code * 2^(base - 24), exact, with
// base = conv_r * (fragment row half) + conv_c * (fragment column half) (mma
// takes subnormal fp16 operands exactly).  The other widths use an fp16 whose
// exponent field makes its value 2^B + code (one rotate + one LOP3 per bit
// plane).  Either way A = 2^(conv_g + base) * (code + conv_off).
__host__ __device__ constexpr bool conv_subn(int b) { return b == 2 || b == 4 || b == 8; }
__host__ __device__ constexpr int conv_g(int b) { return conv_subn(b) ? -24 : 0; }
__host__ __device__ constexpr int conv_r(int b) { return b == 4 ? 4 : (b == 2 ? 2 : 0); }
__host__ __device__ constexpr int conv_c(int b) { return b == 2 ? 4 : 0; }
__host__ __device__ constexpr int conv_off(int b) { return conv_subn(b) ? 0 : (1 << b); }

// Four fp16x2 MMA operand registers (pairs 4j..4j+3 of this lane, register r
// = fragment row half + 2 * column half) of 16-channel chunk j.
template <int BITS, int D>
__device__ __forceinline__ void convert_chunk(const uint32_t* tile, int lane, int j, uint32_t a[4]) {
  if constexpr (BITS == 4) {
    // one word per chunk and lane; pair r at bits 4r (+16)
    const uint32_t w = tile[lane * (D / 16) + j], u = w >> 8;
    a[0] = w & 0x000F000Fu;
    a[1] = w & 0x00F000F0u;
    a[2] = u & 0x000F000Fu;
    a[3] = u & 0x00F000F0u;
  } else if constexpr (BITS == 2) {
    // one word per two chunks; pair 4(j & 1) + r at bits 2(4(j & 1) + r) (+16)
    const uint32_t w0 = tile[lane * (D / 32) + (j >> 1)];
    const uint32_t w = (j & 1) ? (w0 >> 8) : w0;
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = w & (0x00030003u << (2 * r));
  } else if constexpr (BITS == 8) {
    // two words per chunk; pair r at bytes (r & 1) and 2 + (r & 1) of word r / 2
    const uint32_t w0 = tile[lane * (D / 8) + 2 * j], w1 = tile[lane * (D / 8) + 2 * j + 1];
    a[0] = __byte_perm(w0, 0u, 0x4240);
    a[1] = __byte_perm(w0, 0u, 0x4341);
    a[2] = __byte_perm(w1, 0u, 0x4240);
    a[3] = __byte_perm(w1, 0u, 0x4341);
  } else {
    constexpr uint32_t magic = (uint32_t)((BITS + 15) << 10) * 0x00010001u;
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = magic;
#pragma unroll
    for (int p = 0; p < np_of(BITS); ++p) {
      const int w = pw_of(BITS, p), off = po_of(BITS, p);
      const int W = D * w / 64, P = 16 / w;
      const int pos = 10 - BITS + off;
      const uint32_t M = (((1u << w) - 1u) << pos) * 0x00010001u;
      const uint32_t* pl = tile + D * off / 2 + lane * W;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int pi = 4 * j + r;
        const uint32_t word = pl[pi / P];
        const int k = pi % P;
        const int sh = (pos - k * w) & 31;
        a[r] = lop3_and_or(sh ? rotl(word, sh) : word, M, a[r]);
      }
    }
  }
}

template <int D>
__device__ __forceinline__ void convert_dispatch(int bits, const uint32_t* tile, int lane, int j, uint32_t a[4]) {
  switch (bits) {
    case 2: convert_chunk<2, D>(tile, lane, j, a); break;
    case 3: convert_chunk<3, D>(tile, lane, j, a); break;
    case 4: convert_chunk<4, D>(tile, lane, j, a); break;
    case 5: convert_chunk<5, D>(tile, lane, j, a); break;
    case 6: convert_chunk<6, D>(tile, lane, j, a); break;
    case 7: convert_chunk<7, D>(tile, lane, j, a); break;
    default: convert_chunk<8, D>(tile, lane, j, a); break;
  }
}

// Stored metadata entries [0, n) -> fp32 (step * post, zero') with zero' =
// zero - conv_off * step (symmetric: zero = -2^(B-1) step), so that a value is
// step * (code + conv_off) + zero'.  post = post_hi for the entries of the
// upper fragment half (hsel > 0: entries i >= hsel, i.e. tokens 8..15 of a
// per-token tile; hsel <= 0: channels with bit 3 set), else post_lo.  One
// warp, entries strided over the lanes.
// center (per-token values): the codes enter the MMA centred on the middle of
// their range (code - 2^(B-1), see the value kernel's centring MMA), so the
// zero point becomes zero + 2^(B-1) * step (symmetric: exactly 0).
__device__ __forceinline__ void canon_meta(const char* src, int n, int bits, int sym, int meta_f32, float post_lo,
                                           float post_hi, int hsel, float2* dst, int lane, bool center = false) {
  const float off = (float)conv_off(bits);
  const float soff = (float)(1 << (bits - 1));
  for (int i = lane; i < n; i += 32) {
    float z, s;
    load_meta(src, i, meta_f32, sym, &z, &s);
    float zc;
    if (center) zc = sym ? 0.0f : fmaf(soff, s, z);
    else zc = (sym ? -s * soff : z) - off * s;
    const bool hi = hsel > 0 ? (i >= hsel) : ((i & 8) != 0);
    dst[i] = make_float2(s * (hi ? post_hi : post_lo), zc);
  }
}

// Probabilities enter the value MMAs, the row sums and the split-K partials
// as p * 2^kPExp (p <= 1): a probability of a long, flat softmax (1e-5 and
// below) then stays a normal fp16 in both halves of its hi + lo split instead
// of losing its low half to fp16 subnormals.  The scale cancels in out = O / l.
constexpr float kPExp = 14.0f;

template <bool R8>
struct Slots {
  static constexpr int N = R8 ? 4 : 2;
  __device__ static int rh(int s) { return R8 ? (s >> 1) : s; }
  __device__ static int rho(int s, int tig) { return R8 ? (2 * tig + (s & 1)) : tig; }
};

// -------------------------------------------------- query operand build ---

// Stored (zero, step) of entries c and c+1 (c even) in one vector load.
__device__ __forceinline__ void load_meta2(const char* meta, int c, int meta_f32, int sym, float* z0, float* s0,
                                           float* z1, float* s1) {
  if (!meta_f32) {
    if (sym) {
      const __half2 v = *reinterpret_cast<const __half2*>(meta + 2 * c);
      *s0 = __low2float(v);
      *s1 = __high2float(v);
      *z0 = *z1 = 0.0f;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(meta + 4 * c);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
      *z0 = a.x;
      *s0 = a.y;
      *z1 = b.x;
      *s1 = b.y;
    }
  } else {
    if (sym) {
      const float2 v = *reinterpret_cast<const float2*>(meta + 4 * c);
      *s0 = v.x;
      *s1 = v.y;
      *z0 = *z1 = 0.0f;
    } else {
      const float4 v = *reinterpret_cast<const float4*>(meta + 8 * c);
      *z0 = v.x;
      *s0 = v.y;
      *z1 = v.z;
      *s1 = v.w;
    }
  }
}

// Fragment-ordered QK B operand of one warp: q * s_c (kmeta = the stored
// per-channel key metadata of the current group, read straight from the
// stage) or q (kmeta == null), scaled by 2^E, channels of the upper half of
// each 16-channel chunk further by chi (the conversion's column scale), and
// split into fp16 hi + lo; bias[rho] = sum_c q_c zero'_c with zero' = zero -
// conv_off * step (symmetric zero = -2^(B-1) step).  Only valid query columns
// are written; the rest of barea stays zero.  Each lane loads the metadata of
// its channels once for every query, and the per-query bias partials are
// summed by one reduce-scatter butterfly over the warp.
template <int D, bool R8>
__device__ __forceinline__ float build_qb(const float* qs, int rep, const char* kmeta, int kbits, int ksym, int kf32,
                                          uint32_t* barea, float* bias, int E, float chi, int lane) {
  constexpr int IT = D / 64;  // channel pairs per lane
  const float sc = exp2i(E);
  const float koff = (float)conv_off(kbits), ksoff = (float)(1 << (kbits - 1));
  float sm0[IT], sm1[IT], zq0[IT], zq1[IT];  // per channel: operand scale, folded zero point
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int c = 2 * (lane + 32 * it);
    const float scc = (c & 8) ? sc * chi : sc;
    sm0[it] = scc;
    sm1[it] = scc;
    zq0[it] = zq1[it] = 0.0f;
    if (kmeta) {
      float z0, st0, z1, st1;
      load_meta2(kmeta, c, kf32, ksym, &z0, &st0, &z1, &st1);
      if (ksym) {
        z0 = -st0 * ksoff;
        z1 = -st1 * ksoff;
      }
      sm0[it] = st0 * scc;
      sm1[it] = st1 * scc;
      zq0[it] = z0 - koff * st0;
      zq1[it] = z1 - koff * st1;
    }
  }
  float bpart[8];  // this lane's bias partial of each query
#pragma unroll
  for (int rho = 0; rho < 8; ++rho) {
    bpart[rho] = 0.0f;
    if (rho >= rep) continue;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const int c = 2 * (lane + 32 * it);
      const float2 q2 = *reinterpret_cast<const float2*>(qs + rho * D + c);
      if (kmeta) bpart[rho] += q2.x * zq0[it] + q2.y * zq1[it];
      const float v0 = q2.x * sm0[it], v1 = q2.y * sm1[it];
      const __half2 hh = __floats2half2_rn(v0, v1);
      const float2 hf = __half22float2(hh);
      const __half2 ll = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
      const int j = c >> 4, cc = c & 15, ttig = (cc & 7) >> 1, breg = cc >> 3;
      if (!R8) {
        barea[(j * 32 + 4 * (2 * rho) + ttig) * 2 + breg] = *reinterpret_cast<const uint32_t*>(&hh);
        barea[(j * 32 + 4 * (2 * rho + 1) + ttig) * 2 + breg] = *reinterpret_cast<const uint32_t*>(&ll);
      } else {
        barea[((2 * j) * 32 + 4 * rho + ttig) * 2 + breg] = *reinterpret_cast<const uint32_t*>(&hh);
        barea[((2 * j + 1) * 32 + 4 * rho + ttig) * 2 + breg] = *reinterpret_cast<const uint32_t*>(&ll);
      }
    }
  }
  float b1 = 0.0f;
  if (kmeta && rep == 1) {
    // one query: the butterfly leaves the sum in every lane; the caller keeps
    // it in a register (no shared-memory copy)
    b1 = bpart[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b1 += __shfl_xor_sync(0xffffffffu, b1, o);
  } else if (kmeta) {
    // reduce-scatter: after the rounds over lane bits 4, 3, 2 each lane keeps
    // one query's partial (query index from those bits), then the last two
    // rounds finish the sum; lanes with bits 0..1 clear write it
    int nq = 8;
#pragma unroll
    for (int o = 16; o >= 4; o >>= 1) {
      nq >>= 1;
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (k < nq) {
          const float keep = up ? bpart[k + nq] : bpart[k];
          const float give = up ? bpart[k] : bpart[k + nq];
          bpart[k] = keep + __shfl_xor_sync(0xffffffffu, give, o);
        }
      }
    }
    float b = bpart[0];
    b += __shfl_xor_sync(0xffffffffu, b, 2);
    b += __shfl_xor_sync(0xffffffffu, b, 1);
    const int rho = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
    if ((lane & 3) == 0 && rho < rep) bias[rho] = b;
  }
  __syncwarp();
  return b1;
}

template <int V>
struct IntC {
  static constexpr int value = V;
};

// stage index of tile i: i mod stages
struct StageR {
  int mask;
  __device__ int get(int i) const { return i & mask; }
};

// ------------------------------------------------------ configurations ---

// Runtime configuration: every format field comes from the launch arguments
// (the generic kernel, any format the C ABI accepts).
struct DynCfg {
  static constexpr int kStaticStages = 0;  // stage count known only at run time
  static constexpr int kRep = 8;           // largest query heads per KV head
  static constexpr int kRope = 1;          // (layouts come from the launch arguments)
  __device__ static int rep(const DecodeArgs& a) { return a.rep; }
  __device__ static int kbits(const DecodeArgs& a) { return a.K.bits; }
  __device__ static int ksym(const DecodeArgs& a) { return a.K.sym; }
  __device__ static int kf32(const DecodeArgs& a) { return a.K.meta_f32; }
  __device__ static int kwhole(const DecodeArgs& a) { return a.K.whole; }
  __device__ static bool ktok(const DecodeArgs& a) { return a.K.axis == 0; }
  __device__ static int kgpt(const DecodeArgs& a) { return a.K.gpt; }
  __device__ static int klg(const DecodeArgs& a) { return a.K.lg_group; }
  __device__ static int kG(const DecodeArgs& a) { return a.K.group; }
  __device__ static int kmb(const DecodeArgs& a) { return a.K.meta_bytes; }
  __device__ static int vbits(const DecodeArgs& a) { return a.V.bits; }
  __device__ static int vsym(const DecodeArgs& a) { return a.V.sym; }
  __device__ static int vf32(const DecodeArgs& a) { return a.V.meta_f32; }
  __device__ static int vwhole(const DecodeArgs& a) { return a.V.whole; }
  __device__ static int vgpt(const DecodeArgs& a) { return a.V.gpt; }
  __device__ static int vlg(const DecodeArgs& a) { return a.V.lg_group; }
  __device__ static int vG(const DecodeArgs& a) { return a.V.group; }
  __device__ static int vmb(const DecodeArgs& a) { return a.V.meta_bytes; }
  __device__ static int kc_bytes(const DecodeArgs& a) { return a.K.tile_bytes; }
  __device__ static int vc_bytes(const DecodeArgs& a) { return a.V.tile_bytes; }
  __device__ static int km_bytes(const DecodeArgs& a) { return a.K.mtile_bytes; }
  __device__ static int vm_bytes(const DecodeArgs& a) { return a.V.mtile_bytes; }
  __device__ static int st_kc(const DecodeArgs& a) { return a.st_kc; }
  __device__ static int st_km(const DecodeArgs& a) { return a.st_km; }
  __device__ static int st_vc(const DecodeArgs& a) { return a.st_vc; }
  __device__ static int st_vm(const DecodeArgs& a) { return a.st_vm; }
  __device__ static int stage_bytes(const DecodeArgs& a) { return a.stage_bytes; }
  __device__ static int lg_ns(const DecodeArgs& a) { return a.lg_nstages; }
  __device__ static int barea_bytes(const DecodeArgs& a) { return a.barea_bytes; }
  __device__ static int canon_k(const DecodeArgs& a) { return a.canon_k; }
  __device__ static int canon_v(const DecodeArgs& a) { return a.canon_v; }
  __device__ static int stage_off(const DecodeArgs& a) { return a.stage_off; }
  __device__ static int warp_bytes(const DecodeArgs& a) { return a.warp_bytes; }
  __device__ static int head_bytes(const DecodeArgs& a) { return a.head_bytes; }
  __device__ static int stage_f16(const DecodeArgs& a) { return a.stage_f16; }
};

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x >> 1); }

// Compile-time configuration (fp16 metadata, no whole-vector groups): every
// format field and shared-memory offset is a constant, so index arithmetic,
// format branches and group bookkeeping fold away.
template <int D, int REP, int KB, int KAX, int KG, int KSYM, int VB, int VAX, int VG, int VSYM, int ROPEL = 0>
struct StatCfg {
  static constexpr int KGPT = KAX == 0 ? D / KG : 0, VGPT = VAX == 0 ? D / VG : 0;
  static constexpr int KMB = KSYM ? 2 : 4, VMB = VSYM ? 2 : 4;
  static constexpr int kRope = ROPEL;  // the layout includes the rotary tables
  static constexpr DecLayout L = dec_layout(D, REP, KB, KAX, 0, KGPT, KMB, VB, VAX, 0, VGPT, VMB, 0, ROPEL);
  static constexpr int kStaticStages = 1 << L.lg_ns;
  static constexpr int kRep = REP;
  __device__ static constexpr int rep(const DecodeArgs&) { return REP; }
  __device__ static constexpr int kbits(const DecodeArgs&) { return KB; }
  __device__ static constexpr int ksym(const DecodeArgs&) { return KSYM; }
  __device__ static constexpr int kf32(const DecodeArgs&) { return 0; }
  __device__ static constexpr int kwhole(const DecodeArgs&) { return 0; }
  __device__ static constexpr bool ktok(const DecodeArgs&) { return KAX == 0; }
  __device__ static constexpr int kgpt(const DecodeArgs&) { return KGPT; }
  __device__ static constexpr int klg(const DecodeArgs&) { return ilog2(KG); }
  __device__ static constexpr int kG(const DecodeArgs&) { return KG; }
  __device__ static constexpr int kmb(const DecodeArgs&) { return KMB; }
  __device__ static constexpr int vbits(const DecodeArgs&) { return VB; }
  __device__ static constexpr int vsym(const DecodeArgs&) { return VSYM; }
  __device__ static constexpr int vf32(const DecodeArgs&) { return 0; }
  __device__ static constexpr int vwhole(const DecodeArgs&) { return 0; }
  __device__ static constexpr int vgpt(const DecodeArgs&) { return VGPT; }
  __device__ static constexpr int vlg(const DecodeArgs&) { return ilog2(VG); }
  __device__ static constexpr int vG(const DecodeArgs&) { return VG; }
  __device__ static constexpr int vmb(const DecodeArgs&) { return VMB; }
  __device__ static constexpr int kc_bytes(const DecodeArgs&) { return L.kc_bytes; }
  __device__ static constexpr int vc_bytes(const DecodeArgs&) { return L.vc_bytes; }
  __device__ static constexpr int km_bytes(const DecodeArgs&) { return L.km_bytes; }
  __device__ static constexpr int vm_bytes(const DecodeArgs&) { return L.vm_bytes; }
  __device__ static constexpr int st_kc(const DecodeArgs&) { return L.st_kc; }
  __device__ static constexpr int st_km(const DecodeArgs&) { return L.st_km; }
  __device__ static constexpr int st_vc(const DecodeArgs&) { return L.st_vc; }
  __device__ static constexpr int st_vm(const DecodeArgs&) { return L.st_vm; }
  __device__ static constexpr int stage_bytes(const DecodeArgs&) { return L.stage_bytes; }
  __device__ static constexpr int lg_ns(const DecodeArgs&) { return L.lg_ns; }
  __device__ static constexpr int barea_bytes(const DecodeArgs&) { return L.barea_bytes; }
  __device__ static constexpr int canon_k(const DecodeArgs&) { return L.canon_k; }
  __device__ static constexpr int canon_v(const DecodeArgs&) { return L.canon_v; }
  __device__ static constexpr int stage_off(const DecodeArgs&) { return L.stage_off; }
  __device__ static constexpr int warp_bytes(const DecodeArgs&) { return L.warp_bytes; }
  __device__ static constexpr int head_bytes(const DecodeArgs&) { return L.head_bytes; }
  __device__ static constexpr int stage_f16(const DecodeArgs&) { return 0; }
};

// --------------------------------------------------------------- kernel ----

// resident CTAs per SM the register budget is sized for
// (compile-time configurations need fewer registers than the generic kernel;
// measured: 5 at head_dim 128 beats 4, 3 at head_dim 256 loses to 2; per-channel
// values keep their group accumulators and stay at 4 to avoid spills)
__host__ __device__ constexpr int decode_min_blocks(int D, bool is_static, int vaxis = 0, bool rope = false) {
  return is_static ? (D == 64 ? 5 : (D == 128 ? ((vaxis || rope) ? 4 : 5) : 2)) : (D == 64 ? 5 : (D == 128 ? 3 : 2));
}

// FUSED: the launch also appends the new token (kvq_append_decode_attn); the
// plain decode kernel is compiled without any of that code.
// NW: warps per CTA (each warp streams its own token range; the CTA's warps
// merge in shared memory).  One-warp CTAs let the block scheduler spread the
// warps of a launch over the SMs one at a time.
// ROPE: the keys are cached before the rotary position embedding; every
// dequantized key is turned by its token's angles before the QK MMA (runtime
// formats, and compile-time configurations built with the rotary layout).
template <int D, bool R8, int VAXIS, class CFG, bool FUSED = false, bool ROPE = false, int NW = kWarps>
__global__ void __launch_bounds__(NW * 32, decode_min_blocks(D, CFG::kStaticStages != 0, VAXIS, ROPE) * kWarps / NW)
    decode_kernel(const __grid_constant__ DecodeArgs a) {
  static_assert(NW == kWarps || !ROPE, "the rotary tables are built by four warps");
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int NCH = D / 16;                // 16-channel chunks / m-tiles
  constexpr int NB = R8 ? 2 : 1;             // B operands per chunk (hi/lo split over two MMAs)
  // query operand kept in registers at head_dim 64; wider heads read it from
  // shared memory per MMA (measured at head_dim 128: the 16 registers are worth
  // more as a fifth resident CTA per SM, 6-7 % faster)
  constexpr bool BREG = NCH * 2 * NB <= 8;
  constexpr int GV_MAX = D / 32;             // per-token value groups per head row (group >= 32)
  using SL = Slots<R8>;
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int rep = CFG::rep(a), H = a.H, S = a.S;
  // cluster launch: this arrival tells the cluster that this CTA runs; the
  // matching wait comes before the first store into another CTA's shared memory
  if (a.csize) cluster_arrive_relaxed();
  pdl_wait();  // the cache and the query are complete
  const int hq0 = h * rep;
  // the query and the largest steps are requested before the length, so the
  // three loads are in flight together
  // query values per thread (four warps: rep 8)
  constexpr int QPT = NW == kWarps ? D / 16 : (CFG::kRep * D + NW * 32 - 1) / (NW * 32);
  float qv[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = threadIdx.x + u * (NW * 32);
    const long qi = ((long)b * H * rep + hq0) * D + i;
    qv[u] = 0.0f;
    if (i < rep * D)
      qv[u] = a.q_f32 ? reinterpret_cast<const float*>(a.q)[qi] : __half2float(reinterpret_cast<const __half*>(a.q)[qi]);
  }
  float smax_k = __uint_as_float(a.smax_k[(long)b * H + h]);
  float smax_v = __uint_as_float(a.smax_v[(long)b * H + h]);
  // fused append: the cache holds n_old tokens of this (sequence, head) and
  // this launch appends token n_old, then attends over n_old + 1 tokens; the
  // new rows head for L2 now, so the appending warp finds them there
  if (FUSED && warp == 0) {
    const int row_bytes = D * (a.ap.k.x_f32 ? 4 : 2);
    const long xo = ((long)b * H + h) * row_bytes;
    if (lane * 128 < row_bytes) prefetch_l2(static_cast<const char*>(a.ap.k.x) + xo + lane * 128);
    if (lane * 128 < row_bytes) prefetch_l2(static_cast<const char*>(a.ap.v.x) + xo + lane * 128);
  }
  // fused append: one thread reads the old length and hands it to the whole
  // CTA through shared memory, so no thread of the CTA reads the counter after
  // the CTA has counted itself in below
  __shared__ int s_n_old;
  if (FUSED) {
    if (threadIdx.x == 0) s_n_old = a.ap.head_lens[(long)b * H + h];
    __syncthreads();
  }
  const int n_old = FUSED ? s_n_old : 0;
  const int n = FUSED ? n_old + 1 : a.lens[b];
  // tokens held as codes; the newer ones are fp16 rows (unsealed per-channel
  // groups and the full-precision window)
  const bool k_token = CFG::ktok(a);
  const int k_lgG = CFG::klg(a), v_lgG = CFG::vlg(a);
  const int kold = max(n - a.K.window, 0), vold = max(n - a.V.window, 0);
  const int sealed_k = k_token ? (a.K.window ? (kold >> 4) << 4 : n) : ((kold >> k_lgG) << k_lgG);
  const int sealed_v = VAXIS == 0 ? (a.V.window ? (vold >> 4) << 4 : n) : ((vold >> v_lgG) << v_lgG);
  // Work of a (sequence, head): a token from the first fp16 unit on counts
  // a.fw times (its rows are read with direct loads, several times a packed
  // token's bytes), so that the window's tiles spread over several warps
  // instead of piling up in the last one.  Chunks of S and warp ranges of Sw
  // split the work; a range's ends map back to tokens at unit boundaries (a
  // multiple of 16 and of every per-channel group), so a group never straddles
  // two ranges.
  const int unit = max(kTile, max(k_token ? 1 : CFG::kG(a), VAXIS == 0 ? 1 : CFG::vG(a)));
  const int fw = a.fw;
  const int bnd = fw > 1 ? (min(sealed_k, sealed_v) & ~(unit - 1)) : n;
  const int ne = bnd + fw * (n - bnd);
  const int nchunks = (ne + S - 1) / S;
  auto range_end = [&](int e) {  // first token past work e
    e = min(e, ne);
    return e <= bnd ? e : min(n, bnd + (((e - bnd + fw - 1) / fw + unit - 1) & ~(unit - 1)));
  };
  // every CTA of (b, h) counts itself in once its length read is complete (a
  // fence orders the read before the count); the last one to arrive advances
  // the lengths, which no CTA of this launch reads afterwards
  unsigned arrival = 0u;
  if (FUSED && threadIdx.x == 0 && nchunks > 0) {
    __threadfence();
    arrival = atomicAdd(a.arrive + (long)b * H + h, 1u);
  }
  auto advance_lengths = [&]() {
    if (FUSED && threadIdx.x == 0 && arrival == gridDim.x - 1u) {
      __threadfence();  // every other CTA's read precedes its count, which precedes this write
      a.ap.head_lens[(long)b * H + h] = n;
      if (h == 0) a.ap.lens[b] = n;
      a.arrive[(long)b * H + h] = 0u;
    }
  };
  // (in a cluster launch every CTA takes part in the merge: splits past the
  // sequence's end just contribute empty partials)
  if (!a.csize) {
    if (n == 0) {
      if (chunk == 0)
        for (int i = threadIdx.x; i < rep * D; i += blockDim.x) a.out[((long)b * H * rep + hq0) * D + i] = 0.0f;
      return;
    }
    if (chunk >= nchunks) {
      advance_lengths();
      return;
    }
  }

  // ---- tensor formats (constants in a compile-time configuration)
  const int kbits = CFG::kbits(a), ksym = CFG::ksym(a), kf32 = CFG::kf32(a), kwhole = CFG::kwhole(a);
  const int kgpt = CFG::kgpt(a), kG = CFG::kG(a);
  const int vbits = CFG::vbits(a), vsym = CFG::vsym(a), vf32 = CFG::vf32(a), vwhole = CFG::vwhole(a);
  const int vgpt = CFG::vgpt(a), vG = CFG::vG(a);
  const int kmb = CFG::kmb(a), vmb = CFG::vmb(a);
  const int kc_bytes = CFG::kc_bytes(a), vc_bytes = CFG::vc_bytes(a);
  const int km_bytes = CFG::km_bytes(a), vm_bytes = CFG::vm_bytes(a);
  const int st_kc = CFG::st_kc(a), st_km = CFG::st_km(a), st_vc = CFG::st_vc(a), st_vm = CFG::st_vm(a);
  const int stage_bytes = CFG::stage_bytes(a), lg_ns = CFG::lg_ns(a), ns = 1 << lg_ns;
  const int tcap = a.tcap, ntiles = a.ntiles;

  // ---- shared memory carve-up
  float* qs = reinterpret_cast<float*>(smem);  // [rep][D] q * scale * log2(e)
  float* qg = qs + rep * D;                     // [gpt_k][rep] per-token key group sums of q
  unsigned char* wbase = smem + CFG::head_bytes(a) + warp * CFG::warp_bytes(a);
  uint32_t* barea = reinterpret_cast<uint32_t*>(wbase);                    // QK B operand
  float2* canK = reinterpret_cast<float2*>(wbase + CFG::barea_bytes(a));  // canonical key metadata
  float2* canV = canK + CFG::canon_k(a);                                   // canonical value metadata
  float* wbias = reinterpret_cast<float*>(canV + CFG::canon_v(a));         // [8] per-channel key bias
  unsigned char* stages = wbase + CFG::stage_off(a);

  // ---- this warp's token range and its copy sources
  // (fused append: the warp whose range holds token n_old appends it before
  // it stages anything; its range holds every tile and group the append
  // writes, so no other warp or CTA reads them)
  const int w0 = range_end(chunk * S + warp * a.Sw);
  const int w1 = range_end(chunk * S + (warp + 1) * a.Sw);
  const bool appender = FUSED && w0 <= n_old && n_old < w1;
  const int ntl = w1 > w0 ? (w1 - w0 + kTile - 1) / kTile : 0;
  const long bh = (long)b * H + h;
  const char* kc_src = a.K.codes + (bh * ntiles + (w0 >> 4)) * (long)kc_bytes;
  const char* vc_src = a.V.codes + (bh * ntiles + (w0 >> 4)) * (long)vc_bytes;
  // per-token metadata of the range's first tile (whole vector: per sequence), or its first per-channel group
  const char* km_src = k_token ? a.K.meta + (kwhole ? ((long)b * tcap + w0) : ((bh * tcap + w0) * kgpt)) * kmb
                               : a.K.meta + ((bh * (tcap >> k_lgG) + (w0 >> k_lgG)) * D) * kmb;
  const char* vm_src = VAXIS == 0 ? a.V.meta + (vwhole ? ((long)b * tcap + w0) : ((bh * tcap + w0) * vgpt)) * vmb
                                  : a.V.meta + ((bh * (tcap >> v_lgG) + (w0 >> v_lgG)) * D) * vmb;
  const int kring = a.K.ring, vring = a.V.ring;
  const __half* ktail = a.K.tail + bh * kring * D;
  const __half* vtail = a.V.tail + bh * vring * D;
  const int kgmask = k_token ? 0 : kG - 1;
  const int vgmask = VAXIS == 0 ? 0 : vG - 1;

  // Stage i of this warp's range: every lane copies its 16-byte pieces.  Tiles
  // are issued in order, so the sources are running pointers (already offset
  // by the lane) and only the shared-memory slot depends on i.
  const uint32_t st_lane = smem_u32(stages) + lane * 16;
  const char* kc_g = kc_src + lane * 16;
  const char* vc_g = vc_src + lane * 16;
  const char* km_g = km_src + lane * 16;
  const char* vm_g = vm_src + lane * 16;
  auto lane_copy = [&](uint32_t sdst, const char* gsrc, int bytes) {
#pragma unroll 4
    for (int o = 0; o < bytes; o += 512)  // uniform trip count; a lane's last piece is predicated
      if (o + lane * 16 < bytes) cp_async16_s(sdst + o, gsrc + o);
  };
  const int f16st = CFG::stage_f16(a);
  auto issue = [&](int i) {
    const int t0 = w0 + i * kTile;
    const uint32_t sa = st_lane + (i & (ns - 1)) * stage_bytes;
    // fp16 rows of the tile (16 consecutive ring rows): staged (materialised
    // rows), else prefetched into L2 for the direct loads of the tile body
    if (t0 >= sealed_k) {
      const char* src = reinterpret_cast<const char*>(ktail + (long)(t0 % kring) * D);
      if (f16st) lane_copy(sa + st_kc, src + lane * 16, 32 * D);
      else for (int o = lane * 128; o < 32 * D; o += 32 * 128) prefetch_l2(src + o);
    }
    if (t0 >= sealed_v) {
      const char* src = reinterpret_cast<const char*>(vtail + (long)(t0 % vring) * D);
      if (f16st) lane_copy(sa + st_vc, src + lane * 16, 32 * D);
      else for (int o = lane * 128; o < 32 * D; o += 32 * 128) prefetch_l2(src + o);
    }
    if (t0 < sealed_k) {
      lane_copy(sa + st_kc, kc_g, kc_bytes);
      if (k_token || (t0 & kgmask) == 0) {  // per-token: every tile; per-channel: at a group's first tile
        lane_copy(sa + st_km, km_g, km_bytes);
        km_g += km_bytes;
      }
    }
    kc_g += kc_bytes;
    if (t0 < sealed_v) {
      lane_copy(sa + st_vc, vc_g, vc_bytes);
      if (VAXIS == 0 || ((t0 + kTile) & vgmask) == 0) {  // per-channel: at a group's last tile
        lane_copy(sa + st_vm, vm_g, vm_bytes);
        vm_g += vm_bytes;
      }
    }
    vc_g += vc_bytes;
  };

  // Tiles known to be full and packed in both tensors (the bulk of every
  // range) issue their copies with no fp16-row or sealed-range checks
  // (measured: 6-7 % faster on the Llama-2-13B and serving shapes).
  const int lim_fast = min(min(sealed_k, sealed_v), w1);
  const int nfast_tiles = lim_fast > w0 ? (lim_fast - w0) >> 4 : 0;
  auto issue_fast = [&](int i) {
    const int t0 = w0 + i * kTile;
    const uint32_t sa = st_lane + (i & (ns - 1)) * stage_bytes;
    lane_copy(sa + st_kc, kc_g, kc_bytes);
    if (k_token || (t0 & kgmask) == 0) {
      lane_copy(sa + st_km, km_g, km_bytes);
      km_g += km_bytes;
    }
    kc_g += kc_bytes;
    lane_copy(sa + st_vc, vc_g, vc_bytes);
    if (VAXIS == 0 || ((t0 + kTile) & vgmask) == 0) {
      lane_copy(sa + st_vm, vm_g, vm_bytes);
      vm_g += vm_bytes;
    }
    vc_g += vc_bytes;
  };
  // the first stages go out before the query set-up, so their DRAM latency
  // overlaps it
  // (one commit group per stage, empty past the range's end, so that the
  // group of tile i is always the (i+1)-th oldest)
  auto issue_first = [&](int i0, int i1) {
    for (int i = i0; i < i1; ++i) {
      if (i < ntl) issue(i);
      cp_async_commit();
    }
  };
  // the appending warp stages at once the tiles below the first one the
  // append writes (a per-token tensor: the new token's tile; a per-channel
  // tensor: the group it seals, if it seals one) and the rest after it; the
  // append's scratch is the ring's slots from `early` on, which hold nothing
  // until then
  // With a full-precision window the append only stores fp16 rows; the block
  // (per-token tensor: 16 tokens) or group (per-channel tensor) that leaves
  // the window at this step is sealed by the warp whose range holds it
  // (ranges are multiples of 16 and of every per-channel group, so one warp
  // holds all of it, and no other warp or CTA reads it).
  int kseal = -1, vseal = -1;  // first token of the block / group this warp seals
  if (FUSED) {
    const int kw = a.K.window, vw = a.V.window;
    const int ku = k_token ? kTile : kG, vu = VAXIS == 0 ? kTile : vG;
    if (kw && n - kw >= ku && ((n - kw) & (ku - 1)) == 0 && w0 <= n - kw - ku && n - kw - ku < w1)
      kseal = n - kw - ku;
    if (vw && n - vw >= vu && ((n - vw) & (vu - 1)) == 0 && w0 <= n - vw - vu && n - vw - vu < w1)
      vseal = n - vw - vu;
  }
  int early = ns;
  if (appender || kseal >= 0 || vseal >= 0) {
    int prot = 0x7fffffff, need = 0;
    if (appender && !a.K.window) {
      if (k_token) prot = min(prot, n_old & ~(kTile - 1));
      else if (((n_old + 1) & (kG - 1)) == 0) prot = min(prot, n_old + 1 - kG), need = fused_append_scratch(D, 1, 1);
    }
    if (appender && !a.V.window) {
      if (VAXIS == 0) prot = min(prot, n_old & ~(kTile - 1));
      else if (((n_old + 1) & (vG - 1)) == 0) prot = min(prot, n_old + 1 - vG), need = fused_append_scratch(D, 1, 1);
    }
    if (kseal >= 0) prot = min(prot, kseal), need = fused_append_scratch(D, 1, 1);
    if (vseal >= 0) prot = min(prot, vseal), need = fused_append_scratch(D, 1, 1);
    early = min(min(ns, max(0, (prot - w0) / kTile)), ns - (need + stage_bytes - 1) / stage_bytes);
  }
  issue_first(0, early);

#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = threadIdx.x + u * (NW * 32);
    if (i < rep * D) qs[i] = qv[u] * a.scale_log2;
  }
  // rotary tables: pair frequencies theta_i = base^(-2i/D) as fp32 (hi, lo)
  // pairs from one fp64 evaluation each; then (cos, sin)(u * theta_i) for the
  // sixteen token offsets u of a tile
  float2* rth = reinterpret_cast<float2*>(smem + a.rope_off);  // [D/2]
  float2* rtab = rth + D / 2;                                   // [16][rope_row(D)]
  float2* rbase = rtab + 16 * rope_row(D) + warp * (D / 2);     // this warp's tile bases [D/2]
  if (ROPE && threadIdx.x < D / 2) {
    const double th = exp2(-(2.0 * threadIdx.x / D) * a.rope_l2b);
    const float hi = (float)th;
    rth[threadIdx.x] = make_float2(hi, (float)(th - (double)hi));
  }
  __syncthreads();
  if (ROPE) {
    for (int i = threadIdx.x; i < 16 * (D / 2); i += blockDim.x) {
      const int u = i / (D / 2), pr = i - u * (D / 2);
      const float2 th = rth[pr];
      float sn, cs;
      sincosf(fmaf((float)u, th.x, (float)u * th.y), &sn, &cs);
      rtab[u * rope_row(D) + pr] = make_float2(cs, sn);
    }
  }
  if (k_token) {
    const int Gk = kwhole ? D : kG;  // within one head a whole-vector group spans all D channels
    for (int i = threadIdx.x; i < kgpt * rep; i += blockDim.x) {
      const int jg = i / rep, rho = i % rep;
      float s = 0.0f;
      for (int c = jg * Gk; c < (jg + 1) * Gk; ++c) s += qs[rho * D + c];
      qg[jg * rep + rho] = s;
    }
  }
  for (int i = lane; i < CFG::barea_bytes(a) / 4; i += 32) barea[i] = 0u;
  if (lane < 8) wbias[lane] = 0.0f;
  __syncthreads();
  if (FUSED && (appender || kseal >= 0 || vseal >= 0)) {
    // append / seal into the cache (scratch: this warp's idle stage ring), make
    // the writes visible to the copies that follow, then stage the first
    // tiles; this warp's step bounds include the steps just written
    float kst = 0.0f, vst = 0.0f;
    unsigned char* scratch = stages + early * stage_bytes;
    if (appender) fused_append<D>(a.ap, b, h, n_old, scratch, &kst, &vst);
    if (kseal >= 0) kst = fmaxf(kst, seal_window_block<D>(a.ap.k, b, h, kseal, scratch));
    if (vseal >= 0) vst = fmaxf(vst, seal_window_block<D>(a.ap.v, b, h, vseal, scratch));
    smax_k = fmaxf(smax_k, kst);
    smax_v = fmaxf(smax_v, vst);
    __threadfence_block();  // only this warp reads what it wrote
    __syncwarp();
    issue_first(early, ns);
  }


  // ---- per-warp state
  float m_run[SL::N], l_run[SL::N];
#pragma unroll
  for (int s = 0; s < SL::N; ++s) {
    m_run[s] = -INFINITY;
    l_run[s] = 0.0f;
  }
  float O[NCH][4];
#pragma unroll
  for (int j = 0; j < NCH; ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) O[j][r] = 0.0f;
  // Per-token values: zero-point sums sum_t p_t * zero'_{t,g} of this lane's
  // B tokens (2tig, 2tig+1, 2tig+8, 2tig+9) for the query of its B column,
  // one per value group (groups-in-columns: one, for the lane's own group)
  float Zs[VAXIS == 0 ? GV_MAX : 1];
#pragma unroll
  for (int jg = 0; jg < (VAXIS == 0 ? GV_MAX : 1); ++jg) Zs[jg] = 0.0f;
  float Og[VAXIS == 1 ? NCH : 1][4];
  float Pg[SL::N];
#pragma unroll
  for (int j = 0; j < (VAXIS == 1 ? NCH : 1); ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) Og[j][r] = 0.0f;
#pragma unroll
  for (int s = 0; s < SL::N; ++s) Pg[s] = 0.0f;

  uint32_t breg[BREG ? NCH * 2 * NB : 1];
  auto load_b = [&]() {
    if (BREG) {
#pragma unroll
      for (int j = 0; j < NCH; ++j)
#pragma unroll
        for (int hl2 = 0; hl2 < NB; ++hl2) {
          const uint2 v = reinterpret_cast<const uint2*>(barea)[(j * NB + hl2) * 32 + lane];
          breg[BREG ? (j * NB + hl2) * 2 : 0] = v.x;
          breg[BREG ? (j * NB + hl2) * 2 + 1 : 0] = v.y;
        }
    }
  };
  // query operand normalisation: q * step * 2^E stays below 2^15 for every key
  // group (the largest stored key step of this sequence/head bounds the steps)
  float qmax = 0.0f;
  for (int i = lane; i < rep * D; i += 32) qmax = fmaxf(qmax, fabsf(qs[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
  const int E_unit = norm_exp(qmax);
  const int E_chan = k_token ? E_unit : norm_exp(qmax * smax_k);
  int Ek = E_unit;
  int qb_state = -1;  // query operand held: 0 unit with the key conversion's column scale, 1 plain unit, 2 key group
  float kbias1 = 0.0f;  // one query, per-channel keys: the group's bias sum_c q_c zero'_c (query column 0's lanes)
  // conversion exponents of the key and value codes (A = 2^(g + r*rowhalf +
  // c*colhalf) * (code + off)): key columns are channels (compensated in the
  // query operand), key rows tokens (in the score fold); value rows are
  // channels (at the output), value columns tokens (in the P operand)
  const int k_cg = conv_g(kbits), k_cr = conv_r(kbits);
  const float k_chi = exp2i(-conv_c(kbits));
  const int v_cg = conv_g(vbits), v_cr = conv_r(vbits);
  const float v_chi = exp2i(-conv_c(vbits));
  // Per-token values of 3, 5, 6, 7 and 8 bits: a second MMA per chunk with a
  // constant A of -(conv_off + 2^(B-1)) (in each register's conversion scale)
  // and the tile's P operand centres the codes on their mid-range inside the
  // accumulator, so O never holds the large offset sum (up to 1.5 * 2^B steps
  // per token) that the zero points would cancel later (fp32 cancellation
  // over long ranges); the zero points carry the matching + 2^(B-1) * step.
  // Every constant is an exact fp16.  2- and 4-bit codes enter with no offset
  // and a mid-range of at most 7.5 steps: measured, the extra MMA and its
  // registers cost more there (9 % on a 2-bit head_dim 128 batch) than the
  // accuracy it adds.
  const bool vcen = VAXIS == 0 && vbits != 2 && vbits != 4;
  uint32_t acen[4];
  {
    const float cen = (float)(conv_off(vbits) + (1 << (vbits - 1)));
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const __half hv = __float2half_rn(-cen * exp2i(v_cg + v_cr * (r & 1) + conv_c(vbits) * (r >> 1)));
      acen[r] = pack_h2(hv, hv);
    }
  }
  if (ROPE) {
    // dequantized, rotated keys meet the plain query
    build_qb<D, R8>(qs, rep, nullptr, kbits, ksym, kf32, barea, wbias, E_unit, 1.0f, lane);
    qb_state = 1;
    load_b();
  } else if (k_token) {
    build_qb<D, R8>(qs, rep, nullptr, kbits, ksym, kf32, barea, wbias, E_unit, k_chi, lane);
    qb_state = 0;
    load_b();
  }
  // value step normalisation: every folded p * step (p scaled by 2^kPExp) lies below 2^15
  const int E_v = VAXIS == 0 ? norm_exp(smax_v) - (int)kPExp : 0;
  const float sc_v = exp2i(E_v), inv_sc_v = exp2i(-E_v);
  const int hl = g & 1;
  // per-lane rows into the canonical metadata
  const int gs_k = kwhole ? 1 : kgpt, gs_v = vwhole ? 1 : vgpt;
  const int cpgk = k_token ? (kwhole ? NCH : (kG >> 4)) : NCH;  // chunks per key group (per-token keys)
  const int cpgv = VAXIS == 0 ? (vwhole ? NCH : (vG >> 4)) : NCH;
  const int lg_cpgk = 31 - __clz(cpgk), lg_cpgv = 31 - __clz(cpgv);
  const int tk0 = 2 * tig;  // B-operand tokens 2tig, 2tig+1, 2tig+8, 2tig+9
  // Per-token values with few groups per row (2 * rep * groups <= 8): every
  // (query, value group, hi/lo) gets its own B column, so one B operand per
  // tile carries all groups' step-scaled probabilities and each m-tile (one
  // channel group) reads the columns of its group.  Lane column n = g:
  // hi/lo = n & 1, group = (n >> 1) % groups, query = (n >> 1) / groups.
  const bool GC = VAXIS == 0 && !R8 && 2 * rep * gs_v <= 8;
  const int gc_grp = GC ? (g >> 1) % gs_v : 0;
  const int pv_rho = GC ? (g >> 1) / gs_v : (g >> 1);

  // Per-token values: the packed tiles accumulate O in scaled units (2^E_v, the
  // conversion's row exponent) with the zero points apart in Zs; before the
  // first fp16 row of the window, O is turned into plain units (as the
  // epilogue would) so that fp16 rows accumulate directly.
  bool o_real = false;
  // Lane holding, after the reduction over tig, the zero-point sums of
  // (query rho, value group jg): the lanes whose B column is that query's hi
  // column (groups-in-columns: of that group).
  auto zsrc = [&](int rho, int jg) { return 4 * (R8 ? rho : (GC ? 2 * (rho * gs_v + jg) : 2 * rho)); };
  // Add the zero-point sums to O (in plain units), for every output element
  // of this lane: (channel c, query rho0 / rho1).  The group of a channel is
  // the same across the warp for each (j, rr).
  auto add_zero_terms = [&]() {
    float tz[VAXIS == 0 ? GV_MAX : 1];
#pragma unroll
    for (int u = 0; u < (VAXIS == 0 ? GV_MAX : 1); ++u) {
      float v = Zs[u];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      tz[u] = v;
    }
    const int lg_gsz = vwhole ? 30 : v_lgG;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int jg = (16 * j + 8 * rr) >> lg_gsz;
        float zsel = 0.0f;
        if (GC) zsel = tz[0];
        else {
#pragma unroll
          for (int u = 0; u < (VAXIS == 0 ? GV_MAX : 1); ++u)
            if (u == jg) zsel = tz[u];
        }
        const int r0 = R8 ? 2 * tig : (GC ? min(tig / gs_v, rep - 1) : min(tig, rep - 1));
        const float z0 = __shfl_sync(0xffffffffu, zsel, zsrc(r0, jg));
        const float z1 = R8 ? __shfl_sync(0xffffffffu, zsel, zsrc(2 * tig + 1, jg)) : 0.0f;
        const float osc = inv_sc_v * exp2i(-v_cg - (rr ? v_cr : 0));  // 2^-E_v and the row exponent
        O[j][2 * rr] = O[j][2 * rr] * osc + z0;
        O[j][2 * rr + 1] = O[j][2 * rr + 1] * osc + z1;
      }
    }
  };
  // Per-token values: the packed tiles accumulate O in scaled units (2^E_v, the
  // conversion's row exponent) with the zero points apart in Zs; before the
  // first fp16 row of the window, O is turned into plain units (as the
  // epilogue would) so that fp16 rows accumulate directly.
  auto to_real = [&]() {
    add_zero_terms();
#pragma unroll
    for (int jg = 0; jg < (VAXIS == 0 ? GV_MAX : 1); ++jg) Zs[jg] = 0.0f;
    o_real = true;
  };

  // One 16-token tile.  FAST: the tile is full and both its keys and values are
  // packed (the bulk of every range), so the tail and partial-tile checks fold away.
  auto tile_body = [&](const int i, auto stag, auto ftag) {
    constexpr bool FAST = decltype(ftag)::value != 0;
    const int s = stag.get(i);
    const int t0 = w0 + i * kTile;
    // ns groups are younger than tile i's: wait until at most ns - 1 are
    // pending, then the warp barrier makes every lane's copies visible
    if (CFG::kStaticStages == 4 || (CFG::kStaticStages == 0 && lg_ns == 2)) cp_async_wait<3>();
    else cp_async_wait<1>();
    __syncwarp();
    const unsigned char* st = stages + s * stage_bytes;
    const bool kp = FAST || t0 < sealed_k, vp = FAST || t0 < sealed_v;
    const bool vflush = VAXIS == 1 && vp && ((t0 + kTile) & vgmask) == 0;

    // ---- metadata of this stage -> canonical fp32 pairs
    if (ROPE) {
      // keys: (step, zero') per channel of the group (at its first tile) or
      // per (token, group), in plain units; the register scales are applied
      // when each register is dequantized
      if (kp && (k_token || (t0 & kgmask) == 0))
        canon_meta(reinterpret_cast<const char*>(st + st_km), k_token ? kTile * gs_k : D, kbits, ksym, kf32, 1.0f,
                   1.0f, 8 * gs_k, canK, lane);
      // this tile's angle bases (cos, sin)(t0 * theta_i), halved (the rotated
      // keys enter the MMA at half scale so they stay inside fp16's range).
      // Exact two-term reduction of t0 * theta_i modulo 2 pi (Cody and Waite's
      // additive reduction with FMA): t0 < 2^24 is exact, the product's error is
      // recovered with an FMA, 2 pi is split in its nearest float and the rest.
      const float tf = (float)t0;
      for (int pr = lane; pr < D / 2; pr += 32) {
        const float2 th = rth[pr];
        const float p0 = tf * th.x;
        const float pe = fmaf(tf, th.x, -p0);
        const float kq = rintf(p0 * 0.159154943091895335769f);
        float r = fmaf(-kq, 6.28318548202514648438f, p0);
        r = fmaf(-kq, -1.74845553146951715e-7f, r);
        r += pe + tf * th.y;
        float sn, cs;
        __sincosf(r, &sn, &cs);
        rbase[pr] = make_float2(0.5f * cs, 0.5f * sn);
      }
    } else if (kp) {
      if (k_token) {
        if (qb_state != 0) {
          Ek = E_unit;
          build_qb<D, R8>(qs, rep, nullptr, kbits, ksym, kf32, barea, wbias, E_unit, k_chi, lane);
          qb_state = 0;
          load_b();
        }
        // (per-token key metadata is read raw from the stage by the fold below:
        // measured, a shared canonicalisation pass per tile plus its barrier
        // cost more than the per-lane conversions, even at 8 groups a token)
      } else if ((t0 & kgmask) == 0) {
        Ek = E_chan;
        const float b1 = build_qb<D, R8>(qs, rep, reinterpret_cast<const char*>(st + st_km), kbits, ksym, kf32, barea,
                                         wbias, E_chan, k_chi, lane);
        kbias1 = tig == 0 ? b1 : 0.0f;
        qb_state = 2;
        load_b();
      }
    } else if (qb_state != 1) {
      // fp16 rows of the keys: plain operands, no conversion scale
      Ek = E_unit;
      build_qb<D, R8>(qs, rep, nullptr, kbits, ksym, kf32, barea, wbias, E_unit, 1.0f, lane);
      qb_state = 1;
      load_b();
    }
    if (vp) {
      if (VAXIS == 1 && vflush)
        canon_meta(reinterpret_cast<const char*>(st + st_vm), D, vbits, vsym, vf32, exp2i(-v_cg), exp2i(-v_cg - v_cr), 0,
                   canV, lane);
    }
    // the entries written above are read by other lanes below (build_qb and
    // load_b synchronise on their own): a warp barrier only where this tile wrote any
    if (ROPE || (VAXIS == 1 && vflush)) __syncwarp();

    // ------------------------------------------------------------ QK ----
    float score[SL::N];
#pragma unroll
    for (int q = 0; q < SL::N; ++q) score[q] = 0.0f;
    {
      float C[4] = {0.f, 0.f, 0.f, 0.f};
      float C2[4] = {0.f, 0.f, 0.f, 0.f};  // second accumulation chain (odd chunks)
      const uint32_t* ktile = reinterpret_cast<const uint32_t*>(st + st_kc);
      const bool ktok = kp && k_token;
      // packed keys: undo 2^Ek and the conversion's row exponent
      const float inv_e0 = exp2i(-Ek - (kp ? k_cg : 0)), inv_e1 = exp2i(-Ek - (kp ? k_cg + k_cr : 0));
      // per-token keys: the stored (zero, step) of this lane's two score rows
      // for group jg, straight from the stage; the step takes the query and
      // conversion scales of its row half, the zero point (zero - conv_off *
      // step; symmetric -2^(B-1) step) multiplies the group's query sum
      const char* kraw = reinterpret_cast<const char*>(st + st_km);
      const float kpost0 = exp2i(-Ek - k_cg), kpost1 = exp2i(-Ek - k_cg - k_cr);
      const float koff = (float)conv_off(kbits), ksoff = (float)(1 << (kbits - 1));
      auto fold = [&](int jg) {
#pragma unroll
        for (int r = 0; r < 4; ++r) C[r] += C2[r];
        float ks0 = 0.f, kz0 = 0.f, ks1 = 0.f, kz1 = 0.f;
        if (ktok) {
          load_meta(kraw, g * gs_k + jg, kf32, ksym, &kz0, &ks0);
          load_meta(kraw, (g + 8) * gs_k + jg, kf32, ksym, &kz1, &ks1);
          kz0 = ksym ? -ks0 * ksoff : kz0;
          kz1 = ksym ? -ks1 * ksoff : kz1;
          if (koff != 0.0f) {  // (0 * step is not folded away under IEEE rules)
            kz0 -= koff * ks0;
            kz1 -= koff * ks1;
          }
          ks0 *= kpost0;
          ks1 *= kpost1;
        }
#pragma unroll
        for (int q = 0; q < SL::N; ++q) {
          const float v = R8 ? C[q] : (C[2 * q] + C[2 * q + 1]);
          if (ktok) {
            const int rho = min(SL::rho(q, tig), rep - 1);
            score[q] += (SL::rh(q) ? ks1 : ks0) * v + (SL::rh(q) ? kz1 : kz0) * qg[jg * rep + rho];
          } else if (kp) {
            score[q] += v * (SL::rh(q) ? inv_e1 : inv_e0) + (rep == 1 ? kbias1 : wbias[SL::rho(q, tig)]);
          } else {
            score[q] += v * inv_e0;
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          C[r] = 0.0f;
          C2[r] = 0.0f;
        }
      };
      auto mma_chunk = [&](int j, const uint32_t* A) {
#pragma unroll
        for (int hl2 = 0; hl2 < NB; ++hl2) {
          uint32_t b0, b1;
          if (BREG) {
            b0 = breg[BREG ? (j * NB + hl2) * 2 : 0];
            b1 = breg[BREG ? (j * NB + hl2) * 2 + 1 : 0];
          } else {
            const uint2 v = reinterpret_cast<const uint2*>(barea)[(j * NB + hl2) * 32 + lane];
            b0 = v.x;
            b1 = v.y;
          }
          if (j & 1) mma_16816(C2, A[0], A[1], A[2], A[3], b0, b1);
          else mma_16816(C, A[0], A[1], A[2], A[3], b0, b1);
        }
      };
      auto qk_packed = [&](auto kb) {
        constexpr int KB = decltype(kb)::value;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          uint32_t A[4];
          convert_chunk<KB, D>(ktile, lane, j, A);
          mma_chunk(j, A);
          if (ktok && ((j + 1) & (cpgk - 1)) == 0) fold(j >> lg_cpgk);
        }
      };
      if constexpr (ROPE) {
        // Dequantize each key register (row token g + 8 rh, channel pair
        // i = 8j + tig + 4 kh: the two halves are the pair's channels), turn it
        // by the token's angle t * theta_i = (t0 + u) * theta_i with
        // cos/sin(t0 theta + u theta) from this tile's bases and the in-tile
        // table, and feed it as an fp16 hi + lo pair against the plain query.
        auto rope_chunk = [&](int j, const uint32_t* A, bool packed, int kb) {
          uint32_t Ah[4], Al[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int rh = r & 1, kh = r >> 1;
            const int pr = 8 * j + tig + 4 * kh, c0 = 2 * pr;
            float2 x = __half22float2(*reinterpret_cast<const __half2*>(&A[r]));
            if (packed) {
              const float us = exp2i(-(conv_g(kb) + conv_r(kb) * rh + conv_c(kb) * kh));
              if (k_token) {
                const float2 m = canK[(g + 8 * rh) * gs_k + (kwhole ? 0 : (c0 >> k_lgG))];
                x.x = fmaf(x.x * us, m.x, m.y);
                x.y = fmaf(x.y * us, m.x, m.y);
              } else {
                const float4 m = *reinterpret_cast<const float4*>(canK + c0);
                x.x = fmaf(x.x * us, m.x, m.y);
                x.y = fmaf(x.y * us, m.z, m.w);
              }
            }
            const float2 bs = rbase[pr], ut = rtab[(g + 8 * rh) * rope_row(D) + pr];
            const float cs = bs.x * ut.x - bs.y * ut.y, sn = bs.y * ut.x + bs.x * ut.y;
            const float r0 = cs * x.x - sn * x.y, r1 = sn * x.x + cs * x.y;
            const __half2 hh = __floats2half2_rn(r0, r1);
            const float2 hf = __half22float2(hh);
            const __half2 ll = __floats2half2_rn(r0 - hf.x, r1 - hf.y);
            Ah[r] = *reinterpret_cast<const uint32_t*>(&hh);
            Al[r] = *reinterpret_cast<const uint32_t*>(&ll);
          }
#pragma unroll
          for (int hl2 = 0; hl2 < NB; ++hl2) {
            uint32_t b0, b1;
            if (BREG) {
              b0 = breg[BREG ? (j * NB + hl2) * 2 : 0];
              b1 = breg[BREG ? (j * NB + hl2) * 2 + 1 : 0];
            } else {
              const uint2 v = reinterpret_cast<const uint2*>(barea)[(j * NB + hl2) * 32 + lane];
              b0 = v.x;
              b1 = v.y;
            }
            mma_16816(C, Ah[0], Ah[1], Ah[2], Ah[3], b0, b1);
            mma_16816(C2, Al[0], Al[1], Al[2], Al[3], b0, b1);
          }
        };
        auto rope_packed = [&](auto kb) {
          constexpr int KB = decltype(kb)::value;
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            uint32_t A[4];
            convert_chunk<KB, D>(ktile, lane, j, A);
            rope_chunk(j, A, true, KB);
          }
        };
        if (kp) {
          switch (kbits) {
            case 2: rope_packed(IntC<2>{}); break;
            case 3: rope_packed(IntC<3>{}); break;
            case 4: rope_packed(IntC<4>{}); break;
            case 5: rope_packed(IntC<5>{}); break;
            case 6: rope_packed(IntC<6>{}); break;
            case 7: rope_packed(IntC<7>{}); break;
            default: rope_packed(IntC<8>{}); break;
          }
        } else {
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            const __half* tb = (f16st ? reinterpret_cast<const __half*>(st + st_kc) : ktail + (long)(t0 % kring) * D) +
                               16 * j + 2 * tig;
            uint32_t A[4];
            A[0] = *reinterpret_cast<const uint32_t*>(tb + (long)g * D);
            A[1] = *reinterpret_cast<const uint32_t*>(tb + (long)(g + 8) * D);
            A[2] = *reinterpret_cast<const uint32_t*>(tb + (long)g * D + 8);
            A[3] = *reinterpret_cast<const uint32_t*>(tb + (long)(g + 8) * D + 8);
            rope_chunk(j, A, false, 16);
          }
        }
        // keys at half scale, query at 2^E_unit
        const float inv = exp2i(1 - E_unit);
#pragma unroll
        for (int q = 0; q < SL::N; ++q) {
          const float v = R8 ? (C[q] + C2[q]) : (C[2 * q] + C[2 * q + 1] + C2[2 * q] + C2[2 * q + 1]);
          score[q] += v * inv;
        }
      } else if (kp) {
        switch (kbits) {
          case 2: qk_packed(IntC<2>{}); break;
          case 3: qk_packed(IntC<3>{}); break;
          case 4: qk_packed(IntC<4>{}); break;
          case 5: qk_packed(IntC<5>{}); break;
          case 6: qk_packed(IntC<6>{}); break;
          case 7: qk_packed(IntC<7>{}); break;
          default: qk_packed(IntC<8>{}); break;
        }
      } else {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          // fp16 tail rows: token row R = g + 8*rh, channels 16j + 2tig + 8*kh (+1)
          const __half* tb = (f16st ? reinterpret_cast<const __half*>(st + st_kc) : ktail + (long)(t0 % kring) * D) +
                             16 * j + 2 * tig;
          uint32_t A[4];
          A[0] = *reinterpret_cast<const uint32_t*>(tb + (long)g * D);
          A[1] = *reinterpret_cast<const uint32_t*>(tb + (long)(g + 8) * D);
          A[2] = *reinterpret_cast<const uint32_t*>(tb + (long)g * D + 8);
          A[3] = *reinterpret_cast<const uint32_t*>(tb + (long)(g + 8) * D + 8);
          mma_chunk(j, A);
        }
      }
      if (!ROPE && !ktok) fold(0);
    }

    // --------------------------------------------------------- softmax --
    float p[SL::N];
    float alpha[SL::N];
    {
      if (!FAST && t0 + kTile > w1) {  // partial last tile of the range
#pragma unroll
        for (int q = 0; q < SL::N; ++q)
          if (t0 + g + 8 * SL::rh(q) >= w1) score[q] = -INFINITY;
      }
      // the running max only moves when some score of the tile exceeds it
      bool up = false;
#pragma unroll
      for (int q = 0; q < SL::N; ++q) up |= score[q] > m_run[q];
      if (__any_sync(0xffffffffu, up)) {
        float tmax[SL::N];
#pragma unroll
        for (int q = 0; q < SL::N; ++q) tmax[q] = score[q];
#pragma unroll
        for (int q = 0; q < SL::N; ++q) {
          const int q2 = R8 ? (q ^ 2) : (q ^ 1);
          if (q < q2) {
            float m2 = fmaxf(tmax[q], tmax[q2]);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
            tmax[q] = m2;
            tmax[q2] = m2;
          }
        }
#pragma unroll
        for (int q = 0; q < SL::N; ++q) {
          const float mnew = fmaxf(m_run[q], tmax[q]);
          alpha[q] = fast_exp2(m_run[q] - mnew);
          m_run[q] = mnew;
        }
      } else {
#pragma unroll
        for (int q = 0; q < SL::N; ++q) alpha[q] = 1.0f;
      }
#pragma unroll
      for (int q = 0; q < SL::N; ++q) {
        p[q] = fast_exp2(score[q] - m_run[q] + kPExp);
        l_run[q] = l_run[q] * alpha[q] + p[q];
      }
    }
    {
      // O columns of this thread: non-R8 (rho = tig, hi/lo), R8 (rho = 2tig, 2tig+1)
      float a0 = alpha[0], a1 = R8 ? alpha[1] : alpha[0];
      if (GC) {  // this lane's O columns belong to query tig / groups
        a0 = __shfl_sync(0xffffffffu, alpha[0], min(tig / gs_v, rep - 1));
        a1 = a0;
      }
      if (__any_sync(0xffffffffu, (a0 != 1.0f) || (a1 != 1.0f))) {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          O[j][0] *= a0;
          O[j][1] *= a1;
          O[j][2] *= a0;
          O[j][3] *= a1;
          if (VAXIS == 1) {
            Og[VAXIS == 1 ? j : 0][0] *= a0;
            Og[VAXIS == 1 ? j : 0][1] *= a1;
            Og[VAXIS == 1 ? j : 0][2] *= a0;
            Og[VAXIS == 1 ? j : 0][3] *= a1;
          }
        }
#pragma unroll
        for (int q = 0; q < SL::N; ++q) Pg[q] *= alpha[q];
        if (VAXIS == 0) {
          // the zero-point sums follow the query of this lane's B column
          float az;
          if (!R8) {
            az = __shfl_sync(0xffffffffu, alpha[0], min(pv_rho, rep - 1));
          } else {
            const float ae = __shfl_sync(0xffffffffu, alpha[0], g >> 1);
            const float ao = __shfl_sync(0xffffffffu, alpha[1], g >> 1);
            az = (g & 1) ? ao : ae;
          }
#pragma unroll
          for (int jg = 0; jg < (VAXIS == 0 ? GV_MAX : 1); ++jg) Zs[jg] *= az;
        }
      }
    }

    // ------------------------------------------------------------ PV ----
    {
      // p of tokens 2tig, 2tig+1, 2tig+8, 2tig+9 for this lane's B column n = g
      float pv[4];
      {
        const int srcA = 8 * tig, srcB = 8 * tig + 4;
        if (!R8) {
          const int rho = pv_rho;
          pv[0] = __shfl_sync(0xffffffffu, p[0], srcA + rho);
          pv[1] = __shfl_sync(0xffffffffu, p[0], srcB + rho);
          pv[2] = __shfl_sync(0xffffffffu, p[1], srcA + rho);
          pv[3] = __shfl_sync(0xffffffffu, p[1], srcB + rho);
        } else {
          const int src_t = g >> 1, par = g & 1;
          const float e0 = __shfl_sync(0xffffffffu, p[0], srcA + src_t);
          const float e1 = __shfl_sync(0xffffffffu, p[1], srcA + src_t);
          const float f0 = __shfl_sync(0xffffffffu, p[0], srcB + src_t);
          const float f1 = __shfl_sync(0xffffffffu, p[1], srcB + src_t);
          const float e2 = __shfl_sync(0xffffffffu, p[2], srcA + src_t);
          const float e3 = __shfl_sync(0xffffffffu, p[3], srcA + src_t);
          const float f2 = __shfl_sync(0xffffffffu, p[2], srcB + src_t);
          const float f3 = __shfl_sync(0xffffffffu, p[3], srcB + src_t);
          pv[0] = par ? e1 : e0;
          pv[1] = par ? f1 : f0;
          pv[2] = par ? e3 : e2;
          pv[3] = par ? f3 : f2;
        }
      }
      const uint32_t* vtile = reinterpret_cast<const uint32_t*>(st + st_vc);
      if (VAXIS == 1) {
#pragma unroll
        for (int q = 0; q < SL::N; ++q) Pg[q] += p[q];
      }
      uint32_t bh0 = 0, bh1 = 0, bl0 = 0, bl1 = 0;
      auto make_b = [&](float x0, float x1, float x2, float x3) {
        const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        const __half2 l01 = __floats2half2_rn(x0 - f01.x, x1 - f01.y);
        const __half2 l23 = __floats2half2_rn(x2 - f23.x, x3 - f23.y);
        bh0 = *reinterpret_cast<const uint32_t*>(&h01);
        bh1 = *reinterpret_cast<const uint32_t*>(&h23);
        bl0 = *reinterpret_cast<const uint32_t*>(&l01);
        bl1 = *reinterpret_cast<const uint32_t*>(&l23);
      };
      auto mma_v = [&](int j, const uint32_t* A, bool into_group) {
        if (VAXIS == 1 && into_group) {
          if (!R8) {
            mma_16816(Og[VAXIS == 1 ? j : 0], A[0], A[1], A[2], A[3], hl ? bl0 : bh0, hl ? bl1 : bh1);
          } else {
            mma_16816(Og[VAXIS == 1 ? j : 0], A[0], A[1], A[2], A[3], bh0, bh1);
            mma_16816(Og[VAXIS == 1 ? j : 0], A[0], A[1], A[2], A[3], bl0, bl1);
          }
        } else {
          if (!R8) {
            mma_16816(O[j], A[0], A[1], A[2], A[3], hl ? bl0 : bh0, hl ? bl1 : bh1);
          } else {
            mma_16816(O[j], A[0], A[1], A[2], A[3], bh0, bh1);
            mma_16816(O[j], A[0], A[1], A[2], A[3], bl0, bl1);
          }
        }
      };
      // Per-token values: the stored (zero, step) of this lane's B tokens, read
      // straight from the stage; the B operand is p * step (with the value
      // normalisation and, for tokens 8..15, the conversion's column scale) and
      // the zero-point sums take p * zero' (zero' = zero - conv_off * step, or
      // zero + 2^(B-1) * step when the codes are centred).
      const char* vraw = reinterpret_cast<const char*>(st + st_vm);
      const float voff = (float)conv_off(vbits), vsoff = (float)(1 << (vbits - 1));
      auto vgroup = [&](int jg, float* zacc) {
        float sv[4], zv[4];
        const int tk[4] = {tk0, tk0 + 1, tk0 + 8, tk0 + 9};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float z, st;
          load_meta(vraw, tk[k] * gs_v + jg, vf32, vsym, &z, &st);
          sv[k] = st * (k < 2 ? sc_v : sc_v * v_chi);
          zv[k] = vcen ? (vsym ? 0.0f : fmaf(vsoff, st, z)) : (vsym ? -st * vsoff : z);
          if (!vcen && voff != 0.0f) zv[k] -= voff * st;  // (0 * step is not folded away under IEEE rules)
        }
        make_b(pv[0] * sv[0], pv[1] * sv[1], pv[2] * sv[2], pv[3] * sv[3]);
        *zacc += pv[0] * zv[0] + pv[1] * zv[1] + pv[2] * zv[2] + pv[3] * zv[3];
      };
      auto pv_packed = [&](auto vb) {
        constexpr int VB = decltype(vb)::value;
        if (GC) vgroup(gc_grp, &Zs[0]);
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          if (VAXIS == 0 && !GC && (j & (cpgv - 1)) == 0) {
            const int jg = j >> lg_cpgv;
            vgroup(jg, &Zs[VAXIS == 0 ? jg : 0]);
          }
          uint32_t A[4];
          convert_chunk<VB, D>(vtile, lane, j, A);
          mma_v(j, A, true);
          if (VAXIS == 0 && vcen) mma_v(j, acen, true);
        }
      };
      if (vp) {
        if (VAXIS == 1) make_b(pv[0], pv[1], pv[2] * v_chi, pv[3] * v_chi);
        switch (vbits) {
          case 2: pv_packed(IntC<2>{}); break;
          case 3: pv_packed(IntC<3>{}); break;
          case 4: pv_packed(IntC<4>{}); break;
          case 5: pv_packed(IntC<5>{}); break;
          case 6: pv_packed(IntC<6>{}); break;
          case 7: pv_packed(IntC<7>{}); break;
          default: pv_packed(IntC<8>{}); break;
        }
      } else {
        if (VAXIS == 0 && !o_real) to_real();  // per-token values: the packed part is complete
        make_b(pv[0], pv[1], pv[2], pv[3]);
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          // fp16 rows: rows = channels 16j + g (+8), columns = tokens 2tig (+1) (+8)
          const __half* tb = (f16st ? reinterpret_cast<const __half*>(st + st_vc) : vtail + (long)(t0 % vring) * D) +
                             16 * j + g;
          auto pr = [&](int t, int coff) -> uint32_t {
            return pack_h2(tb[(long)t * D + coff], tb[(long)(t + 1) * D + coff]);
          };
          uint32_t A[4];
          A[0] = pr(2 * tig, 0);
          A[1] = pr(2 * tig, 8);
          A[2] = pr(2 * tig + 8, 0);
          A[3] = pr(2 * tig + 8, 8);
          mma_v(j, A, false);
        }
      }
      // per-channel values: apply the group's steps and zero points at its last tile
      if (vflush) {
        float ps[SL::N];
#pragma unroll
        for (int q = 0; q < SL::N; ++q) {
          float v = Pg[q];
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          ps[q] = v;
        }
        const float pc0 = R8 ? (ps[0] + ps[2]) : (ps[0] + ps[1]);
        const float pc1 = R8 ? (ps[1] + ps[3]) : 0.0f;  // non-R8: the lo column carries no zero term
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const float2 m = canV[16 * j + g + 8 * rr];
            O[j][2 * rr + 0] += m.x * Og[VAXIS == 1 ? j : 0][2 * rr + 0] + m.y * pc0;
            O[j][2 * rr + 1] += m.x * Og[VAXIS == 1 ? j : 0][2 * rr + 1] + m.y * pc1;
            Og[VAXIS == 1 ? j : 0][2 * rr + 0] = 0.0f;
            Og[VAXIS == 1 ? j : 0][2 * rr + 1] = 0.0f;
          }
        }
#pragma unroll
        for (int q = 0; q < SL::N; ++q) Pg[q] = 0.0f;
      }
    }

    __syncwarp();  // every lane is done with stage s before it is refilled
    if (FAST && i + ns < nfast_tiles) issue_fast(i + ns);
    else if (i + ns < ntl) issue(i + ns);
    cp_async_commit();
  };

  {
    // fully packed, full tiles first, then the tail / partial tiles.  One tile
    // body per loop (no unrolling by the stage count): measured on GB300, the
    // four-body loop overflowed the instruction cache (the top stall was "no
    // instruction") and ran 20-27 % slower on every benchmarked workload.
    const int nfast = nfast_tiles;
    int i = 0;
    for (; i < nfast; ++i) tile_body(i, StageR{ns - 1}, IntC<1>{});
    for (; i < ntl; ++i) tile_body(i, StageR{ns - 1}, IntC<0>{});
  }
  cp_async_wait<0>();  // (only empty groups remain) before the stages are reused

  pdl_trigger();  // only the merge and the combine remain: the next kernel may start launching
  advance_lengths();

  // ---- warp epilogue: complete l and the per-token value zero-point sums
#pragma unroll
  for (int q = 0; q < SL::N; ++q) {
    float v = l_run[q];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    l_run[q] = v;
  }
  float lq0, lq1, mq0, mq1;  // per O column query
  if (!R8) {
    lq0 = l_run[0] + l_run[1];
    lq1 = lq0;
    mq0 = m_run[0];
    mq1 = m_run[0];
  } else {
    lq0 = l_run[0] + l_run[2];
    lq1 = l_run[1] + l_run[3];
    mq0 = m_run[0];
    mq1 = m_run[1];
  }
  // per-token values still in scaled units: O becomes plain units plus the zero terms
  if (VAXIS == 0 && !o_real) to_real();
  __syncthreads();  // stages are free: reuse them for the CTA merge
  float* mw = reinterpret_cast<float*>(smem + CFG::head_bytes(a));  // [4][rep][D+2]
  const int rowlen = D + 2;
  {
    const int lg_gsz = (VAXIS == 0 && !vwhole) ? v_lgG : 30;  // channel group of an output column
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int c = 16 * j + g + 8 * rr;
        float v0, v1;
        int rho0, rho1;
        if (!R8) {
          v0 = O[j][2 * rr] + O[j][2 * rr + 1];
          rho0 = tig;
          if (VAXIS == 0 && GC) rho0 = (tig % gs_v == (c >> lg_gsz)) ? tig / gs_v : -1;
          v1 = 0.0f;
          rho1 = -1;
        } else {
          v0 = O[j][2 * rr];
          v1 = O[j][2 * rr + 1];
          rho0 = 2 * tig;
          rho1 = 2 * tig + 1;
        }
        if (rho0 >= 0 && rho0 < rep) mw[(warp * rep + rho0) * rowlen + c] = v0;
        if (rho1 >= 0 && rho1 < rep) mw[(warp * rep + rho1) * rowlen + c] = v1;
      }
    }
    if (g == 0) {
      if (!R8) {
        if (tig < rep) {
          mw[(warp * rep + tig) * rowlen + D] = mq0;
          mw[(warp * rep + tig) * rowlen + D + 1] = lq0;
        }
      } else {
        mw[(warp * rep + 2 * tig) * rowlen + D] = mq0;
        mw[(warp * rep + 2 * tig) * rowlen + D + 1] = lq0;
        mw[(warp * rep + 2 * tig + 1) * rowlen + D] = mq1;
        mw[(warp * rep + 2 * tig + 1) * rowlen + D + 1] = lq1;
      }
    }
  }
  __syncthreads();
  // CTA merge -> chunk partial in the workspace (cluster launch: straight
  // into the gather area of the cluster's first CTA)
  constexpr int wrow = D + 4;  // workspace row: D outputs, m, l, two pad (16-byte aligned rows)
  const long hqb = (long)b * H * rep + hq0;
  const int max_chunks = a.max_chunks;
  namespace cg = cooperative_groups;
  float* gath = reinterpret_cast<float*>(smem + a.gath_off);  // [csize][rep][rowlen] (first CTA)
  float* part = gath;
  if (a.csize) {
    cg::cluster_group cl = cg::this_cluster();
    part = cl.map_shared_rank(gath, 0) + (int)cl.block_rank() * rep * rowlen;
    cluster_wait();  // every CTA of the cluster has started: its shared memory may be written
  }
  for (int i = threadIdx.x; i < rep * rowlen; i += blockDim.x) {
    const int rho = i / rowlen, c = i % rowlen;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mw[(w * rep + rho) * rowlen + D]);
    float acc = 0.0f;
    if (c == D) acc = M;
    else {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float mwv = mw[(w * rep + rho) * rowlen + D];
        const float f = (mwv == -INFINITY) ? 0.0f : fast_exp2(mwv - M);
        acc += f * mw[(w * rep + rho) * rowlen + c];
      }
    }
    if (a.csize) part[rho * rowlen + c] = acc;
    else a.work[((hqb + rho) * max_chunks + chunk) * wrow + c] = acc;
  }
  if (a.csize) {
    // Cluster merge: the splits of this (sequence, head) are the CTAs of one
    // cluster and have stored their partials (m_k, l_k, O_k) in the first
    // CTA's gather area; once the barrier has made them visible, that CTA
    // merges them and the others leave (nobody reads their shared memory).
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();
    if (cl.block_rank() != 0) return;
    const int K = a.csize;
    for (int i = threadIdx.x; i < rep * D; i += blockDim.x) {
      const int rho = i / D, c = i - rho * D;
      const float* pr = gath + rho * rowlen;
      float M = -INFINITY;
      for (int k = 0; k < K; ++k) M = fmaxf(M, pr[k * rep * rowlen + D]);
      float num = 0.0f, den = 0.0f;
      for (int k = 0; k < K; ++k) {
        const float* pk = pr + k * rep * rowlen;
        const float mk = pk[D];
        const float f = (mk == -INFINITY) ? 0.0f : fast_exp2(mk - M);
        den += f * pk[D + 1];
        num += f * pk[c];
      }
      a.out[(hqb + rho) * D + c] = den > 0.0f ? num / den : 0.0f;
    }
    return;
  }
  // Two-level combine behind atomic tickets (no CTA ever waits): the last CTA
  // of each group of up to kCombineGroup chunks merges the group's partials;
  // with one group it writes the output, otherwise the group result goes to
  // the group workspace and the last group merges those.
  __shared__ int last;
  uint32_t* tk = a.tickets + bh * (1 + a.max_groups);
  const int grp = chunk / kCombineGroup;
  const int ngroups = (nchunks + kCombineGroup - 1) / kCombineGroup;
  const int gsize = min(kCombineGroup, nchunks - grp * kCombineGroup);
  // every thread's partial is written before the barrier; one thread then
  // releases them all (the fence is cumulative over the writes the barrier
  // ordered before it) and takes the ticket
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = atomicAdd(tk + 1 + grp, 1u) == (unsigned)gsize - 1u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  float* sw = mw;  // combine scratch (the merge area is free again)
  // Merge K partials (m_k, l_k, O_k) per query: the (m, l) pairs are staged in
  // shared memory by all threads at once, and every output column loads its K
  // partial values as independent, unrolled loads.
  auto merge = [&](const float* src0, long qstride, int K, bool final_out, float* dst0, long dst_qstride) {
    float* wts = sw;                 // [rep][K] m_k, then weights
    float* lks = sw + rep * K;       // [rep][K] l_k
    float* tot = sw + 2 * rep * K;   // [rep][2] (M, den)
    for (int i = threadIdx.x; i < rep * K; i += blockDim.x) {
      const int rho = i / K, k = i - rho * K;
      const float* e = src0 + rho * qstride + (long)k * wrow + D;
      wts[i] = __ldcg(e);
      lks[i] = __ldcg(e + 1);
    }
    __syncthreads();
    for (int rho = threadIdx.x; rho < rep; rho += blockDim.x) {
      float M = -INFINITY;
      for (int k = 0; k < K; ++k) M = fmaxf(M, wts[rho * K + k]);
      float den = 0.0f;
      for (int k = 0; k < K; ++k) {
        const float mk = wts[rho * K + k];
        const float f = (mk == -INFINITY) ? 0.0f : fast_exp2(mk - M);
        den += f * lks[rho * K + k];
        wts[rho * K + k] = f;
      }
      tot[2 * rho] = M;
      tot[2 * rho + 1] = den;
    }
    __syncthreads();
    // four output columns per thread, up to kCombineGroup 16-byte loads in flight
    for (int i4 = threadIdx.x; i4 < rep * D / 4; i4 += blockDim.x) {
      const int rho = (4 * i4) / D, c = 4 * i4 - rho * D;
      const float4* src = reinterpret_cast<const float4*>(src0 + rho * qstride + c);
      const float* w = wts + rho * K;
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k0 = 0; k0 < K; k0 += kCombineGroup) {
        float4 v[kCombineGroup];
#pragma unroll
        for (int u = 0; u < kCombineGroup; ++u)
          v[u] = (k0 + u < K) ? __ldcg(src + (long)(k0 + u) * (wrow / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kCombineGroup; ++u)
          if (k0 + u < K) {
            const float f = w[k0 + u];
            num.x += f * v[u].x;
            num.y += f * v[u].y;
            num.z += f * v[u].z;
            num.w += f * v[u].w;
          }
      }
      if (final_out) {
        const float den = tot[2 * rho + 1];
        const float inv = den > 0.0f ? 1.0f / den : 0.0f;
        float* o = a.out + (hqb + rho) * D + c;
        o[0] = num.x * inv;
        o[1] = num.y * inv;
        o[2] = num.z * inv;
        o[3] = num.w * inv;
      } else {
        *reinterpret_cast<float4*>(dst0 + rho * dst_qstride + c) = num;
      }
    }
    if (!final_out)
      for (int rho = threadIdx.x; rho < rep; rho += blockDim.x) {
        dst0[rho * dst_qstride + D] = tot[2 * rho];
        dst0[rho * dst_qstride + D + 1] = tot[2 * rho + 1];
      }
  };
  const float* part0 = a.work + (hqb * max_chunks + (long)grp * kCombineGroup) * wrow;
  if (ngroups == 1) {
    merge(part0, (long)max_chunks * wrow, gsize, true, nullptr, 0);
    if (threadIdx.x == 0) tk[1 + grp] = 0u;
    return;
  }
  float* g0 = a.gwork + (hqb * a.max_groups + grp) * wrow;
  merge(part0, (long)max_chunks * wrow, gsize, false, g0, (long)a.max_groups * wrow);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    tk[1 + grp] = 0u;
    last = atomicAdd(tk, 1u) == (unsigned)ngroups - 1u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  merge(a.gwork + hqb * a.max_groups * wrow, (long)a.max_groups * wrow, ngroups, true, nullptr, 0);
  if (threadIdx.x == 0) tk[0] = 0u;
}

}  // namespace kvq
