// kvq_decode.cuh — split-K decode attention over the packed KV cache (sm_103a).
//
// One CTA = one (sequence, kv head, token chunk); 4 warps, each an independent
// flash-decoding pass over a contiguous, group-aligned sub-range, merged at the
// end of the CTA; the last CTA of a (sequence, kv head) merges all chunks
// (log-sum-exp combine) behind an atomic ticket, so no kernel ever waits on
// another CTA.
//
// Per 16-token tile a warp:
//   1. waits for its stage: packed codes + metadata copied global -> shared by
//      the TMA engine (cp.async.bulk, mbarrier completion, bounded waits);
//   2. QK: converts the key codes of each 16-channel chunk to exact fp16
//      operands in registers (rotate + one LOP3 per code pair: the code lands
//      in the top mantissa bits of an fp16 whose exponent makes its value
//      2^B + code) and runs mma.sync m16n8k16 against the query split into
//      fp16 hi + lo parts (~22-bit operand, fp32 accumulation); scales, zero
//      points and the 2^B offset are folded into the query (per-channel keys)
//      or applied to the fp32 accumulators (per-token keys);
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

#include "kvq_decode_args.h"

namespace kvq {

// ---------------------------------------------------------------- planes ---

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

// Four fp16x2 MMA operand registers (pairs 4j..4j+3 of this lane) holding
// 2^BITS + code, exact.
template <int BITS, int D>
__device__ __forceinline__ void convert_chunk(const uint32_t* tile, int lane, int j, uint32_t a[4]) {
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

// per-tensor metadata entry -> (zero', step) with zero' = zero - 2^B step (asym) or the
// symmetric equivalent: the value is step * (2^B + code) + zero'
__device__ __forceinline__ void meta_fold(const char* m, int idx, const TensorLayout& L, float* zf, float* st) {
  float z, s;
  load_meta(m, idx, L.meta_f32, L.sym, &z, &s);
  const float off = (float)(1 << L.bits);
  if (L.sym) z = -s * (float)(1 << (L.bits - 1));
  *st = s;
  *zf = z - off * s;
}

template <bool R8>
struct Slots {
  static constexpr int N = R8 ? 4 : 2;
  __device__ static int rh(int s) { return R8 ? (s >> 1) : s; }
  __device__ static int rho(int s, int tig) { return R8 ? (2 * tig + (s & 1)) : tig; }
};

// -------------------------------------------------- query operand build ---

// Build the fragment-ordered QK B operand of one warp for a set of channel
// scales (per-channel keys: this group's steps; per-token keys / fp16 tail:
// unit scales), with the power-of-two normalisation E and the bias
// sum_c q_c zero'_c per query.  Values (rho >= rep) stay zero.
template <int D, bool R8>
__device__ void build_qb(const float* qs, int rep, const char* kmeta_grp, const TensorLayout& K, bool unit,
                         uint32_t* barea, float* bias, int* Eout) {
  const int lane = threadIdx.x & 31;
  // pass 1: max |q * s|
  float mx = 0.0f;
  for (int i = lane; i < rep * D; i += 32) {
    int rho = i / D, c = i % D;
    float s = 1.0f, z = 0.0f;
    if (!unit) meta_fold(kmeta_grp, c, K, &z, &s);
    mx = fmaxf(mx, fabsf(qs[rho * D + c] * s));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const int E = norm_exp(mx);
  const float sc = exp2i(E);
  // pass 2: channel pairs -> hi/lo fp16 pairs scattered to fragment positions
  float bsum[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) bsum[r] = 0.0f;
  for (int i = lane; i < rep * (D / 2); i += 32) {
    int rho = i / (D / 2), c = 2 * (i % (D / 2));
    float s0 = 1.0f, z0 = 0.0f, s1 = 1.0f, z1 = 0.0f;
    if (!unit) {
      meta_fold(kmeta_grp, c, K, &z0, &s0);
      meta_fold(kmeta_grp, c + 1, K, &z1, &s1);
    }
    float q0 = qs[rho * D + c], q1 = qs[rho * D + c + 1];
    float v0 = q0 * s0 * sc, v1 = q1 * s1 * sc;
    __half h0, l0, h1, l1;
    split_hl(v0, &h0, &l0);
    split_hl(v1, &h1, &l1);
    if (!unit) {
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r == rho) bsum[r] += q0 * z0 + q1 * z1;
    }
    // fragment position of channel pair (c, c+1): chunk j, tig, b0/b1
    int j = c >> 4, cc = c & 15, tig = (cc & 7) >> 1, breg = cc >> 3;
    if (!R8) {
      int ghi = 2 * rho, glo = 2 * rho + 1;
      barea[(j * 32 + 4 * ghi + tig) * 2 + breg] = pack_h2(h0, h1);
      barea[(j * 32 + 4 * glo + tig) * 2 + breg] = pack_h2(l0, l1);
    } else {
      barea[((j * 2 + 0) * 32 + 4 * rho + tig) * 2 + breg] = pack_h2(h0, h1);
      barea[((j * 2 + 1) * 32 + 4 * rho + tig) * 2 + breg] = pack_h2(l0, l1);
    }
  }
  if (!unit) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float v = bsum[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && r < rep) bias[r] = v;
    }
  }
  *Eout = E;
  __syncwarp();
}

// --------------------------------------------------------------- kernel ----

template <int D, bool R8, int VAXIS>
__global__ void __launch_bounds__(128) decode_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int NCH = D / 16;  // 16-channel chunks / m-tiles
  using SL = Slots<R8>;
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int rep = a.rep;
  const int n = a.lens[b];
  const int nchunks = (n + a.S - 1) / a.S;
  const int hq0 = h * rep;
  if (n == 0) {
    if (chunk == 0)
      for (int i = threadIdx.x; i < rep * D; i += blockDim.x) a.out[((long)b * a.H * rep + hq0) * D + i] = 0.0f;
    return;
  }
  if (chunk >= nchunks) return;

  // ---- shared memory carve-up
  float* qs = reinterpret_cast<float*>(smem);          // [rep][D] q * scale * log2(e)
  float* qg = qs + rep * D;                              // [gpt_k][rep] per-token key group sums of q
  unsigned char* wbase = smem + a.head_bytes + warp * a.warp_bytes;
  uint32_t* barea = reinterpret_cast<uint32_t*>(wbase);  // QK B operand
  float* wbias = reinterpret_cast<float*>(wbase + a.barea_bytes);  // [8] per-channel key bias
  unsigned char* stages = wbase + a.barea_bytes + 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stages + a.nstages * a.stage_bytes);

  for (int i = threadIdx.x; i < rep * D; i += blockDim.x) {
    const long qi = ((long)b * a.H * rep + hq0) * D + i;
    qs[i] = (a.q_f32 ? reinterpret_cast<const float*>(a.q)[qi] : __half2float(reinterpret_cast<const __half*>(a.q)[qi])) *
            a.scale_log2;
  }
  const int gpt_k = a.K.gpt;
  const bool k_token = a.K.axis == 0, k_whole = a.K.whole;
  __syncthreads();
  if (k_token) {
    const int Gk = k_whole ? D : a.K.group;  // within one head a whole-vector group spans all D channels
    for (int i = threadIdx.x; i < gpt_k * rep; i += blockDim.x) {
      int jg = i / rep, rho = i % rep;
      float s = 0.0f;
      for (int c = jg * Gk; c < (jg + 1) * Gk; ++c) s += qs[rho * D + c];
      qg[jg * rep + rho] = s;
    }
  }
  // zero this warp's B operand area (unused query columns must stay zero)
  for (int i = lane; i < a.barea_bytes / 4; i += 32) barea[i] = 0u;
  if (lane == 0)
    for (int s = 0; s < a.nstages; ++s) mbar_init(&bars[s], 1);
  fence_mbar_init();
  __syncthreads();

  // ---- this warp's token range
  const int w0 = chunk * a.S + warp * a.Sw;
  const int w1 = min(w0 + a.Sw, n);
  const int ntl = w1 > w0 ? (w1 - w0 + kTile - 1) / kTile : 0;
  const int sealed_k = a.K.axis == 1 ? (n / a.K.group) * a.K.group : n;
  const int sealed_v = a.V.axis == 1 ? (n / a.V.group) * a.V.group : n;
  const long bh = (long)b * a.H + h;
  const char* kcodes = a.base + a.K.codes_off + a.layer * a.K.codes_layer + bh * a.ntiles * (long)a.kc_bytes;
  const char* vcodes = a.base + a.V.codes_off + a.layer * a.V.codes_layer + bh * a.ntiles * (long)a.vc_bytes;
  const char* kmeta = a.base + a.K.meta_off + a.layer * a.K.meta_layer;
  const char* vmeta = a.base + a.V.meta_off + a.layer * a.V.meta_layer;
  const __half* ktail = reinterpret_cast<const __half*>(a.base + a.K.tail_off + a.layer * a.K.tail_layer) +
                        bh * a.K.group * D;
  const __half* vtail = reinterpret_cast<const __half*>(a.base + a.V.tail_off + a.layer * a.V.tail_layer) +
                        bh * a.V.group * D;

  auto meta_src = [&](const TensorLayout& L, const char* mbase, int t0, int per_tile_bytes) -> const char* {
    long idx;
    if (L.whole) idx = (long)b * a.tcap + t0;
    else idx = (bh * a.tcap + t0) * L.gpt;
    (void)per_tile_bytes;
    return mbase + idx * L.meta_bytes;
  };

  auto issue = [&](int i) {
    const int s = i % a.nstages;
    const int t0 = w0 + i * kTile;
    unsigned char* st = stages + s * a.stage_bytes;
    uint32_t bytes = 0;
    const bool kp = t0 < sealed_k, vp = t0 < sealed_v;
    const bool kgrp = kp && a.K.axis == 1 && (t0 % a.K.group) == 0;
    const bool vgrp = vp && a.V.axis == 1 && ((t0 + kTile) % a.V.group) == 0;
    if (kp) bytes += a.kc_bytes + (a.K.axis == 1 ? (kgrp ? a.km_group_bytes : 0) : a.km_tile_bytes);
    if (vp) bytes += a.vc_bytes + (a.V.axis == 1 ? (vgrp ? a.vm_group_bytes : 0) : a.vm_tile_bytes);
    mbar_expect_tx(&bars[s], bytes);
    if (kp) {
      bulk_g2s(st + a.st_kc, kcodes + (long)(t0 / kTile) * a.kc_bytes, a.kc_bytes, &bars[s]);
      if (a.K.axis == 0) bulk_g2s(st + a.st_km, meta_src(a.K, kmeta, t0, a.km_tile_bytes), a.km_tile_bytes, &bars[s]);
      else if (kgrp)
        bulk_g2s(st + a.st_km, kmeta + ((bh * (a.tcap / a.K.group) + t0 / a.K.group) * D) * a.K.meta_bytes,
                 a.km_group_bytes, &bars[s]);
    }
    if (vp) {
      bulk_g2s(st + a.st_vc, vcodes + (long)(t0 / kTile) * a.vc_bytes, a.vc_bytes, &bars[s]);
      if (a.V.axis == 0) bulk_g2s(st + a.st_vm, meta_src(a.V, vmeta, t0, a.vm_tile_bytes), a.vm_tile_bytes, &bars[s]);
      else if (vgrp)
        bulk_g2s(st + a.st_vm, vmeta + ((bh * (a.tcap / a.V.group) + t0 / a.V.group) * D) * a.V.meta_bytes,
                 a.vm_group_bytes, &bars[s]);
    }
  };

  if (lane == 0)
    for (int i = 0; i < min(ntl, a.nstages); ++i) issue(i);

  // ---- per-warp state
  float m_run[SL::N], l_run[SL::N];  // per slot (slots with equal rho hold equal m)
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
  // per-token values: zero-point sums per group and slot-query; per-channel values: group accumulators
  constexpr int GV_MAX = D / 32;
  float Zs[GV_MAX][SL::N];
#pragma unroll
  for (int jg = 0; jg < GV_MAX; ++jg)
#pragma unroll
    for (int s = 0; s < SL::N; ++s) Zs[jg][s] = 0.0f;
  float Og[VAXIS == 1 ? NCH : 1][4];
  float Pg[SL::N];
#pragma unroll
  for (int j = 0; j < (VAXIS == 1 ? NCH : 1); ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) Og[j][r] = 0.0f;
#pragma unroll
  for (int s = 0; s < SL::N; ++s) Pg[s] = 0.0f;

  int Eq = 0;
  bool qb_unit = false;  // barea holds plain q (per-token keys or key tail)
  if (k_token) {
    build_qb<D, R8>(qs, rep, nullptr, a.K, true, barea, wbias, &Eq);
    qb_unit = true;
  }
  const float inv_eq_tok = exp2i(-Eq);
  int E_v = 0;
  if (a.V.axis == 0) {
    float smax = __uint_as_float(a.smax_v[bh]);
    E_v = norm_exp(smax);
  }
  const float sc_v = exp2i(E_v), inv_sc_v = exp2i(-E_v);
  int Ek = Eq;
  bool failed = false;

  for (int i = 0; i < ntl; ++i) {
    const int s = i % a.nstages;
    const int t0 = w0 + i * kTile;
    if (!failed && !mbar_wait_bounded(&bars[s], (uint32_t)((i / a.nstages) & 1), a.err)) failed = true;
    if (failed) break;
    const unsigned char* st = stages + s * a.stage_bytes;
    const bool kp = t0 < sealed_k, vp = t0 < sealed_v;

    // ------------------------------------------------------------ QK ----
    float score[SL::N];
#pragma unroll
    for (int q = 0; q < SL::N; ++q) score[q] = 0.0f;
    if (kp && a.K.axis == 1 && (t0 % a.K.group) == 0) {
      build_qb<D, R8>(qs, rep, reinterpret_cast<const char*>(st + a.st_km), a.K, false, barea, wbias, &Ek);
      qb_unit = false;
    } else if (!kp && !qb_unit) {
      build_qb<D, R8>(qs, rep, nullptr, a.K, true, barea, wbias, &Ek);
      qb_unit = true;
    }
    {
      float C[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t* ktile = reinterpret_cast<const uint32_t*>(st + a.st_kc);
      const int cpg = k_token ? (k_whole ? NCH : a.K.group / 16) : NCH;
      const float inv_e = exp2i(-Ek);
      auto fold_group = [&](int jg) {
#pragma unroll
        for (int q = 0; q < SL::N; ++q) {
          float v = R8 ? C[q] : (C[2 * q] + C[2 * q + 1]);
          if (kp && k_token) {
            const int row = g + 8 * SL::rh(q);
            float zf, stp;
            meta_fold(reinterpret_cast<const char*>(st + a.st_km), k_whole ? row : row * gpt_k + jg, a.K, &zf, &stp);
            const int rho = SL::rho(q, tig);
            const float qsum = rho < rep ? qg[jg * rep + rho] : 0.0f;
            score[q] += stp * v * inv_e + zf * qsum;
          } else if (kp) {
            const int rho = SL::rho(q, tig);
            score[q] += v * inv_e + (rho < rep ? wbias[rho] : 0.0f);
          } else {
            score[q] += v * inv_e;
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) C[r] = 0.0f;
      };
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        uint32_t A[4];
        if (kp) {
          switch (a.K.bits) {
            case 2: convert_chunk<2, D>(ktile, lane, j, A); break;
            case 3: convert_chunk<3, D>(ktile, lane, j, A); break;
            case 4: convert_chunk<4, D>(ktile, lane, j, A); break;
            case 5: convert_chunk<5, D>(ktile, lane, j, A); break;
            case 6: convert_chunk<6, D>(ktile, lane, j, A); break;
            case 7: convert_chunk<7, D>(ktile, lane, j, A); break;
            default: convert_chunk<8, D>(ktile, lane, j, A); break;
          }
        } else {
          // fp16 tail rows: token row R = g + 8*rh, channels 16j + 2tig + 8*kh (+1)
          const __half* tb = ktail + (long)(t0 - sealed_k) * D + 16 * j + 2 * tig;
          A[0] = *reinterpret_cast<const uint32_t*>(tb + (long)g * D);
          A[1] = *reinterpret_cast<const uint32_t*>(tb + (long)(g + 8) * D);
          A[2] = *reinterpret_cast<const uint32_t*>(tb + (long)g * D + 8);
          A[3] = *reinterpret_cast<const uint32_t*>(tb + (long)(g + 8) * D + 8);
        }
        if (!R8) {
          uint2 bb = reinterpret_cast<const uint2*>(barea)[j * 32 + lane];
          mma_16816(C, A[0], A[1], A[2], A[3], bb.x, bb.y);
        } else {
          uint2 bh2 = reinterpret_cast<const uint2*>(barea)[(j * 2) * 32 + lane];
          uint2 bl2 = reinterpret_cast<const uint2*>(barea)[(j * 2 + 1) * 32 + lane];
          mma_16816(C, A[0], A[1], A[2], A[3], bh2.x, bh2.y);
          mma_16816(C, A[0], A[1], A[2], A[3], bl2.x, bl2.y);
        }
        if (kp && k_token) {
          if ((j + 1) % cpg == 0) fold_group(j / cpg);
        }
      }
      if (!(kp && k_token)) fold_group(0);
    }

    // --------------------------------------------------------- softmax --
    float p[SL::N];
    float alpha[SL::N];
    {
      float tmax[SL::N];
#pragma unroll
      for (int q = 0; q < SL::N; ++q) {
        const int t = t0 + g + 8 * SL::rh(q);
        const int rho = SL::rho(q, tig);
        if (t >= w1 || rho >= rep) score[q] = -INFINITY;
        tmax[q] = score[q];
      }
      // combine the two row-halves of the same query, then across the 8 token rows
#pragma unroll
      for (int q = 0; q < SL::N; ++q) {
        const int q2 = R8 ? (q ^ 2) : (q ^ 1);
        if (q < q2) {
          float m2 = fmaxf(tmax[q], tmax[q2]);
          tmax[q] = m2;
          tmax[q2] = m2;
        }
      }
#pragma unroll
      for (int q = 0; q < SL::N; ++q) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) tmax[q] = fmaxf(tmax[q], __shfl_xor_sync(0xffffffffu, tmax[q], o));
      }
#pragma unroll
      for (int q = 0; q < SL::N; ++q) {
        const float mnew = fmaxf(m_run[q], tmax[q]);
        alpha[q] = (mnew == -INFINITY) ? 1.0f : fast_exp2(m_run[q] - mnew);
        p[q] = (mnew == -INFINITY) ? 0.0f : fast_exp2(score[q] - mnew);
        m_run[q] = mnew;
        l_run[q] = l_run[q] * alpha[q] + p[q];
      }
    }
    // rescale accumulators: O columns of this thread belong to its slot queries
    {
      // non-R8: columns (2tig, 2tig+1) = (rho = tig, hi/lo) -> alpha[0] (== alpha[1])
      // R8    : columns (2tig, 2tig+1) = rho 2tig, 2tig+1   -> alpha[0], alpha[1]
      const float a0 = alpha[0], a1 = R8 ? alpha[1] : alpha[0];
      const bool need = (a0 != 1.0f) || (a1 != 1.0f);
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          O[j][0] *= a0;
          O[j][1] *= a1;
          O[j][2] *= a0;
          O[j][3] *= a1;
          if (VAXIS == 1) {
            Og[j][0] *= a0;
            Og[j][1] *= a1;
            Og[j][2] *= a0;
            Og[j][3] *= a1;
          }
        }
#pragma unroll
        for (int q = 0; q < SL::N; ++q) {
          Pg[q] *= alpha[q];
#pragma unroll
          for (int jg = 0; jg < GV_MAX; ++jg) Zs[jg][q] *= alpha[q];
        }
      }
    }

    // ------------------------------------------------------------ PV ----
    {
      // gather p for the B operand: tokens 2tig, 2tig+1, 2tig+8, 2tig+9 of column n = g
      float pv[4];
      {
        const int srcA = 8 * tig, srcB = 8 * tig + 4;
        if (!R8) {
          const int rho = g >> 1;
          float x0 = __shfl_sync(0xffffffffu, p[0], srcA + (rho & 3));
          float x1 = __shfl_sync(0xffffffffu, p[0], srcB + (rho & 3));
          float x2 = __shfl_sync(0xffffffffu, p[1], srcA + (rho & 3));
          float x3 = __shfl_sync(0xffffffffu, p[1], srcB + (rho & 3));
          pv[0] = x0; pv[1] = x1; pv[2] = x2; pv[3] = x3;
        } else {
          const int src_t = g >> 1, par = g & 1;
          float e0 = __shfl_sync(0xffffffffu, p[0], srcA + src_t);
          float e1 = __shfl_sync(0xffffffffu, p[1], srcA + src_t);
          float f0 = __shfl_sync(0xffffffffu, p[0], srcB + src_t);
          float f1 = __shfl_sync(0xffffffffu, p[1], srcB + src_t);
          float e2 = __shfl_sync(0xffffffffu, p[2], srcA + src_t);
          float e3 = __shfl_sync(0xffffffffu, p[3], srcA + src_t);
          float f2 = __shfl_sync(0xffffffffu, p[2], srcB + src_t);
          float f3 = __shfl_sync(0xffffffffu, p[3], srcB + src_t);
          pv[0] = par ? e1 : e0;
          pv[1] = par ? f1 : f0;
          pv[2] = par ? e3 : e2;
          pv[3] = par ? f3 : f2;
        }
      }
      const int hl = g & 1;  // non-R8: this lane's column is the lo part when odd
      const int tok[4] = {2 * tig, 2 * tig + 1, 2 * tig + 8, 2 * tig + 9};
      const uint32_t* vtile = reinterpret_cast<const uint32_t*>(st + a.st_vc);
      const char* vm = reinterpret_cast<const char*>(st + a.st_vm);
      // zero-point sums (per-token values) at the score owners
      if (vp && VAXIS == 0) {
#pragma unroll
        for (int jg = 0; jg < GV_MAX; ++jg) {
          if (jg >= (a.V.whole ? 1 : a.V.gpt)) break;
#pragma unroll
          for (int q = 0; q < SL::N; ++q) {
            const int row = g + 8 * SL::rh(q);
            float zf, stp;
            meta_fold(vm, a.V.whole ? row : row * a.V.gpt + jg, a.V, &zf, &stp);
            Zs[jg][q] += p[q] * zf;
          }
        }
      }
      if (VAXIS == 1) {
#pragma unroll
        for (int q = 0; q < SL::N; ++q) Pg[q] += p[q];
      }
      uint32_t bh0 = 0, bh1 = 0, bl0 = 0, bl1 = 0;
      auto make_b = [&](int jg, bool fold) {
        float x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float v = pv[u];
          if (fold) {
            float zf, stp;
            meta_fold(vm, a.V.whole ? tok[u] : tok[u] * a.V.gpt + jg, a.V, &zf, &stp);
            v = v * stp * sc_v;
          }
          x[u] = v;
        }
        __half h[4], l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) split_hl(x[u], &h[u], &l[u]);
        bh0 = pack_h2(h[0], h[1]);
        bh1 = pack_h2(h[2], h[3]);
        bl0 = pack_h2(l[0], l[1]);
        bl1 = pack_h2(l[2], l[3]);
      };
      const int cpg_v = (VAXIS == 0) ? (a.V.whole ? NCH : a.V.group / 16) : NCH;
      if (!vp || VAXIS == 1) make_b(0, false);
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        if (vp && VAXIS == 0 && (j % cpg_v) == 0) make_b(j / cpg_v, true);
        uint32_t A[4];
        if (vp) {
          switch (a.V.bits) {
            case 2: convert_chunk<2, D>(vtile, lane, j, A); break;
            case 3: convert_chunk<3, D>(vtile, lane, j, A); break;
            case 4: convert_chunk<4, D>(vtile, lane, j, A); break;
            case 5: convert_chunk<5, D>(vtile, lane, j, A); break;
            case 6: convert_chunk<6, D>(vtile, lane, j, A); break;
            case 7: convert_chunk<7, D>(vtile, lane, j, A); break;
            default: convert_chunk<8, D>(vtile, lane, j, A); break;
          }
        } else {
          // fp16 tail: rows = channels 16j + g (+8), columns = tokens 2tig (+1) (+8)
          const __half* tb = vtail + (long)(t0 - sealed_v) * D + 16 * j + g;
          auto pr = [&](int t, int coff) -> uint32_t {
            return pack_h2(tb[(long)t * D + coff], tb[(long)(t + 1) * D + coff]);
          };
          A[0] = pr(2 * tig, 0);
          A[1] = pr(2 * tig, 8);
          A[2] = pr(2 * tig + 8, 0);
          A[3] = pr(2 * tig + 8, 8);
        }
        if (vp && VAXIS == 1) {
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
      }
      // per-channel values: flush the group at its last tile
      if (VAXIS == 1 && vp && ((t0 + kTile) % a.V.group) == 0) {
        // P sums per query: reduce over the 8 token rows and both row halves
        float ps[SL::N];
#pragma unroll
        for (int q = 0; q < SL::N; ++q) {
          float v = Pg[q];
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          ps[q] = v;
        }
        float pc0, pc1;  // query sums for this thread's two O columns
        if (!R8) {
          pc0 = ps[0] + ps[1];
          pc1 = 0.0f;  // lo column carries no zero-point term
        } else {
          pc0 = ps[0] + ps[2];
          pc1 = ps[1] + ps[3];
        }
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int c = 16 * j + g + 8 * rr;
            float zf, stp;
            meta_fold(vm, c, a.V, &zf, &stp);
            O[j][2 * rr + 0] += stp * Og[VAXIS == 1 ? j : 0][2 * rr + 0] + zf * pc0;
            O[j][2 * rr + 1] += stp * Og[VAXIS == 1 ? j : 0][2 * rr + 1] + zf * pc1;
            Og[VAXIS == 1 ? j : 0][2 * rr + 0] = 0.0f;
            Og[VAXIS == 1 ? j : 0][2 * rr + 1] = 0.0f;
          }
        }
#pragma unroll
        for (int q = 0; q < SL::N; ++q) Pg[q] = 0.0f;
      }
    }

    __syncwarp();
    if (lane == 0 && i + a.nstages < ntl) {
      fence_proxy_async();
      issue(i + a.nstages);
    }
  }
  if (failed) {
    // give copies still in flight a bounded chance to land before the CTA exits
    if (lane == 0)
      for (int i = 0; i < min(ntl, a.nstages); ++i) {
        const int s = i % a.nstages;
        mbar_wait_bounded(&bars[s], 0u, nullptr);
      }
  }

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
  // per-token values: O (in units of 2^E_v) -> true units, plus zero-point sums
  if (VAXIS == 0) {
#pragma unroll
    for (int jg = 0; jg < GV_MAX; ++jg)
#pragma unroll
      for (int q = 0; q < SL::N; ++q) {
        float v = Zs[jg][q];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        Zs[jg][q] = v;
      }
  }
  __syncthreads();  // stages are free: reuse them for the CTA merge
  float* mw = reinterpret_cast<float*>(smem + a.head_bytes);  // [4][rep][D+2]
  const int rowlen = D + 2;
  // write this warp's (m, l, O) per query
  {
    const int gcnt = (VAXIS == 0) ? (a.V.whole ? 1 : a.V.gpt) : 1;
    const int gsz = (VAXIS == 0) ? (a.V.whole ? D : a.V.group) : D;
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
          v1 = 0.0f;
          rho1 = -1;
        } else {
          v0 = O[j][2 * rr];
          v1 = O[j][2 * rr + 1];
          rho0 = 2 * tig;
          rho1 = 2 * tig + 1;
        }
        if (VAXIS == 0) {
          const int jg = c / gsz;
          float z0 = 0.f, z1 = 0.f;
#pragma unroll
          for (int u = 0; u < GV_MAX; ++u)
            if (u == jg) {
              z0 = R8 ? (Zs[u][0] + Zs[u][2]) : (Zs[u][0] + Zs[u][1]);
              z1 = R8 ? (Zs[u][1] + Zs[u][3]) : 0.0f;
            }
          (void)gcnt;
          v0 = v0 * inv_sc_v + z0;
          v1 = v1 * inv_sc_v + z1;
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
  // CTA merge -> chunk partial in the workspace
  const long hqb = (long)b * a.H * rep + hq0;
  for (int i = threadIdx.x; i < rep * rowlen; i += blockDim.x) {
    const int rho = i / rowlen, c = i % rowlen;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[(w * rep + rho) * rowlen + D]);
    float acc = 0.0f;
    if (c == D) acc = M;
    else {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mwv = mw[(w * rep + rho) * rowlen + D];
        const float f = (mwv == -INFINITY) ? 0.0f : fast_exp2(mwv - M);
        acc += f * mw[(w * rep + rho) * rowlen + c];
      }
    }
    a.work[((hqb + rho) * a.max_chunks + chunk) * rowlen + c] = acc;
  }
  // the last CTA of (b, h) combines all chunks
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev = atomicAdd(a.tickets + bh, 1u);
    last = (prev == (unsigned)nchunks - 1u);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = threadIdx.x; i < rep * D; i += blockDim.x) {
    const int rho = i / D, c = i % D;
    const float* pbase = a.work + (hqb + rho) * a.max_chunks * (long)rowlen;
    float M = -INFINITY;
    for (int k = 0; k < nchunks; ++k) M = fmaxf(M, __ldcg(pbase + (long)k * rowlen + D));
    float num = 0.0f, den = 0.0f;
    for (int k = 0; k < nchunks; ++k) {
      const float mk = __ldcg(pbase + (long)k * rowlen + D);
      const float f = (mk == -INFINITY) ? 0.0f : fast_exp2(mk - M);
      num += f * __ldcg(pbase + (long)k * rowlen + c);
      den += f * __ldcg(pbase + (long)k * rowlen + D + 1);
    }
    a.out[(hqb + rho) * D + c] = den > 0.0f ? num / den : 0.0f;
  }
  if (threadIdx.x == 0) a.tickets[bh] = 0u;
}

}  // namespace kvq
