/*
 * kvq_oracle.c — plain, slow, scalar CPU oracle for group-wise integer KV-cache
 * quantization and single-token decode attention over the dequantized cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, import or
 * execute this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no source with the CUDA library.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC (no FMA
 * contraction, IEEE fp32 division), so every float operation below is one
 * correctly rounded IEEE-754 operation in the order written.
 *
 * What each function follows (page title, section):
 *  - Cache size: "Kuantisasi KV Cache untuk Mengurangi Memory Inferensi Long
 *    Context", section "Ukuran cache bertambah mengikuti token, layer, dan KV
 *    head" (elements = 2 * layers * cached_tokens * kv_heads * head_dim) and
 *    section "Pengecualian recent-token mengubah perhitungan memory" (total =
 *    recent high-precision part + packed codes + scales/metadata + workspace).
 *  - Symmetric quantizer: same page, section "Scale menentukan sistem koordinat
 *    kuantisasi" (q = clamp(round(x/scale), q_min, q_max), x_hat = q*scale).
 *  - Asymmetric quantizer: "O Seu Cache KV Nao Tem um Problema de Bits...",
 *    section "O Que o Erro de Quantizacao E Realmente Feito" (zero point = the
 *    group minimum, step = group range / (2^B - 1), round to the nearest step,
 *    error at most half a step).
 *  - Axes: same page, sections "Chaves: Os Valores Extremos Vivem em Canais
 *    Fixos" (keys grouped per channel, along tokens) and "Valores: Onde a
 *    Intuicao Quebra" (values grouped per token, along channels); section
 *    "O Imposto dos Sistemas..." (per-channel groups are only formed once G
 *    tokens exist; newer tokens stay in full precision).
 *  - "Whole vector" groups: "Asymetrie kvantizace KV cache", section "Vychozi
 *    zjisteni na GPT-2" (scaling over the whole vector vs per head).
 *
 * Readings where the pages are silent, taken as follows:
 *  - ties round half to even (rintf in the default rounding mode);
 *  - metadata stored as fp16: zero rounded toward -inf, step rounded toward +inf,
 *    step recomputed from the stored zero, so every input lies in
 *    [z, z + (2^B-1) s] and the half-step bound survives storage; fp32 metadata
 *    is the literal formula;
 *  - a zero point or step of -0 is canonicalised to +0;
 *  - step == 0 (all values equal the stored zero) gives code 0;
 *  - symmetric range is +-(2^(B-1)-1) with scale = absmax / (2^(B-1)-1); the
 *    stored code is q + 2^(B-1);
 *  - the fp16 recent-token tail holds the input rounded to nearest fp16, and a
 *    per-channel group is quantized from those fp16 values (so a prefill and a
 *    token-by-token append of the same tokens build the same cache);
 *  - full-precision recent window of R tokens for both tensors (same page,
 *    section "O Imposto dos Sistemas e Por Que Nao E um Detalhe": the most
 *    recent tokens, up to 128, stay in full precision and are quantized in
 *    groups once enough have accumulated): with R > 0 a per-channel group is
 *    sealed once all its tokens are older than the newest R, and a per-token
 *    tensor quantizes a 16-token block once all of it is older than the newest
 *    R (tokens in between stay fp16); tokens quantized after a stay in the
 *    window are quantized from their fp16 values.  R = 0 is the cache without
 *    a window (per-token tensors quantize every token on arrival).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KVQO_PER_TOKEN 0
#define KVQO_PER_CHANNEL 1
#define KVQO_ROUND_NEAREST 0
#define KVQO_ROUND_DOWN 1 /* toward -infinity */
#define KVQO_ROUND_UP 2   /* toward +infinity */

/* ---------------------------------------------------------------- fp16 ---- */

/* Exact binary16 -> binary32 (IEEE 754-2008 binary16: 1 sign, 5 exponent
 * bits with bias 15, 10 fraction bits; subnormals have exponent -14). */
float kvqo_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0x1f) {
    v = f ? NAN : INFINITY;
  } else if (e == 0) {
    v = ldexp((double)f, -24);
  } else {
    v = ldexp((double)(f + 1024), e - 25);
  }
  return (float)(sign ? -v : v);
}

/* binary32 -> binary16 under one of three rounding rules, from the definition:
 * the result is the representable binary16 value selected by the rule among
 * the two that bracket x (overflow handled as IEEE 754 specifies). */
uint16_t kvqo_f32_to_f16(float xf, int mode) {
  double x = (double)xf;
  if (isnan(x)) return 0x7e00;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isinf(x)) return sign | 0x7c00;
  if (a == 0.0) return sign;
  /* quantum (spacing of binary16 values) at the magnitude of a */
  int e2;
  frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1) */
  int exp_unb = e2 - 1;   /* a in [2^exp_unb, 2^(exp_unb+1)) */
  if (exp_unb < -14) exp_unb = -14;
  double quantum = ldexp(1.0, exp_unb - 10);
  double r = a / quantum; /* exact: division by a power of two */
  double n = floor(r);
  double frac = r - n;    /* exact */
  int up; /* round magnitude up? */
  if (mode == KVQO_ROUND_NEAREST) {
    up = frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0);
  } else if (mode == KVQO_ROUND_DOWN) {
    up = sign ? (frac > 0.0) : 0;
  } else {
    up = sign ? 0 : (frac > 0.0);
  }
  double mag = (n + (up ? 1.0 : 0.0)) * quantum; /* exact */
  if (mag > 65504.0) {
    /* overflow: nearest -> inf (a value here is >= 65520 after rounding);
       directed rules saturate toward the finite side */
    int to_inf;
    if (mode == KVQO_ROUND_NEAREST) to_inf = 1;
    else if (mode == KVQO_ROUND_DOWN) to_inf = sign ? 1 : 0;
    else to_inf = sign ? 0 : 1;
    return to_inf ? (sign | 0x7c00) : (sign | 0x7bff);
  }
  /* encode the exactly representable magnitude */
  if (mag < ldexp(1.0, -14)) {
    int f = (int)(mag / ldexp(1.0, -24));
    return sign | (uint16_t)f;
  }
  int e2m;
  double m = frexp(mag, &e2m); /* mag = m * 2^e2m */
  int E = e2m - 1 + 15;
  int f = (int)(ldexp(m, 11) - 1024.0);
  return sign | (uint16_t)(E << 10) | (uint16_t)f;
}

void kvqo_f32_to_f16_array(const float* x, long n, int mode, uint16_t* out) {
  for (long i = 0; i < n; ++i) out[i] = kvqo_f32_to_f16(x[i], mode);
}

void kvqo_f16_to_f32_array(const uint16_t* h, long n, float* out) {
  for (long i = 0; i < n; ++i) out[i] = kvqo_f16_to_f32(h[i]);
}

/* ------------------------------------------------------- one group -------- */

/* Quantize one group of n values x[i*stride].  Writes the stored metadata
 * (z, s) as floats (exact values of the stored fp16 or fp32 numbers; z = 0 for
 * the symmetric form) and one code per element into codes[i*cstride]. */
void kvqo_quant_group(const float* x, long n, long stride, int bits, int sym, int meta_f32,
                      uint8_t* codes, long cstride, float* z_out, float* s_out) {
  const int levels = (1 << bits) - 1;
  if (!sym) {
    float mn = x[0], mx = x[0];
    for (long i = 1; i < n; ++i) {
      float v = x[i * stride];
      if (v < mn) mn = v;
      if (v > mx) mx = v;
    }
    float z, s;
    if (meta_f32) {
      z = mn + 0.0f;                      /* -0 -> +0 */
      s = (mx - z) / (float)levels + 0.0f;
    } else {
      z = kvqo_f16_to_f32(kvqo_f32_to_f16(mn + 0.0f, KVQO_ROUND_DOWN));
      float s32 = (mx - z) / (float)levels + 0.0f; /* -0 -> +0 */
      s = kvqo_f16_to_f32(kvqo_f32_to_f16(s32, KVQO_ROUND_UP));
    }
    for (long i = 0; i < n; ++i) {
      int q = 0;
      if (s != 0.0f) {
        float d = x[i * stride] - z;
        float t = rintf(d / s);
        if (t < 0.0f) t = 0.0f;
        if (t > (float)levels) t = (float)levels;
        q = (int)t;
      }
      codes[i * cstride] = (uint8_t)q;
    }
    *z_out = z;
    *s_out = s;
  } else {
    const int qmax = (1 << (bits - 1)) - 1;
    const int off = 1 << (bits - 1);
    float a = 0.0f;
    for (long i = 0; i < n; ++i) {
      float v = fabsf(x[i * stride]);
      if (v > a) a = v;
    }
    float s = a / (float)qmax;
    if (!meta_f32) s = kvqo_f16_to_f32(kvqo_f32_to_f16(s, KVQO_ROUND_UP));
    for (long i = 0; i < n; ++i) {
      int q = 0;
      if (s != 0.0f) {
        float t = rintf(x[i * stride] / s);
        if (t < (float)-qmax) t = (float)-qmax;
        if (t > (float)qmax) t = (float)qmax;
        q = (int)t;
      }
      codes[i * cstride] = (uint8_t)(q + off);
    }
    *z_out = 0.0f;
    *s_out = s;
  }
}

/* Reconstruction of one code: x_hat = q*s + z (asymmetric) or
 * (u - 2^(B-1))*s (symmetric), in double: exact for fp16 metadata. */
double kvqo_dequant_one(int code, float z, float s, int bits, int sym) {
  if (sym) return (double)(code - (1 << (bits - 1))) * (double)s;
  return (double)code * (double)s + (double)z;
}

/* ------------------------------------------------ layer-level tensors ----- */

/* Number of tokens of a sequence of length n whose codes are sealed, with a
 * full-precision window of the newest `window` tokens (0: none). */
long kvqo_sealed(long n, int axis, int group, int window) {
  long old = n - window > 0 ? n - window : 0;
  if (axis == KVQO_PER_CHANNEL) return (old / group) * group;
  return window ? (old / 16) * 16 : n;
}

/* fp16 rows per (sequence, head) that the unsealed tokens can occupy. */
long kvqo_tail_rows(int axis, int group, int window) {
  if (axis == KVQO_PER_CHANNEL) return (long)group + window;
  return window ? (long)window + 16 : 0;
}

/* Number of metadata groups in the canonical layout of one layer. */
long kvqo_meta_groups(int batch, int heads, int dim, int tcap, int axis, int group) {
  if (axis == KVQO_PER_CHANNEL) return (long)batch * heads * (tcap / group) * dim;
  if (group == heads * dim) return (long)batch * tcap;
  return (long)batch * heads * tcap * (dim / group);
}

/* Quantize one tensor (K or V) of one layer.
 *   x     : [batch][tstride][heads][dim] input values (exact fp32 copies of the
 *           source numbers); sequence b has lens[b] valid tokens.
 *   codes : [batch][heads][tcap][dim] canonical codes (tokens >= sealed are 0)
 *   meta  : [groups][2] (z, s), group order as kvqo_meta_groups() describes:
 *           per channel : ((b*heads + h)*(tcap/G) + t/G)*dim + c
 *           per token   : ((b*heads + h)*tcap + t)*(dim/G) + c/G
 *           whole vector: b*tcap + t
 *   tail  : [batch][heads][tail_rows][dim] fp16 bits of the unsealed tokens
 *           (slot = t - sealed; tail_rows = kvqo_tail_rows()), or NULL when
 *           there are none.
 * Returns 0, or -1 on an unsupported shape. */
int kvqo_quantize_tensor(const float* x, int batch, int tstride, int heads, int dim, const int* lens, int tcap,
                         int bits, int group, int axis, int sym, int meta_f32, int window, uint8_t* codes, float* meta,
                         uint16_t* tail) {
  if (bits < 2 || bits > 8 || window < 0 || window % 16) return -1;
  const long rows = kvqo_tail_rows(axis, group, window);
  const long xs_t = (long)heads * dim;      /* stride between tokens */
  const long xs_b = (long)tstride * xs_t;   /* stride between sequences */
  memset(codes, 0, sizeof(uint8_t) * (size_t)batch * heads * tcap * dim);
  memset(meta, 0, sizeof(float) * 2 * (size_t)kvqo_meta_groups(batch, heads, dim, tcap, axis, group));
  for (int b = 0; b < batch; ++b) {
    long n = lens[b];
    if (n > tcap || n > tstride) return -1;
    const float* xb = x + b * xs_b;
    const long ns = kvqo_sealed(n, axis, group, window);
    /* unsealed tokens: the input rounded to nearest fp16 */
    if (ns < n) {
      if (!tail) return -1;
      for (int h = 0; h < heads; ++h)
        for (long t = ns; t < n; ++t)
          for (int c = 0; c < dim; ++c)
            tail[(((long)b * heads + h) * rows + (t - ns)) * dim + c] =
                kvqo_f32_to_f16(xb[t * xs_t + (long)h * dim + c], KVQO_ROUND_NEAREST);
    }
    if (axis == KVQO_PER_CHANNEL) {
      long ng = ns / group;
      float* col = (float*)malloc(sizeof(float) * (size_t)group);
      for (int h = 0; h < heads; ++h) {
        for (long g = 0; g < ng; ++g) {
          for (int c = 0; c < dim; ++c) {
            /* a per-channel group is formed from its tokens as held in the fp16
               staging tail: the values are rounded to nearest fp16 first */
            for (long t = 0; t < group; ++t)
              col[t] = kvqo_f16_to_f32(
                  kvqo_f32_to_f16(xb[(g * group + t) * xs_t + (long)h * dim + c], KVQO_ROUND_NEAREST));
            uint8_t* dst = codes + (((long)b * heads + h) * tcap + g * group) * dim + c;
            long mi = (((long)b * heads + h) * (tcap / group) + g) * dim + c;
            kvqo_quant_group(col, group, 1, bits, sym, meta_f32, dst, dim, &meta[2 * mi], &meta[2 * mi + 1]);
          }
        }
      }
      free(col);
    } else if (group == heads * dim) {
      float* vec = (float*)malloc(sizeof(float) * (size_t)heads * dim);
      for (long t = 0; t < ns; ++t) {
        /* the whole token vector (all heads) is one group; codes land per head.
           After a stay in the window the token is quantized from its fp16 values. */
        for (long i = 0; i < (long)heads * dim; ++i) {
          float v = xb[t * xs_t + i];
          vec[i] = window ? kvqo_f16_to_f32(kvqo_f32_to_f16(v, KVQO_ROUND_NEAREST)) : v;
        }
        uint8_t* tmp = (uint8_t*)malloc((size_t)heads * dim);
        long mi = (long)b * tcap + t;
        kvqo_quant_group(vec, (long)heads * dim, 1, bits, sym, meta_f32, tmp, 1, &meta[2 * mi], &meta[2 * mi + 1]);
        for (int h = 0; h < heads; ++h)
          for (int c = 0; c < dim; ++c)
            codes[(((long)b * heads + h) * tcap + t) * dim + c] = tmp[(long)h * dim + c];
        free(tmp);
      }
      free(vec);
    } else {
      if (dim % group) return -1;
      int gpd = dim / group;
      float* vec = (float*)malloc(sizeof(float) * (size_t)group);
      for (long t = 0; t < ns; ++t) {
        for (int h = 0; h < heads; ++h) {
          for (int j = 0; j < gpd; ++j) {
            const float* src = xb + t * xs_t + (long)h * dim + (long)j * group;
            for (int i = 0; i < group; ++i)
              vec[i] = window ? kvqo_f16_to_f32(kvqo_f32_to_f16(src[i], KVQO_ROUND_NEAREST)) : src[i];
            uint8_t* dst = codes + (((long)b * heads + h) * tcap + t) * dim + (long)j * group;
            long mi = (((long)b * heads + h) * tcap + t) * gpd + j;
            kvqo_quant_group(vec, group, 1, bits, sym, meta_f32, dst, 1, &meta[2 * mi], &meta[2 * mi + 1]);
          }
        }
      }
      free(vec);
    }
  }
  return 0;
}

/* Reconstruct one tensor of one layer into xhat [batch][heads][tcap][dim]
 * (double): sealed tokens from codes and metadata, unsealed tokens from the
 * fp16 tail, tokens >= lens[b] set to 0. */
int kvqo_dequant_tensor(const uint8_t* codes, const float* meta, const uint16_t* tail, int batch, int heads,
                        int dim, const int* lens, int tcap, int bits, int group, int axis, int sym, int window,
                        double* xhat) {
  memset(xhat, 0, sizeof(double) * (size_t)batch * heads * tcap * dim);
  const long rows = kvqo_tail_rows(axis, group, window);
  for (int b = 0; b < batch; ++b) {
    long n = lens[b];
    long ns = kvqo_sealed(n, axis, group, window);
    for (int h = 0; h < heads; ++h) {
      for (long t = 0; t < n; ++t) {
        for (int c = 0; c < dim; ++c) {
          long o = (((long)b * heads + h) * tcap + t) * dim + c;
          if (t >= ns) {
            if (!tail) return -1;
            xhat[o] = (double)kvqo_f16_to_f32(tail[(((long)b * heads + h) * rows + (t - ns)) * dim + c]);
            continue;
          }
          long mi;
          if (axis == KVQO_PER_CHANNEL) mi = (((long)b * heads + h) * (tcap / group) + t / group) * dim + c;
          else if (group == heads * dim) mi = (long)b * tcap + t;
          else mi = (((long)b * heads + h) * tcap + t) * (dim / group) + c / group;
          xhat[o] = kvqo_dequant_one(codes[o], meta[2 * mi], meta[2 * mi + 1], bits, sym);
        }
      }
    }
  }
  return 0;
}

/* Single-token decode attention, fp64 throughout, plain definition:
 *   for each sequence b and query head hq (KV head h = hq / (q_heads/kv_heads)):
 *   s_t = scale * sum_c q[c] * khat[t][c]  over t < lens[b],
 *   p_t = exp(s_t - max_t s_t),  out[c] = sum_t p_t vhat[t][c] / sum_t p_t.
 * An empty sequence gives zeros.  q: [batch][q_heads][dim] (fp32 values);
 * khat, vhat: [batch][kv_heads][tcap][dim]; out: [batch][q_heads][dim]. */
int kvqo_attention(const double* khat, const double* vhat, const float* q, const int* lens, int batch,
                   int q_heads, int kv_heads, int dim, int tcap, float scale, double* out) {
  if (kv_heads <= 0 || q_heads % kv_heads) return -1;
  int rep = q_heads / kv_heads;
  double* s = (double*)malloc(sizeof(double) * (size_t)(tcap > 0 ? tcap : 1));
  for (int b = 0; b < batch; ++b) {
    long n = lens[b];
    for (int hq = 0; hq < q_heads; ++hq) {
      int h = hq / rep;
      const float* qv = q + ((long)b * q_heads + hq) * dim;
      double* o = out + ((long)b * q_heads + hq) * dim;
      for (int c = 0; c < dim; ++c) o[c] = 0.0;
      if (n == 0) continue;
      const double* kb = khat + ((long)b * kv_heads + h) * tcap * dim;
      const double* vb = vhat + ((long)b * kv_heads + h) * tcap * dim;
      double m = -INFINITY;
      for (long t = 0; t < n; ++t) {
        double acc = 0.0;
        for (int c = 0; c < dim; ++c) acc += (double)qv[c] * kb[t * dim + c];
        s[t] = (double)scale * acc;
        if (s[t] > m) m = s[t];
      }
      double l = 0.0;
      for (long t = 0; t < n; ++t) {
        double p = exp(s[t] - m);
        l += p;
        for (int c = 0; c < dim; ++c) o[c] += p * vb[t * dim + c];
      }
      for (int c = 0; c < dim; ++c) o[c] /= l;
    }
  }
  free(s);
  return 0;
}

/* ------------------------------------------------------------- RoPE ------ */

/* Rotary position embedding applied to dequantized keys ("O Seu Cache KV Nao
 * Tem um Problema de Bits. Tem um Problema de Geometria", section "Embebedos
 * Rotatorios Complicam as Chaves": RoPE turns pairs of channels by an angle
 * set by the token's position, which spreads a fixed outlier channel into its
 * neighbour; the remedy there is to quantize keys before the rotation and to
 * rotate after dequantization; section "O Que Fazer Com Isso", item 2).
 * Readings where the page is silent: the pairs are adjacent channels
 * (2i, 2i+1); pair i of the token at position t turns by t * theta_i with
 * theta_i = base^(-2i/dim); a token's position is its index in the sequence.
 *   (x0, x1) -> (x0 cos a - x1 sin a, x0 sin a + x1 cos a),  a = t * theta_i.
 * In place on x [batch][heads][tcap][dim] (fp64), rows t < lens[b]. */
void kvqo_rope(double* x, int batch, int heads, int dim, int tcap, const int* lens, double base) {
  for (int b = 0; b < batch; ++b) {
    for (int h = 0; h < heads; ++h) {
      for (long t = 0; t < lens[b]; ++t) {
        double* row = x + (((long)b * heads + h) * tcap + t) * dim;
        for (int i = 0; i < dim / 2; ++i) {
          double theta = pow(base, -2.0 * (double)i / (double)dim);
          double a = (double)t * theta;
          double c = cos(a), sn = sin(a);
          double x0 = row[2 * i], x1 = row[2 * i + 1];
          row[2 * i] = x0 * c - x1 * sn;
          row[2 * i + 1] = x0 * sn + x1 * c;
        }
      }
    }
  }
}

/* ------------------------------------------------------------ sizes ------ */

/* Bytes of one layer-tensor holding lens[b] tokens, split into the terms of
 * the memory model: packed codes (bits per sealed element), metadata (per
 * group: 4 bytes asym / 2 bytes sym with fp16 metadata, twice that with fp32),
 * fp16 tail (2 bytes per unsealed element).  out[0..2] = packed, meta, tail.
 * Packed bytes are counted exactly: elements*bits/8 (rounded up per tensor). */
void kvqo_tensor_bytes(int batch, int heads, int dim, const int* lens, int bits, int group, int axis, int sym,
                       int meta_f32, int window, double* out) {
  double packed_bits = 0.0, meta = 0.0, tail = 0.0;
  double per_group = (sym ? 2.0 : 4.0) * (meta_f32 ? 2.0 : 1.0);
  for (int b = 0; b < batch; ++b) {
    long n = lens[b];
    long ns = kvqo_sealed(n, axis, group, window);
    packed_bits += (double)ns * heads * dim * bits;
    tail += (double)(n - ns) * heads * dim * 2.0;
    if (axis == KVQO_PER_CHANNEL) meta += (double)(ns / group) * heads * dim * per_group;
    else if (group == heads * dim) meta += (double)ns * per_group;
    else meta += (double)ns * heads * (dim / group) * per_group;
  }
  out[0] = ceil(packed_bits / 8.0);
  out[1] = meta;
  out[2] = tail;
}

/* Element count of the uncompressed cache: 2 * layers * tokens * kv_heads * dim. */
double kvqo_cache_elements(int layers, double tokens, int kv_heads, int dim) {
  return 2.0 * layers * tokens * kv_heads * dim;
}
