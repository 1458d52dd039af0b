/*
 * kvq.h — C ABI of libkvq: group-wise integer KV-cache quantization and
 * single-token decode attention over the packed cache, on one NVIDIA GB300
 * (sm_103a).  Plain C types only; every device pointer is a CUDA device
 * address owned by the caller; `stream` is a cudaStream_t passed as void*.
 *
 * Method (source pages, by title and section):
 *  - Asymmetric quantizer: "O Seu Cache KV Nao Tem um Problema de Bits. Tem um
 *    Problema de Geometria", section "O Que o Erro de Quantizacao E Realmente
 *    Feito": zero point = group minimum, step = range/(2^B-1), every element
 *    rounded to the nearest step, error at most half a step.
 *  - Symmetric quantizer: "Kuantisasi KV Cache untuk Mengurangi Memory
 *    Inferensi Long Context", section "Scale menentukan sistem koordinat
 *    kuantisasi": q = clamp(round(x/scale), q_min, q_max), x_hat = q*scale.
 *  - Axes: first page above, sections "Chaves: Os Valores Extremos Vivem em
 *    Canais Fixos" (keys grouped per channel along tokens) and "Valores: Onde
 *    a Intuicao Quebra" (values grouped per token along channels).
 *  - Unsealed per-channel groups stay in full precision: same page, section
 *    "O Imposto dos Sistemas e Por Que Nao E um Detalhe".
 *  - Memory model: second page above, sections "Ukuran cache bertambah
 *    mengikuti token, layer, dan KV head" and "Pengecualian recent-token
 *    mengubah perhitungan memory".
 *  - Fused unpack + scale inside attention: same page, section "Kuantisasi
 *    dapat memindahkan pekerjaan ke decode path".
 *
 * Numerical contract (readings where the pages are silent):
 *  - min/max/absmax are exact; zero point z = min rounded toward -inf to fp16
 *    (-0 stored as +0); step s = ((max - z) / (2^B-1)) in IEEE fp32 (round to
 *    nearest), then rounded toward +inf to fp16; with KVQ_F32 metadata z = min
 *    and s = (max - min)/(2^B-1) in fp32.
 *  - code = s == 0 ? 0 : clamp(rint((x - z) / s), 0, 2^B-1) with IEEE fp32
 *    subtraction and division, ties to even.
 *  - symmetric: s = absmax / (2^(B-1)-1) (fp32, then rounded up to fp16),
 *    q = clamp(rint(x/s), -(2^(B-1)-1), 2^(B-1)-1), stored code q + 2^(B-1).
 *  - inputs must be finite; with fp16 metadata |x| <= 65504.
 *  - decode attention: s_t = scale * q . k_hat_t, softmax over all cached
 *    tokens of the sequence (fp32 accumulation), out = sum_t p_t v_hat_t.
 *
 * Errors: every entry point validates on the host before launching anything
 * and returns a kvq_status; on error nothing is launched and no state
 * changes.  Asynchronous CUDA errors surface as KVQ_ERR_CUDA from the call
 * that observes them.  Nothing throws across the ABI.  A cache handle is not
 * thread-safe, and calls on one handle must be ordered on one stream: they
 * share the handle's workspace.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,    /* NULL pointer, out-of-range index, bad shape */
  KVQ_ERR_UNSUPPORTED = 2,    /* legal per the method, not built (e.g. head_dim 96) */
  KVQ_ERR_CAPACITY = 3,       /* a sequence would exceed max_tokens */
  KVQ_ERR_BUFFER_TOO_SMALL = 4, /* device buffer smaller than kvq_bytes.alloc */
  KVQ_ERR_CUDA = 5,           /* a CUDA runtime error (launch or asynchronous) */
  KVQ_ERR_DEVICE_TIMEOUT = 6  /* a device-side wait gave up (reserved: no kernel waits today) */
} kvq_status;

typedef enum { KVQ_PER_TOKEN = 0, KVQ_PER_CHANNEL = 1 } kvq_axis; /* group along channels / along tokens */
typedef enum { KVQ_ASYM = 0, KVQ_SYM = 1 } kvq_mode;
typedef enum { KVQ_F16 = 0, KVQ_F32 = 1 } kvq_dtype;

/* group value meaning "all kv_heads*head_dim channels of one token" (per-token axis only) */
#define KVQ_WHOLE_VECTOR (-1)

typedef struct {
  int bits;   /* 2..8 */
  int group;  /* per-token axis: channels per group, one of 32, 64, 128, 256 dividing head_dim,
                 or KVQ_WHOLE_VECTOR (kv_heads*head_dim <= 2560); per-channel axis: tokens
                 per group, one of 16, 32, 64, 128 */
  int axis;   /* kvq_axis */
  int mode;   /* kvq_mode */
} kvq_tensor_cfg;

typedef struct {
  int layers;      /* >= 1 */
  int batch;       /* sequences, 1..1024 */
  int q_heads;     /* query heads; q_heads / kv_heads in {1, 2, 4, 8} */
  int kv_heads;    /* >= 1 */
  int head_dim;    /* 64, 128 or 256 */
  int max_tokens;  /* capacity per sequence, >= 1 */
  kvq_tensor_cfg k, v;
  int meta_dtype;  /* kvq_dtype of the stored zero point / step: KVQ_F16 (default) or KVQ_F32 */
  int max_splits;  /* split-K partitions per sequence for decode, <= 1024; 0 = default (about
                      4864 / (batch * kv_heads), at least 8, at most one per 64 tokens) */
  int recent_window; /* full-precision window R of the newest tokens of both tensors, a multiple of 16,
                        0..1024; 0 = none ("O Seu Cache KV Nao Tem um Problema de Bits...", section "O
                        Imposto dos Sistemas e Por Que Nao E um Detalhe": the newest tokens, up to 128,
                        stay in full precision and are quantized in groups once enough accumulate).  With
                        R > 0 a per-channel group is sealed once all its tokens are older than the newest
                        R, a per-token tensor quantizes a 16-token block once all of it is older than the
                        newest R (from the tokens' fp16 values); the newer tokens are held in fp16.  With
                        R = 0 per-token tensors quantize every token on arrival. */
  float rope_theta; /* 0 = keys are cached and attended as given.  > 0: pre-RoPE key quantization ("O Seu
                       Cache KV Nao Tem um Problema de Bits...", sections "Embebedos Rotatorios Complicam
                       as Chaves" and "O Que Fazer Com Isso", item 2): the caller passes keys BEFORE the
                       rotary position embedding, they are quantized as given, and decode attention turns
                       every dequantized key of token t (its index in the sequence) by the embedding:
                       channel pair (2i, 2i+1) by the angle t * rope_theta^(-2i/head_dim).  The query is
                       passed as the model rotates it (post-RoPE).  Finite, 0 or > 1; positions below
                       2^24. */
} kvq_config;

/* Byte accounting.  The first four terms follow the memory model total =
 * high-precision recent part + packed codes + scales/metadata + workspace,
 * evaluated for the given lengths over all layers; `alloc` is the size of the
 * device buffer kvq_cache_create needs (capacity layout, alignment padding,
 * lengths and control words included). */
typedef struct {
  double tail;       /* fp16 elements of unsealed per-channel groups, 2 bytes each */
  double packed;     /* bits/8 per sealed element */
  double metadata;   /* per group: 4 bytes (asym) or 2 (sym) with fp16 metadata, twice with fp32 */
  double workspace;  /* decode split-K partials at max_splits */
  double total;      /* tail + packed + metadata + workspace */
  double elements;   /* 2 * layers * tokens * kv_heads * head_dim (uncompressed element count) */
  size_t alloc;      /* bytes for kvq_cache_create */
} kvq_bytes;

typedef struct kvq_cache* kvq_cache_t;

/* Size accounting for `cfg` holding lens_host[b] tokens in every layer
 * (lens_host NULL: max_tokens for every sequence).  Host only, no CUDA call.
 * Errors: KVQ_ERR_INVALID_ARG / KVQ_ERR_UNSUPPORTED for a bad config,
 * KVQ_ERR_CAPACITY if a length exceeds max_tokens. */
kvq_status kvq_cache_bytes(const kvq_config* cfg, const int32_t* lens_host, kvq_bytes* out);

/* Create a cache inside the caller's device buffer (size >= kvq_bytes.alloc,
 * 256-byte aligned).  The library never allocates device memory; it zero-fills
 * `device_buf` on `stream` and carves it into packed codes, metadata, fp16
 * tails, lengths and decode workspace.  All sequences start empty.  The buffer
 * must outlive the handle.  Must be called with the buffer's device current. */
kvq_status kvq_cache_create(const kvq_config* cfg, void* device_buf, size_t buf_bytes, void* stream,
                            kvq_cache_t* out);

/* Release the host-side handle (the device buffer stays the caller's). */
kvq_status kvq_cache_destroy(kvq_cache_t cache);

/* Replace layer `layer`'s contents with a prefill of lens_host[b] tokens per
 * sequence.  k, v: device [batch][t_stride][kv_heads][head_dim] of in_dtype
 * (KVQ_F16 or KVQ_F32), token-major; lens_host[b] <= min(t_stride, max_tokens).
 * Keys and values are quantized per their kvq_tensor_cfg; for a per-channel
 * tensor, floor(len/G)*G tokens are sealed and the rest go to its fp16 tail
 * (rounded to nearest).  Asynchronous on `stream`. */
kvq_status kvq_prefill_quantize(kvq_cache_t cache, int layer, const void* k, const void* v, int in_dtype,
                                const int32_t* lens_host, int64_t t_stride, void* stream);

/* Append one token to every sequence of layer `layer`.  k_new, v_new: device
 * [batch][kv_heads][head_dim] of in_dtype.  Per-token tensors quantize the new
 * token at once; per-channel tensors store it in the fp16 tail and seal the
 * group (quantize its G tokens) when the tail reaches G.  All-or-nothing:
 * KVQ_ERR_CAPACITY (nothing launched) if any sequence is full. */
kvq_status kvq_append(kvq_cache_t cache, int layer, const void* k_new, const void* v_new, int in_dtype,
                      void* stream);

/* Decode attention of one query token per sequence over everything cached in
 * layer `layer` (including tokens just appended).  q: device
 * [batch][q_heads][head_dim] of q_dtype; out: device [batch][q_heads][head_dim]
 * fp32.  Query head hq reads KV head hq / (q_heads/kv_heads).  softmax_scale
 * <= 0 means 1/sqrt(head_dim).  An empty sequence yields zeros.  Split-K over
 * tokens (tensor-core dequant-in-register kernel) then a log-sum-exp combine,
 * both on `stream`; partials live in the cache's workspace. */
kvq_status kvq_decode_attn(kvq_cache_t cache, int layer, const void* q, int q_dtype, float softmax_scale,
                           float* out, void* stream);

/* kvq_append followed by kvq_decode_attn on the same layer, in one launch:
 * same arguments as the two calls (k_new / v_new: device [batch][kv_heads]
 * [head_dim] of in_dtype; q / out as for kvq_decode_attn), same resulting
 * cache contents, lengths and output up to fp32 summation order.  This is one
 * decode step of a layer as the pages describe it: the new token's key and
 * value enter the cache (section "O Imposto dos Sistemas e Por Que Nao E um
 * Detalhe" of "O Seu Cache KV Nao Tem um Problema de Bits. Tem um Problema de
 * Geometria": per-channel groups keep new tokens in fp16 until G exist), then
 * the query attends over every cached token.  Inside the launch the warp
 * whose token range holds the new token writes it (and seals a per-channel
 * group that just filled) before it reads its tiles; nothing else waits.
 * Formats without a compile-time specialisation, layouts with a
 * full-precision window or whole-vector groups, and k_new / v_new not 8-byte
 * aligned run the two kernels back to back instead (same results);
 * kvq_last_launches tells which (1 or 2).  All-or-nothing:
 * KVQ_ERR_CAPACITY (nothing launched) if any sequence is full. */
kvq_status kvq_append_decode_attn(kvq_cache_t cache, int layer, const void* k_new, const void* v_new, int in_dtype,
                                  const void* q, int q_dtype, float softmax_scale, float* out, void* stream);

/* kvq_decode_attn without scratch memory from the caller: identical inputs,
 * output and numerics, but the split-K partials and combine tickets live in a
 * 16 MiB array compiled into libkvq (static device memory, held by every GPU
 * that loads the library until the process exits).  For callers that cannot
 * allocate or reserve device memory beyond what they already planned: e.g. a
 * runtime whose device memory is laid out once by another component, or a
 * plugin that must not call cudaMalloc.  Allocates nothing.  The source pages
 * have no counterpart of this call; it is a deployment convenience.
 *  - Needs batch * q_heads * (max_splits + ceil(max_splits/16)) * (head_dim + 4)
 *    * 4 bytes (rounded up to 256) + batch * kv_heads * (1 + ceil(max_splits/16))
 *    * 4 bytes <= 16 MiB, else KVQ_ERR_BUFFER_TOO_SMALL
 *    (nothing launched; kvq_last_error says how much was needed).
 *  - The first call on a device looks up the array's device address with that
 *    device current (cudaGetSymbolAddress); make that first call before any
 *    stream capture.
 *  - Every call shares the one array and finds the last call's contents in it.
 *    The combine tickets are cleared on `stream` at each call (one memset
 *    before the launch): a completed call leaves them at zero, but a call whose
 *    launch failed or was aborted may not.  Calls that overlap on the GPU
 *    (different streams, handles or threads) race with each other.
 *  - Argument checks are those of kvq_decode_attn (KVQ_ERR_INVALID_ARG for a bad
 *    layer, a null pointer, an unknown dtype or a non-finite softmax_scale). */
kvq_status kvq_decode_attn_static(kvq_cache_t cache, int layer, const void* q, int q_dtype, float softmax_scale,
                                  float* out, void* stream);

/* Canonical copy of layer `layer` for inspection and tests (device pointers,
 * any may be NULL to skip):
 *   codes_k/v : uint8  [batch][kv_heads][tcap][head_dim], one code per element
 *               (0 beyond the sealed tokens);
 *   meta_k/v  : float  [groups][2] = (zero, step) as stored (zero = 0 when
 *               symmetric); group order: per channel ((b*H+h)*(tcap/G)+t/G)*D+c,
 *               per token ((b*H+h)*tcap+t)*(D/G)+c/G, whole vector b*tcap+t;
 *   tail_k/v  : uint16 [batch][kv_heads][rows][head_dim] fp16 bits of the
 *               tokens held in fp16 (row t - sealed); rows = G + recent_window
 *               for a per-channel tensor, recent_window + 16 for a per-token
 *               tensor with a window; null / unused when a tensor has none;
 *   lens      : int32  [batch].
 * tcap is kvq_cache_tcap(). */
kvq_status kvq_export(kvq_cache_t cache, int layer, uint8_t* codes_k, uint8_t* codes_v, float* meta_k,
                      float* meta_v, uint16_t* tail_k, uint16_t* tail_v, int32_t* lens, void* stream);

/* Token capacity of the canonical export layout (max_tokens rounded up to the tile / group size). */
int kvq_cache_tcap(kvq_cache_t cache);

/* Host mirror of the lengths of layer `layer` (lens_host: int32[batch]). */
kvq_status kvq_get_lens(kvq_cache_t cache, int layer, int32_t* lens_host);

/* Materialised baseline, step 1: dequantize layer `layer` into fp16 rows
 * k_out, v_out [batch][kv_heads][tcap][head_dim] (tcap = kvq_cache_tcap(); device, 16-byte aligned; caller-owned;
 * token t of sequence b at row t; rows >= the sequence's length are not
 * written): x_hat = z + code * s as one fp32 fma (asymmetric), (code -
 * 2^(B-1)) * s (symmetric), the stored fp16 value for tail tokens, rounded to
 * nearest fp16.  This is the design that dequantizes a cached block into a
 * temporary floating-point tensor before attention ("Kuantisasi KV Cache untuk
 * Mengurangi Memory Inferensi Long Context", section "Kuantisasi dapat
 * memindahkan pekerjaan ke decode path"); it exists to measure the fused
 * kvq_decode_attn against.  Asynchronous on `stream`; KVQ_ERR_INVALID_ARG for
 * a bad layer or null output. */
kvq_status kvq_dequantize(kvq_cache_t cache, int layer, void* k_out, void* v_out, void* stream);

/* Materialised baseline, step 2: decode attention (same definition, query
 * layout, scale and output as kvq_decode_attn) over fp16 rows k16, v16 in the
 * kvq_dequantize layout (16-byte aligned), for the lengths of `layer` in `cache`.  Uses the same
 * split-K kernel with every token read as fp16 (no packed codes, no metadata)
 * and the cache's workspace, so it must not overlap a kvq_decode_attn on the
 * same cache. */
kvq_status kvq_decode_attn_materialized(kvq_cache_t cache, int layer, const void* k16, const void* v16,
                                        const void* q, int q_dtype, float softmax_scale, float* out, void* stream);

/* Bytes one kvq_decode_attn call on `layer` must read at minimum with the
 * current lengths: packed codes + metadata + fp16 tail + q (q_dtype bytes per
 * element), the algorithmic traffic of the path.  Host only. */
kvq_status kvq_decode_traffic(kvq_cache_t cache, int layer, int q_dtype, double* bytes);

/* Synchronise `stream` and report whether a kernel on this handle recorded a
 * device-side failure in the handle's error word (KVQ_ERR_DEVICE_TIMEOUT; the
 * word is then cleared; the current kernels contain no device-side wait that
 * could set it) or a CUDA error is pending (KVQ_ERR_CUDA). */
kvq_status kvq_device_status(kvq_cache_t cache, void* stream);

/* Decode split plan hint: when plan_tokens > 0, kvq_decode_attn sizes its
 * split-K launch as if every sequence held max(its length, plan_tokens) tokens
 * (CTAs past a sequence's real length do no work).  A launch planned this way
 * stays valid while the cache grows up to plan_tokens, which is what a CUDA
 * graph that captured kvq_append + kvq_decode_attn (or kvq_append_decode_attn)
 * and is replayed step after step needs.  0 (default) plans for the current
 * lengths. */
kvq_status kvq_set_decode_plan(kvq_cache_t cache, int plan_tokens);

/* Decode kernel choice, three bits.  Bit 0: 0 (default) uses a compile-time
 * specialisation of the decode kernel when the cache's formats match one (fp16
 * metadata, no whole-vector groups, formats of the benchmarked workloads), else
 * the generic kernel; 1 always uses the generic (runtime-format) kernel.
 * Bit 1: 0 (default) merges the split-K partials of a (sequence, kv head)
 * inside one thread-block cluster when there are at most 8 splits (through
 * distributed shared memory), else through the global workspace; 1 always uses
 * the global workspace.  Bit 2: 1 uses one-warp CTAs (each CTA streams one
 * token range; the ranges of a (sequence, kv head) merge through the global
 * workspace) where a compile-time specialisation exists in that shape, 0
 * (default) four-warp CTAs.  Every choice computes the same result (up to fp32
 * summation order); they only affect speed.  which outside 0..7:
 * KVQ_ERR_INVALID_ARG. */
kvq_status kvq_set_decode_kernel(kvq_cache_t cache, int which);

/* 1 if kvq_decode_attn currently runs a compile-time specialisation, else 0. */
int kvq_decode_kernel_specialized(kvq_cache_t cache);

/* Warps per CTA of the kernel kvq_decode_attn (fused == 0) or
 * kvq_append_decode_attn (fused != 0) currently launches: 4 or 1 (see bit 2 of
 * kvq_set_decode_kernel); 0 for a null handle, or for fused != 0 when that call
 * runs the append and decode kernels one after the other. */
int kvq_decode_cta_warps(kvq_cache_t cache, int fused);

/* Replayed graphs advance the device lengths only; this copies them back into
 * the host mirror (synchronises `stream`). */
kvq_status kvq_refresh_lens(kvq_cache_t cache, void* stream);

/* Number of kernel launches the last kvq_decode_attn / kvq_append /
 * kvq_append_decode_attn / kvq_prefill_quantize call on this handle issued. */
int kvq_last_launches(kvq_cache_t cache);

/* Human-readable name of a status code (static string). */
const char* kvq_status_string(kvq_status status);

/* Message of the last CUDA error seen by this handle ("" if none). */
const char* kvq_last_error(kvq_cache_t cache);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
