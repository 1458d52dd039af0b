// kvq_api.cu — the extern "C" boundary of libkvq: host-side validation, the
// device-buffer carve-up, byte accounting and dispatch to the kernels.
//
// Byte accounting follows "Kuantisasi KV Cache untuk Mengurangi Memory
// Inferensi Long Context", sections "Ukuran cache bertambah mengikuti token,
// layer, dan KV head" (elements = 2 * layers * cached_tokens * kv_heads *
// head_dim) and "Pengecualian recent-token mengubah perhitungan memory"
// (total = high-precision recent part + packed codes + scales/metadata +
// temporary workspace).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>

#include "kvq_internal.h"

using namespace kvq;

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool valid_tensor(const kvq_tensor_cfg& t, int D, int H) {
  if (t.bits < 2 || t.bits > 8) return false;
  if (t.mode != KVQ_ASYM && t.mode != KVQ_SYM) return false;
  if (t.axis == KVQ_PER_TOKEN) {
    if (t.group == KVQ_WHOLE_VECTOR) return true;
    if (t.group != 32 && t.group != 64 && t.group != 128 && t.group != 256) return false;
    return D % t.group == 0;
  }
  if (t.axis == KVQ_PER_CHANNEL) return t.group == 16 || t.group == 32 || t.group == 64 || t.group == 128;
  return false;
}

kvq_status validate(const kvq_config* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->layers < 1 || c->batch < 1 || c->kv_heads < 1 || c->q_heads < 1 || c->max_tokens < 1 ||
      c->max_splits < 0 || c->max_splits > kMaxSplits || c->recent_window < 0 || c->recent_window % 16 ||
      c->recent_window > 1024)
    return KVQ_ERR_INVALID_ARG;
  if (c->batch > kMaxBatch) return KVQ_ERR_UNSUPPORTED;
  if (c->q_heads % c->kv_heads) return KVQ_ERR_INVALID_ARG;
  int rep = c->q_heads / c->kv_heads;
  if (rep != 1 && rep != 2 && rep != 4 && rep != 8) return KVQ_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  if (c->meta_dtype != KVQ_F16 && c->meta_dtype != KVQ_F32) return KVQ_ERR_INVALID_ARG;
  const kvq_tensor_cfg* ts[2] = {&c->k, &c->v};
  for (int i = 0; i < 2; ++i) {
    const kvq_tensor_cfg& t = *ts[i];
    if (t.axis != KVQ_PER_TOKEN && t.axis != KVQ_PER_CHANNEL) return KVQ_ERR_INVALID_ARG;
    if (t.mode != KVQ_ASYM && t.mode != KVQ_SYM) return KVQ_ERR_INVALID_ARG;
    if (t.bits < 2 || t.bits > 8) return KVQ_ERR_INVALID_ARG;
    if (t.axis == KVQ_PER_CHANNEL && t.group == KVQ_WHOLE_VECTOR) return KVQ_ERR_INVALID_ARG;
    if (t.group == 0 || (t.group < 0 && t.group != KVQ_WHOLE_VECTOR)) return KVQ_ERR_INVALID_ARG;
    if (!valid_tensor(t, c->head_dim, c->kv_heads)) return KVQ_ERR_UNSUPPORTED;
    // a whole-vector group of one token is quantized in one CTA's shared memory
    if (t.axis == KVQ_PER_TOKEN && t.group == KVQ_WHOLE_VECTOR && (long)c->kv_heads * c->head_dim > 2560)
      return KVQ_ERR_UNSUPPORTED;
  }
  if ((long)c->max_tokens > (1L << 30)) return KVQ_ERR_UNSUPPORTED;
  if (!std::isfinite(c->rope_theta) || c->rope_theta < 0.0f || (c->rope_theta > 0.0f && c->rope_theta <= 1.0f))
    return KVQ_ERR_INVALID_ARG;
  if (c->rope_theta > 0.0f && c->max_tokens > (1 << 24)) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

TensorLayout make_layout(const kvq_tensor_cfg& t, const kvq_config& c) {
  TensorLayout L;
  std::memset(&L, 0, sizeof(L));
  L.bits = t.bits;
  L.axis = t.axis;
  L.sym = t.mode == KVQ_SYM;
  L.whole = t.axis == KVQ_PER_TOKEN && t.group == KVQ_WHOLE_VECTOR;
  L.group = L.whole ? c.kv_heads * c.head_dim : t.group;
  L.meta_f32 = c.meta_dtype == KVQ_F32;
  L.meta_bytes = (L.sym ? 2 : 4) * (L.meta_f32 ? 2 : 1);
  L.gpt = (t.axis == KVQ_PER_TOKEN) ? (L.whole ? 1 : c.head_dim / t.group) : 0;
  L.tile_words = c.head_dim * t.bits / 2;
  L.planes = planes_of(t.bits);
  L.window = c.recent_window;
  L.ring = t.axis == KVQ_PER_CHANNEL ? L.group + L.window : (L.window ? L.window + kTile : 0);
  return L;
}

int tcap_of(const kvq_config& c) {
  int unit = kTile;
  if (c.k.axis == KVQ_PER_CHANNEL) unit = std::max(unit, c.k.group);
  if (c.v.axis == KVQ_PER_CHANNEL) unit = std::max(unit, c.v.group);
  return (c.max_tokens + unit - 1) / unit * unit;
}

// Default split-K capacity per sequence: enough partitions that a batch fills
// several waves of a GB300 (152 SMs x ~8 resident CTAs) even when it holds few
// (sequence, kv head) pairs, never finer than 64 tokens per partition.
int max_chunks_of(const kvq_config& c, int tcap) {
  if (c.max_splits > 0) return c.max_splits;
  const long want = (4L * 152 * 8 + (long)c.batch * c.kv_heads - 1) / ((long)c.batch * c.kv_heads);
  const long cap = std::max(1, (tcap + 63) / 64);
  return (int)std::max(1L, std::min(std::min(std::max(want, 8L), cap), (long)kMaxSplits));
}

// carve the buffer: returns the total size; fills offsets when C != null
size_t carve(const kvq_config& c, kvq_cache* C) {
  TensorLayout K = make_layout(c.k, c), V = make_layout(c.v, c);
  const int tcap = tcap_of(c);
  const long B = c.batch, H = c.kv_heads, D = c.head_dim, L = c.layers;
  size_t off = 0;
  TensorLayout* ls[2] = {&K, &V};
  for (int i = 0; i < 2; ++i) {
    TensorLayout& T = *ls[i];
    T.codes_layer = align256((size_t)B * H * (tcap / kTile) * T.tile_words * 4);
    T.codes_off = off;
    off += T.codes_layer * L;
    long groups;
    if (T.axis == 1) groups = B * H * (tcap / T.group) * D;
    else if (T.whole) groups = B * tcap;
    else groups = B * H * tcap * T.gpt;
    T.meta_layer = align256((size_t)groups * T.meta_bytes);
    T.meta_off = off;
    off += T.meta_layer * L;
    if (T.ring) {
      T.tail_layer = align256((size_t)B * H * T.ring * D * 2);
      T.tail_off = off;
      off += T.tail_layer * L;
    }
  }
  size_t lens_off = off;
  off += align256((size_t)L * B * 4);
  size_t smax_off = off;
  off += align256((size_t)2 * L * B * H * 4);
  size_t hl_off = off;
  off += align256((size_t)L * B * H * 4);
  size_t ar_off = off;
  off += align256((size_t)B * H * 4);
  const int mc = max_chunks_of(c, tcap);
  size_t dt_off = off;
  off += align256(decode_ticket_words(B, H, mc) * 4);
  size_t err_off = off;
  off += 256;
  size_t work_off = off;
  off += align256(decode_work_floats(B, c.q_heads, (int)D, mc) * 4);
  if (C) {
    C->k = K;
    C->v = V;
    C->tcap = tcap;
    C->max_chunks = mc;
    C->d_lens = reinterpret_cast<int32_t*>(C->base + lens_off);
    C->d_smax = reinterpret_cast<uint32_t*>(C->base + smax_off);
    C->d_head_lens = reinterpret_cast<int32_t*>(C->base + hl_off);
    C->d_arrive = reinterpret_cast<uint32_t*>(C->base + ar_off);
    C->d_decode_tickets = reinterpret_cast<uint32_t*>(C->base + dt_off);
    C->d_err = reinterpret_cast<int*>(C->base + err_off);
    C->d_work = reinterpret_cast<float*>(C->base + work_off);
  }
  return off;
}

// Algorithmic terms of the memory model for one layer-tensor.
void tensor_terms(const TensorLayout& T, const kvq_config& c, const int32_t* lens, double* packed, double* meta,
                  double* tail) {
  const double H = c.kv_heads, D = c.head_dim;
  double pb = 0, m = 0, tl = 0;
  for (int b = 0; b < c.batch; ++b) {
    long n = lens[b];
    long ns = sealed_tokens(T, n);
    pb += (double)ns * H * D * T.bits;
    tl += (double)(n - ns) * H * D * 2.0;
    if (T.axis == 1) m += (double)(ns / T.group) * H * D * T.meta_bytes;
    else if (T.whole) m += (double)ns * T.meta_bytes;
    else m += (double)ns * H * T.gpt * T.meta_bytes;
  }
  *packed = std::ceil(pb / 8.0);
  *meta = m;
  *tail = tl;
}

kvq_status cuda_status(kvq_cache* C, cudaError_t e) {
  if (e == cudaSuccess) return KVQ_OK;
  if (C) C->last_error = cudaGetErrorString(e);
  return KVQ_ERR_CUDA;
}

kvq_status layer_ok(kvq_cache* C, int layer) {
  if (!C) return KVQ_ERR_INVALID_ARG;
  if (layer < 0 || layer >= C->cfg.layers) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_cache_bytes(const kvq_config* cfg, const int32_t* lens_host, kvq_bytes* out) {
  kvq_status s = validate(cfg);
  if (s != KVQ_OK) return s;
  if (!out) return KVQ_ERR_INVALID_ARG;
  std::vector<int32_t> lens(cfg->batch, cfg->max_tokens);
  if (lens_host) {
    for (int b = 0; b < cfg->batch; ++b) {
      if (lens_host[b] < 0) return KVQ_ERR_INVALID_ARG;
      if (lens_host[b] > cfg->max_tokens) return KVQ_ERR_CAPACITY;
      lens[b] = lens_host[b];
    }
  }
  TensorLayout K = make_layout(cfg->k, *cfg), V = make_layout(cfg->v, *cfg);
  double pk, mk, tk, pv, mv, tv;
  tensor_terms(K, *cfg, lens.data(), &pk, &mk, &tk);
  tensor_terms(V, *cfg, lens.data(), &pv, &mv, &tv);
  const int tcap = tcap_of(*cfg);
  out->packed = (pk + pv) * cfg->layers;
  out->metadata = (mk + mv) * cfg->layers;
  out->tail = (tk + tv) * cfg->layers;
  out->workspace = (double)decode_work_floats(cfg->batch, cfg->q_heads, cfg->head_dim, max_chunks_of(*cfg, tcap)) * 4.0;
  out->total = out->packed + out->metadata + out->tail + out->workspace;
  double tokens = 0;
  for (int b = 0; b < cfg->batch; ++b) tokens += lens[b];
  out->elements = 2.0 * cfg->layers * tokens * cfg->kv_heads * cfg->head_dim;
  out->alloc = carve(*cfg, nullptr);
  return KVQ_OK;
}

kvq_status kvq_cache_create(const kvq_config* cfg, void* device_buf, size_t buf_bytes, void* stream,
                            kvq_cache_t* out) {
  kvq_status s = validate(cfg);
  if (s != KVQ_OK) return s;
  if (!device_buf || !out) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(device_buf) & 255) return KVQ_ERR_INVALID_ARG;
  size_t need = carve(*cfg, nullptr);
  if (buf_bytes < need) return KVQ_ERR_BUFFER_TOO_SMALL;
  kvq_cache* C = new (std::nothrow) kvq_cache();
  if (!C) return KVQ_ERR_INVALID_ARG;
  C->cfg = *cfg;
  C->base = static_cast<char*>(device_buf);
  C->bytes = buf_bytes;
  carve(*cfg, C);
  C->lens.assign((size_t)cfg->layers * cfg->batch, 0);
  cudaError_t e = cudaGetDevice(&C->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&C->sm_count, cudaDevAttrMultiProcessorCount, C->device);
  if (e == cudaSuccess) e = quant_setup(C);
  if (e == cudaSuccess) e = decode_setup(C);
  if (e == cudaSuccess) e = cudaMemsetAsync(device_buf, 0, need, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    delete C;
    return KVQ_ERR_CUDA;
  }
  *out = C;
  return KVQ_OK;
}

kvq_status kvq_cache_destroy(kvq_cache_t cache) {
  if (!cache) return KVQ_ERR_INVALID_ARG;
  delete cache;
  return KVQ_OK;
}

kvq_status kvq_prefill_quantize(kvq_cache_t C, int layer, const void* k, const void* v, int in_dtype,
                                const int32_t* lens_host, int64_t t_stride, void* stream) {
  kvq_status s = layer_ok(C, layer);
  if (s != KVQ_OK) return s;
  if (!lens_host || (in_dtype != KVQ_F16 && in_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  int maxn = 0;
  for (int b = 0; b < C->cfg.batch; ++b) {
    if (lens_host[b] < 0) return KVQ_ERR_INVALID_ARG;
    if (lens_host[b] > C->cfg.max_tokens) return KVQ_ERR_CAPACITY;
    maxn = std::max(maxn, (int)lens_host[b]);
  }
  if (t_stride < maxn || t_stride < 0) return KVQ_ERR_INVALID_ARG;
  if (maxn > 0 && (!k || !v)) return KVQ_ERR_INVALID_ARG;
  C->last_launches = 0;
  cudaError_t e = launch_prefill(C, layer, k, v, in_dtype == KVQ_F32, lens_host, (long)t_stride,
                                 static_cast<cudaStream_t>(stream), &C->last_launches);
  if (e != cudaSuccess) return cuda_status(C, e);
  std::copy(lens_host, lens_host + C->cfg.batch, C->lens.begin() + (long)layer * C->cfg.batch);
  return KVQ_OK;
}

kvq_status kvq_append(kvq_cache_t C, int layer, const void* k_new, const void* v_new, int in_dtype, void* stream) {
  kvq_status s = layer_ok(C, layer);
  if (s != KVQ_OK) return s;
  if (!k_new || !v_new || (in_dtype != KVQ_F16 && in_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  int32_t* lens = C->lens.data() + (long)layer * C->cfg.batch;
  for (int b = 0; b < C->cfg.batch; ++b)
    if (lens[b] + 1 > C->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  C->last_launches = 0;
  cudaError_t e = launch_append(C, layer, k_new, v_new, in_dtype == KVQ_F32, static_cast<cudaStream_t>(stream),
                                &C->last_launches);
  if (e != cudaSuccess) return cuda_status(C, e);
  for (int b = 0; b < C->cfg.batch; ++b) lens[b] += 1;
  return KVQ_OK;
}

kvq_status kvq_decode_attn(kvq_cache_t C, int layer, const void* q, int q_dtype, float softmax_scale, float* out,
                           void* stream) {
  kvq_status s = layer_ok(C, layer);
  if (s != KVQ_OK) return s;
  if (!q || !out || (q_dtype != KVQ_F16 && q_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f)) softmax_scale = 1.0f / std::sqrt((float)C->cfg.head_dim);
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  C->last_launches = 0;
  cudaError_t e = launch_decode(C, layer, q, q_dtype == KVQ_F32, softmax_scale, out,
                                static_cast<cudaStream_t>(stream), &C->last_launches);
  return cuda_status(C, e);
}

kvq_status kvq_append_decode_attn(kvq_cache_t C, int layer, const void* k_new, const void* v_new, int in_dtype,
                                  const void* q, int q_dtype, float softmax_scale, float* out, void* stream) {
  kvq_status s = layer_ok(C, layer);
  if (s != KVQ_OK) return s;
  if (!k_new || !v_new || (in_dtype != KVQ_F16 && in_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  if (!q || !out || (q_dtype != KVQ_F16 && q_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f)) softmax_scale = 1.0f / std::sqrt((float)C->cfg.head_dim);
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  int32_t* lens = C->lens.data() + (long)layer * C->cfg.batch;
  for (int b = 0; b < C->cfg.batch; ++b)
    if (lens[b] + 1 > C->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  C->last_launches = 0;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the fused append reads each lane's channels as 4- / 8-byte pairs
  const bool aligned = (reinterpret_cast<uintptr_t>(k_new) % 8) == 0 && (reinterpret_cast<uintptr_t>(v_new) % 8) == 0;
  if (!C->fused_ok || !aligned) {
    cudaError_t e = launch_append(C, layer, k_new, v_new, in_dtype == KVQ_F32, st, &C->last_launches);
    if (e != cudaSuccess) return cuda_status(C, e);
    for (int b = 0; b < C->cfg.batch; ++b) lens[b] += 1;
    e = launch_decode(C, layer, q, q_dtype == KVQ_F32, softmax_scale, out, st, &C->last_launches);
    return cuda_status(C, e);
  }
  // the launch is planned for the new lengths
  for (int b = 0; b < C->cfg.batch; ++b) lens[b] += 1;
  cudaError_t e = launch_append_decode(C, layer, k_new, v_new, in_dtype == KVQ_F32, q, q_dtype == KVQ_F32,
                                       softmax_scale, out, st, &C->last_launches);
  if (e != cudaSuccess) {
    for (int b = 0; b < C->cfg.batch; ++b) lens[b] -= 1;
    return cuda_status(C, e);
  }
  return KVQ_OK;
}

kvq_status kvq_dequantize(kvq_cache_t C, int layer, void* k_out, void* v_out, void* stream) {
  kvq_status s = layer_ok(C, layer);
  if (s != KVQ_OK) return s;
  if (!k_out || !v_out) return KVQ_ERR_INVALID_ARG;
  C->last_launches = 0;
  cudaError_t e = launch_dequantize(C, layer, k_out, v_out, static_cast<cudaStream_t>(stream), &C->last_launches);
  return cuda_status(C, e);
}

kvq_status kvq_decode_attn_materialized(kvq_cache_t C, int layer, const void* k16, const void* v16, const void* q,
                                        int q_dtype, float softmax_scale, float* out, void* stream) {
  kvq_status s = layer_ok(C, layer);
  if (s != KVQ_OK) return s;
  if (!k16 || !v16 || !q || !out || (q_dtype != KVQ_F16 && q_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f)) softmax_scale = 1.0f / std::sqrt((float)C->cfg.head_dim);
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  C->last_launches = 0;
  cudaError_t e = launch_decode_materialized(C, layer, k16, v16, q, q_dtype == KVQ_F32, softmax_scale, out,
                                             static_cast<cudaStream_t>(stream), &C->last_launches);
  return cuda_status(C, e);
}

kvq_status kvq_export(kvq_cache_t C, int layer, uint8_t* codes_k, uint8_t* codes_v, float* meta_k, float* meta_v,
                      uint16_t* tail_k, uint16_t* tail_v, int32_t* lens, void* stream) {
  kvq_status s = layer_ok(C, layer);
  if (s != KVQ_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_export(C, layer, 0, codes_k, meta_k, tail_k, st);
  if (e == cudaSuccess) e = launch_export(C, layer, 1, codes_v, meta_v, tail_v, st);
  if (e == cudaSuccess && lens)
    e = cudaMemcpyAsync(lens, C->d_lens + (long)layer * C->cfg.batch, sizeof(int32_t) * C->cfg.batch,
                        cudaMemcpyDeviceToDevice, st);
  return cuda_status(C, e);
}

int kvq_cache_tcap(kvq_cache_t C) { return C ? C->tcap : 0; }

kvq_status kvq_get_lens(kvq_cache_t C, int layer, int32_t* lens_host) {
  kvq_status s = layer_ok(C, layer);
  if (s != KVQ_OK) return s;
  if (!lens_host) return KVQ_ERR_INVALID_ARG;
  std::copy(C->lens.begin() + (long)layer * C->cfg.batch, C->lens.begin() + (long)(layer + 1) * C->cfg.batch,
            lens_host);
  return KVQ_OK;
}

kvq_status kvq_decode_traffic(kvq_cache_t C, int layer, int q_dtype, double* bytes) {
  kvq_status s = layer_ok(C, layer);
  if (s != KVQ_OK) return s;
  if (!bytes || (q_dtype != KVQ_F16 && q_dtype != KVQ_F32)) return KVQ_ERR_INVALID_ARG;
  const int32_t* lens = C->lens.data() + (long)layer * C->cfg.batch;
  double pk, mk, tk, pv, mv, tv;
  tensor_terms(C->k, C->cfg, lens, &pk, &mk, &tk);
  tensor_terms(C->v, C->cfg, lens, &pv, &mv, &tv);
  double qb = (double)C->cfg.batch * C->cfg.q_heads * C->cfg.head_dim * (q_dtype == KVQ_F32 ? 4.0 : 2.0);
  *bytes = pk + mk + tk + pv + mv + tv + qb;
  return KVQ_OK;
}

kvq_status kvq_device_status(kvq_cache_t C, void* stream) {
  if (!C) return KVQ_ERR_INVALID_ARG;
  int flag = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&flag, C->d_err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(C, e);
  if (flag) {
    cudaMemsetAsync(C->d_err, 0, sizeof(int), st);
    return KVQ_ERR_DEVICE_TIMEOUT;
  }
  return KVQ_OK;
}

int kvq_last_launches(kvq_cache_t C) { return C ? C->last_launches : 0; }

kvq_status kvq_set_decode_plan(kvq_cache_t C, int plan_tokens) {
  if (!C || plan_tokens < 0) return KVQ_ERR_INVALID_ARG;
  C->plan_tokens = plan_tokens;
  return KVQ_OK;
}

kvq_status kvq_set_decode_kernel(kvq_cache_t C, int which) {
  if (!C || which < 0 || which > 7) return KVQ_ERR_INVALID_ARG;
  C->generic_decode = which & 1;
  C->global_combine = (which >> 1) & 1;
  C->one_warp = (which >> 2) & 1;
  return cuda_status(C, decode_setup(C));
}

int kvq_decode_cta_warps(kvq_cache_t C, int fused) {
  if (!C || !C->dec_fn) return 0;
  if (fused) return C->fused_ok ? C->dec_nw_fused : 0;
  return C->dec_nw;
}

int kvq_decode_kernel_specialized(kvq_cache_t C) {
  if (!C || !C->dec_fn || C->generic_decode) return 0;
  void* fast = C->cfg.rope_theta > 0.0f ? decode_kernel_rope_fast(C) : decode_kernel_fast(C);
  return C->dec_fn == fast ? 1 : 0;
}

kvq_status kvq_refresh_lens(kvq_cache_t C, void* stream) {
  if (!C) return KVQ_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(C->lens.data(), C->d_lens, sizeof(int32_t) * C->lens.size(),
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_status(C, e);
}

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CAPACITY: return "sequence capacity exceeded";
    case KVQ_ERR_BUFFER_TOO_SMALL: return "device buffer too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* kvq_last_error(kvq_cache_t C) { return C ? C->last_error.c_str() : ""; }

}  // extern "C"
