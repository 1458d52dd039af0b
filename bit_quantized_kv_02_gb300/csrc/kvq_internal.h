// kvq_internal.h — host-side cache handle and internal launcher declarations.
#pragma once

#include <string>
#include <vector>

#include "../../include/kvq.h"
#include "kvq_common.cuh"

struct kvq_cache {
  kvq_config cfg;
  int tcap = 0;          // token capacity of the tile / group layout
  char* base = nullptr;  // caller's device buffer
  size_t bytes = 0;
  kvq::TensorLayout k, v;
  int32_t* d_lens = nullptr;            // [layers][batch]
  uint32_t* d_smax = nullptr;           // [2][layers][batch][kv_heads] largest step (float bits), K then V
  int32_t* d_head_lens = nullptr;       // [layers][batch][kv_heads] per-head copies of the lengths (append)
  uint32_t* d_decode_tickets = nullptr; // [batch][kv_heads]
  int* d_err = nullptr;                 // device error word
  float* d_work = nullptr;              // split-K partials [batch][q_heads][max_chunks][head_dim + 4], then group partials
  int max_chunks = 0;
  std::vector<int32_t> lens;  // host mirror [layers][batch]
  int last_launches = 0;
  std::string last_error;
  int device = 0;
  int sm_count = 0;
  int plan_tokens = 0;  // decode split plan assumes at least this many tokens per sequence
  size_t dec_smem = 0;  // dynamic shared memory of the decode kernel
  int dec_occ = 1;      // resident decode CTAs per SM
  int dec_cluster_ok = 0;  // split-K partials may merge inside a thread-block cluster
  int global_combine = 0;  // 1: always merge split-K partials through the global workspace
  void* dec_fn = nullptr;  // decode kernel in use (compile-time specialisation or generic)
  int generic_decode = 0;  // 1: always use the generic (runtime-format) decode kernel
  int fused_ok = 0;        // the append can run inside the decode launch (kvq_append_decode_attn)
  void* dec_fn_fused = nullptr;  // the decode kernel's specialisation with the append fused in
  int dec_nw = kvq::kWarps;        // warps per CTA of dec_fn
  int dec_nw_fused = kvq::kWarps;  // warps per CTA of dec_fn_fused
  int dec_occ_fused = 1;           // resident CTAs per SM of dec_fn_fused
  int one_warp = 0;                // 1: one-warp-CTA specialisations where a format has them
  uint32_t* d_arrive = nullptr;  // [batch][kv_heads] arrival counters of the fused append
};

namespace kvq {

// Launch with programmatic stream serialisation: the kernel's CTAs may be
// scheduled while the previous kernel of the stream finishes; every such
// kernel calls pdl_wait() before it touches global memory.
// cluster_x > 0 also groups the grid's x dimension into clusters of that size.
inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args,
                              int cluster_x = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int na = 1;
  if (cluster_x > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

struct LensArg {
  int v[kMaxBatch];
};

inline long meta_groups(const kvq_cache* C, const TensorLayout& L) {
  const long B = C->cfg.batch, H = C->cfg.kv_heads, D = C->cfg.head_dim;
  if (L.axis == 1) return B * H * (C->tcap / L.group) * D;
  if (L.whole) return B * C->tcap;
  return B * H * C->tcap * L.gpt;
}

cudaError_t launch_prefill(kvq_cache* C, int layer, const void* k, const void* v, int x_f32,
                           const int32_t* lens_host, long t_stride, cudaStream_t st, int* launches);
cudaError_t launch_append(kvq_cache* C, int layer, const void* k, const void* v, int x_f32, cudaStream_t st,
                          int* launches);
cudaError_t launch_dequantize(kvq_cache* C, int layer, void* k_out, void* v_out, cudaStream_t st, int* launches);
cudaError_t launch_decode_materialized(kvq_cache* C, int layer, const void* k16, const void* v16, const void* q,
                                       int q_f32, float scale, float* out, cudaStream_t st, int* launches);
cudaError_t launch_export(kvq_cache* C, int layer, int is_value, uint8_t* codes, float* meta, uint16_t* tail,
                          cudaStream_t st);
size_t append_smem(const kvq_cache* C);

// fast prefill kernels (kvq_prefill.cu): fp16 inputs, no window, no whole-vector groups
struct QuantArgs;
bool prefill_fast_ok(const QuantArgs& a);
cudaError_t launch_prefill_fast(const QuantArgs& a, int maxn, cudaStream_t st);
cudaError_t prefill_fast_setup();

// one-time kernel attribute set-up at cache creation (keeps launches capturable)
cudaError_t quant_setup(kvq_cache* C);
cudaError_t decode_setup(kvq_cache* C);
// (nw, if not null, receives the kernel's warps per CTA)
void* decode_kernel_fast(const kvq_cache* C, int* nw = nullptr);
void* decode_kernel_fused(const kvq_cache* C, int* nw = nullptr);
void* decode_kernel_rope_fast(const kvq_cache* C);

// decode: plans the split, launches the split-K kernel (which also combines)
cudaError_t launch_decode(kvq_cache* C, int layer, const void* q, int q_f32, float scale, float* out,
                          cudaStream_t st, int* launches);

cudaError_t launch_append_decode(kvq_cache* C, int layer, const void* k, const void* v, int x_f32, const void* q,
                                 int q_f32, float scale, float* out, cudaStream_t st, int* launches);

cudaError_t launch_decode_scratch(kvq_cache* C, int layer, const void* q, int q_f32, float scale, float* out,
                                  cudaStream_t st, int* launches, float* work, uint32_t* tickets);

}  // namespace kvq
