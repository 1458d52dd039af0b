// kvq_decode.cu — split planning and launch of the decode attention kernel.
#include <algorithm>
#include <cmath>
#include <vector>

#include "kvq_decode_args.h"

namespace kvq {

namespace {

struct Plan {
  DecodeArgs a;
  size_t smem;
  dim3 grid;
};

// Shared memory a cluster launch adds after the kernel's plan: the first
// CTA's gather area of the csize split partials ([csize][rep][D+2] floats).
static size_t gather_bytes(int csize, int rep, int D) { return (size_t)csize * rep * (D + 2) * 4; }

// Raise (never lower) a kernel's dynamic shared-memory limit: several caches
// may share one kernel with different plans.
static cudaError_t raise_smem_limit(const void* fn, size_t bytes) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  if ((size_t)fa.maxDynamicSharedSizeBytes >= bytes) return cudaSuccess;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Whether a cluster launch of fn keeps the residency the planner counts on
// (min(occ, 4) CTAs per SM) with the largest gather area added.
static bool cluster_fits(const void* fn, size_t smem, int rep, int D, int occ, int warp_bytes) {
  const size_t full = smem + gather_bytes(kMaxCluster, rep, D);
  if (full > 227 * 1024) return false;
  if (4L * rep * (D + 2) * 4 > 4L * warp_bytes) return false;  // the CTA merge's four warp partials
  if (raise_smem_limit(fn, full) != cudaSuccess) return false;
  int occ2 = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, fn, kWarps * 32, full) != cudaSuccess) return false;
  return occ2 >= std::min(occ, 4);
}

void* pick_kernel_rope(int D, bool r8, int vaxis) {
  if (D == 64) return decode_kernel_ptr_rope_d64(r8, vaxis);
  if (D == 128) return decode_kernel_ptr_rope_d128(r8, vaxis);
  if (D == 256) return decode_kernel_ptr_rope_d256(r8, vaxis);
  return nullptr;
}

void* pick_kernel(int D, bool r8, int vaxis) {
  if (D == 64) return decode_kernel_ptr_d64(r8, vaxis);
  if (D == 128) return decode_kernel_ptr_d128(r8, vaxis);
  if (D == 256) return decode_kernel_ptr_d256(r8, vaxis);
  return nullptr;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// bytes of one tile's (per-token) or one group's (per-channel) metadata
int meta_tile_bytes(const TensorLayout& L) { return kTile * (L.whole ? 1 : L.gpt) * L.meta_bytes; }

// Work weight of a token in fp16 rows (see plan_launch): 1 without a window.
int window_weight(const kvq_cache* C) {
  if (C->k.window == 0 && C->v.window == 0) return 1;
  const int D = C->cfg.head_dim;
  auto packed = [&](const TensorLayout& L) {
    const double meta = L.axis == 0 ? meta_tile_bytes(L) : (double)D * L.meta_bytes * kTile / L.group;
    return L.tile_words * 4.0 + meta;
  };
  const double ratio = 2.0 * kTile * D * 2.0 / (packed(C->k) + packed(C->v));
  return std::max(1, std::min(8, (int)std::lround(ratio)));
}

}  // namespace

// Shared-memory plan and per-call split of the token range.
static cudaError_t make_plan(kvq_cache* C, int layer, Plan* P, int* occ_out, int nw = kWarps) {
  const kvq_config& cfg = C->cfg;
  const int D = cfg.head_dim, rep = cfg.q_heads / cfg.kv_heads;
  const bool r8 = rep == 8;
  DecodeArgs& a = P->a;
  auto fill = [&](DecTensor& d, const TensorLayout& L) {
    d.codes = C->base + L.codes_off + (size_t)layer * L.codes_layer;
    d.meta = C->base + L.meta_off + (size_t)layer * L.meta_layer;
    d.tail = reinterpret_cast<const __half*>(C->base + L.tail_off + (size_t)layer * L.tail_layer);
    d.bits = L.bits;
    d.sym = L.sym;
    d.meta_f32 = L.meta_f32;
    d.axis = L.axis;
    d.whole = L.whole;
    d.group = L.whole ? D : L.group;
    int lg = 0;
    while ((1 << lg) < d.group) ++lg;
    d.lg_group = L.whole ? 30 : lg;
    d.gpt = L.gpt;
    d.meta_bytes = L.meta_bytes;
    d.tile_bytes = L.tile_words * 4;
    d.mtile_bytes = L.axis == 0 ? meta_tile_bytes(L) : D * L.meta_bytes;
    d.window = L.window;
    d.ring = L.ring;
  };
  fill(a.K, C->k);
  fill(a.V, C->v);
  a.B = cfg.batch;
  a.H = cfg.kv_heads;
  a.rep = rep;
  a.tcap = C->tcap;
  a.ntiles = C->tcap / kTile;
  a.lens = C->d_lens + (long)layer * cfg.batch;
  a.smax_k = C->d_smax + ((long)0 * cfg.layers + layer) * cfg.batch * cfg.kv_heads;
  a.smax_v = C->d_smax + ((long)1 * cfg.layers + layer) * cfg.batch * cfg.kv_heads;
  a.max_chunks = C->max_chunks;
  a.work = C->d_work;
  a.max_groups = combine_groups(C->max_chunks);
  a.gwork = C->d_work + (size_t)cfg.batch * cfg.q_heads * C->max_chunks * (D + 4);
  a.tickets = C->d_decode_tickets;
  a.err = C->d_err;
  // the cache's fp16 rows (window, unsealed groups) are read straight from
  // global memory, prefetched into L2 when their tile is issued
  a.stage_f16 = 0;
  a.fw = 1;
  a.arrive = C->d_arrive;
  const int rope = cfg.rope_theta > 0.0f;
  a.rope_l2b = rope ? std::log2((double)cfg.rope_theta) : 0.0;
  const DecLayout L = dec_layout(D, rep, C->k.bits, C->k.axis, C->k.whole, C->k.gpt, C->k.meta_bytes, C->v.bits,
                                 C->v.axis, C->v.whole, C->v.gpt, C->v.meta_bytes, 0, rope);
  a.rope_off = L.rope_off;
  a.st_kc = L.st_kc;
  a.st_km = L.st_km;
  a.st_vc = L.st_vc;
  a.st_vm = L.st_vm;
  a.stage_bytes = L.stage_bytes;
  a.lg_nstages = L.lg_ns;
  a.barea_bytes = L.barea_bytes;
  a.canon_k = L.canon_k;
  a.canon_v = L.canon_v;
  a.stage_off = L.stage_off;
  a.warp_bytes = L.warp_bytes;
  a.head_bytes = L.head_bytes;
  P->smem = (size_t)a.head_bytes + (size_t)nw * a.warp_bytes;
  if (!C->dec_fn) return cudaErrorInvalidValue;
  *occ_out = C->dec_occ;
  return cudaSuccess;
}

cudaError_t decode_setup(kvq_cache* C) {
  // pre-RoPE caches run the rotary instances of the runtime-format kernel
  const bool rope = C->cfg.rope_theta > 0.0f;
  int nw = kWarps;
  void* fn = C->generic_decode ? nullptr : (rope ? decode_kernel_rope_fast(C) : decode_kernel_fast(C, &nw));
  if (!fn) nw = kWarps;
  if (!fn && rope) fn = pick_kernel_rope(C->cfg.head_dim, C->cfg.q_heads / C->cfg.kv_heads == 8, C->v.axis);
  if (!fn) fn = pick_kernel(C->cfg.head_dim, C->cfg.q_heads / C->cfg.kv_heads == 8, C->v.axis);
  if (!fn) return cudaErrorInvalidValue;
  C->dec_fn = fn;
  C->dec_nw = nw;
  Plan P;
  int occ = 1;
  cudaError_t e = make_plan(C, 0, &P, &occ, nw);
  if (e != cudaSuccess) return e;
  if (P.smem > 227 * 1024) return cudaErrorInvalidValue;
  e = raise_smem_limit(fn, P.smem);
  if (e != cudaSuccess) return e;
  // the same (largest) shared-memory carve-out as the append kernel, so that
  // alternating append / decode launches need no L1 / shared reconfiguration
  e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, nw * 32, P.smem);
  if (e != cudaSuccess) return e;
  C->dec_smem = P.smem;
  C->dec_occ = std::max(occ, 1);
  const int rep = C->cfg.q_heads / C->cfg.kv_heads;
  // (one-warp CTAs merge through the global workspace only)
  C->dec_cluster_ok = !C->global_combine && nw == kWarps &&
                      cluster_fits(fn, P.smem, rep, C->cfg.head_dim, C->dec_occ, P.a.warp_bytes);
  // the fused append needs a fused specialisation, layouts where each
  // (sequence, head) owns all it writes (no whole-vector groups; with a
  // window the block or group leaving it is sealed by the warp whose range
  // holds it), its scratch inside one warp's stage ring, and the plain
  // kernel's residency and cluster merge (the launch is planned for the plain kernel)
  const int ring = (1 << P.a.lg_nstages) * P.a.stage_bytes;
  C->fused_ok = 0;
  int nwf = kWarps;
  C->dec_fn_fused = (C->generic_decode || rope) ? nullptr : decode_kernel_fused(C, &nwf);
  C->dec_nw_fused = nwf;
  const int window = C->k.window || C->v.window;
  if (C->dec_fn_fused && !C->k.whole && !C->v.whole &&
      fused_append_scratch(C->cfg.head_dim, C->k.axis, C->v.axis, window) <= ring) {
    void* ff = C->dec_fn_fused;
    Plan Pf;
    int occ_f = 0, occ_unused = 1;
    e = make_plan(C, 0, &Pf, &occ_unused, nwf);
    if (e == cudaSuccess) e = raise_smem_limit(ff, Pf.smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ff, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_f, ff, nwf * 32, Pf.smem);
    if (e != cudaSuccess) return e;
    C->dec_occ_fused = std::max(occ_f, 1);
    if (nwf == nw) {
      // same CTA shape: planned like the plain kernel, whose residency and cluster merge it must keep
      const bool cl_same =
          !C->dec_cluster_ok || cluster_fits(ff, P.smem, rep, C->cfg.head_dim, C->dec_occ, P.a.warp_bytes);
      C->fused_ok = occ_f >= C->dec_occ && cl_same;
    } else {
      C->fused_ok = occ_f > 0;  // planned for its own residency, merged through the global workspace
    }
  }
  return cudaSuccess;
}

// Choose tokens per CTA (a multiple of nw warps x the alignment unit) so that
// the CTAs fill whole waves of the GPU with as little imbalance as possible.
// Cost = waves x (tokens per CTA + a fixed cost per CTA).  The fixed cost (the
// prologue's first-data latency, the split-K merge) is worth about 96 tokens
// of streaming per warp of the CTA: on a Llama-2-13B-shaped batch (16 x 40
// heads x 4113 tokens) three splits of 1408 tokens in four-warp CTAs ran 13 %
// faster than seven of 640.  Candidates are even fractions of the whole job
// and even splits of the longest sequence.
static int choose_split(const kvq_cache* C, const int32_t* lens, int unit, int slots, int max_chunks,
                        int nw = kWarps) {
  const int step = nw * unit;
  const double fixed = 96.0 * nw;
  const int B = C->cfg.batch, H = C->cfg.kv_heads;
  long total = 0;
  int maxn = 0;
  for (int b = 0; b < B; ++b) {
    total += lens[b];
    maxn = std::max(maxn, (int)lens[b]);
  }
  if (maxn == 0) return step;
  const int s_min_cap = round_up((maxn + max_chunks - 1) / max_chunks, step);
  int best = 0;
  double best_cost = 1e300;
  auto eval = [&](int S) {
    if (S < s_min_cap) S = s_min_cap;
    long ctas = 0;
    for (int b = 0; b < B; ++b) ctas += (lens[b] + S - 1) / S;
    ctas *= H;
    const double waves = std::ceil((double)ctas / slots);
    const double cost = waves * (S + fixed);
    if (cost < best_cost - 1e-9 || (std::fabs(cost - best_cost) < 1e-9 && S > best)) {
      best_cost = cost;
      best = S;
    }
  };
  const double ideal = (double)total * H / slots;
  for (int k = 1; k <= 4096; k *= 2) eval(step * k);
  for (int m = 1; m <= 8; ++m) eval(round_up((int)std::ceil(ideal / m), step));
  for (int n = 1; n <= 64; ++n) eval(round_up((maxn + n - 1) / n, step));
  return best;
}

// Plan one decode launch on the host length mirror, raised to the plan hint (a
// launch planned for the hint stays valid while the cache grows up to it):
// split size, grid, and how the split-K partials merge.
static cudaError_t plan_launch(kvq_cache* C, int layer, const void* q, int q_f32, float scale, float* out, Plan* P,
                               dim3* grid, bool fused = false) {
  const int nw = fused ? C->dec_nw_fused : C->dec_nw;
  int occ = 1;
  cudaError_t e = make_plan(C, layer, P, &occ, nw);
  if (e != cudaSuccess) return e;
  if (fused && nw != C->dec_nw) occ = C->dec_occ_fused;
  DecodeArgs& a = P->a;
  const kvq_config& cfg = C->cfg;
  int unit = kTile;
  if (C->k.axis == 1) unit = std::max(unit, C->k.group);
  if (C->v.axis == 1) unit = std::max(unit, C->v.group);
  std::vector<int32_t> plan(C->lens.begin() + (long)layer * cfg.batch, C->lens.begin() + (long)(layer + 1) * cfg.batch);
  for (auto& x : plan) x = std::max(x, (int32_t)std::min(C->plan_tokens, C->cfg.max_tokens));
  // With a full-precision window, a token still in fp16 rows counts as the
  // ratio of an fp16 tile's bytes to a packed tile's (codes and metadata of
  // both tensors), at most 8, so that the split spreads the window's tiles
  // over several warps.  The kernel weighs the fp16 part from the first unit
  // below its sealed tokens, at most window + 2 units of a sequence; the plan
  // uses that bound (the work only grows with the length, so a launch planned
  // for a length covers every shorter one).
  a.fw = window_weight(C);
  if (a.fw > 1) {
    const int span = std::max(C->k.window, C->v.window) + 2 * unit;
    for (auto& x : plan) x += (int32_t)((a.fw - 1) * std::min((int)x, span));
  }
  // about four resident CTAs (16 warps) per SM already keep the issue slots
  // busy; planning for more only adds per-CTA fixed work.  The fused append +
  // decode launch is planned for every resident CTA: fewer, longer ranges
  // hide the appending warp's quantization better (measured on Llama-2-13B:
  // one split of 4224 tokens per (sequence, head), one wave of 640 CTAs, 5 %
  // faster per step than three splits of 1408, while the plain decode is 4 %
  // slower that way)
  // (in warps: about 16 resident warps per SM; the four-warp fused launch
  // takes every resident CTA)
  const int slots =
      C->sm_count * ((fused && nw == kWarps) ? occ : std::max(1, std::min(occ * nw, 4 * kWarps) / nw));
  a.S = choose_split(C, plan.data(), unit, slots, C->max_chunks, nw);
  a.Sw = a.S / nw;
  int maxn = 0;
  for (int b = 0; b < cfg.batch; ++b) maxn = std::max(maxn, (int)plan[b]);
  const int nch = std::max(1, (maxn + a.S - 1) / a.S);
  // up to kMaxCluster splits of a (sequence, head) form one thread-block
  // cluster and merge through distributed shared memory; more go through the
  // global workspace and atomic tickets
  // (only when the whole grid is resident at once: with several waves, CTAs
  // that wait for their cluster would hold slots that later CTAs need)
  const long ctas = (long)nch * cfg.kv_heads * cfg.batch;
  a.csize = (C->dec_cluster_ok && nw == kWarps && nch <= kMaxCluster && ctas <= slots) ? nch : 0;
  a.gath_off = (int)P->smem;
  P->smem += gather_bytes(a.csize, cfg.q_heads / cfg.kv_heads, cfg.head_dim);
  a.q = q;
  a.q_f32 = q_f32;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  *grid = dim3(nch, cfg.kv_heads, cfg.batch);
  return cudaSuccess;
}

cudaError_t launch_decode(kvq_cache* C, int layer, const void* q, int q_f32, float scale, float* out,
                          cudaStream_t st, int* launches) {
  Plan P;
  dim3 grid;
  cudaError_t e = plan_launch(C, layer, q, q_f32, scale, out, &P, &grid);
  if (e != cudaSuccess) return e;
  void* args[] = {&P.a};
  e = launch_pdl(C->dec_fn, grid, dim3(C->dec_nw * 32), P.smem, st, args, P.a.csize);
  ++*launches;
  return e;
}

// Append of one token per (sequence, head) fused into the decode launch.  The
// host mirror of the lengths already counts the new token.
cudaError_t launch_append_decode(kvq_cache* C, int layer, const void* k, const void* v, int x_f32, const void* q,
                                 int q_f32, float scale, float* out, cudaStream_t st, int* launches) {
  Plan P;
  dim3 grid;
  cudaError_t e = plan_launch(C, layer, q, q_f32, scale, out, &P, &grid, true);
  if (e != cudaSuccess) return e;
  P.a.ap = make_append_args(C, layer, k, v, x_f32);
  void* args[] = {&P.a};
  e = launch_pdl(C->dec_fn_fused, grid, dim3(C->dec_nw_fused * 32), P.smem, st, args, P.a.csize);
  ++*launches;
  return e;
}

// Same plan and kernel as launch_decode, with the split-K partials and the
// combine tickets placed in caller-chosen scratch (used by the entry point
// whose scratch is a static device array).
cudaError_t launch_decode_scratch(kvq_cache* C, int layer, const void* q, int q_f32, float scale, float* out,
                                  cudaStream_t st, int* launches, float* work, uint32_t* tickets) {
  Plan P;
  dim3 grid;
  cudaError_t e = plan_launch(C, layer, q, q_f32, scale, out, &P, &grid);
  if (e != cudaSuccess) return e;
  DecodeArgs& a = P.a;
  a.work = work;
  a.gwork = work + (size_t)C->cfg.batch * C->cfg.q_heads * C->max_chunks * (C->cfg.head_dim + 4);
  a.tickets = tickets;
  void* args[] = {&a};
  e = launch_pdl(C->dec_fn, grid, dim3(C->dec_nw * 32), P.smem, st, args, a.csize);
  ++*launches;
  return e;
}

// Decode over fp16 K / V rows materialised by kvq_dequantize ([B][Hkv][tcap][D]):
// the same kernel (runtime formats, per-channel axis for both tensors) with
// every token in its fp16 tail path, i.e. no packed tiles and no metadata.
cudaError_t launch_decode_materialized(kvq_cache* C, int layer, const void* k16, const void* v16, const void* q,
                                       int q_f32, float scale, float* out, cudaStream_t st, int* launches) {
  const kvq_config& cfg = C->cfg;
  const int D = cfg.head_dim, rep = cfg.q_heads / cfg.kv_heads;
  const int rope = cfg.rope_theta > 0.0f;  // the rows hold pre-RoPE keys: rotate them as the fused path does
  void* fn = rope ? pick_kernel_rope(D, rep == 8, 1) : pick_kernel(D, rep == 8, 1);
  if (!fn) return cudaErrorInvalidValue;
  Plan P;
  int occ_unused = 1;
  cudaError_t e = make_plan(C, layer, &P, &occ_unused);
  if (e != cudaSuccess) return e;
  DecodeArgs& a = P.a;
  auto tail_only = [&](DecTensor& d, const void* rows) {
    d.tail = static_cast<const __half*>(rows);
    d.axis = 1;
    d.whole = 0;
    d.group = C->tcap;         // row stride of a (sequence, head)
    d.lg_group = 30;           // nothing is ever sealed
    d.gpt = 0;
    d.window = 0;
    d.ring = C->tcap;          // token t at row t
  };
  tail_only(a.K, k16);
  tail_only(a.V, v16);
  a.stage_f16 = 1;
  const DecLayout L = dec_layout(D, rep, a.K.bits, 1, 0, 0, a.K.meta_bytes, a.V.bits, 1, 0, 0, a.V.meta_bytes, 1, rope);
  a.rope_off = L.rope_off;
  a.st_kc = L.st_kc;
  a.st_km = L.st_km;
  a.st_vc = L.st_vc;
  a.st_vm = L.st_vm;
  a.stage_bytes = L.stage_bytes;
  a.lg_nstages = L.lg_ns;
  a.barea_bytes = L.barea_bytes;
  a.canon_k = L.canon_k;
  a.canon_v = L.canon_v;
  a.stage_off = L.stage_off;
  a.warp_bytes = L.warp_bytes;
  a.head_bytes = L.head_bytes;
  const size_t smem = (size_t)a.head_bytes + (size_t)kWarps * a.warp_bytes;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  e = raise_smem_limit(fn, smem);
  if (e != cudaSuccess) return e;
  int occ = 1;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kWarps * 32, smem);
  if (e != cudaSuccess) return e;
  std::vector<int32_t> plan(C->lens.begin() + (long)layer * cfg.batch, C->lens.begin() + (long)(layer + 1) * cfg.batch);
  for (auto& x : plan) x = std::max(x, (int32_t)std::min(C->plan_tokens, C->cfg.max_tokens));
  const int slots = C->sm_count * std::min(std::max(occ, 1), 4);
  a.S = choose_split(C, plan.data(), kTile, slots, C->max_chunks);
  a.Sw = a.S / kWarps;
  int maxn = 0;
  for (int b = 0; b < cfg.batch; ++b) maxn = std::max(maxn, (int)plan[b]);
  const int nch = std::max(1, (maxn + a.S - 1) / a.S);
  const long ctas = (long)nch * cfg.kv_heads * cfg.batch;
  const bool cl_ok = !C->global_combine && nch <= kMaxCluster && ctas <= slots &&
                     cluster_fits(fn, smem, rep, D, std::max(occ, 1), a.warp_bytes);
  a.csize = cl_ok ? nch : 0;
  a.gath_off = (int)smem;
  const size_t lsmem = smem + gather_bytes(a.csize, rep, D);
  a.q = q;
  a.q_f32 = q_f32;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  void* args[] = {&a};
  e = launch_pdl(fn, dim3(nch, cfg.kv_heads, cfg.batch), dim3(kWarps * 32), lsmem, st, args, a.csize);
  ++*launches;
  return e;
}

}  // namespace kvq
