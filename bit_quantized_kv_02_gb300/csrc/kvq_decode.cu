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

void* pick_kernel(int D, bool r8, int vaxis) {
  if (D == 64) return decode_kernel_ptr_d64(r8, vaxis);
  if (D == 128) return decode_kernel_ptr_d128(r8, vaxis);
  if (D == 256) return decode_kernel_ptr_d256(r8, vaxis);
  return nullptr;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// bytes of one tile's (per-token) or one group's (per-channel) metadata
int meta_tile_bytes(const TensorLayout& L) { return kTile * (L.whole ? 1 : L.gpt) * L.meta_bytes; }

}  // namespace

// Shared-memory plan and per-call split of the token range.
static cudaError_t make_plan(kvq_cache* C, int layer, Plan* P, int* occ_out) {
  const kvq_config& cfg = C->cfg;
  const int D = cfg.head_dim, rep = cfg.q_heads / cfg.kv_heads;
  const bool r8 = rep == 8;
  DecodeArgs& a = P->a;
  a.K = C->k;
  a.V = C->v;
  a.layer = layer;
  a.B = cfg.batch;
  a.H = cfg.kv_heads;
  a.rep = rep;
  a.tcap = C->tcap;
  a.ntiles = C->tcap / kTile;
  a.base = C->base;
  a.lens = C->d_lens + (long)layer * cfg.batch;
  a.smax_v = C->d_smax + ((long)1 * cfg.layers + layer) * cfg.batch * cfg.kv_heads;
  a.max_chunks = C->max_chunks;
  a.work = C->d_work;
  a.tickets = C->d_decode_tickets;
  a.err = C->d_err;
  a.kc_bytes = C->k.tile_words * 4;
  a.vc_bytes = C->v.tile_words * 4;
  a.km_tile_bytes = C->k.axis == 0 ? meta_tile_bytes(C->k) : 0;
  a.vm_tile_bytes = C->v.axis == 0 ? meta_tile_bytes(C->v) : 0;
  a.km_group_bytes = C->k.axis == 1 ? D * C->k.meta_bytes : 0;
  a.vm_group_bytes = C->v.axis == 1 ? D * C->v.meta_bytes : 0;
  a.st_kc = 0;
  a.st_km = round_up(a.st_kc + a.kc_bytes, 16);
  a.st_vc = round_up(a.st_km + std::max(a.km_tile_bytes, a.km_group_bytes), 16);
  a.st_vm = round_up(a.st_vc + a.vc_bytes, 16);
  a.stage_bytes = round_up(a.st_vm + std::max(a.vm_tile_bytes, a.vm_group_bytes), 128);
  a.nstages = a.stage_bytes <= 4096 ? 4 : 3;
  a.barea_bytes = (D / 16) * 32 * 8 * (r8 ? 2 : 1);
  a.warp_bytes = round_up(a.barea_bytes + 128 + a.nstages * a.stage_bytes + a.nstages * 8, 128);
  const int merge_bytes = kWarps * rep * (D + 2) * 4;
  if (a.warp_bytes * kWarps < merge_bytes) a.warp_bytes = round_up((merge_bytes + kWarps - 1) / kWarps, 128);
  a.head_bytes = round_up((rep * D + (C->k.axis == 0 ? C->k.gpt * rep : 0)) * 4, 128);
  P->smem = (size_t)a.head_bytes + (size_t)kWarps * a.warp_bytes;
  if (!pick_kernel(D, r8, C->v.axis)) return cudaErrorInvalidValue;
  *occ_out = C->dec_occ;
  return cudaSuccess;
}

cudaError_t decode_setup(kvq_cache* C) {
  Plan P;
  int occ = 1;
  cudaError_t e = make_plan(C, 0, &P, &occ);
  if (e != cudaSuccess) return e;
  void* fn = pick_kernel(C->cfg.head_dim, C->cfg.q_heads / C->cfg.kv_heads == 8, C->v.axis);
  if (P.smem > 227 * 1024) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P.smem);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kWarps * 32, P.smem);
  if (e != cudaSuccess) return e;
  C->dec_smem = P.smem;
  C->dec_occ = std::max(occ, 1);
  return cudaSuccess;
}

// Choose tokens per CTA (a multiple of 4 warps x the alignment unit) so that
// the CTAs fill whole waves of the GPU with as little imbalance as possible.
static int choose_split(const kvq_cache* C, const int32_t* lens, int unit, int slots, int max_chunks) {
  const int B = C->cfg.batch, H = C->cfg.kv_heads;
  long total = 0;
  int maxn = 0;
  for (int b = 0; b < B; ++b) {
    total += lens[b];
    maxn = std::max(maxn, (int)lens[b]);
  }
  if (maxn == 0) return 4 * unit;
  const int s_min_cap = round_up((maxn + max_chunks - 1) / max_chunks, 4 * unit);
  int best = 0;
  double best_cost = 1e300;
  auto eval = [&](int S) {
    if (S < s_min_cap) S = s_min_cap;
    long ctas = 0;
    for (int b = 0; b < B; ++b) ctas += (lens[b] + S - 1) / S;
    ctas *= H;
    const double waves = std::ceil((double)ctas / slots);
    // per-CTA fixed cost ~ 96 tokens of streaming
    const double cost = waves * (S + 96.0);
    if (cost < best_cost - 1e-9 || (std::fabs(cost - best_cost) < 1e-9 && S > best)) {
      best_cost = cost;
      best = S;
    }
  };
  const double ideal = (double)total * H / slots;
  for (int k = 1; k <= 4096; k *= 2) eval(4 * unit * k);
  for (int m = 1; m <= 8; ++m) eval(round_up((int)std::ceil(ideal / m), 4 * unit));
  return best;
}

cudaError_t launch_decode(kvq_cache* C, int layer, const void* q, int q_f32, float scale, float* out,
                          cudaStream_t st, int* launches) {
  Plan P;
  int occ = 1;
  cudaError_t e = make_plan(C, layer, &P, &occ);
  if (e != cudaSuccess) return e;
  DecodeArgs& a = P.a;
  const kvq_config& cfg = C->cfg;
  int unit = kTile;
  if (C->k.axis == 1) unit = std::max(unit, C->k.group);
  if (C->v.axis == 1) unit = std::max(unit, C->v.group);
  // plan on the host length mirror, raised to the plan hint (a launch planned
  // for the hint stays valid while the cache grows up to it)
  std::vector<int32_t> plan(C->lens.begin() + (long)layer * cfg.batch, C->lens.begin() + (long)(layer + 1) * cfg.batch);
  for (auto& x : plan) x = std::max(x, (int32_t)std::min(C->plan_tokens, C->cfg.max_tokens));
  const int32_t* lens = plan.data();
  const int slots = C->sm_count * occ;
  a.S = choose_split(C, lens, unit, slots, C->max_chunks);
  a.Sw = a.S / kWarps;
  int maxn = 0;
  for (int b = 0; b < cfg.batch; ++b) maxn = std::max(maxn, (int)lens[b]);
  const int nch = std::max(1, (maxn + a.S - 1) / a.S);
  a.q = q;
  a.q_f32 = q_f32;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  void* fn = pick_kernel(cfg.head_dim, cfg.q_heads / cfg.kv_heads == 8, C->v.axis);
  dim3 grid(nch, cfg.kv_heads, cfg.batch);
  void* args[] = {&a};
  e = cudaLaunchKernel(fn, grid, dim3(kWarps * 32), args, C->dec_smem, st);
  ++*launches;
  return e;
}

// Same plan and kernel as launch_decode, with the split-K partials and the
// combine tickets placed in caller-chosen scratch (used by the entry point
// whose scratch is a static device array).
cudaError_t launch_decode_scratch(kvq_cache* C, int layer, const void* q, int q_f32, float scale, float* out,
                                  cudaStream_t st, int* launches, float* work, uint32_t* tickets) {
  Plan P;
  int occ = 1;
  cudaError_t e = make_plan(C, layer, &P, &occ);
  if (e != cudaSuccess) return e;
  DecodeArgs& a = P.a;
  a.work = work;
  a.tickets = tickets;
  const kvq_config& cfg = C->cfg;
  int unit = kTile;
  if (C->k.axis == 1) unit = std::max(unit, C->k.group);
  if (C->v.axis == 1) unit = std::max(unit, C->v.group);
  std::vector<int32_t> plan(C->lens.begin() + (long)layer * cfg.batch, C->lens.begin() + (long)(layer + 1) * cfg.batch);
  for (auto& x : plan) x = std::max(x, (int32_t)std::min(C->plan_tokens, C->cfg.max_tokens));
  const int slots = C->sm_count * occ;
  a.S = choose_split(C, plan.data(), unit, slots, C->max_chunks);
  a.Sw = a.S / kWarps;
  int maxn = 0;
  for (int b = 0; b < cfg.batch; ++b) maxn = std::max(maxn, (int)plan[b]);
  const int nch = std::max(1, (maxn + a.S - 1) / a.S);
  a.q = q;
  a.q_f32 = q_f32;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  void* fn = pick_kernel(cfg.head_dim, cfg.q_heads / cfg.kv_heads == 8, C->v.axis);
  dim3 grid(nch, cfg.kv_heads, cfg.batch);
  void* args[] = {&a};
  e = cudaLaunchKernel(fn, grid, dim3(kWarps * 32), args, C->dec_smem, st);
  ++*launches;
  return e;
}

}  // namespace kvq
