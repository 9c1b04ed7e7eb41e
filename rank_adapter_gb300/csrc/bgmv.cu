// Host side of the BGMV family: CTA geometry of a layer, work lists, and the
// launch sequences of lora_shrink / lora_expand / lora_apply (kernels in
// bgmv_kernels.cuh, instantiated by bgmv_shrink_k.cu and bgmv_expand_k.cu).
#include <map>
#include <mutex>
#include <utility>

#include "bgmv_kernels.cuh"

namespace ra {
namespace bgmvk {
namespace {

int align16(int v) { return (v + 15) & ~15; }

constexpr int kBySlotMaxWaves = 2;  // see fill_common

// Multiprocessors of the current device (cached per device).
int sm_count_cached() {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  return cache[dev] = n;
}

// Geometry of the shrink and expand CTAs for a layer.
Geo make_geo(const lora_layer_desc &d, bool wide = false) {
  Geo g{};
  const int es = d.dtype == LORA_BF16 ? 2 : 4;
  g.d_in = d.d_in;
  g.r_max = d.r_max;
  const int row_bytes = d.r_max * es;
  int sc = (kAStageBytes / row_bytes) & ~7;
  if (sc < 8) sc = 8;
  if (sc > d.d_in) sc = d.d_in;
  g.sc = sc;
  g.kchunk = kStretches * sc;
  g.kc_count = (d.d_in + g.kchunk - 1) / g.kchunk;
  int pw = ((wide ? 2 * kBPassBytes : kBPassBytes) / row_bytes) & ~7;
  if (pw < 8) pw = 8;
  int max_out = 0;
  for (int s = 0; s < d.n_slices; ++s) max_out = d.out_sizes[s] > max_out ? d.out_sizes[s] : max_out;
  if (pw > max_out) pw = max_out;
  g.pw = pw;
  g.a_stage = align16(sc * row_bytes);
  g.x_stage = align16(kTT * sc * es);
  int off = 0;
  g.off_rs = off;
  off += align16(2 * kSmallTable * 4);
  g.off_rows = off;
  off += align16(kRowsWin * 4);
  const int common = off;
  // shrink: ring + reduction buffer
  g.off_ring = off;
  off += kStretches * (g.a_stage + g.x_stage);
  g.off_red = off;
  off += align16(kSWarps * kTT * d.r_max * 4);
  g.smem_shrink = off;
  // expand: u of two passes (of up to kExpandNG tiles where the chunk is
  // narrow enough for tiles side by side), one B chunk (+ the zero partner
  // row of an odd rank)
  g.off_u = common;
  g.off_b = common + align16(2 * (pw * 2 <= kReach ? kExpandNG : 1) * kTT * d.r_max * 4);
  g.smem_expand = g.off_b + align16((d.r_max + 1) * pw * es);
  g.smem_reduce = common;
  return g;
}

void fill_common(BgmvArgs &a, const lora_layer_desc &d, const MetaView &mv, ListSel sel) {
  a.list = WorkLists::list(mv.num_slots, sel);
  // Slot-indexed shrink CTAs (A prefetched before the metadata is known) when
  // most slots are likely live in the list: a whole batch of at least one
  // token per slot, or AUTO's short segments when the batch averages fewer
  // than LORA_SGMV_MIN_ROWS tokens per slot (most slots are then short).
  const int S1 = mv.num_slots - 1;
  a.by_slot = (sel == kListAll && mv.num_tokens >= S1) ||
                      (sel == kListSmall && mv.num_tokens >= S1 && mv.num_tokens <= LORA_SGMV_MIN_ROWS * S1)
                  ? 1 : 0;
  a.small_only = sel == kListSmall ? 1 : 0;
  a.x_div = d.x_row_div > 1 ? d.x_row_div : 1;
  a.n_slices = d.n_slices;
  a.max_items = std::min(mv.num_slots - 1, mv.num_tokens);
  a.mv = mv;
  int off = 0;
  for (int s = 0; s < d.n_slices; ++s) {
    a.A[s] = d.A[s];
    a.B[s] = d.B[s];
    a.out_sizes[s] = d.out_sizes[s];
    a.out_off[s] = off;
    off += d.out_sizes[s];
    a.slice_order[s] = s;
  }
  for (int i = 1; i < d.n_slices; ++i)  // widest slices first
    for (int j = i; j > 0 && d.out_sizes[a.slice_order[j]] > d.out_sizes[a.slice_order[j - 1]]; --j)
      std::swap(a.slice_order[j], a.slice_order[j - 1]);
  a.slot_rank = d.slot_rank;
  a.slot_scale = d.slot_scale;
  for (int wide = 0; wide < 2; ++wide) {
    a.g = make_geo(d, wide != 0);
    int chunks = 0;
    for (int s = 0; s < d.n_slices; ++s) {
      a.chunk_start[s] = chunks;
      chunks += (d.out_sizes[s] + a.g.pw - 1) / a.g.pw;
    }
    a.chunk_start[d.n_slices] = chunks;
    if ((int64_t)chunks * a.max_items <= kWideGrid) break;  // a shallow expand grid keeps the narrow CTAs
  }
  // A slot-indexed shrink grid of a whole batch several waves deep gains
  // little from reading A before the metadata wait (only its first wave does)
  // and reads the A of every slot without tokens; such grids are
  // record-indexed instead (MoE step 124.9 -> 123.9 us). AUTO's short list
  // keeps its slot-indexed grid: there the first wave's early A measured
  // better (mixed batch 83.1 vs 84.8 us).
  if (a.by_slot && !a.small_only &&
      (int64_t)S1 * a.n_slices * a.g.kc_count > (int64_t)kBySlotMaxWaves * kSMinBlocks * sm_count_cached())
    a.by_slot = 0;
}

}  // namespace
}  // namespace bgmvk

using namespace bgmvk;

size_t bgmv_workspace_bytes(const lora_layer_desc &d, int max_tokens) {
  const Geo g = make_geo(d);
  if (max_tokens <= 0) return 0;
  return (size_t)d.n_slices * max_tokens * g.kc_count * d.r_max * sizeof(float);
}

cudaError_t launch_bgmv_shrink(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const void *x,
                               int64_t ldx, float *buf, float *ws, cudaStream_t st) {
  if (std::min(mv.num_slots - 1, mv.num_tokens) <= 0) return cudaSuccess;
  BgmvArgs a{};
  fill_common(a, d, mv, sel);
  a.x = x;
  a.ldx = ldx;
  a.buf = buf;
  a.part = ws;
  a.to_parts = a.g.kc_count > 1;  // one chunk: the CTA writes u rows itself
  cudaError_t e = d.dtype == LORA_BF16 ? dispatch_shrink_bf16(a, st) : dispatch_shrink_f32(a, st);
  if (e != cudaSuccess || !a.to_parts) return e;
  a.u_in = ws;
  return launch_reduce(a, st);
}

cudaError_t launch_bgmv_apply_shrink(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const void *x,
                                     int64_t ldx, float *buf, float *ws, cudaStream_t st) {
  if (std::min(mv.num_slots - 1, mv.num_tokens) <= 0) return cudaSuccess;
  BgmvArgs a{};
  fill_common(a, d, mv, sel);
  a.x = x;
  a.ldx = ldx;
  a.part = ws;
  a.buf = buf;
  a.to_parts = 1;  // the expand forms u from the partials; buf is optional
  cudaError_t e = d.dtype == LORA_BF16 ? dispatch_shrink_bf16(a, st) : dispatch_shrink_f32(a, st);
  if (e != cudaSuccess || buf == nullptr) return e;
  a.u_in = ws;  // the caller also wants the u rows
  return launch_reduce(a, st);
}

cudaError_t launch_bgmv_apply_expand(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const float *ws,
                                     void *y, int64_t ldy, int y_dtype, cudaStream_t st) {
  if (std::min(mv.num_slots - 1, mv.num_tokens) <= 0) return cudaSuccess;
  BgmvArgs a{};
  fill_common(a, d, mv, sel);
  a.u_in = ws;
  a.u_parts = 1;
  a.pre = 1;
  a.y = y;
  a.ldy = ldy;
  return launch_expand(a, d.dtype, y_dtype, st);
}

cudaError_t launch_bgmv_apply(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const void *x,
                              int64_t ldx, float *buf, float *ws, void *y, int64_t ldy, int y_dtype,
                              cudaStream_t st) {
  cudaError_t e = launch_bgmv_apply_shrink(d, mv, sel, x, ldx, buf, ws, st);
  if (e != cudaSuccess) return e;
  return launch_bgmv_apply_expand(d, mv, sel, ws, y, ldy, y_dtype, st);
}

cudaError_t launch_bgmv_expand(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const float *buf,
                               void *y, int64_t ldy, int y_dtype, cudaStream_t st) {
  if (std::min(mv.num_slots - 1, mv.num_tokens) <= 0) return cudaSuccess;
  BgmvArgs a{};
  fill_common(a, d, mv, sel);
  a.u_in = buf;
  a.u_parts = 0;
  a.y = y;
  a.ldy = ldy;
  return launch_expand(a, d.dtype, y_dtype, st);
}

}  // namespace ra
