// Host side of the C ABI declared in include/lora.h: argument validation,
// dispatch to the kernel families, status codes. Nothing here allocates
// device memory or keeps state between calls beyond per-(kernel, device)
// launch attributes.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <map>
#include <utility>

#include "common.cuh"

namespace ra {

namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

cudaError_t set_max_dynamic_smem(const void *kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void *, int>, int> granted;  // (kernel, device) -> limit set so far
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = granted.find({kernel, dev});
  if (it != granted.end() && it->second >= bytes) return cudaSuccess;
  if (bytes <= 48 * 1024) return cudaSuccess;  // within the default limit
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) granted[{kernel, dev}] = bytes;
  return e;
}

}  // namespace ra

namespace {

thread_local int g_last_cuda_error = 0;

// Clear a launch error left in this library's runtime state by an earlier
// failed call, so that it is not reported against the next one.
void clear_stale_error() { (void)cudaGetLastError(); }

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return LORA_OK;
  g_last_cuda_error = (int)e;
  return LORA_ECUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_size(int dtype) { return dtype == LORA_BF16 ? 2 : 4; }

int check_desc(const lora_layer_desc *d) {
  if (d == nullptr) return LORA_EINVAL;
  if (d->dtype != LORA_F32 && d->dtype != LORA_BF16) return LORA_EINVAL;
  if (d->n_slices < 1 || d->n_slices > LORA_MAX_SLICES) return LORA_ERANGE;
  if (d->d_in < 8 || d->d_in % 8 != 0) return LORA_EINVAL;
  if (d->r_max < 8 || d->r_max > LORA_MAX_RANK || (d->r_max & (d->r_max - 1)) != 0) return LORA_ERANGE;
  if (d->num_slots < 1 || d->num_slots > LORA_MAX_NUM_SLOTS) return LORA_ERANGE;
  for (int s = 0; s < d->n_slices; ++s) {
    if (d->out_sizes[s] < 8 || d->out_sizes[s] % 8 != 0) return LORA_EINVAL;
    if (d->A[s] == nullptr || d->B[s] == nullptr) return LORA_EINVAL;
    if (!aligned16(d->A[s]) || !aligned16(d->B[s])) return LORA_EALIGN;
  }
  if (d->slot_rank == nullptr || d->slot_scale == nullptr) return LORA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(d->slot_rank) & 3u) || (reinterpret_cast<uintptr_t>(d->slot_scale) & 3u))
    return LORA_EALIGN;
  if (d->x_row_div < 0) return LORA_EINVAL;
  return LORA_OK;
}

int check_meta(const lora_meta *m) {
  if (m == nullptr) return LORA_EINVAL;
  if (m->num_slots < 1 || m->num_slots > LORA_MAX_NUM_SLOTS) return LORA_ERANGE;
  if (m->num_tokens < 0 || m->num_tokens > LORA_MAX_TOKENS) return LORA_ERANGE;
  if (m->num_tokens > 0 && (m->token_slot == nullptr || m->sorted_rows == nullptr)) return LORA_EINVAL;
  if (!m->seg_slot || !m->seg_count || !m->seg_start || !m->num_segs || !m->no_lora || !m->status || !m->tiles)
    return LORA_EINVAL;
  if (m->tiles_bytes < lora_meta_tiles_bytes(m->num_slots)) return LORA_EINVAL;
  if (!aligned16(m->tiles)) return LORA_EALIGN;
  return LORA_OK;
}

// The SGMV family exists for bf16 tables with r_max >= 16 (the MMA N / K granularity).
bool sgmv_available(const lora_layer_desc *d) {
  return d->dtype == LORA_BF16 && d->r_max >= 16 && ra::sgmv_supported();
}

// AUTO sends its large segments to SGMV only in batches of at least
// LORA_AUTO_SGMV_MIN_TOKENS tokens that average at least
// LORA_AUTO_SGMV_MIN_AVG tokens per adapter slot; other batches run entirely on BGMV.
bool auto_uses_sgmv(const lora_layer_desc *d, int num_tokens) {
  return num_tokens >= LORA_AUTO_SGMV_MIN_TOKENS &&
         (int64_t)num_tokens >= (int64_t)LORA_AUTO_SGMV_MIN_AVG * (d->num_slots - 1) && sgmv_available(d);
}

// Which families a (kind, batch) runs and where their scratch lives in the
// workspace: [BGMV chunk partials | SGMV split partials (256-byte aligned)].
struct Plan {
  bool bgmv, sgmv, split;  // split: AUTO with segments on both families
  size_t bgmv_bytes, sgmv_off, sgmv_bytes, total;
};

Plan plan_of(const lora_layer_desc *d, int num_tokens, int kind) {
  Plan p{};
  p.sgmv = kind == LORA_SGMV || (kind == LORA_AUTO && auto_uses_sgmv(d, num_tokens)) ||
           (kind == LORA_MIXED && sgmv_available(d));
  p.bgmv = kind != LORA_SGMV;
  p.split = p.bgmv && p.sgmv;
  p.bgmv_bytes = p.bgmv ? ra::bgmv_workspace_bytes(*d, num_tokens) : 0;
  p.sgmv_off = (p.bgmv_bytes + 255) & ~(size_t)255;
  p.sgmv_bytes = p.sgmv ? ra::sgmv_workspace_bytes(*d, num_tokens) : 0;
  p.total = p.sgmv_bytes ? p.sgmv_off + p.sgmv_bytes : p.bgmv_bytes;
  return p;
}

int check_ws(const Plan &p, const void *ws, size_t ws_bytes) {
  if (p.total == 0) return LORA_OK;
  if (ws == nullptr || ws_bytes < p.total) return LORA_EINVAL;
  if (!aligned16(ws)) return LORA_EALIGN;
  return LORA_OK;
}

ra::MetaView view_of(const lora_meta *m) {
  ra::MetaView v;
  v.sorted_rows = m->sorted_rows;
  v.seg_slot = m->seg_slot;
  v.seg_count = m->seg_count;
  v.seg_start = m->seg_start;
  v.work = static_cast<const int32_t *>(m->tiles);
  v.num_tokens = m->num_tokens;
  v.num_slots = m->num_slots;
  return v;
}

}  // namespace

extern "C" {

const char *lora_strerror(int status) {
  switch (status) {
    case LORA_OK: return "success";
    case LORA_EINVAL: return "invalid argument (null pointer, shape or size mismatch)";
    case LORA_ERANGE: return "value out of range (slot, rank, num_slots, num_tokens or n_slices)";
    case LORA_EALIGN: return "pointer or leading dimension not 16-byte aligned";
    case LORA_EUNSUPPORTED: return "unsupported combination (e.g. SGMV on an fp32 table)";
    case LORA_ECUDA: return "CUDA launch or copy failed (see lora_last_cuda_error)";
    case LORA_EBADSLOT: return "some token slot ids were outside [0, num_slots) and were treated as slot 0";
    case LORA_EDEVICE: return "a kernel stopped waiting on its own pipeline; the outputs since the last lora_prepare_meta are invalid";
    case LORA_EBADTOKEN: return "some token ids were outside the embedding vocabulary; their rows got no delta";
    default: return "unknown lora_status";
  }
}

int lora_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t lora_launch_count(void) { return ra::g_launches.load(std::memory_order_relaxed); }

size_t lora_meta_tiles_bytes(int32_t num_slots) {
  if (num_slots < 1) return 0;
  return ra::WorkLists::ints(num_slots) * sizeof(int32_t);
}

size_t lora_workspace_bytes(const lora_layer_desc *desc, int32_t max_tokens, int32_t kind) {
  if (check_desc(desc) != LORA_OK || max_tokens <= 0) return 0;
  if (kind != LORA_AUTO && kind != LORA_BGMV && kind != LORA_SGMV && kind != LORA_MIXED) return 0;
  if (kind == LORA_SGMV && !sgmv_available(desc)) return 0;
  return plan_of(desc, max_tokens, kind).total;
}

int lora_set_slot(const lora_layer_desc *desc, int32_t slot, int32_t rank, float scale,
                  const void *const *A_src, const void *const *B_src, lora_stream_t stream) {
  clear_stale_error();
  int st = check_desc(desc);
  if (st != LORA_OK) return st;
  if (slot < 1 || slot >= desc->num_slots) return LORA_ERANGE;
  if (rank < 1 || rank > desc->r_max) return LORA_ERANGE;
  if (A_src == nullptr || B_src == nullptr) return LORA_EINVAL;
  for (int s = 0; s < desc->n_slices; ++s) {
    if ((A_src[s] == nullptr) != (B_src[s] == nullptr)) return LORA_EINVAL;
    if (B_src[s] != nullptr && !aligned16(B_src[s])) return LORA_EALIGN;
    if (A_src[s] != nullptr && (reinterpret_cast<uintptr_t>(A_src[s]) % elem_size(desc->dtype))) return LORA_EALIGN;
  }
  return cuda_status(ra::launch_slot_write(*desc, slot, rank, scale, A_src, B_src, (cudaStream_t)stream));
}

int lora_reset_slot(const lora_layer_desc *desc, int32_t slot, lora_stream_t stream) {
  clear_stale_error();
  int st = check_desc(desc);
  if (st != LORA_OK) return st;
  if (slot < 1 || slot >= desc->num_slots) return LORA_ERANGE;
  return cuda_status(ra::launch_slot_write(*desc, slot, 0, 0.f, nullptr, nullptr, (cudaStream_t)stream));
}

int lora_prepare_meta(const lora_meta *meta, lora_stream_t stream) {
  clear_stale_error();
  int st = check_meta(meta);
  if (st != LORA_OK) return st;
  return cuda_status(ra::launch_prepare_meta(*meta, (cudaStream_t)stream));
}

int lora_prepare_meta_unshared(const lora_meta *meta, lora_stream_t stream) {
  clear_stale_error();
  int st = check_meta(meta);
  if (st != LORA_OK) return st;
  return cuda_status(ra::launch_prepare_meta(*meta, (cudaStream_t)stream, true));
}

int lora_shrink(const lora_layer_desc *desc, const lora_meta *meta, const void *x, int64_t ldx,
                float *buf, int32_t kind, void *ws, size_t ws_bytes, lora_stream_t stream) {
  clear_stale_error();
  int st = check_desc(desc);
  if (st != LORA_OK) return st;
  st = check_meta(meta);
  if (st != LORA_OK) return st;
  if (meta->num_slots != desc->num_slots) return LORA_EINVAL;
  if (kind != LORA_AUTO && kind != LORA_BGMV && kind != LORA_SGMV && kind != LORA_MIXED) return LORA_EINVAL;
  if (kind == LORA_SGMV && !sgmv_available(desc)) return LORA_EUNSUPPORTED;
  if (meta->num_tokens == 0) return LORA_OK;
  if (x == nullptr || buf == nullptr) return LORA_EINVAL;
  if (ldx < desc->d_in) return LORA_EINVAL;
  if (!aligned16(x) || !aligned16(buf) || (ldx * (int64_t)elem_size(desc->dtype)) % 16 != 0) return LORA_EALIGN;
  const Plan p = plan_of(desc, meta->num_tokens, kind);
  st = check_ws(p, ws, ws_bytes);
  if (st != LORA_OK) return st;
  const ra::MetaView mv = view_of(meta);
  cudaStream_t s = (cudaStream_t)stream;
  float *wb = static_cast<float *>(ws);
  float *wsg = reinterpret_cast<float *>(static_cast<char *>(ws) + p.sgmv_off);
  if (!p.sgmv) return cuda_status(ra::launch_bgmv_shrink(*desc, mv, ra::kListAll, x, ldx, buf, wb, s));
  const ra::ListSel sel = p.split ? ra::kListLarge : ra::kListAll;
  if (p.split) {
    st = cuda_status(ra::launch_bgmv_shrink(*desc, mv, ra::kListSmall, x, ldx, buf, wb, s));
    if (st != LORA_OK) return st;
  }
  st = cuda_status(ra::launch_sgmv_shrink(*desc, mv, sel, x, ldx, wsg, s, p.split));
  if (st != LORA_OK) return st;
  return cuda_status(ra::launch_sgmv_reduce(*desc, mv, sel, wsg, buf, s));
}

int lora_expand(const lora_layer_desc *desc, const lora_meta *meta, const float *buf, void *y,
                int64_t ldy, int32_t y_dtype, int32_t kind, lora_stream_t stream) {
  clear_stale_error();
  int st = check_desc(desc);
  if (st != LORA_OK) return st;
  st = check_meta(meta);
  if (st != LORA_OK) return st;
  if (meta->num_slots != desc->num_slots) return LORA_EINVAL;
  if (kind != LORA_AUTO && kind != LORA_BGMV && kind != LORA_SGMV && kind != LORA_MIXED) return LORA_EINVAL;
  if (y_dtype != LORA_F32 && y_dtype != LORA_BF16) return LORA_EINVAL;
  if (desc->dtype == LORA_F32 && y_dtype != LORA_F32) return LORA_EUNSUPPORTED;
  if (kind == LORA_SGMV && !sgmv_available(desc)) return LORA_EUNSUPPORTED;
  if (meta->num_tokens == 0) return LORA_OK;
  if (y == nullptr || buf == nullptr) return LORA_EINVAL;
  int64_t total = 0;
  for (int s = 0; s < desc->n_slices; ++s) total += desc->out_sizes[s];
  if (ldy < total) return LORA_EINVAL;
  if (!aligned16(y) || !aligned16(buf) || (ldy * (int64_t)elem_size(y_dtype)) % 16 != 0) return LORA_EALIGN;
  const Plan p = plan_of(desc, meta->num_tokens, kind);
  const ra::MetaView mv = view_of(meta);
  cudaStream_t s = (cudaStream_t)stream;
  if (!p.sgmv) return cuda_status(ra::launch_bgmv_expand(*desc, mv, ra::kListAll, buf, y, ldy, y_dtype, s));
  if (p.split) {
    st = cuda_status(ra::launch_bgmv_expand(*desc, mv, ra::kListSmall, buf, y, ldy, y_dtype, s));
    if (st != LORA_OK) return st;
  }
  return cuda_status(ra::launch_sgmv_expand(*desc, mv, p.split ? ra::kListLarge : ra::kListAll, buf, 0, y, ldy,
                                            y_dtype, s, p.split));
}

int lora_apply(const lora_layer_desc *desc, const lora_meta *meta, const void *x, int64_t ldx, float *buf,
               void *y, int64_t ldy, int32_t y_dtype, int32_t kind, void *ws, size_t ws_bytes,
               lora_stream_t stream) {
  clear_stale_error();
  int st = check_desc(desc);
  if (st != LORA_OK) return st;
  st = check_meta(meta);
  if (st != LORA_OK) return st;
  if (meta->num_slots != desc->num_slots) return LORA_EINVAL;
  if (kind != LORA_AUTO && kind != LORA_BGMV && kind != LORA_SGMV && kind != LORA_MIXED) return LORA_EINVAL;
  if (y_dtype != LORA_F32 && y_dtype != LORA_BF16) return LORA_EINVAL;
  if (desc->dtype == LORA_F32 && y_dtype != LORA_F32) return LORA_EUNSUPPORTED;
  if (kind == LORA_SGMV && !sgmv_available(desc)) return LORA_EUNSUPPORTED;
  if (meta->num_tokens == 0) return LORA_OK;
  if (x == nullptr || y == nullptr) return LORA_EINVAL;
  int64_t total = 0;
  for (int s = 0; s < desc->n_slices; ++s) total += desc->out_sizes[s];
  if (ldx < desc->d_in || ldy < total) return LORA_EINVAL;
  if (!aligned16(x) || !aligned16(y) || (buf != nullptr && !aligned16(buf)) ||
      (ldx * (int64_t)elem_size(desc->dtype)) % 16 != 0 || (ldy * (int64_t)elem_size(y_dtype)) % 16 != 0)
    return LORA_EALIGN;
  const Plan p = plan_of(desc, meta->num_tokens, kind);
  st = check_ws(p, ws, ws_bytes);
  if (st != LORA_OK) return st;
  const ra::MetaView mv = view_of(meta);
  cudaStream_t s = (cudaStream_t)stream;
  float *wb = static_cast<float *>(ws);
  float *wsg = reinterpret_cast<float *>(static_cast<char *>(ws) + p.sgmv_off);
  if (!p.sgmv)
    return cuda_status(ra::launch_bgmv_apply(*desc, mv, ra::kListAll, x, ldx, buf, wb, y, ldy, y_dtype, s));
  const ra::ListSel sel = p.split ? ra::kListLarge : ra::kListAll;
  // Both shrinks first, then both expands: each expand reads partials that
  // are at least one launch old.
  if (p.split) {
    st = cuda_status(ra::launch_bgmv_apply_shrink(*desc, mv, ra::kListSmall, x, ldx, buf, wb, s));
    if (st != LORA_OK) return st;
  }
  st = cuda_status(ra::launch_sgmv_shrink(*desc, mv, sel, x, ldx, wsg, s, p.split));
  if (st != LORA_OK) return st;
  if (buf != nullptr) {
    st = cuda_status(ra::launch_sgmv_reduce(*desc, mv, sel, wsg, buf, s));
    if (st != LORA_OK) return st;
  }
  if (p.split) {
    st = cuda_status(ra::launch_bgmv_apply_expand(*desc, mv, ra::kListSmall, wb, y, ldy, y_dtype, s));
    if (st != LORA_OK) return st;
  }
  return cuda_status(ra::launch_sgmv_expand(*desc, mv, sel, wsg, 1, y, ldy, y_dtype, s, p.split));
}

int lora_query_status(const lora_meta *meta, int32_t *out, lora_stream_t stream) {
  if (meta == nullptr || meta->status == nullptr || out == nullptr) return LORA_EINVAL;
  int32_t v[2] = {0, 0};
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&v[0], meta->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && meta->tiles != nullptr)
    e = cudaMemcpyAsync(&v[1], static_cast<const int32_t *>(meta->tiles) + ra::WorkLists::kErrWord, sizeof(int32_t),
                        cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e);
  *out = v[0];
  if ((v[1] & ~ra::kErrBadToken) != 0) return LORA_EDEVICE;
  if (v[1] != 0) return LORA_EBADTOKEN;
  return v[0] == 0 ? LORA_OK : LORA_EBADSLOT;
}

int lora_probe_bounded_wait(const lora_meta *meta, uint32_t limit_us, lora_stream_t stream) {
  clear_stale_error();
  const int st = check_meta(meta);
  if (st != LORA_OK) return st;
  if (limit_us < 1 || limit_us > 1000000) return LORA_ERANGE;
  return cuda_status(ra::launch_wait_probe(view_of(meta), limit_us, (cudaStream_t)stream));
}

int lora_embed_shrink(const lora_layer_desc *desc, const lora_meta *meta, const int32_t *token_id, float *buf,
                      lora_stream_t stream) {
  clear_stale_error();
  int st = check_desc(desc);
  if (st != LORA_OK) return st;
  st = check_meta(meta);
  if (st != LORA_OK) return st;
  if (meta->num_slots != desc->num_slots || desc->n_slices != 1) return LORA_EINVAL;
  if (meta->num_tokens == 0) return LORA_OK;
  if (token_id == nullptr || buf == nullptr) return LORA_EINVAL;
  if (!aligned16(buf) || reinterpret_cast<uintptr_t>(token_id) % sizeof(int32_t) != 0) return LORA_EALIGN;
  return cuda_status(ra::launch_embed_shrink(*desc, view_of(meta), meta->token_slot, token_id, buf,
                                             (cudaStream_t)stream));
}

int lora_moe_pair_slots(const int32_t *token_slot, const int32_t *topk_ids, int32_t num_tokens, int32_t topk,
                        int32_t num_loras, int32_t num_experts, int32_t local_experts, const int32_t *expert_map,
                        int32_t *pair_slot, lora_stream_t stream) {
  clear_stale_error();
  if (topk < 1 || topk > 64 || num_tokens < 0 || (int64_t)num_tokens * topk > LORA_MAX_TOKENS) return LORA_ERANGE;
  if (num_loras < 0 || num_experts < 1 || local_experts < 1 || local_experts > num_experts) return LORA_ERANGE;
  if (1 + (int64_t)num_loras * local_experts > LORA_MAX_NUM_SLOTS) return LORA_ERANGE;
  if (num_tokens == 0) return LORA_OK;
  if (token_slot == nullptr || topk_ids == nullptr || pair_slot == nullptr) return LORA_EINVAL;
  auto misaligned = [](const void *p) { return reinterpret_cast<uintptr_t>(p) % sizeof(int32_t) != 0; };
  if (misaligned(token_slot) || misaligned(topk_ids) || misaligned(pair_slot) ||
      (expert_map != nullptr && misaligned(expert_map)))
    return LORA_EALIGN;
  return cuda_status(ra::launch_moe_pair_slots(token_slot, topk_ids, num_tokens, topk, num_loras, num_experts,
                                               local_experts, expert_map, pair_slot, (cudaStream_t)stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free shrink.
//
// Some callers cannot allocate device memory at the point where they run the
// shrink: code that executes inside another framework's memory pool or under
// an allocator that forbids new device allocations, or latency-critical
// serving paths that must not call into an allocator at all. For them this
// entry point keeps the shrink's per-chunk partial rows in a fixed array
// that is part of the library's device image instead of a caller-provided
// workspace. Every GPU that loads the library holds this array (8 MiB) until
// the process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB of partial rows
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// Device address of g_noalloc_scratch on the current device. In host code the
// array's name only stands in for the symbol, so the address is looked up
// (once per device, with that device current) and cached.
cudaError_t noalloc_scratch(float **out) {
  static std::mutex mu;
  static std::map<int, float *> addr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = addr.find(dev);
  if (it == addr.end()) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    it = addr.emplace(dev, static_cast<float *>(p)).first;
  }
  *out = it->second;
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t lora_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int lora_shrink_noalloc(const lora_layer_desc *desc, const lora_meta *meta, const void *x, int64_t ldx, float *buf,
                        lora_stream_t stream) {
  clear_stale_error();
  int st = check_desc(desc);
  if (st != LORA_OK) return st;
  st = check_meta(meta);
  if (st != LORA_OK) return st;
  if (meta->num_slots != desc->num_slots) return LORA_EINVAL;
  if (meta->num_tokens == 0) return LORA_OK;
  if (x == nullptr || buf == nullptr) return LORA_EINVAL;
  if (ldx < desc->d_in) return LORA_EINVAL;
  if (!aligned16(x) || !aligned16(buf) || (ldx * (int64_t)elem_size(desc->dtype)) % 16 != 0) return LORA_EALIGN;
  if (ra::bgmv_workspace_bytes(*desc, meta->num_tokens) > kNoAllocScratchBytes) return LORA_ERANGE;
  float *scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(
      ra::launch_bgmv_shrink(*desc, view_of(meta), ra::kListAll, x, ldx, buf, scratch, (cudaStream_t)stream));
}

}  // extern "C"
