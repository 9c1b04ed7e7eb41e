// Shared device helpers and internal launcher declarations for the sm_103a
// multi-LoRA kernels. Nothing here is part of the C ABI (include/lora.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "lora.h"

namespace ra {

// ------------------------------------------------------------------ element types

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ static inline float to_f(float v) { return v; }
  __device__ static inline float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static inline float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static inline __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// 8 consecutive elements widened to fp32 (one 16-byte vector of bf16, two of fp32).
__device__ __forceinline__ void load8_f32(const __nv_bfloat16 *p, float (&v)[8]) {
  uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8_f32(const float *p, float (&v)[8]) {
  float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// Plain (coherent) loads for buffers the same grid may also write (y).
__device__ __forceinline__ void load8_rw(const __nv_bfloat16 *p, float (&v)[8]) {
  uint4 u = *reinterpret_cast<const uint4 *>(p);
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8_rw(const float *p, float (&v)[8]) {
  float4 a = reinterpret_cast<const float4 *>(p)[0];
  float4 b = reinterpret_cast<const float4 *>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&v)[8]) {
  uint4 u;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(p) = u;
}
__device__ __forceinline__ void store8(float *p, const float (&v)[8]) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// ------------------------------------------------------------------ cluster / shared memory

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Full cluster barrier with release/acquire ordering of shared-memory writes.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Load a float4 from the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote) : "memory");
  return v;
}

// ------------------------------------------------------------------ asynchronous copies
// 16-byte global -> shared copies (cp.async, L2-only caching). Completion is
// waited for per commit group; no thread spins on memory.

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Ask the memory system to bring [p, p + bytes) into L2 (no completion to wait for).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// Wait until at most n of the most recently committed groups are still pending.
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  if (n <= 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
  else if (n == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
  else if (n == 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
  else asm volatile("cp.async.wait_group 3;" ::: "memory");
}

// ------------------------------------------------------------------ work lists (meta->tiles)
//
// int32 layout written by the metadata kernel and read by shrink / expand:
//   [0] n_all    LoRA segments (slot != 0)
//   [1] n_small  LoRA segments not on the large list
//   [2] n_large  LoRA segments with >= LORA_SGMV_MIN_ROWS tokens, when some LoRA
//                segment has >= LORA_AUTO_LONG_ROWS tokens (else none)
//   [3] tiles_all    sum over all LoRA segments of ceil(count / LORA_SGMV_TILE_M)
//   [4] tiles_large  the same over the large segments
//   [5..6] reserved (0)
//   [7] device error bits (0 when written; a kernel whose pipeline wait ran
//       out sets a bit, read back by lora_query_status)
//   then three lists of S = num_slots unit records (all, small, large), each
//   record 8 ints: {segment, slot, count, first sorted row, first 4 token rows}
//   (rows past the count are -1; unused records are all -1),
//   then S records indexed by slot (slot s's record of the "all" list, or all -1),
//   then all_tile_start[S+1] and large_tile_start[S+1] (cumulative tile counts),
//   then for each list, slot_rec[S]: the index of slot s's record in that list, or -1.
struct WorkLists {
  static constexpr int kHeader = 8;
  static constexpr int kRec = 8;
  static constexpr int kErrWord = 7;  // device error bits; kErrBadToken marks a token id outside the vocabulary
  __host__ __device__ static inline size_t ints(int S) {
    return kHeader + 4 * (size_t)kRec * S + 2 * ((size_t)S + 1) + 3 * (size_t)S;
  }
  __host__ __device__ static inline int list(int S, int which) { return kHeader + which * kRec * S; }
  __host__ __device__ static inline int by_slot(int S) { return kHeader + 3 * kRec * S; }
  __host__ __device__ static inline int all_tile_start(int S) { return kHeader + 4 * kRec * S; }
  __host__ __device__ static inline int large_tile_start(int S) { return kHeader + 4 * kRec * S + S + 1; }
  __host__ __device__ static inline int slot_rec(int S, int which) { return kHeader + 4 * kRec * S + 2 * (S + 1) + which * S; }
};

enum ListSel { kListAll = 0, kListSmall = 1, kListLarge = 2 };

// Error bit of the embedding lookup in the work lists' device error word: a
// token id was outside the vocabulary (its row got no delta). The other bits
// are pipeline waits that ran out.
constexpr int32_t kErrBadToken = 1 << 8;

// Device-side view of the metadata used by the compute kernels.
struct MetaView {
  const int32_t *sorted_rows;
  const int32_t *seg_slot;
  const int32_t *seg_count;
  const int32_t *seg_start;
  const int32_t *work;
  int32_t num_tokens;
  int32_t num_slots;
};

// ------------------------------------------------------------------ programmatic dependent launch
// Every kernel of this library is launched with programmatic stream
// serialization, so it may be scheduled while its predecessor on the stream
// drains. Each kernel therefore waits for the predecessor's completion (and
// memory flush) before it touches data a predecessor may still be writing.
// Protocol:
// * every slot write is followed by a fence kernel that waits for it and
//   never triggers early, so the slot table (A, B, ranks, scales) is complete
//   and visible whenever a later kernel starts;
// * every kernel waits before it exits, so a kernel's completion implies the
//   completion of everything before it on the stream;
// * the metadata kernel triggers its successor at once (it only sorts in
//   shared memory before its wait); an SGMV kernel launched right behind
//   this library's BGMV kernel of the same call triggers at once too and its
//   first CTA waits just before it exits (the families touch disjoint rows and
//   workspace parts, and everything older than the BGMV kernel is complete
//   when it starts); every other kernel triggers only after its own wait;
// * apart from those SGMV kernels, a kernel reads before its wait only the
//   slot table, and (the expand launched behind this library's shrink) the
//   metadata, which is then complete.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ host helpers

// Raise a kernel's dynamic shared-memory limit to at least `bytes` (per kernel and device).
cudaError_t set_max_dynamic_smem(const void *kernel, int bytes);

// Kernels this library has launched in the process (launch_pdl counts them).
void count_launch();

// Launch with programmatic stream serialization (see pdl_wait) and, when
// cluster_x > 1, thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e == cudaSuccess) count_launch();
  return e;
}

// ------------------------------------------------------------------ internal launchers
// Each returns a cudaError_t from the launch (cudaSuccess if nothing to launch).

cudaError_t launch_slot_write(const lora_layer_desc &d, int slot, int rank, float scale,
                              const void *const *A_src, const void *const *B_src, cudaStream_t st);
cudaError_t launch_prepare_meta(const lora_meta &m, cudaStream_t st, bool early = false);
// BGMV family (bgmv.cu). ws: chunk partials, bgmv_workspace_bytes() bytes (may be null when 0).
size_t bgmv_workspace_bytes(const lora_layer_desc &d, int max_tokens);
cudaError_t launch_bgmv_shrink(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const void *x,
                               int64_t ldx, float *buf, float *ws, cudaStream_t st);
cudaError_t launch_bgmv_expand(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const float *buf,
                               void *y, int64_t ldy, int y_dtype, cudaStream_t st);
cudaError_t launch_bgmv_apply(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const void *x,
                              int64_t ldx, float *buf, float *ws, void *y, int64_t ldy, int y_dtype,
                              cudaStream_t st);
// The expand half of launch_bgmv_apply's work and its shrink half, for callers
// that launch other kernels in between (AUTO batches with SGMV segments).
cudaError_t launch_bgmv_apply_shrink(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const void *x,
                                     int64_t ldx, float *buf, float *ws, cudaStream_t st);
cudaError_t launch_bgmv_apply_expand(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const float *ws,
                                     void *y, int64_t ldy, int y_dtype, cudaStream_t st);
// Embedding lookup (embed.cu): buf rows of the one-hot token ids, see lora_embed_shrink.
// Mixture-of-experts (moe.cu): composite slot of every (token, choice) pair.
cudaError_t launch_moe_pair_slots(const int32_t *token_slot, const int32_t *topk_ids, int T, int topk, int num_loras,
                                  int num_experts, int local_experts, const int32_t *expert_map, int32_t *pair_slot,
                                  cudaStream_t st);
cudaError_t launch_embed_shrink(const lora_layer_desc &d, const MetaView &mv, const int32_t *token_slot,
                                const int32_t *token_id, float *buf, cudaStream_t st);
// SGMV family (sgmv.cu, tcgen05). part: split partials, sgmv_workspace_bytes() bytes.
bool sgmv_supported();
// The pipelines' bounded wait, run against a barrier nothing arms (see lora_probe_bounded_wait).
cudaError_t launch_wait_probe(const MetaView &mv, uint32_t limit_us, cudaStream_t st);
size_t sgmv_workspace_bytes(const lora_layer_desc &d, int max_tokens);
// behind: launched right behind this library's BGMV kernel(s) of the same
// call over the other segments (the kernel then works before its wait).
cudaError_t launch_sgmv_shrink(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const void *x,
                               int64_t ldx, float *part, cudaStream_t st, bool behind = false);
cudaError_t launch_sgmv_reduce(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const float *part,
                               float *buf, cudaStream_t st);
// u_parts: u_src holds the shrink's split partials (else the u buffer [n_slices, T, r_max]).
cudaError_t launch_sgmv_expand(const lora_layer_desc &d, const MetaView &mv, ListSel sel, const float *u_src,
                               int u_parts, void *y, int64_t ldy, int y_dtype, cudaStream_t st, bool behind = false);

}  // namespace ra
