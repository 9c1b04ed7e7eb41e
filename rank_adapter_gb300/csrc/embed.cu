// Embedding LoRA (page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section
// "embedding 的 LoRA 是一个查表增量"): for an embedding layer the shrink is a
// row lookup in the stacked A table -- slot a's r-vector for token id v is row
// v of A[a] ([num_slots, vocab, r_max], the page's lora_a_stacked; the page
// indexes the flattened table at v + a * vocab) -- and the expand that follows
// is the ordinary one. The lookup is lora_shrink's arithmetic for the one-hot
// row of v: buf[0, t, k] = scale[a] * A[a][v, k] for k < rank a, 0 for the
// rank tail, rows of slot-0 tokens not written.
#include <algorithm>

#include "common.cuh"

namespace ra {
namespace {

constexpr int kEmbThreads = 256;
constexpr int kEmbMaxBlocks = 1184;  // 8 per SM on 152 SMs; the work is a few rows per token

// One thread per (token, rank index): consecutive threads read consecutive
// elements of a row. An id outside the vocabulary gives a zero row (no delta)
// and sets the work lists' bad-token bit, reported by lora_query_status.
template <typename TW>
__global__ void __launch_bounds__(kEmbThreads) embed_shrink_kernel(const TW *A, const int32_t *token_slot,
                                                                   const int32_t *token_id,
                                                                   const int32_t *slot_rank,
                                                                   const float *slot_scale, float *buf,
                                                                   int32_t *work, int T, int S, int vocab,
                                                                   int r_max) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)T * r_max;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / r_max), k = (int)(i - (int64_t)t * r_max);
    const int a = token_slot[t];
    if (a <= 0 || a >= S) continue;  // no LoRA (ids outside the table count as slot 0): row not written
    const int v = token_id[t];
    const int r_a = min(max(slot_rank[a], 0), r_max);
    float val = 0.f;
    if (v < 0 || v >= vocab) {
      if (k == 0) atomicOr(&work[WorkLists::kErrWord], kErrBadToken);
    } else if (k < r_a) {
      val = slot_scale[a] * Elem<TW>::to_f(A[((int64_t)a * vocab + v) * r_max + k]);
    }
    buf[i] = val;
  }
}

}  // namespace

cudaError_t launch_embed_shrink(const lora_layer_desc &d, const MetaView &mv, const int32_t *token_slot,
                                const int32_t *token_id, float *buf, cudaStream_t st) {
  if (mv.num_tokens <= 0) return cudaSuccess;
  const int64_t total = (int64_t)mv.num_tokens * d.r_max;
  const int grid = (int)std::min<int64_t>((total + kEmbThreads - 1) / kEmbThreads, kEmbMaxBlocks);
  int32_t *work = const_cast<int32_t *>(mv.work);
  if (d.dtype == LORA_BF16)
    return launch_pdl(embed_shrink_kernel<__nv_bfloat16>, dim3((unsigned)grid), dim3(kEmbThreads), 0, st, 1u,
                      static_cast<const __nv_bfloat16 *>(d.A[0]), token_slot, token_id,
                      (const int32_t *)d.slot_rank, (const float *)d.slot_scale, buf, work, mv.num_tokens,
                      mv.num_slots, d.d_in, d.r_max);
  return launch_pdl(embed_shrink_kernel<float>, dim3((unsigned)grid), dim3(kEmbThreads), 0, st, 1u,
                    static_cast<const float *>(d.A[0]), token_slot, token_id, (const int32_t *)d.slot_rank,
                    (const float *)d.slot_scale, buf, work, mv.num_tokens, mv.num_slots, d.d_in, d.r_max);
}

}  // namespace ra
