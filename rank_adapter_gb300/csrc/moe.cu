// Composite (adapter, local expert) slot of every (token, choice) pair of a
// mixture-of-experts layer (page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section
// "MoE 的 LoRA:按专家挂载、融合 kernel 与 EP 切片"): the pairs, grouped by this
// slot through the ordinary token metadata, take the place of the pages'
// (adapter, expert) blocks of moe_lora_align_block_size.
#include "common.cuh"

namespace ra {
namespace {

struct MoeArgs {
  const int32_t *token_slot, *topk_ids, *expert_map;
  int32_t *pair_slot;
  int T, topk, num_loras, num_experts, local_experts;
};

__global__ void __launch_bounds__(256) moe_pair_slots_kernel(MoeArgs a) {
  // Inputs may come from the previous kernel; the output is read by the next
  // one before its wait, so this kernel releases it only by completing.
  pdl_wait();
  const int64_t n = (int64_t)a.T * a.topk;
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n; p += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(p / a.topk);
    const int s = a.token_slot[t], e = a.topk_ids[p];
    int out;
    if (s < 0 || s > a.num_loras || e < 0 || e >= a.num_experts) {
      out = -1;
    } else {
      const int el = a.expert_map != nullptr ? a.expert_map[e] : e;
      if (el >= a.local_experts) out = -1;
      else if (s == 0 || el < 0) out = 0;
      else out = 1 + (s - 1) * a.local_experts + el;
    }
    a.pair_slot[p] = out;
  }
}

}  // namespace

cudaError_t launch_moe_pair_slots(const int32_t *token_slot, const int32_t *topk_ids, int T, int topk, int num_loras,
                                  int num_experts, int local_experts, const int32_t *expert_map, int32_t *pair_slot,
                                  cudaStream_t st) {
  MoeArgs a{token_slot, topk_ids, expert_map, pair_slot, T, topk, num_loras, num_experts, local_experts};
  const int64_t n = (int64_t)T * topk;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 4 * 152);
  return launch_pdl(moe_pair_slots_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1u, a);
}

}  // namespace ra
