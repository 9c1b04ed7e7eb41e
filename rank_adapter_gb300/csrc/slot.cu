// Slot write / reset (set_lora / reset_lora of the vLLM page "vLLM 源码完全拆解(十八):
// 多 LoRA 服务", section "activate_adapter:把 CPU 上的低秩矩阵搬进 GPU 槽位"):
// copy one adapter's per-slice A [d_in, r] and B [r, d_out_s] into slot k of the
// stacked [num_slots, d_in, r_max] / [num_slots, r_max, d_out_s] buffers and
// zero the rank tail, so a rank-r adapter in an r_max table stays exact.
// Off the per-step path: it runs once per adapter activation.
#include "common.cuh"

namespace ra {
namespace {

struct SlotArgs {
  void *dstA[LORA_MAX_SLICES];        // slot k of A[s]
  void *dstB[LORA_MAX_SLICES];        // slot k of B[s]
  const void *srcA[LORA_MAX_SLICES];  // [d_in, rank] or NULL (zero the slice)
  const void *srcB[LORA_MAX_SLICES];  // [rank, out_s] or NULL
  int out_sizes[LORA_MAX_SLICES];
  int n_slices, d_in, r_max, rank, slot;
  float scale;
  int32_t *slot_rank;
  float *slot_scale;
};

// blockIdx.y = 2 * slice + {0: A, 1: B}. Each thread writes 8 consecutive
// destination elements with one vector store.
template <typename T>
__global__ void __launch_bounds__(256) slot_write_kernel(SlotArgs a) {
  pdl_wait();  // no early trigger: successors start only once the table is complete
  const int s = blockIdx.y >> 1;
  const bool isB = blockIdx.y & 1;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    a.slot_rank[a.slot] = a.rank;
    a.slot_scale[a.slot] = a.scale;
  }
  T *dst = static_cast<T *>(isB ? a.dstB[s] : a.dstA[s]);
  const T *src = static_cast<const T *>(isB ? a.srcB[s] : a.srcA[s]);
  const int rows = isB ? a.r_max : a.d_in;
  const int cols = isB ? a.out_sizes[s] : a.r_max;
  const int64_t nvec = (int64_t)rows * cols / 8;  // cols % 8 == 0
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = v * 8;
    const int i = (int)(e / cols);
    const int j0 = (int)(e % cols);
    float out[8];
    if (isB) {
      // B rows are contiguous in both layouts: rows < rank copy, the rest are 0.
      if (src != nullptr && i < a.rank) {
        load8_f32(src + (int64_t)i * cols + j0, out);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) out[q] = 0.f;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int j = j0 + q;
        out[q] = (src != nullptr && j < a.rank) ? Elem<T>::to_f(src[(int64_t)i * a.rank + j]) : 0.f;
      }
    }
    store8(dst + e, out);
  }
}

// Launched right after every slot write. Kernels of this library may start
// while their predecessor on the stream drains and read the slot table before
// their own dependency wait; this kernel waits for the slot write to complete
// and flush, and triggers nothing, so the next kernel starts only after the
// table is visible.
__global__ void slot_fence_kernel() { pdl_wait(); }

}  // namespace

cudaError_t launch_slot_write(const lora_layer_desc &d, int slot, int rank, float scale,
                              const void *const *A_src, const void *const *B_src, cudaStream_t st) {
  SlotArgs a{};
  const size_t es = d.dtype == LORA_BF16 ? 2 : 4;
  int64_t max_elems = 0;
  for (int s = 0; s < d.n_slices; ++s) {
    a.dstA[s] = static_cast<char *>(d.A[s]) + (size_t)slot * d.d_in * d.r_max * es;
    a.dstB[s] = static_cast<char *>(d.B[s]) + (size_t)slot * d.r_max * d.out_sizes[s] * es;
    a.srcA[s] = A_src ? A_src[s] : nullptr;
    a.srcB[s] = B_src ? B_src[s] : nullptr;
    a.out_sizes[s] = d.out_sizes[s];
    int64_t ea = (int64_t)d.d_in * d.r_max, eb = (int64_t)d.r_max * d.out_sizes[s];
    max_elems = ea > max_elems ? ea : max_elems;
    max_elems = eb > max_elems ? eb : max_elems;
  }
  a.n_slices = d.n_slices;
  a.d_in = d.d_in;
  a.r_max = d.r_max;
  a.rank = rank;
  a.slot = slot;
  a.scale = scale;
  a.slot_rank = d.slot_rank;
  a.slot_scale = d.slot_scale;
  int64_t blocks = (max_elems / 8 + 255) / 256;
  if (blocks > 1216) blocks = 1216;  // 8 CTAs per SM x 152 SMs, grid-stride beyond
  if (blocks < 1) blocks = 1;
  dim3 grid((unsigned)blocks, 2 * d.n_slices);
  cudaError_t e = d.dtype == LORA_BF16 ? launch_pdl(slot_write_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, 1u, a)
                                      : launch_pdl(slot_write_kernel<float>, grid, dim3(256), 0, st, 1u, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(slot_fence_kernel, dim3(1), dim3(32), 0, st, 1u);
}

}  // namespace ra
