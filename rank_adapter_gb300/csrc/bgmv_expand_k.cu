// Instantiations of the BGMV expand kernel and the split path's reduce kernel (see bgmv_kernels.cuh).
#include "bgmv_kernels.cuh"

namespace ra {
namespace bgmvk {
namespace {

// Split path: u rows of every token of a unit from its chunk partials. Grid: max_items * n_slices.
__global__ void __launch_bounds__(kThreads) bgmv_reduce_kernel(BgmvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_wait();
  pdl_trigger();
  const int item = (int)blockIdx.x % a.max_items;
  const int slice = a.slice_order[blockIdx.x / a.max_items];
  int *rows = reinterpret_cast<int *>(smem + a.g.off_rows);
  Unit u;
  if (!load_unit(a, item, u, smem, rows)) return;
  const int r_max = a.g.r_max;
  for (int i = threadIdx.x; i < u.cnt * r_max; i += kThreads) {
    const int t = i / r_max, k = i - t * r_max;
    const int row = a.mv.sorted_rows[u.start + t];
    a.buf[((int64_t)slice * a.mv.num_tokens + row) * r_max + k] = u_from_partials(a, slice, u.start + t, k, u);
  }
}

}  // namespace

cudaError_t launch_expand(const BgmvArgs &a, int dtype, int y_dtype, cudaStream_t st) {
  void (*k)(BgmvArgs);
  const bool groups = a.g.pw * 2 <= kReach;  // column chunks that leave threads idle: tiles side by side
  if (dtype == LORA_BF16 && y_dtype == LORA_BF16)
    k = groups ? bgmv_expand_kernel<__nv_bfloat16, __nv_bfloat16, true>
               : bgmv_expand_kernel<__nv_bfloat16, __nv_bfloat16, false>;
  else if (dtype == LORA_BF16)
    k = groups ? bgmv_expand_kernel<__nv_bfloat16, float, true> : bgmv_expand_kernel<__nv_bfloat16, float, false>;
  else
    k = groups ? bgmv_expand_kernel<float, float, true> : bgmv_expand_kernel<float, float, false>;
  cudaError_t e = set_max_dynamic_smem((const void *)k, a.g.smem_expand);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3((unsigned)a.chunk_start[a.n_slices], (unsigned)a.max_items), dim3(kThreads),
                    (size_t)a.g.smem_expand, st, 1u, a);
}

cudaError_t launch_reduce(const BgmvArgs &a, cudaStream_t st) {
  return launch_pdl(bgmv_reduce_kernel, dim3((unsigned)(a.max_items * a.n_slices)), dim3(kThreads),
                    (size_t)a.g.smem_reduce, st, 1u, a);
}

}  // namespace bgmvk
}  // namespace ra
