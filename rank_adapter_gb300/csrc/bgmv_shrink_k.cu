// Instantiations of the BGMV shrink kernel (see bgmv_kernels.cuh).
#include <map>
#include <mutex>
#include <tuple>

#include "bgmv_kernels.cuh"

namespace ra {
namespace bgmvk {
namespace {

// CTAs of a shrink kernel resident at once on the whole GPU (cached per kernel and shared-memory size).
int resident_ctas(const void *k, int smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void *, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(dev, k, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kSThreads, (size_t)smem) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return cache[key] = per_sm * sms;
}

template <typename TW, int NV>
cudaError_t launch_shrink_nv(const BgmvArgs &a0, cudaStream_t st) {
  auto k = bgmv_shrink_kernel<TW, NV>;
  cudaError_t e = set_max_dynamic_smem((const void *)k, a0.g.smem_shrink);
  if (e != cudaSuccess) return e;
  BgmvArgs a = a0;
  const int rows_per = a.by_slot ? a.mv.num_slots - 1 : a.max_items;
  const int64_t grid = (int64_t)rows_per * a.n_slices * a.g.kc_count;
  // (not for AUTO's short-segment list: there it measured no better)
  const int wave = a.by_slot && !a.small_only ? resident_ctas((const void *)k, a.g.smem_shrink) : 0;
  a.wave = wave > 0 && grid > wave ? wave : 0;
  return launch_pdl(k, dim3((unsigned)(rows_per * a.n_slices), (unsigned)a.g.kc_count), dim3(kSThreads),
                    (size_t)a.g.smem_shrink, st, 1u, a);
}

template <typename TW>
cudaError_t dispatch_shrink(const BgmvArgs &a, cudaStream_t st) {
  const int nv = a.g.r_max / Elem<TW>::kVec;
  if constexpr (sizeof(TW) == 2) {
    switch (nv) {
      case 1: return launch_shrink_nv<TW, 1>(a, st);
      case 2: return launch_shrink_nv<TW, 2>(a, st);
      case 4: return launch_shrink_nv<TW, 4>(a, st);
      case 8: return launch_shrink_nv<TW, 8>(a, st);
      case 16: return launch_shrink_nv<TW, 16>(a, st);
    }
  } else {
    switch (nv) {
      case 2: return launch_shrink_nv<TW, 2>(a, st);
      case 4: return launch_shrink_nv<TW, 4>(a, st);
      case 8: return launch_shrink_nv<TW, 8>(a, st);
      case 16: return launch_shrink_nv<TW, 16>(a, st);
      case 32: return launch_shrink_nv<TW, 32>(a, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t dispatch_shrink_bf16(const BgmvArgs &a, cudaStream_t st) { return dispatch_shrink<__nv_bfloat16>(a, st); }
cudaError_t dispatch_shrink_f32(const BgmvArgs &a, cudaStream_t st) { return dispatch_shrink<float>(a, st); }

}  // namespace bgmvk
}  // namespace ra
