// SGMV shrink / expand on the tcgen05 tensor cores (prefill form). Not built yet:
// the launchers report "not supported" and the ABI answers LORA_EUNSUPPORTED for
// an explicit SGMV request, while AUTO runs every segment through BGMV.
#include "common.cuh"

namespace ra {

bool sgmv_supported() { return false; }

cudaError_t launch_sgmv_shrink(const lora_layer_desc &, const MetaView &, ListSel, const void *, int64_t,
                               float *, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t launch_sgmv_expand(const lora_layer_desc &, const MetaView &, ListSel, const float *, void *,
                               int64_t, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ra
