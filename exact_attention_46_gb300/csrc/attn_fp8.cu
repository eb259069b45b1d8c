// attn_fp8.cu -- E4M3 instantiations of the fused attention forward (D = 64, 128, 256;
// with and without the causal mask).  The kernel itself is in attn_kernel.cuh.
#include "attn_kernel.cuh"

namespace ea46 {
#define EA46_INST(D, CAUSAL)                                                                 \
  template cudaError_t launch_attn<D, true, CAUSAL>(const CUtensorMap&, const CUtensorMap&, \
                                                    const CUtensorMap&, const CUtensorMap&, const AttnParams&,  \
                                                    cudaStream_t, const SplitParams*);
EA46_INST(64, false)
EA46_INST(64, true)
EA46_INST(128, false)
EA46_INST(128, true)
EA46_INST(256, false)
EA46_INST(256, true)
#undef EA46_INST
}  // namespace ea46
