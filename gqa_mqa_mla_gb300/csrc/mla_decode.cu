// mla_decode.cu -- absorbed MLA decode partial kernel (tcgen05 / TMEM).
#include "internal.h"
#include "ptx.cuh"

namespace decattn {

cudaError_t launch_mla_partial(const MlaParams&, const CUtensorMap&, const CUtensorMap&,
                               const CUtensorMap&, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace decattn
