// decode_latent.cu -- split-K decode attention over a latent (MLA-style)
// e4m3 cache on the tcgen05 tensor cores.  Not built yet: the entry point
// reports zero resident CTAs, which makes paged_decode_attn return
// KV_ERR_UNSUPPORTED for the latent layout.
#include "common.cuh"
#include "internal.h"

namespace kvfp8 {

int latent_split_ctas_per_sm() { return 0; }

cudaError_t launch_latent_split(const DecodeArgs&, cudaStream_t, int*) {
  return cudaErrorNotSupported;
}

}  // namespace kvfp8
