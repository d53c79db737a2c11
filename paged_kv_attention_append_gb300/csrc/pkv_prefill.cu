// Tensor-core (tcgen05 + TMEM) causal prefill tiles.  Not enabled yet: the
// planner emits no prefill tiles, so every row runs on the split-KV kernel.
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {

int launch_prefill(const AttnArgs &a, int *launches) {
  (void)launches;
  return a.num_prefill_tiles > 0 ? (int)cudaErrorNotSupported : 0;
}

}  // namespace pkv
