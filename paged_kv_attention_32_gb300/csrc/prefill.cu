// Ragged causal prefill kernel (tcgen05 / TMEM).  Not built yet: the launcher
// reports PKA_ERR_UNSUPPORTED.
#include "host_common.h"
#include "prefill.h"

namespace pka {

int launch_prefill(const pka_prefill_plan&, const PrefillArgs&, const CUtensorMap&,
                   const CUtensorMap&, const CUtensorMap&, cudaStream_t) {
  return fail(PKA_ERR_UNSUPPORTED, "the prefill kernel is not built yet");
}

}  // namespace pka
