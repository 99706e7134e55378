// markov_tc.cu -- tcgen05 Markov producer (placeholder until the tensor-core kernel lands).
#include "kernels.h"

namespace spec {

bool markov_tc_supported(int, int, int, int, const void*, const void*, const void*, const void*) {
  return false;
}

cudaError_t launch_markov_tc(const RowJob&, float*, float*, int*, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace spec
