// attn_tc.cu — tensor-core sliding-window attention (placeholder until the
// tensor-core kernels land): reports "not supported".
#include "kernels.h"

namespace ttt {
int attn_fwd_tc(const AttnArgs&, cudaStream_t) { return (int)cudaErrorNotSupported; }
int attn_bwd_tc(const AttnArgs&, cudaStream_t) { return (int)cudaErrorNotSupported; }
}  // namespace ttt
