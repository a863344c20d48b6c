// attn_bwd.cu -- causal context-parallel attention backward (placeholder
// until the tcgen05 backward kernel lands).
#include "cp_attn.h"
#include "kernels.h"

namespace cpattn {

int launch_attn_bwd(const BwdArgs&, cudaStream_t) { return CP_ERR_UNSUPPORTED; }

}  // namespace cpattn
