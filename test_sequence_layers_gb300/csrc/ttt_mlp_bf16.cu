// ttt_mlp_bf16.cu -- TTT-MLP forward on sm_103a (bf16 operands, fp32 state).
#include "ttt_internal.h"

namespace ttt {

int launch_mlp_bf16(const MlpArgs &, const CUtensorMap *) { return -2; }

}  // namespace ttt
