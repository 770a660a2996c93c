// K3 dispatch: causal softmax attention by head_dim and group size.
//   head_dim 64            attn_pair.cu     (two query tiles per item; any GQA)
//   head_dim 128, MHA      attn_pair128.cu  (two query tiles, shared S buffer)
//   head_dim 128, GQA      attn_gqa.cu      (the group's query heads packed
//   head_dim 160, any      attn_gqa.cu       into one 128-row tile)
#include "internal.h"

namespace blk {

cudaError_t launch_attention(DType dt, const AttnArgs& a, cudaStream_t s) {
    if (a.B == 0 || a.S == 0) return cudaSuccess;
    switch (a.d) {
        case 64: return launch_attention_pair64(dt, a, s);
        case 128:
            return a.H == a.Hk ? launch_attention_pair128(dt, a, s) : launch_attention_gqa(dt, a, s);
        case 160: return launch_attention_gqa(dt, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace blk
