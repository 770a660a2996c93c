// K7: token-embedding gather for the model-level wrap (model.cu).
#pragma once
#include "internal.h"

namespace blk {

// x[t, :] = table[tokens[t], :] for t < n_tokens (hidden % 8 == 0, rows
// 16-byte aligned); ids outside [0, vocab) read row 0.
cudaError_t launch_embed_gather(DType dt, const int32_t* tokens, const void* table, void* x,
                                int64_t n_tokens, int hidden, int64_t vocab, int num_sms,
                                cudaStream_t s);

}  // namespace blk
