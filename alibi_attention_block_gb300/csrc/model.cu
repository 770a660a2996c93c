// K7: token-embedding gather for the model-level wrap: x[t, :] =
// embed[tokens[t], :] ("Bloom in a sovereign engine", Contribution; nnterp
// "stablelm" Printout: embed_tokens). HBM bound: one 16-byte load and store
// per 8 elements, a row per group of threads. Token ids come from device
// memory; an id outside [0, vocab) is clamped to row 0 so nothing outside the
// table is read.
#include "model.h"

namespace blk {

namespace {

template <typename T>
__global__ void __launch_bounds__(256) embed_gather_kernel(const int32_t* tokens, const T* table,
                                                           T* x, int64_t n_tokens, int hidden,
                                                           int64_t vocab) {
    const int vpr = hidden / 8;  // 16-byte vectors per row
    const int64_t total = n_tokens * vpr;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / vpr;
        const int c = static_cast<int>(i - t * vpr);
        int64_t id = tokens[t];
        if (id < 0 || id >= vocab) id = 0;
        const uint4 v = *reinterpret_cast<const uint4*>(table + id * hidden + c * 8);
        *reinterpret_cast<uint4*>(x + t * hidden + c * 8) = v;
    }
}

}  // namespace

cudaError_t launch_embed_gather(DType dt, const int32_t* tokens, const void* table, void* x,
                                int64_t n_tokens, int hidden, int64_t vocab, int num_sms,
                                cudaStream_t s) {
    if (n_tokens == 0) return cudaSuccess;
    const int64_t total = n_tokens * (hidden / 8);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (dt == DType::F16)
        embed_gather_kernel<__half><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            tokens, static_cast<const __half*>(table), static_cast<__half*>(x), n_tokens, hidden,
            vocab);
    else
        embed_gather_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            tokens, static_cast<const __nv_bfloat16*>(table), static_cast<__nv_bfloat16*>(x),
            n_tokens, hidden, vocab);
    return cudaGetLastError();
}

}  // namespace blk
