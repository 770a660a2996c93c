// K1: row norms. LayerNorm with bias ("StableLM-2: partial RoPE and a first
// LayerNorm-with-bias path", section 1) and RMSNorm ("OLMo-2: reordered (post)
// normalization", section 1), with an optional residual added after the norm
// (the OLMo-2 post-norm add). Inside the block the input or the residual may
// be the fp32 mid-block residual stream, and an fp32 copy of the output can be
// written alongside the storage-dtype one.
//
// HBM-bound: each row is read once into registers with 16-byte loads (a group
// of TPR threads per row, VPT 8-element vectors per thread), reduced with warp
// shuffles (plus shared memory when a row spans several warps), normalised
// from registers (two-pass mean/variance, fp32) and written once.
#include "internal.h"

namespace blk {

namespace {

constexpr int kNormThreads = 256;

template <int TPR>
__device__ __forceinline__ float row_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if constexpr (TPR > 32) {
        constexpr int kWarpsPerRow = TPR / 32;
        const int warp = threadIdx.x / 32;
        const int first = (warp / kWarpsPerRow) * kWarpsPerRow;
        __syncthreads();
        if ((threadIdx.x & 31) == 0) red[warp] = v;
        __syncthreads();
        v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarpsPerRow; ++w) v += red[first + w];
    }
    return v;
}

// T: gains/shifts; TX: input rows; TR: residual rows; y is T, y32 an
// optional fp32 copy of y.
template <typename T, typename TX, typename TR, int TPR, int VPT, bool RMS>
__global__ void __launch_bounds__(kNormThreads) norm_kernel(const TX* x,
                                                            const TR* __restrict__ res,
                                                            const T* __restrict__ gamma,
                                                            const T* __restrict__ beta,
                                                            T* y,
                                                            float* __restrict__ y32, int64_t rows,
                                                            int cols, float eps, int pdl) {
    __shared__ float red[kNormThreads / 32];
    if (pdl) {  // launched for programmatic dependent launch
        pdl_wait();
        pdl_launch_dependents();
    }
    constexpr int kRowsPerBlock = kNormThreads / TPR;
    const int sub = threadIdx.x % TPR;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + threadIdx.x / TPR;
    const bool active = row < rows;
    const int nvec = cols / 8;
    const TX* xr = x + (active ? row : 0) * cols;

    float v[VPT][8];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int vi = sub + i * TPR;
        if (active && vi < nvec) {
            load8(xr + vi * 8, v[i]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[i][e] = 0.f;
        }
    }
    // eight independent partial sums per thread keep the adds pipelined
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += v[i][e];
    const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    float mean = 0.f;
    if constexpr (!RMS) mean = row_sum<TPR>(sum, red) / static_cast<float>(cols);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int vi = sub + i * TPR;
        if (vi < nvec) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float c = v[i][e] - mean;
                acc[e] = fmaf(c, c, acc[e]);
            }
        }
    }
    const float sq = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    const float rstd = rsqrtf(row_sum<TPR>(sq, red) / static_cast<float>(cols) + eps);
    if (!active) return;
    T* yr = y + row * cols;
    float* y32r = y32 ? y32 + row * cols : nullptr;
    const TR* rr = res ? res + row * cols : nullptr;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int vi = sub + i * TPR;
        if (vi >= nvec) continue;
        float g[8], o[8];
        load8(gamma + vi * 8, g);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = (v[i][e] - mean) * rstd * g[e];
        if (!RMS && beta) {
            float b[8];
            load8(beta + vi * 8, b);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] += b[e];
        }
        if (rr) {
            float r[8];
            load8(rr + vi * 8, r);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] += r[e];
        }
        store8(yr + vi * 8, o);
        if (y32r) store8(y32r + vi * 8, o);
    }
}

template <typename T, typename TX, typename TR, int TPR, int VPT>
cudaError_t launch_tv(bool rms, const NormIO& io, const void* g, const void* b, int64_t rows,
                      int cols, float eps, cudaStream_t s) {
    constexpr int kRowsPerBlock = kNormThreads / TPR;
    const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    const bool pdl = pdl_allowed(s);
    auto go = [&](auto kern) {
        return launch_pdl(pdl, kern, dim3(static_cast<unsigned>(blocks)), dim3(kNormThreads), 0, s,
                          static_cast<const TX*>(io.x), static_cast<const TR*>(io.res),
                          static_cast<const T*>(g), static_cast<const T*>(b),
                          static_cast<T*>(io.y), io.y32, rows, cols, eps, pdl ? 1 : 0);
    };
    return rms ? go(norm_kernel<T, TX, TR, TPR, VPT, true>)
               : go(norm_kernel<T, TX, TR, TPR, VPT, false>);
}

template <typename T, typename TX, typename TR>
cudaError_t launch_t(bool rms, const NormIO& io, const void* g, const void* b, int64_t rows,
                     int cols, float eps, cudaStream_t s) {
    const int nvec = cols / 8;
    // At most four 8-element vectors per thread (measured: a 2048-wide bf16
    // row runs ~25% faster on two warps than on one), more threads for wider
    // rows.
#define BLK_NORM_CASE(TPR, VPT) \
    if (nvec <= (TPR) * (VPT)) return launch_tv<T, TX, TR, TPR, VPT>(rms, io, g, b, rows, cols, eps, s)
    BLK_NORM_CASE(32, 1);
    BLK_NORM_CASE(32, 2);
    BLK_NORM_CASE(32, 4);
    // fp32 rows up to 2048 wide: four warps of two vectors (64 bytes) per
    // thread, the bytes a 16-bit row's thread holds at four vectors. Measured
    // at 8192 x 2048: OLMo-2's post-norm over the fp32 attention output
    // 37.1 -> 33.4 us; on 16-bit rows the same split was slower (22.0 -> 22.4).
    if constexpr (sizeof(TX) == 4) BLK_NORM_CASE(128, 2);
    BLK_NORM_CASE(64, 4);
    BLK_NORM_CASE(128, 4);
    BLK_NORM_CASE(256, 4);
    BLK_NORM_CASE(256, 8);
#undef BLK_NORM_CASE
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_io(bool rms, const NormIO& io, const void* g, const void* b, int64_t rows,
                      int cols, float eps, cudaStream_t s) {
    if (io.x_f32 && io.res_f32) return launch_t<T, float, float>(rms, io, g, b, rows, cols, eps, s);
    if (io.x_f32) return launch_t<T, float, T>(rms, io, g, b, rows, cols, eps, s);
    if (io.res_f32) return launch_t<T, T, float>(rms, io, g, b, rows, cols, eps, s);
    return launch_t<T, T, T>(rms, io, g, b, rows, cols, eps, s);
}

}  // namespace

cudaError_t launch_norm(DType dt, bool rms, const NormIO& io, const void* gamma, const void* beta,
                        int64_t rows, int cols, float eps, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    if (dt == DType::F16) return launch_io<__half>(rms, io, gamma, beta, rows, cols, eps, s);
    return launch_io<__nv_bfloat16>(rms, io, gamma, beta, rows, cols, eps, s);
}

}  // namespace blk
