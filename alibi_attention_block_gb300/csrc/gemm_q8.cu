// Q8_0 weights: the quantizer (weights -> int8 codes + fp16 scales) and the
// W8A16 GEMM C = A dequant(W)^T on tcgen05 tensor cores with the block's
// fused epilogues.
//
// Format: Q8_0 as published with GGML, the format the "RoFormer HIP FP32
// layout optimization" report names (BS-RoFormer Q8_0); the q8/int8 results
// are on "StableLM-2: partial RoPE ...", section 3 (Results) and "OLMo-2:
// reordered (post) normalization ...", section 4. Each row of W[N, K] is cut
// into blocks of 32 consecutive inputs; per block, in float32, d = absmax/127
// and codes q = round(w * (1/d)) (half away from zero), then d is stored as
// fp16. Here the codes are int8 q[N, K] row-major and the scales fp16
// d[K/32, N] block-major (one row of N scales per 32 inputs), so a tile's
// scales are rows of contiguous bytes that TMA can move.
//
// The GEMM (A bf16/fp16 [M, K], both operands K-major) is the K2 kernel with
// its B operand built on chip: TMA brings the A tile, the int8 code tile and
// the fp16 scales of one 64-wide k-block into a 4-stage ring; eight
// converter warps expand the codes to the storage type (q * d exactly in
// fp32, one rounding to the storage type) and write them in the
// 128-byte-swizzled K-major layout the MMA reads, into a 2-stage ring of B
// tiles. The conversion, not the tensor core, sets the pace: eight converter
// warps (two per scheduler) measured 6-11% faster than four with eight
// epilogue warps. 14 warps:
//   warp 0       TMA producer (A, codes, scales)
//   warp 1       TMEM allocator and single-thread MMA issuer (M=128, N=256,
//                K=16, fp32 accumulators double-buffered in TMEM)
//   warps 2..5   epilogue (the K2 epilogues: bias, residuals, SwiGLU, GELU,
//                QKV scatter with rotary), each warp both column halves of
//                its TMEM lane quarter
//   warps 6..13  converters
// Weight bytes per output element fall from 2 to 1 + 1/16 (codes + scales).
#include "gemm_epi.cuh"

namespace blk {

namespace {

using namespace gemm;

constexpr int kQBN = 256;                  // B tile rows (output columns, or gate|up rows)
constexpr int kConvWarps = 8;
constexpr int kQ8EpiWarps = 4;  // each takes both column halves of its lane quarter
constexpr int kQ8Threads = 64 + 32 * kQ8EpiWarps + 32 * kConvWarps;
constexpr int kTmaStages = 4;
constexpr int kBStages = 2;
constexpr int kABytes = kBM * kBK * 2;            // 16 KB
constexpr int kCodeBytes = kQBN * kBK;            // 16 KB of int8 codes
constexpr int kScaleBytes = 2 * kQBN * 2;         // two 32-input blocks x 256 rows of fp16
constexpr int kTmaStageBytes = kABytes + kCodeBytes + 1024;  // scales padded to 1 KB
constexpr int kBTileBytes = kQBN * kBK * 2;       // 32 KB, 128-byte swizzled
constexpr int kOffB = kTmaStages * kTmaStageBytes;
constexpr int kOffBar = kOffB + kBStages * kBTileBytes;
constexpr int kOffEpi = kOffBar + 256;
constexpr int kQ8Smem = kOffEpi + kQ8EpiWarps * 32 * 128 + 1024;
static_assert(kScaleBytes <= 1024, "scales exceed their slot");
static_assert(kTmaStageBytes % 1024 == 0 && kOffB % 1024 == 0, "tiles must stay 1 KB aligned");

struct Q8Maps {
    CUtensorMap q, q2;  // int8 codes [N, K]: gate (or the only weight) and up
    CUtensorMap d, d2;  // fp16 scales [K/32, N]
};

// 16 int8 codes and their scale -> 8 words of packed storage-type values
// q * d. A code byte u ^ 0x80 placed in the low byte of the float 2^23 gives
// 2^23 + 128 + q exactly; subtracting 2^23 + 128 leaves q.
template <typename T>
__device__ __forceinline__ void expand16(uint4 w, float d, uint32_t (&out)[8]) {
    const uint32_t words[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u,
                               w.w ^ 0x80808080u};
    const uint64_t bias2 = f2_pack(-8388736.0f, -8388736.0f);
    const uint64_t d2 = f2_pack(d, d);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float b0 = __uint_as_float(__byte_perm(words[i], 0x4B000000u, 0x7540));
        const float b1 = __uint_as_float(__byte_perm(words[i], 0x4B000000u, 0x7541));
        const float b2 = __uint_as_float(__byte_perm(words[i], 0x4B000000u, 0x7542));
        const float b3 = __uint_as_float(__byte_perm(words[i], 0x4B000000u, 0x7543));
        float q0, q1, q2, q3;
        // (b + bias) * d with one rounding each: q is exact, q * d is exact in
        // fp32 (7 + 11 significant bits), so the only rounding is the pack
        ffma2(b0, b1, f2_pack(1.f, 1.f), bias2, q0, q1);
        ffma2(b2, b3, f2_pack(1.f, 1.f), bias2, q2, q3);
        float v0, v1, v2, v3;
        ffma2(q0, q1, d2, f2_pack(0.f, 0.f), v0, v1);
        ffma2(q2, q3, d2, f2_pack(0.f, 0.f), v2, v3);
        out[2 * i] = dt_traits<T>::pack2(v0, v1);
        out[2 * i + 1] = dt_traits<T>::pack2(v2, v3);
    }
}

__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
}

template <typename T, int EPI, int ROT>
__global__ void __launch_bounds__(kQ8Threads, 1)
    gemm_q8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ Q8Maps qm,
                   const GemmArgs g, const __grid_constant__ RopeParams rp) {
    constexpr int BN = kQBN;
    constexpr int kBNOut = EPI == EPI_SWIGLU ? BN / 2 : BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + kOffBar;
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kTmaStages + i); };
    auto bfull = [&](int i) { return bar0 + 8u * (2 * kTmaStages + i); };
    auto bempty = [&](int i) { return bar0 + 8u * (2 * kTmaStages + kBStages + i); };
    auto tfull = [&](int i) { return bar0 + 8u * (2 * kTmaStages + 2 * kBStages + i); };
    auto tempty = [&](int i) { return bar0 + 8u * (2 * kTmaStages + 2 * kBStages + 2 + i); };
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * (2 * kTmaStages + 2 * kBStages + 4));
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTmaStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1 + kConvWarps);  // the MMA commit and every converter warp
        }
        for (int i = 0; i < kBStages; ++i) {
            mbar_init(bfull(i), kConvWarps);
            mbar_init(bempty(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull(i), 1);
            mbar_init(tempty(i), kQ8EpiWarps);
        }
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&qm.q);
        tma_prefetch_desc(&qm.d);
        if (EPI == EPI_SWIGLU) {
            tma_prefetch_desc(&qm.q2);
            tma_prefetch_desc(&qm.d2);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 2 * BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (g.pdl) {  // launched for programmatic dependent launch
        pdl_wait();  // inputs written by the previous kernel are visible from here on
        pdl_launch_dependents();
    }
    const int m_tiles = (g.M + kBM - 1) / kBM;
    const int n_tiles = (g.N + kBNOut - 1) / kBNOut;
    const int num_units = m_tiles * n_tiles;
    const int kb_count = (g.K + kBK - 1) / kBK;
    auto tile_of = [&](int u, int& mt, int& nt) {
        mt = g.n_fastest ? u / n_tiles : u % m_tiles;
        nt = g.n_fastest ? u % n_tiles : u / m_tiles;
    };
    if (warp == 0) {
        if (lane == 0) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
                int mt, nt;
                tile_of(u, mt, nt);
                // rows of the two 128-row halves of the B tile, in their maps
                const int r0 = EPI == EPI_SWIGLU ? nt * kBNOut : nt * BN;
                const int r1 = EPI == EPI_SWIGLU ? nt * kBNOut : nt * BN + BN / 2;
                const CUtensorMap* mq1 = EPI == EPI_SWIGLU ? &qm.q2 : &qm.q;
                const CUtensorMap* md1 = EPI == EPI_SWIGLU ? &qm.d2 : &qm.d;
                for (int kb = 0; kb < kb_count; ++kb) {
                    if (!mbar_wait(empty(st), ph ^ 1u, g.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + st * kTmaStageBytes;
                    const uint32_t sq = sa + kABytes;
                    const uint32_t sd = sq + kCodeBytes;
                    mbar_expect_tx(full(st), kABytes + kCodeBytes + kScaleBytes);
                    tma_load_2d(sa, &tmA, full(st), kb * kBK, mt * kBM);
                    tma_load_2d(sq, &qm.q, full(st), kb * kBK, r0);
                    tma_load_2d(sq + (BN / 2) * kBK, mq1, full(st), kb * kBK, r1);
                    tma_load_2d(sd, &qm.d, full(st), r0, kb * 2);
                    tma_load_2d(sd + kScaleBytes / 2, md1, full(st), r1, kb * 2);
                    if (++st == kTmaStages) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc_f16(dt_traits<T>::mma_fmt, kBM, BN, false);
            const uint64_t da0 = make_sdesc_sw128(sbase, 16, 1024);
            const uint64_t db0 = make_sdesc_sw128(sbase + kOffB, 16, 1024);
            constexpr uint64_t kAStep = kTmaStageBytes >> 4;
            constexpr uint64_t kBStep = kBTileBytes >> 4;
            int st = 0, bs = 0;
            uint32_t ph = 0, bph = 0;
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++it) {
                const int acc = it & 1;
                if (!mbar_wait(tempty(acc), ((it >> 1) & 1) ^ 1u, g.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < kb_count; ++kb) {
                    if (!mbar_wait(full(st), ph, g.err) || !mbar_wait(bfull(bs), bph, g.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = da0 + st * kAStep;
                    const uint64_t bd = db0 + bs * kBStep;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc_mma_ss(d_tmem, ad + k * 2, bd + k * 2, idesc, (kb > 0 || k != 0) ? 1u : 0u);
                    tc_commit(empty(st));
                    tc_commit(bempty(bs));
                    if (++st == kTmaStages) {
                        st = 0;
                        ph ^= 1u;
                    }
                    if (++bs == kBStages) {
                        bs = 0;
                        bph ^= 1u;
                    }
                }
                if (ok) tc_commit(tfull(acc));
            }
        }
    } else if (warp < 2 + kQ8EpiWarps) {
        const int ew = warp - 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t stg0 = sbase + kOffEpi;
        int it = 0;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++it) {
            const int acc = it & 1;
            if (!mbar_wait(tfull(acc), (it >> 1) & 1, g.err)) break;
            tc_fence_after();
            int mt, nt;
            tile_of(u, mt, nt);
            const uint32_t tbase =
                tmem_base + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
            for (int half = 0; half < 2; ++half)
                epilogue_tile<T, BN, EPI, ROT, false>(g, rp, tbase, mt * kBM + row, nt,
                                                      stg0 + ew * (32 * 128), lane,
                                                      mt * kBM + quarter * 32, nullptr, 0, row,
                                                      half);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(acc));
        }
    } else {
        // converters: 1024 16-byte chunks of codes per k-block, 4 per thread;
        // a warp's 32 chunks are 8 rows x 64 contiguous bytes
        const int tid = threadIdx.x - (64 + 32 * kQ8EpiWarps);
        int st = 0, bs = 0;
        uint32_t ph = 0, bph = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
            for (int kb = 0; kb < kb_count; ++kb) {
                if (!mbar_wait(full(st), ph, g.err) || !mbar_wait(bempty(bs), bph ^ 1u, g.err)) {
                    ok = false;
                    break;
                }
                const uint32_t sq = sbase + st * kTmaStageBytes + kABytes;
                const uint32_t sd = sq + kCodeBytes;
                const uint32_t sb = sbase + kOffB + bs * kBTileBytes;
                // all of this thread's loads first, then the arithmetic and
                // stores: two converter warps per scheduler have little else to
                // hide shared-memory latency behind
                constexpr int kIters = (BN * kBK / 16) / (32 * kConvWarps);
                const int c16 = tid & 3;   // 16 codes: k = 16 c16 .. 16 c16 + 15
                uint4 w[kIters];
                uint32_t dh[kIters];
#pragma unroll
                for (int i = 0; i < kIters; ++i) {
                    const int r = (i * (32 * kConvWarps) + tid) >> 2;  // B row
                    w[i] = ld_shared_u4(sq + r * kBK + c16 * 16);
                    // scale of 32-input block c16 / 2 of row r ([half][block][128] fp16)
                    dh[i] = ld_shared_u16(
                        sd + ((r >> 7) * (kScaleBytes / 4) + (c16 >> 1) * 128 + (r & 127)) * 2);
                }
#pragma unroll
                for (int i = 0; i < kIters; ++i) {
                    const int r = (i * (32 * kConvWarps) + tid) >> 2;
                    const float d =
                        __half2float(__ushort_as_half(static_cast<unsigned short>(dh[i])));
                    uint32_t o[8];
                    expand16<T>(w[i], d, o);
                    const uint32_t rb = sb + r * 128;
                    st_shared_v4(rb + (((2 * c16) ^ (r & 7)) << 4), o[0], o[1], o[2], o[3]);
                    st_shared_v4(rb + (((2 * c16 + 1) ^ (r & 7)) << 4), o[4], o[5], o[6], o[7]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bfull(bs));
                    mbar_arrive(empty(st));
                }
                if (++st == kTmaStages) {
                    st = 0;
                    ph ^= 1u;
                }
                if (++bs == kBStages) {
                    bs = 0;
                    bph ^= 1u;
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 2 * BN);
    }
}

template <typename T, int EPI, int ROT = 0>
cudaError_t launch_q8_cfg(const CUtensorMap& ta, const Q8Maps& qm, const GemmArgs& g,
                          const RopeParams& rp, int num_sms, cudaStream_t s) {
    constexpr int kBNOut = EPI == EPI_SWIGLU ? kQBN / 2 : kQBN;
    auto kern = gemm_q8_kernel<T, EPI, ROT>;
    const cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), kQ8Smem);
    if (e != cudaSuccess) return e;
    const int64_t units =
        static_cast<int64_t>((g.M + kBM - 1) / kBM) * ((g.N + kBNOut - 1) / kBNOut);
    const int64_t grid = units < num_sms ? units : num_sms;
    GemmArgs gp = g;
    gp.pdl = pdl_allowed(s);
    (void)launch_pdl(gp.pdl != 0, kern, dim3(static_cast<unsigned>(grid)), dim3(kQ8Threads), kQ8Smem,
                     s, ta, qm, gp, rp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_q8_t(DType dt, int epi, const void* a, const int8_t* q, const void* d,
                        const int8_t* q2, const void* d2, const GemmArgs& g, const RopeParams& rp,
                        int num_sms, cudaStream_t s) {
    CUtensorMap ta;
    Q8Maps qm;
    if (!make_tmap_2d(&ta, dt, a, g.M, g.K, kBM)) return cudaErrorInvalidValue;
    // codes [N, K] in 128-row x 64-byte boxes; scales [K/32, N] in 128 x 2 boxes
    if (!make_tmap_2d_plain(&qm.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q, g.N, g.K, kBK, kQBN / 2) ||
        !make_tmap_2d_plain(&qm.d, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, d, g.K / 32, g.N, kQBN / 2, 2))
        return cudaErrorInvalidValue;
    qm.q2 = qm.q;
    qm.d2 = qm.d;
    if (epi == EPI_SWIGLU &&
        (!make_tmap_2d_plain(&qm.q2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q2, g.N, g.K, kBK, kQBN / 2) ||
         !make_tmap_2d_plain(&qm.d2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, d2, g.K / 32, g.N, kQBN / 2,
                             2)))
        return cudaErrorInvalidValue;
    switch (epi) {
        case EPI_LINEAR: return launch_q8_cfg<T, EPI_LINEAR>(ta, qm, g, rp, num_sms, s);
        case EPI_SWIGLU: return launch_q8_cfg<T, EPI_SWIGLU>(ta, qm, g, rp, num_sms, s);
        case EPI_GELU: return launch_q8_cfg<T, EPI_GELU>(ta, qm, g, rp, num_sms, s);
        case EPI_QKV:
            switch (rp.span) {
                case 0: return launch_q8_cfg<T, EPI_QKV, 0>(ta, qm, g, rp, num_sms, s);
                case 16: return launch_q8_cfg<T, EPI_QKV, 16>(ta, qm, g, rp, num_sms, s);
                case 32: return launch_q8_cfg<T, EPI_QKV, 32>(ta, qm, g, rp, num_sms, s);
                default: return cudaErrorInvalidValue;
            }
        default: return cudaErrorInvalidValue;
    }
}

// One thread per (row n, 32-input block j), n fastest so that the scale
// stores of a warp are contiguous. The float32 steps are GGML's: d =
// absmax / 127, 1 / d, w * (1 / d), rounded half away from zero; d is
// stored in fp16 afterwards.
template <typename T>
__global__ void q8_quantize_kernel(const T* __restrict__ w, int64_t rows, int64_t cols,
                                   int8_t* __restrict__ q, __half* __restrict__ d) {
    const int64_t nblk = cols / 32;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= rows * nblk) return;
    const int64_t j = t / rows, n = t - j * rows;
    const T* src = w + n * cols + j * 32;
    float f[32];
#pragma unroll
    for (int v = 0; v < 4; ++v) load8(src + v * 8, *reinterpret_cast<float(*)[8]>(&f[v * 8]));
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
    const float d32 = __fdiv_rn(amax, 127.0f);
    const float inv = d32 > 0.f ? __fdiv_rn(1.0f, d32) : 0.f;
    uint32_t packed[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int code = static_cast<int>(roundf(__fmul_rn(f[4 * i + b], inv)));
            word |= (static_cast<uint32_t>(code) & 0xFFu) << (8 * b);
        }
        packed[i] = word;
    }
    uint4* dst = reinterpret_cast<uint4*>(q + n * cols + j * 32);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    d[j * rows + n] = __float2half_rn(d32);
}

// Dequantize once: W[n, k] = q[n, k] * d[k/32, n] in the storage type,
// written to memory for the dense GEMM (the path of large token counts,
// where the W8A16 kernel would expand every weight tile once per 128-row
// tile of x). The product is exact in fp32 and rounded once, as in the
// converter warps, so the two paths see the same weights. A block covers 32
// rows x 256 inputs of one matrix: the tile's 8 x 32 scales come in as
// contiguous 64-byte runs through shared memory, and each thread expands one
// 32-input block (two 16-byte code loads, 64 bytes written), eight threads
// per row, so that a warp reads and writes whole 256-byte row segments. (One
// thread per row and block, rows fastest, read 32 bytes from each of 32 rows
// K bytes apart per warp and reached ~2.2 TB/s.) One launch takes all of a
// block's matrices: the tiles of job i are blocks [tile0_i, tile0_{i+1}),
// 256-input column tiles fastest so that consecutive blocks read on along
// the same rows.
constexpr int kDqRows = 32, kDqBlocks = 8;

struct Q8DequantArgs {
    Q8DequantJob job[kQ8DequantMaxJobs];
    int64_t tile0[kQ8DequantMaxJobs];
    int n_jobs;
    int pdl;
};

template <typename T>
__global__ void __launch_bounds__(kDqRows * kDqBlocks) q8_dequant_kernel(const Q8DequantArgs a) {
    __shared__ float sc[kDqBlocks][kDqRows];
    if (a.pdl) {  // launched for programmatic dependent launch
        pdl_wait();
        pdl_launch_dependents();
    }
    // this block's matrix, picked with static indices only (indexing the
    // parameter arrays by a runtime value would copy them to local memory)
    const int64_t t = blockIdx.x;
    Q8DequantJob jb = a.job[0];
    int64_t lt = t;
#pragma unroll
    for (int i = 1; i < kQ8DequantMaxJobs; ++i)
        if (i < a.n_jobs && t >= a.tile0[i]) {
            jb = a.job[i];
            lt = t - a.tile0[i];
        }
    const int64_t nblk = jb.cols / 32;
    const int64_t tiles_k = (nblk + kDqBlocks - 1) / kDqBlocks;
    const int64_t n0 = (lt / tiles_k) * kDqRows;
    const int64_t j0 = (lt % tiles_k) * kDqBlocks;
    const __half* dsc = static_cast<const __half*>(jb.d);
    {
        const int jj = threadIdx.x / kDqRows, r = threadIdx.x % kDqRows;
        const int64_t n = n0 + r, j = j0 + jj;
        sc[jj][r] = n < jb.rows && j < nblk ? __half2float(dsc[j * jb.rows + n]) : 0.f;
    }
    __syncthreads();
    const int r = threadIdx.x / kDqBlocks, jj = threadIdx.x % kDqBlocks;
    const int64_t n = n0 + r, j = j0 + jj;
    if (n >= jb.rows || j >= nblk) return;
    const uint4* src = reinterpret_cast<const uint4*>(jb.q + n * jb.cols + j * 32);
    const uint4 c[2] = {src[0], src[1]};
    const float d = sc[jj][r];
    T* dst = static_cast<T*>(jb.w) + n * jb.cols + j * 32;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint32_t lo = v & 1 ? (v & 2 ? c[1].z : c[0].z) : (v & 2 ? c[1].x : c[0].x);
        const uint32_t hi = v & 1 ? (v & 2 ? c[1].w : c[0].w) : (v & 2 ? c[1].y : c[0].y);
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[e] = static_cast<float>(static_cast<int8_t>((lo >> (8 * e)) & 0xFFu)) * d;
            f[4 + e] = static_cast<float>(static_cast<int8_t>((hi >> (8 * e)) & 0xFFu)) * d;
        }
        store8(dst + v * 8, f);
    }
}

}  // namespace

cudaError_t launch_q8_dequant(DType dt, const Q8DequantJob* jobs, int n_jobs, cudaStream_t s) {
    if (n_jobs < 1 || n_jobs > kQ8DequantMaxJobs) return cudaErrorInvalidValue;
    Q8DequantArgs a{};
    int64_t tiles = 0;
    for (int i = 0; i < n_jobs; ++i) {
        a.job[i] = jobs[i];
        a.tile0[i] = tiles;
        const int64_t nblk = jobs[i].cols / 32;
        tiles += (jobs[i].rows + kDqRows - 1) / kDqRows * ((nblk + kDqBlocks - 1) / kDqBlocks);
    }
    if (tiles == 0) return cudaSuccess;
    if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
    a.n_jobs = n_jobs;
    a.pdl = pdl_allowed(s);
    const dim3 grid(static_cast<unsigned>(tiles)), block(kDqRows * kDqBlocks);
    if (dt == DType::F16)
        (void)launch_pdl(a.pdl != 0, q8_dequant_kernel<__half>, grid, block, 0, s, a);
    else
        (void)launch_pdl(a.pdl != 0, q8_dequant_kernel<__nv_bfloat16>, grid, block, 0, s, a);
    return cudaGetLastError();
}

cudaError_t launch_gemm_q8(DType dt, int epi, const void* a, const int8_t* q, const void* d,
                           const int8_t* q2, const void* d2, const GemmArgs& args,
                           const RopeParams& rp, int num_sms, cudaStream_t s) {
    if (args.M == 0 || args.N == 0) return cudaSuccess;
    GemmArgs g = args;
    const double a_bytes = 2.0 * args.M * args.K;
    const double b_bytes = 1.0625 * args.N * args.K * (epi == EPI_SWIGLU ? 2 : 1);
    g.n_fastest = a_bytes > 48.0 * (1 << 20) && a_bytes > b_bytes;
    g.split_s = 1;
    g.split_base = 0;
    g.split_ws = nullptr;
    g.split_cnt = nullptr;
    if (dt == DType::F16) return launch_q8_t<__half>(dt, epi, a, q, d, q2, d2, g, rp, num_sms, s);
    return launch_q8_t<__nv_bfloat16>(dt, epi, a, q, d, q2, d2, g, rp, num_sms, s);
}

cudaError_t launch_q8_quantize(DType dt, const void* w, int64_t rows, int64_t cols, int8_t* q,
                               void* d, cudaStream_t s) {
    const int64_t n = rows * (cols / 32);
    if (n == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((n + 255) / 256);
    if (dt == DType::F16)
        q8_quantize_kernel<__half><<<grid, 256, 0, s>>>(static_cast<const __half*>(w), rows, cols,
                                                         q, static_cast<__half*>(d));
    else
        q8_quantize_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(w), rows, cols, q, static_cast<__half*>(d));
    return cudaGetLastError();
}

}  // namespace blk
