// K2: C = A B^T on tcgen05 tensor cores, with the block's epilogues fused.
//
// A [M, K] (activations) and B [N, K] (a torch-convention weight W[out, in])
// are both K-major. Persistent kernel, one CTA per SM, 10 warps:
//   warp 0      TMA producer: 128x64 A tile and BNx64 B tile per stage
//               (128-byte swizzle) into a STAGES-deep shared-memory ring
//   warp 1      TMEM allocator and single-thread MMA issuer:
//               tcgen05.mma.cta_group::1.kind::f16, M=128, N=BN, K=16 per
//               instruction, fp32 accumulators in TMEM, double-buffered so
//               the epilogue of tile i overlaps the mainloop of tile i+1
//   warps 2..9  epilogue, two warps per TMEM lane quarter (a warp reaches
//               the quarter of its index mod 4), each with half of the tile's
//               columns: tcgen05.ld 32 lanes x 32 columns per load (one
//               thread per output row), fused op, 16-byte global stores per
//               row; fp32 outputs go through 4 KB of shared memory per warp
//               so that each store instruction writes whole lines
// When the work units end in a partial round, the units of that round may
// be split in two along K (long K only): each half publishes an fp32
// partial tile and the half that finishes second sums both and runs the
// epilogue (a separate kernel instance; see launch_cfg).
// Epilogues (the block's steps after each projection):
//   EPI_LINEAR  + bias, + up to two residuals (o_proj and down_proj residual
//               adds); residuals and output may be fp32 (the block keeps its
//               mid-block residual stream in fp32)
//   EPI_SWIGLU  B tile = [gate rows | up rows]; out = silu(gate) * up
//               (nnterp "stablelm" 02 support(): mlp_neurons = act(gate)*up)
//   EPI_GELU    gelu_tanh(acc + bias) (Bloom's MLP)
//   EPI_QKV     + bias, optional partial NeoX rotary on q/k heads (span 16 or 32),
//               scatter of the [M, (H+2Hk)d] projection into head-split q, k, v
//               for stacked or per-head interleaved ([head][q,k,v][d]) rows
//               ("Bloom in a sovereign engine", Contribution: de-interleave).
#include "gemm_epi.cuh"

namespace blk {

namespace {

using namespace gemm;

template <int BN>
struct GemmCfg {
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBarBytes = 256;
    static constexpr int kEpiBytes = kEpiWarps * 32 * 128;  // per epilogue warp: 32 rows x 32 fp32
    static constexpr int kSmem = kStages * kStageBytes + 1024 + kBarBytes + kEpiBytes;
    static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
};

// Every CTA loads its own A and B tiles with plain (per-CTA) TMA loads.
template <typename T, int BN, int EPI, int ROT, bool SPLIT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB2, const GemmArgs g,
                const __grid_constant__ RopeParams rp) {
    using Cfg = GemmCfg<BN>;
    constexpr int kStages = Cfg::kStages;
    constexpr int kBNOut = EPI == EPI_SWIGLU ? BN / 2 : BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * Cfg::kStageBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kStages + i); };
    auto tfull = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
    auto tempty = [&](int i) { return bar0 + 8u * (2 * kStages + 2 + i); };
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull(i), 1);
            mbar_init(tempty(i), kEpiWarps);
        }
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (EPI == EPI_SWIGLU) tma_prefetch_desc(&tmB2);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
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
    // work units (output tiles), numbered M-fastest (the CTAs running at any
    // time share a few columns of B and all of A stays in L2) or, when A is
    // too large to stay in L2, N-fastest (they share rows of A, read from
    // DRAM once; B stays in L2)
    const int m_units = m_tiles;
    const int num_units = m_units * n_tiles;
    const int unit0 = static_cast<int>(blockIdx.x);
    const int unit_step = static_cast<int>(gridDim.x);
    const int kb_count = (g.K + kBK - 1) / kBK;
    const int num_work =
        SPLIT ? g.split_base + (num_units - g.split_base) * g.split_s : num_units;
    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int v = unit0; v < num_work && ok; v += unit_step) {
                const Unit un = decode_unit<SPLIT>(g, v, kb_count);
                const int u = un.u;
                const int mt = g.n_fastest ? u / n_tiles : u % m_units;
                const int nt = g.n_fastest ? u % n_tiles : u / m_units;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!mbar_wait(empty(stage), phase ^ 1u, g.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + stage * Cfg::kStageBytes;
                    const uint32_t sb = sa + Cfg::kABytes;
                    mbar_expect_tx(full(stage), Cfg::kStageBytes);
                    tma_load_2d(sa, &tmA, full(stage), kb * kBK, mt * kBM);
                    if constexpr (EPI == EPI_SWIGLU) {
                        tma_load_2d(sb, &tmB, full(stage), kb * kBK, nt * kBNOut);
                        tma_load_2d(sb + (BN / 2) * 128, &tmB2, full(stage), kb * kBK, nt * kBNOut);
                    } else {
                        tma_load_2d(sb, &tmB, full(stage), kb * kBK, nt * BN);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc_f16(dt_traits<T>::mma_fmt, kBM, BN, false);
            const uint64_t da0 = make_sdesc_sw128(sbase, 16, 1024);
            const uint64_t db0 = make_sdesc_sw128(sbase + Cfg::kABytes, 16, 1024);
            constexpr uint64_t kStageStep = Cfg::kStageBytes >> 4;
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int v = unit0; v < num_work && ok; v += unit_step, ++it) {
                const Unit un = decode_unit<SPLIT>(g, v, kb_count);
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!mbar_wait(tempty(acc), acc_phase ^ 1u, g.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!mbar_wait(full(stage), phase, g.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = da0 + stage * kStageStep;
                    const uint64_t bd = db0 + stage * kStageStep;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc_mma_ss(d_tmem, ad + k * 2, bd + k * 2, idesc,
                                  (kb > un.kb0 || k != 0) ? 1u : 0u);
                    tc_commit(empty(stage));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit(tfull(acc));
            }
        }
    } else {
        // epilogue warp ew: TMEM lanes 32 (warp % 4) .. +31 (a warp reaches
        // only the lane quarter of its index mod 4), columns of half ew / 4
        const int ew = warp - 2;
        const int quarter = warp & 3;
        const int half = ew / 4;
        const int row = quarter * 32 + lane;
        const uint32_t stg0 = smem_u32(smem) + kStages * Cfg::kStageBytes + Cfg::kBarBytes;
        int it = 0;
        for (int v = unit0; v < num_work; v += unit_step, ++it) {
            const Unit un = decode_unit<SPLIT>(g, v, kb_count);
            const int u = un.u;
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            if (!mbar_wait(tfull(acc), acc_phase, g.err)) break;
            tc_fence_after();
            const int mt = g.n_fastest ? u / n_tiles : u % m_units;
            const int nt = g.n_fastest ? u % n_tiles : u / m_units;
            const uint32_t tbase =
                tmem_base + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
            const float* part = nullptr;
            unsigned* cnt = nullptr;
            if (SPLIT && v >= g.split_base) {
                // a segment of a split unit: publish this warp's 32 rows of
                // the partial tile ([column][row], coalesced per column), then
                // count the warp in; the warp that arrives last for these
                // rows sums every segment and runs the epilogue
                const int t = (v - g.split_base) / g.split_s;
                float* slot0 = g.split_ws + static_cast<size_t>(t * g.split_s) * (kBM * BN);
                float* mine = slot0 + static_cast<size_t>(un.q) * (kBM * BN) + row;
#pragma unroll 1
                for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
                    uint32_t r[32];
                    tmem_ld32(tbase + c * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        __stcg(mine + (c * 32 + i) * kBM, __uint_as_float(r[i]));
                }
                __threadfence();
                __syncwarp();
                cnt = g.split_cnt + (t * kEpiWarps + ew);
                unsigned old = 0;
                if (lane == 0) old = atomicAdd(cnt, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old != static_cast<unsigned>(g.split_s - 1)) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty(acc));
                    continue;
                }
                __threadfence();  // the other segments' partials are visible
                part = slot0;
            }
            epilogue_tile<T, BN, EPI, ROT, SPLIT>(g, rp, tbase, mt * kBM + row, nt,
                                                  stg0 + ew * (32 * 128), lane,
                                                  mt * kBM + quarter * 32, part, un.q, row, half);
            if (cnt && lane == 0) *cnt = 0u;  // every segment has arrived: ready for the next launch
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(acc));
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

template <typename T, int BN, int EPI, int ROT = 0>
cudaError_t launch_cfg(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb2,
                       const GemmArgs& g, const RopeParams& rp, int num_sms, cudaStream_t s) {
    using Cfg = GemmCfg<BN>;
    constexpr int kBNOut = EPI == EPI_SWIGLU ? BN / 2 : BN;
    // the split instance exists only where a split is possible
    constexpr bool kCanSplit = EPI != EPI_SWIGLU;
    auto kern = gemm_kernel<T, BN, EPI, ROT, false>;
    auto kern_split = gemm_kernel<T, BN, EPI, ROT, kCanSplit>;
    cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), Cfg::kSmem);
    if (e == cudaSuccess && kCanSplit)
        e = set_smem_attr_once(reinterpret_cast<const void*>(kern_split), Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t units = static_cast<int64_t>((g.M + kBM - 1) / kBM) * ((g.N + kBNOut - 1) / kBNOut);
    const int64_t grid_units = units < num_sms ? units : num_sms;
    const dim3 grid(static_cast<unsigned>(grid_units), 1, 1);
    // With scratch, split each unit of a last round that would leave at
    // least half of the CTAs idle (G units per round, R <= G/2 in the last)
    // into two halves along K, when each half still has at least
    // kSplitMinKb k-blocks: the unit that finishes second reads the other's
    // partial tile back from L2, one round trip per 32 columns, which only a
    // long mainloop pays for (measured: the down projections gain, shorter
    // K loses).
    GemmArgs ga = g;
    ga.split_s = 1;
    ga.split_base = 0;
    const bool pdl = pdl_allowed(s);
    ga.pdl = pdl;
    if (kCanSplit && g.split_ws && g.split_cnt) {
        const int64_t G = grid_units;
        const int64_t rounds = (units + G - 1) / G;
        const int64_t R = units - (rounds - 1) * G;
        const int64_t sp = 2;
        const int64_t kb_count = (g.K + kBK - 1) / kBK;
        if (rounds >= 2 && R * sp <= G && kb_count >= sp * kSplitMinKb &&
            R * sp <= kGemmSplitSlots && R * kEpiWarps <= kGemmSplitCounters) {
            ga.split_s = static_cast<int>(sp);
            ga.split_base = static_cast<int>((rounds - 1) * G);
            (void)launch_pdl(pdl, kern_split, dim3(grid), dim3(kGemmThreads), Cfg::kSmem, s, ta, tb, tb2, ga, rp);
            return cudaGetLastError();
        }
    }
    (void)launch_pdl(pdl, kern, dim3(grid), dim3(kGemmThreads), Cfg::kSmem, s, ta, tb, tb2, ga, rp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(DType dt, int epi, const void* a, const void* b, const void* b2,
                     const GemmArgs& g, const RopeParams& rp, int num_sms, cudaStream_t s) {
    constexpr int BN = 256;
    CUtensorMap ta, tb, tb2;
    // the B box is half a tile when the tile stacks gate and up rows (SWIGLU)
    const uint32_t b_box = epi == EPI_SWIGLU ? BN / 2 : BN;
    if (!make_tmap_2d(&ta, dt, a, g.M, g.K, kBM)) return cudaErrorInvalidValue;
    if (!make_tmap_2d(&tb, dt, b, g.N, g.K, b_box)) return cudaErrorInvalidValue;
    tb2 = tb;
    if (epi == EPI_SWIGLU && !make_tmap_2d(&tb2, dt, b2, g.N, g.K, b_box))
        return cudaErrorInvalidValue;
    switch (epi) {
        case EPI_LINEAR: return launch_cfg<T, BN, EPI_LINEAR>(ta, tb, tb2, g, rp, num_sms, s);
        case EPI_SWIGLU: return launch_cfg<T, BN, EPI_SWIGLU>(ta, tb, tb2, g, rp, num_sms, s);
        case EPI_GELU: return launch_cfg<T, BN, EPI_GELU>(ta, tb, tb2, g, rp, num_sms, s);
        case EPI_QKV:
            switch (rp.span) {
                case 0: return launch_cfg<T, BN, EPI_QKV, 0>(ta, tb, tb2, g, rp, num_sms, s);
                case 16: return launch_cfg<T, BN, EPI_QKV, 16>(ta, tb, tb2, g, rp, num_sms, s);
                case 32: return launch_cfg<T, BN, EPI_QKV, 32>(ta, tb, tb2, g, rp, num_sms, s);
                default: return cudaErrorInvalidValue;
            }
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gemm(DType dt, int epi, const void* a, const void* b, const void* b2,
                        const GemmArgs& args, const RopeParams& rp, int num_sms, cudaStream_t s) {
    if (args.M == 0 || args.N == 0) return cudaSuccess;
    // N-fastest units when A alone would take more than about a third of L2
    // and is the larger operand (B rows: N, or 2N for gate + up)
    GemmArgs g = args;
    const double a_bytes = 2.0 * args.M * args.K;
    const double b_bytes = 2.0 * args.N * args.K * (epi == EPI_SWIGLU ? 2 : 1);
    g.n_fastest = a_bytes > 48.0 * (1 << 20) && a_bytes > b_bytes;
    if (g.M > kBM) return launch_gemm_pair(dt, epi, a, b, b2, g, rp, num_sms, s);
    if (dt == DType::F16) return launch_t<__half>(dt, epi, a, b, b2, g, rp, num_sms, s);
    return launch_t<__nv_bfloat16>(dt, epi, a, b, b2, g, rp, num_sms, s);
}

}  // namespace blk
