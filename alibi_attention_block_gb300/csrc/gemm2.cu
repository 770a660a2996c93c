// K2 on a pair of SMs: C = A B^T with the block's fused epilogues, each
// tcgen05 MMA issued once for a 256 x 256 output tile that two CTAs (a
// cluster of two, one per SM) compute together (cta_group::2).
//
// Why: at N = 256 one SM's MMA reads its 128 x 64 A tile and all of the
// 256 x 64 B tile from shared memory per k-block, and TMA writes both; the
// shared-memory port, not the tensor core, then sets the pace. With the pair
// instruction each CTA holds and TMA-loads only its own 128 rows of A and
// its own half (128 rows) of B, so per SM the operand reads and the TMA
// writes per k-block fall by a third while the MMA work per SM stays the
// same. Every TMA load lands in the issuing CTA's own shared memory; only
// barrier signals cross between the two CTAs:
//   - each CTA's TMA loads of a stage count their bytes on the even CTA's
//     "full" barrier (cta_group::2 completion), whose single arrival (with
//     the whole stage's byte count) comes from the even CTA's producer;
//   - the even CTA's MMA thread issues the pair MMAs (M = 256: A rows 0..127
//     from the even CTA, 128..255 from the odd one; B rows 0..127 / 128..255
//     likewise; D rows land in each CTA's own TMEM) and commits their
//     completion once to each CTA's "empty" barrier and, per tile, to each
//     CTA's "tfull" barrier;
//   - the odd CTA's epilogue warps report a consumed accumulator by arriving
//     on the even CTA's "tempty" barrier.
// For SwiGLU the B tile is [gate rows | up rows]: the even CTA loads the 128
// gate rows, the odd one the 128 up rows. Roles per CTA (10 warps) and the
// epilogues are those of gemm.cu: warp 0 TMA, warp 1 TMEM allocation (and,
// in the even CTA, MMA issue), warps 2..9 epilogue.
#include <map>
#include <mutex>
#include <utility>

#include "gemm_epi.cuh"

namespace blk {

namespace {

using namespace gemm;

constexpr int kPairBN = 256;                 // MMA N: output columns (or gate|up rows)
constexpr int kBoxBytes = kBM * 64 * 2;      // one 64-column swizzled box of 128 rows

// The mainloop's k-block and ring depth, by epilogue: 128 inputs (two
// 64-column boxes per operand, eight MMAs per barrier round trip) in three
// 64 KB stages for QKV, SwiGLU and GELU; 64 inputs in six 32 KB stages for
// LINEAR. Same-box A/B: qkv 128.0 -> 121.3 us, gate/up 209.5 -> 200.0,
// Bloom's GELU up 71.0 -> 67.5 with 128; but o_proj 59.5 -> 61.7 and down
// 121.4 -> 127.0 (their heavier residual epilogues want the finer ring).
template <int EPI>
struct PairK {
    static constexpr int kBKp = EPI == EPI_LINEAR ? 64 : 128;
    static constexpr int kBoxes = kBKp / 64;
    static constexpr int kStages = EPI == EPI_LINEAR ? 6 : 3;
    static constexpr int kABytes = kBM * kBKp * 2;             // this CTA's 128 rows of A
    static constexpr int kBBytes = (kPairBN / 2) * kBKp * 2;   // this CTA's half of B
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kOffBar = kStages * kStageBytes;
    static constexpr int kOffEpi = kOffBar + 1024;  // staging boxes 1024-byte aligned (swizzle)
    static constexpr int kSmem = kOffEpi + kEpiWarps * 32 * 128 + 1024;
};
constexpr uint32_t kPairTmemCols = 2 * kPairBN;  // two accumulators

template <typename T, int EPI, int ROT, bool SPLIT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmB2,
                     const __grid_constant__ CUtensorMap tmO,
                     const __grid_constant__ CUtensorMap tmO2,
                     const __grid_constant__ CUtensorMap tmO3, const GemmArgs g,
                     const __grid_constant__ RopeParams rp) {
    constexpr int BN = kPairBN;
    constexpr int kBNOut = EPI == EPI_SWIGLU ? BN / 2 : BN;
    constexpr int kPM = 2 * kBM;  // output rows per pair tile
    using PK = PairK<EPI>;
    constexpr int kPairStages = PK::kStages;
    constexpr int kPairABytes = PK::kABytes;
    constexpr int kPairStageBytes = PK::kStageBytes;
    constexpr int kPairOffBar = PK::kOffBar;
    constexpr int kPairOffEpi = PK::kOffEpi;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + kPairOffBar;
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kPairStages + i); };
    auto tfull = [&](int i) { return bar0 + 8u * (2 * kPairStages + i); };
    auto tempty = [&](int i) { return bar0 + 8u * (2 * kPairStages + 2 + i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kPairOffBar + 8 * (2 * kPairStages + 4));
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool lead = rank == 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kPairStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull(i), 1);
            mbar_init(tempty(i), 2 * kEpiWarps);  // both CTAs' epilogue warps (even CTA's only)
        }
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (EPI == EPI_SWIGLU) tma_prefetch_desc(&tmB2);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), kPairTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers and TMEM exist before any signal crosses
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (g.pdl) {  // launched for programmatic dependent launch
        pdl_wait();  // inputs written by the previous kernel are visible from here on
        pdl_launch_dependents();
    }
    const int m_units = (g.M + kPM - 1) / kPM;
    const int n_tiles = (g.N + kBNOut - 1) / kBNOut;
    const int num_units = m_units * n_tiles;
    const int unit0 = static_cast<int>(blockIdx.x) / 2;
    const int unit_step = static_cast<int>(gridDim.x) / 2;
    const int kb_count = (g.K + PK::kBKp - 1) / PK::kBKp;
    const int num_work =
        SPLIT ? g.split_base + (num_units - g.split_base) * g.split_s : num_units;
    auto tile_of = [&](int u, int& mt, int& nt) {
        mt = g.n_fastest ? u / n_tiles : u % m_units;
        nt = g.n_fastest ? u % n_tiles : u / m_units;
    };
    // With a bias (LINEAR, GELU, QKV), a tile's accumulator starts as the
    // bias row, written into TMEM by the epilogue warps once it is free,
    // before the tile's first MMA (which then accumulates): the epilogue no
    // longer adds it. The TMEM-empty barriers then carry one more arrival
    // each, the first two before any tile. Split segments start from zero
    // and take the bias in the last one's epilogue, as before.
    const bool pre = EPI != EPI_SWIGLU && g.bias != nullptr;
    auto preloaded = [&](int v) {
        return pre && v < num_work && !(SPLIT && g.split_s > 1 && v >= g.split_base);
    };
    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t full_lead0 = peer_addr(full(0), 0);
            for (int v = unit0; v < num_work && ok; v += unit_step) {
                const Unit un = decode_unit<SPLIT>(g, v, kb_count);
                int mt, nt;
                tile_of(un.u, mt, nt);
                const int arow = mt * kPM + static_cast<int>(rank) * kBM;
                const CUtensorMap* mb = (EPI == EPI_SWIGLU && rank) ? &tmB2 : &tmB;
                const int brow = EPI == EPI_SWIGLU ? nt * kBNOut : nt * BN + static_cast<int>(rank) * (BN / 2);
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!mbar_wait_cluster(empty(stage), phase ^ 1u, g.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + stage * kPairStageBytes;
                    const uint32_t fb = full_lead0 + 8u * stage;
                    if (lead) mbar_expect_tx(full(stage), 2 * kPairStageBytes);
#pragma unroll
                    for (int bx = 0; bx < PK::kBoxes; ++bx) {
                        tma_load_2d_pair(sa + bx * kBoxBytes, &tmA, fb, kb * PK::kBKp + bx * 64, arow);
                        tma_load_2d_pair(sa + kPairABytes + bx * kBoxBytes, mb, fb,
                                         kb * PK::kBKp + bx * 64, brow);
                    }
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lead && lane == 0) {
            constexpr uint32_t idesc = make_idesc_f16(dt_traits<T>::mma_fmt, kPM, BN, false);
            const uint64_t da0 = make_sdesc_sw128(sbase, 16, 1024);
            const uint64_t db0 = make_sdesc_sw128(sbase + kPairABytes, 16, 1024);
            constexpr uint64_t kStageStep = kPairStageBytes >> 4;
            const uint32_t empty0[2] = {peer_addr(empty(0), 0), peer_addr(empty(0), 1)};
            const uint32_t tfull0[2] = {peer_addr(tfull(0), 0), peer_addr(tfull(0), 1)};
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int v = unit0; v < num_work && ok; v += unit_step, ++it) {
                const Unit un = decode_unit<SPLIT>(g, v, kb_count);
                const int acc = it & 1;
                const uint32_t tpar = pre ? ((it >> 1) & 1) : (((it >> 1) & 1) ^ 1u);
                if (!mbar_wait_cluster(tempty(acc), tpar, g.err)) break;
                const bool start = !preloaded(v);  // the first MMA overwrites
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!mbar_wait_cluster(full(stage), phase, g.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = da0 + stage * kStageStep;
                    const uint64_t bd = db0 + stage * kStageStep;
#pragma unroll
                    for (int k = 0; k < PK::kBKp / 16; ++k) {
                        const uint64_t off = (k / 4) * (kBoxBytes >> 4) + (k % 4) * 2;
                        tc_mma_ss_pair(d_tmem, ad + off, bd + off, idesc,
                                       (kb > un.kb0 || k != 0 || !start) ? 1u : 0u);
                    }
                    tc_commit_pair(empty0[0] + 8u * stage);
                    tc_commit_pair(empty0[1] + 8u * stage);
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) {
                    tc_commit_pair(tfull0[0] + 8u * acc);
                    tc_commit_pair(tfull0[1] + 8u * acc);
                }
            }
        }
    } else {
        const int ew = warp - 2;
        const int quarter = warp & 3;
        const int half = ew / 4;
        const int row = quarter * 32 + lane;
        const uint32_t stg0 = sbase + kPairOffEpi;
        const uint32_t tempty_lead0 = peer_addr(tempty(0), 0);
        const uint32_t lane_q = static_cast<uint32_t>(quarter * 32) << 16;
        auto preload = [&](int v, int acc) {
            const Unit u2 = decode_unit<SPLIT>(g, v, kb_count);
            int mt2, nt2;
            tile_of(u2.u, mt2, nt2);
            preload_bias<T, BN>(g, tmem_base + acc * BN + lane_q, nt2, half);
        };
        if (pre) {
            // the first two tiles' accumulators
            for (int a = 0; a < 2; ++a) {
                if (preloaded(unit0 + a * unit_step)) preload(unit0 + a * unit_step, a);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_lead0 + 8u * a);
            }
        }
        int it = 0;
        for (int v = unit0; v < num_work; v += unit_step, ++it) {
            const Unit un = decode_unit<SPLIT>(g, v, kb_count);
            const int acc = it & 1;
            if (!mbar_wait_cluster(tfull(acc), (it >> 1) & 1, g.err)) break;
            tc_fence_after();
            int mt, nt;
            tile_of(un.u, mt, nt);
            const int m0 = mt * kPM + static_cast<int>(rank) * kBM;  // this CTA's first row
            const uint32_t tbase =
                tmem_base + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
            const float* part = nullptr;
            unsigned* cnt = nullptr;
            bool run = true;
            if (SPLIT && v >= g.split_base) {
                // a segment of a split unit: publish this warp's 32 rows of the
                // partial tile, count in; the last to arrive sums and stores
                const int t = (v - g.split_base) / g.split_s;
                const int slot = t * 2 + static_cast<int>(rank);
                float* slot0 = g.split_ws + static_cast<size_t>(slot * g.split_s) * (kBM * BN);
                float* mine = slot0 + static_cast<size_t>(un.q) * (kBM * BN) + row;
#pragma unroll 1
                for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
                    uint32_t r[32];
                    tmem_ld32(tbase + c * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) __stcg(mine + (c * 32 + i) * kBM, __uint_as_float(r[i]));
                }
                __threadfence();
                __syncwarp();
                cnt = g.split_cnt + (slot * kEpiWarps + ew);
                unsigned old = 0;
                if (lane == 0) old = atomicAdd(cnt, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old != static_cast<unsigned>(g.split_s - 1)) {
                    run = false;
                } else {
                    __threadfence();  // the other segments' partials are visible
                    part = slot0;
                }
            }
            if (run) {
                epilogue_tile<T, BN, EPI, ROT, SPLIT>(g, rp, tbase, m0 + row, nt,
                                                      stg0 + ew * (32 * 128), lane,
                                                      m0 + quarter * 32, part, un.q, row, half,
                                                      g.tma_out ? &tmO : nullptr, &tmO2, &tmO3,
                                                      preloaded(v));
                if (cnt && lane == 0) *cnt = 0u;  // every segment has arrived: ready for reuse
            }
            tc_fence_before();
            __syncwarp();
            // the accumulator's next tile (two on) starts as its bias row
            if (preloaded(v + 2 * unit_step)) {
                preload(v + 2 * unit_step, acc);
                tc_fence_before();
                __syncwarp();
            }
            if (lane == 0) mbar_arrive_cluster(tempty_lead0 + 8u * acc);
        }
        // the warp's TMA stores have read their staging boxes and written
        // the output before the CTA ends
        if (lane == 0) bulk_wait<0>();
    }
    // every MMA of the pair has completed (both epilogues consumed the last
    // accumulators) and every cross-CTA signal has landed
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kPairTmemCols);
    }
}

// cudaOccupancyMaxActiveClusters per (kernel, device): how many CTA pairs
// can be resident at once.
int max_pairs(const void* kern, const cudaLaunchConfig_t& cfg_in, int num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return num_sms / 2;
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({kern, dev});
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = cfg_in;
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms / 2 * 2), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        n = num_sms / 2;
    }
    cache[{kern, dev}] = n;
    return n;
}

template <typename T, int EPI, int ROT = 0>
cudaError_t launch_pair_cfg(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb2,
                            const CUtensorMap (&to)[3], const GemmArgs& g, const RopeParams& rp,
                            int num_sms, cudaStream_t s) {
    constexpr int kBNOut = EPI == EPI_SWIGLU ? kPairBN / 2 : kPairBN;
    constexpr bool kCanSplit = EPI != EPI_SWIGLU;
    auto kern = gemm_pair_kernel<T, EPI, ROT, false>;
    auto kern_split = gemm_pair_kernel<T, EPI, ROT, kCanSplit>;
    constexpr int kPairSmem = PairK<EPI>::kSmem;
    cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), kPairSmem);
    if (e == cudaSuccess && kCanSplit)
        e = set_smem_attr_once(reinterpret_cast<const void*>(kern_split), kPairSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start (set-up only) while the previous kernel drains, outside
    // graph capture (pdl_allowed)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = kPairSmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query below sees the cluster shape only
    const int64_t units =
        static_cast<int64_t>((g.M + 2 * kBM - 1) / (2 * kBM)) * ((g.N + kBNOut - 1) / kBNOut);
    const int64_t slots = max_pairs(reinterpret_cast<const void*>(kern), cfg, num_sms);
    const bool pdl = pdl_allowed(s);
    cfg.numAttrs = pdl ? 2 : 1;
    const int64_t pairs = units < slots ? units : slots;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    GemmArgs ga = g;
    ga.split_s = 1;
    ga.split_base = 0;
    ga.pdl = pdl;
    // the split of a last, partial round along K, as in gemm.cu (each CTA of
    // a pair publishes its own 128-row partial tiles)
    if (kCanSplit && g.split_ws && g.split_cnt) {
        const int64_t G = pairs;
        const int64_t rounds = (units + G - 1) / G;
        const int64_t R = units - (rounds - 1) * G;
        const int64_t sp = 2;
        // (kSplitMinKb counts 64-wide k-blocks)
        const int64_t kbw = PairK<EPI>::kBKp;
        const int64_t kb_count = (g.K + kbw - 1) / kbw;
        if (rounds >= 2 && R * sp <= G && kb_count * kbw >= sp * kSplitMinKb * kBK &&
            R * 2 * sp <= kGemmSplitSlots && R * 2 * kEpiWarps <= kGemmSplitCounters) {
            ga.split_s = static_cast<int>(sp);
            ga.split_base = static_cast<int>((rounds - 1) * G);
            return cudaLaunchKernelEx(&cfg, kern_split, ta, tb, tb2, to[0], to[1], to[2], ga, rp);
        }
    }
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tb2, to[0], to[1], to[2], ga, rp);
}

template <typename T>
cudaError_t launch_pair_t(DType dt, int epi, const void* a, const void* b, const void* b2,
                          const GemmArgs& g, const RopeParams& rp, int num_sms, cudaStream_t s) {
    CUtensorMap ta, tb, tb2, to[3];
    if (!make_tmap_2d(&ta, dt, a, g.M, g.K, kBM)) return cudaErrorInvalidValue;
    if (!make_tmap_2d(&tb, dt, b, g.N, g.K, kPairBN / 2)) return cudaErrorInvalidValue;
    tb2 = tb;
    if (epi == EPI_SWIGLU && !make_tmap_2d(&tb2, dt, b2, g.N, g.K, kPairBN / 2))
        return cudaErrorInvalidValue;
    // TMA stores of the epilogue's staged boxes (32 rows x 64 16-bit values,
    // 128-byte swizzle): the [M, N] output of LINEAR, GELU and SWIGLU, or
    // QKV's q, k, v ([B * heads, S, d]) when a box holds 64 columns of one
    // head (head_dim % 64 == 0) and 32 positions of one sequence (S % 32 ==
    // 0). fp32 outputs keep their staged per-warp stores of whole lines;
    // they measured faster than the TMA's.
    GemmArgs gt = g;
    gt.tma_out = 0;
    to[0] = to[1] = to[2] = ta;
    const CUtensorMapDataType ty =
        dt == DType::F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (epi == EPI_QKV) {
        // boxes of 32 columns (64-byte swizzle) when head_dim % 32 == 0
        if (g.d % 32 == 0 && g.S > 0 && g.S % 32 == 0 && g.M % g.S == 0) {
            const uint64_t B = static_cast<uint64_t>(g.M / g.S);
            if (!make_tmap_3d(&to[0], dt, g.q, B * g.H, g.S, g.d, 32, 32) ||
                !make_tmap_3d(&to[1], dt, g.k, B * g.Hk, g.S, g.d, 32, 32) ||
                !make_tmap_3d(&to[2], dt, g.v, B * g.Hk, g.S, g.d, 32, 32))
                return cudaErrorInvalidValue;
            gt.tma_out = 2;
        }
    } else if (!(epi == EPI_LINEAR && g.out_f32)) {
        if (!make_tmap_2d_plain(&to[0], ty, 2, g.out, g.M, g.N, 64, 32, true))
            return cudaErrorInvalidValue;
        gt.tma_out = 1;
    }
    switch (epi) {
        case EPI_LINEAR: return launch_pair_cfg<T, EPI_LINEAR>(ta, tb, tb2, to, gt, rp, num_sms, s);
        case EPI_SWIGLU: return launch_pair_cfg<T, EPI_SWIGLU>(ta, tb, tb2, to, gt, rp, num_sms, s);
        case EPI_GELU: return launch_pair_cfg<T, EPI_GELU>(ta, tb, tb2, to, gt, rp, num_sms, s);
        case EPI_QKV:
            switch (rp.span) {
                case 0: return launch_pair_cfg<T, EPI_QKV, 0>(ta, tb, tb2, to, gt, rp, num_sms, s);
                case 16: return launch_pair_cfg<T, EPI_QKV, 16>(ta, tb, tb2, to, gt, rp, num_sms, s);
                case 32: return launch_pair_cfg<T, EPI_QKV, 32>(ta, tb, tb2, to, gt, rp, num_sms, s);
                default: return cudaErrorInvalidValue;
            }
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gemm_pair(DType dt, int epi, const void* a, const void* b, const void* b2,
                             const GemmArgs& g, const RopeParams& rp, int num_sms,
                             cudaStream_t s) {
    if (dt == DType::F16) return launch_pair_t<__half>(dt, epi, a, b, b2, g, rp, num_sms, s);
    return launch_pair_t<__nv_bfloat16>(dt, epi, a, b, b2, g, rp, num_sms, s);
}

}  // namespace blk
