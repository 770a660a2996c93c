// K3: causal softmax attention, flash-style, on tcgen05 tensor cores.
//
// One CTA per (128-query tile, head, batch), heaviest (latest) query tiles
// scheduled first; at head_dim 64 two CTAs share an SM, so one CTA's MMAs
// run while the other's softmax warps compute. 6 warps:
//   warp 0      TMA: the Q tile once, then K and V tiles of 128 keys into a
//               STAGES-deep ring (128-byte swizzle, 64-column boxes). A K
//               slot is refilled once its QK^T has completed and a V slot once
//               its PV has, so S_{j+1} never waits on PV_j (even with one stage).
//   warp 1      TMEM allocator and single-thread MMA issuer:
//                 S  = Q K^T  (M=128, N=128, K=d; Q and K K-major in smem)  -> TMEM S
//                 O += P V    (M=128, N=d, K=128; P read from TMEM,
//                              V MN-major in smem)                          -> TMEM O
//               S_{j+1} is issued as soon as the softmax warps have read S_j,
//               so the next QK^T overlaps the exponentials of this tile.
//   warps 2..5  softmax, one thread per query row: one tcgen05.ld of the
//               row's 128 scores (S is released at once), the causal
//               mask on the diagonal (and ragged last) tile only, the row max
//               on the raw scores (3-input max), one paired (f32x2) FMA per two
//               scores into ex2 (scale log2(e)/sqrt(d) folded in; for ALiBi the
//               bias -slope*(i-j), "Bloom in a sovereign engine",
//               Contribution, enters as +slope*j, the -slope*i part being
//               constant along the row), P rounded to the storage type and
//               written to TMEM (32 keys at a time) as the A operand of PV,
//               after PV_{j-1} has finished reading the previous P. O is rescaled in TMEM
//               only when the running max grows by more than 2^8. Finally
//               O / l is written as [B, S, H, d].
// TMEM columns: S [0, 128), P [128, 192) (two 16-bit values per column),
// O [192, 192 + d).
// Query scale head_dim^-0.5 and GQA (kv head = h / (H/Hk)) follow nnterp
// "stablelm" 03 Notes.
#include "internal.h"

namespace blk {

namespace {

constexpr int kAttnThreads = 192;
constexpr int kBQ = 128;
constexpr int kBKV = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest unnormalised p
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;

template <int D>
struct AttnCfg {
    static constexpr int kSub = (D + 63) / 64;          // 64-column boxes per row
    static constexpr int kTileBytes = kSub * kBQ * 128;  // 128 rows x kSub x 128 B
    static constexpr int kStages = D > 128 ? 1 : 2;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmem = kTileBytes * (1 + 2 * kStages) + 1024 + kBarBytes;
    static constexpr uint32_t kTmemCols = (kColO + D) <= 256 ? 256 : 512;
    static constexpr int kMinBlocks = kTmemCols == 256 ? 2 : 1;
};

template <typename T, int D, bool ALIBI>
__global__ void __launch_bounds__(kAttnThreads, AttnCfg<D>::kMinBlocks)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
    using Cfg = AttnCfg<D>;
    constexpr int kStages = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sKV = sQ + Cfg::kTileBytes;  // stage i: K at +2i, V at +2i+1 tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (1 + 2 * kStages) * Cfg::kTileBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8 + 4 * kStages);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t q_full = bar0;
    const uint32_t s_full = bar0 + 8;
    const uint32_t s_free = bar0 + 16;
    const uint32_t p_full = bar0 + 24;
    const uint32_t o_done = bar0 + 32;
    auto k_full = [&](int i) { return bar0 + 64u + 8u * i; };
    auto v_full = [&](int i) { return bar0 + 64u + 8u * (kStages + i); };
    auto k_empty = [&](int i) { return bar0 + 64u + 8u * (2 * kStages + i); };
    auto v_empty = [&](int i) { return bar0 + 64u + 8u * (3 * kStages + i); };

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;

    // tile decode: heaviest query tiles first
    const int nq = (a.S + kBQ - 1) / kBQ;
    const int bh_count = a.B * a.H;
    const int qt = nq - 1 - static_cast<int>(blockIdx.x) / bh_count;
    const int bh = static_cast<int>(blockIdx.x) % bh_count;
    const int b = bh / a.H;
    const int h = bh - b * a.H;
    const int g = h / (a.H / a.Hk);
    const int nkv = qt + 1;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(v_full(i), 1);
            mbar_init(k_empty(i), 1);
            mbar_init(v_empty(i), 1);
        }
        fence_barrier_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t tS = tmem_base + kColS;
    const uint32_t tP = tmem_base + kColP;
    const uint32_t tO = tmem_base + kColO;

    if (warp == 0) {
        if (lane == 0) {
            mbar_expect_tx(q_full, Cfg::kTileBytes);
#pragma unroll
            for (int sub = 0; sub < Cfg::kSub; ++sub)
                tma_load_3d(sQ + sub * kBQ * 128, &tmQ, q_full, sub * 64, qt * kBQ, b * a.H + h);
            for (int j = 0; j < nkv; ++j) {
                const int st = j % kStages;
                const uint32_t ph = (j / kStages) & 1;
                const uint32_t sK = sKV + (2 * st) * Cfg::kTileBytes;
                const uint32_t sV = sK + Cfg::kTileBytes;
                if (!mbar_wait(k_empty(st), ph ^ 1u, a.err)) break;
                mbar_expect_tx(k_full(st), Cfg::kTileBytes);
#pragma unroll
                for (int sub = 0; sub < Cfg::kSub; ++sub)
                    tma_load_3d(sK + sub * kBKV * 128, &tmK, k_full(st), sub * 64, j * kBKV,
                                b * a.Hk + g);
                if (!mbar_wait(v_empty(st), ph ^ 1u, a.err)) break;
                mbar_expect_tx(v_full(st), Cfg::kTileBytes);
#pragma unroll
                for (int sub = 0; sub < Cfg::kSub; ++sub)
                    tma_load_3d(sV + sub * kBKV * 128, &tmV, v_full(st), sub * 64, j * kBKV,
                                b * a.Hk + g);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t fmt = dt_traits<T>::mma_fmt;
            constexpr uint32_t idesc_s = make_idesc_f16(fmt, kBQ, kBKV, false);
            constexpr uint32_t idesc_o = make_idesc_f16(fmt, kBQ, D, true);
            bool ok = mbar_wait(q_full, 0, a.err);
            auto issue_s = [&](int j) -> bool {
                const int st = j % kStages;
                if (!mbar_wait(k_full(st), (j / kStages) & 1, a.err)) return false;
                tc_fence_after();
                const uint32_t sK = sKV + (2 * st) * Cfg::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks / 4) * (kBQ * 128) + (ks % 4) * 32;
                    tc_mma_ss(tS, make_sdesc_sw128(sQ + off, 16, 1024),
                              make_sdesc_sw128(sK + off, 16, 1024), idesc_s, ks > 0 ? 1u : 0u);
                }
                tc_commit(s_full);
                tc_commit(k_empty(st));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; j < nkv && ok; ++j) {
                const int st = j % kStages;
                if (j + 1 < nkv) {
                    if (!mbar_wait(s_free, j & 1, a.err)) break;
                    tc_fence_after();
                    if (!issue_s(j + 1)) break;
                }
                if (!mbar_wait(p_full, j & 1, a.err)) break;
                if (!mbar_wait(v_full(st), (j / kStages) & 1, a.err)) break;
                tc_fence_after();
                const uint32_t sV = sKV + (2 * st + 1) * Cfg::kTileBytes;
#pragma unroll
                for (int ks = 0; ks < kBKV / 16; ++ks) {
                    tc_mma_ts(tO, tP + ks * 8, make_sdesc_sw128(sV + ks * 16 * 128, kBKV * 128, 1024),
                              idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
                }
                tc_commit(o_done);
                tc_commit(v_empty(st));
            }
        }
    } else {
        // softmax warps: thread owns query row `row` of the tile
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int qpos = qt * kBQ + row;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float scale_l2 = a.scale * kLog2e;
        float slope_l2 = 0.f;
        if constexpr (ALIBI) {
            const float slope = a.slopes ? a.slopes[h]
                                         : exp2f(-8.0f * static_cast<float>(h + 1) /
                                                 static_cast<float>(a.H));
            slope_l2 = slope * kLog2e;
        }
        float m_used = -INFINITY;  // running max, log2 domain (scores * scale * log2 e)
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            if (!mbar_wait(s_full, j & 1, a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int kbase = j * kBKV;
            const bool masked = j == qt || kbase + kBKV > a.S;
            const int lim = min(qpos, a.S - 1) - kbase;  // keys <= lim are visible
            const float sk = slope_l2 * static_cast<float>(kbase);
            // scores in the log2 domain before the max subtraction: s*scale for
            // plain attention (applied after the max, which commutes with a
            // positive scale), s*scale + slope*key_pos for ALiBi (the
            // -slope*query_pos part is constant along the row and cancels)
            auto logit = [&](uint32_t raw, int i) -> float {
                const float v = __uint_as_float(raw);
                if constexpr (ALIBI)
                    return fmaf(v, scale_l2, fmaf(slope_l2, static_cast<float>(i), sk));
                else
                    return v;
            };
            // the whole row of S in registers, so S can be overwritten by the
            // next QK^T while this tile's exponentials run
            uint32_t r[kBKV];
            tmem_ld128(tS + lane_off, r);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            if constexpr (ALIBI) {
#pragma unroll
                for (int i = 0; i < kBKV; ++i) r[i] = __float_as_uint(logit(r[i], i));
            }
            if (masked) {
#pragma unroll
                for (int i = 0; i < kBKV; ++i)
                    if (i > lim) r[i] = __float_as_uint(-INFINITY);
            }
            float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
            for (int i = 0; i < kBKV; i += 4) {
                m0 = fmax3f(m0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                m1 = fmax3f(m1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
            }
            float mx = fmaxf(m0, m1);
            if constexpr (!ALIBI) mx *= scale_l2;  // scale > 0: max commutes with it
            float corr = 1.f;
            if (mx > m_used + kRescaleThreshold) {
                corr = ex2_approx(m_used - mx);
                m_used = mx;
            }
            // PV_{j-1} must be done before O is rescaled and before P_j
            // overwrites P_{j-1}, which it reads
            if (j > 0) {
                if (!mbar_wait(o_done, (j - 1) & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + lane_off + c * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                        tmem_st32_nowait(tO + lane_off + c * 32, o);
                    }
                }
            }
            // p = 2^(logit - m), row sum, P (storage type) into TMEM 32 keys at a time
            const uint64_t mul2 = f2_pack(ALIBI ? 1.f : scale_l2, ALIBI ? 1.f : scale_l2);
            const uint64_t neg2 = f2_pack(-m_used, -m_used);
            uint64_t acc2 = f2_pack(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kBKV / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float e0, e1;
                    ffma2(__uint_as_float(r[c * 32 + i]), __uint_as_float(r[c * 32 + i + 1]),
                          mul2, neg2, e0, e1);
                    const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
                    fadd2_acc(acc2, p0, p1);
                    pk[i / 2] = dt_traits<T>::pack2(p0, p1);
                }
                tmem_st16_nowait(tP + lane_off + c * 16, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            float sum0, sum1;
            f2_unpack(acc2, sum0, sum1);
            l = l * corr + (sum0 + sum1);
        }
        if (ok && mbar_wait(o_done, (nkv - 1) & 1, a.err)) {
            tc_fence_after();
            const float inv_l = 1.0f / l;
            T* dst = static_cast<T*>(a.o) +
                     ((static_cast<int64_t>(b) * a.S + qpos) * a.H + h) * static_cast<int64_t>(D);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tO + lane_off + c * 32, r);
                if (qpos < a.S) {
                    float o[8];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = __uint_as_float(r[v * 8 + e]) * inv_l;
                        store8(dst + c * 32 + v * 8, o);
                    }
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

template <typename T, int D, bool ALIBI>
cudaError_t launch_d(DType dt, const AttnArgs& a, cudaStream_t s) {
    using Cfg = AttnCfg<D>;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_3d(&tq, dt, a.q, static_cast<uint64_t>(a.B) * a.H, a.S, D, kBQ) ||
        !make_tmap_3d(&tk, dt, a.k, static_cast<uint64_t>(a.B) * a.Hk, a.S, D, kBKV) ||
        !make_tmap_3d(&tv, dt, a.v, static_cast<uint64_t>(a.B) * a.Hk, a.S, D, kBKV))
        return cudaErrorInvalidValue;
    auto kern = attn_kernel<T, D, ALIBI>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t grid = static_cast<int64_t>((a.S + kBQ - 1) / kBQ) * a.B * a.H;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    kern<<<static_cast<unsigned>(grid), kAttnThreads, Cfg::kSmem, s>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_a(DType dt, const AttnArgs& a, cudaStream_t s) {
    return a.alibi ? launch_d<T, D, true>(dt, a, s) : launch_d<T, D, false>(dt, a, s);
}

template <typename T>
cudaError_t launch_t(DType dt, const AttnArgs& a, cudaStream_t s) {
    switch (a.d) {
        case 64: return launch_a<T, 64>(dt, a, s);
        case 128: return launch_a<T, 128>(dt, a, s);
        case 160: return launch_a<T, 160>(dt, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_attention(DType dt, const AttnArgs& a, cudaStream_t s) {
    if (a.B == 0 || a.S == 0) return cudaSuccess;
    if (dt == DType::F16) return launch_t<__half>(dt, a, s);
    return launch_t<__nv_bfloat16>(dt, a, s);
}

}  // namespace blk
