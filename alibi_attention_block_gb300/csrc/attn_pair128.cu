// K3 at head_dim 128: causal softmax attention on tcgen05 tensor cores, two
// 128-query tiles per work item (as attn_pair.cu does at head_dim 64).
//
// At head_dim 128 two query tiles' S, P and O do not fit 512 TMEM columns
// twice over, so the tiles share one S buffer: S [0, 128) holds S_A or S_B,
// P_A [128, 192) and P_B [192, 256) (bf16 pairs), O_A [256, 384),
// O_B [384, 512). One thread issues every MMA in a fixed order,
//     S_A(0), S_B(0), then per key tile j:
//     PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
// so each QK^T follows the other tile's PV: by the time the tensor core is
// free for S_x(j+1), the other tile's softmax has read S out of the shared
// buffer, and each PV finds its P written while the tensor core ran the
// other tile's PV and QK^T.
// 12 warps:
//   warp 0      TMA: each query tile's Q (its own buffer, reloaded once the
//               tile's last QK^T of the item has completed), K and V tiles of
//               128 keys into a two-stage ring (128-byte swizzle, 64-column
//               boxes, zero fill past S). K and V load with an evict-last L2
//               policy (the head's other query-tile pairs read the same key
//               prefix), Q evict-first.
//   warp 1      TMEM allocator and MMA issuer: S (M=128, N=128, K=128: Q and
//               K K-major in shared memory), PV (N=128: P from TMEM, V
//               MN-major).
//   warps 2, 3  idle.
//   warps 4..7  softmax of tile A, 8..11 of tile B, one thread per query row:
//               one tcgen05.ld of the row's 128 scores (the shared S is
//               released at once), causal mask on the diagonal (and ragged
//               last) tile, 3-input max, paired f32x2 FMA into ex2 (scale
//               log2(e)/sqrt(d); ALiBi as +slope*key), P packed to the storage
//               type in registers; once the previous PV has read P_x, one
//               64-column store, and O rescaled in TMEM when the running max
//               grew by more than 2^8. An item's O / l is read out during the
//               warpgroup's first tile of its next item.
// Query scale head_dim^-0.5 and GQA (kv head = h / (H/Hk)) follow nnterp
// "stablelm" 03 Notes; ALiBi "Bloom in a sovereign engine", Contribution.
#include "internal.h"

namespace blk {

namespace {

constexpr int kP128Threads = 384;
constexpr int kTQ = 128;
constexpr int kTK = 128;
constexpr int D = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kLaunchRegs = 168, kRegsControl = 96, kRegsSoftmax = 192;

struct Cfg {
    static constexpr int kSub = D / 64;
    static constexpr int kQBytes = kSub * kTQ * 128;   // 32 KB
    static constexpr int kKVBytes = kSub * kTK * 128;  // 32 KB
    static constexpr int kStages = 2;
    static constexpr int kOffKV = 2 * kQBytes;         // Q_A, Q_B
    static constexpr int kOffBar = kOffKV + kStages * 2 * kKVBytes;
    // ALiBi: per softmax warpgroup an mbarrier (its four warps' arrivals)
    // and two 128-float tables slope*log2(e)*i (i = key column within a
    // tile), one per item parity
    static constexpr int kOffTabBar = kOffBar + 256;
    static constexpr int kOffBias = kOffTabBar + 16;
    static constexpr int kSmem = kOffBias + 2 * 2 * kTK * 4 + 1024;
    static constexpr uint32_t kColP = 128;             // P_x at kColP + 64 x
    static constexpr uint32_t kColO = 256;             // O_x at kColO + D x
    static constexpr uint32_t kTmemCols = 512;
};

struct PairCursor {
    int item, it, i, b, h, g, nA, nB;
    bool valid;
    __device__ __forceinline__ int item_of(int round) const {
        const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
        return round * G + ((round & 1) ? G - 1 - c : c);
    }
    __device__ __forceinline__ void decode(const AttnArgs& a, int nq, int np) {
        const int bh_count = a.B * a.H;
        i = np - 1 - item / bh_count;
        const int bh = item % bh_count;
        b = bh / a.H;
        h = bh - b * a.H;
        g = h / (a.H / a.Hk);
        nA = 2 * i + 1;
        nB = (2 * i + 1 < nq) ? 2 * i + 2 : 0;
    }
    __device__ __forceinline__ void start(const AttnArgs& a, int nq, int np, int n_items) {
        it = 0;
        item = item_of(0);
        valid = item < n_items;
        if (valid) decode(a, nq, np);
    }
    __device__ __forceinline__ void next(const AttnArgs& a, int nq, int np, int n_items) {
        ++it;
        item = item_of(it);
        valid = item < n_items;
        if (valid) decode(a, nq, np);
    }
    __device__ __forceinline__ int n_kv() const { return nB ? nB : nA; }
};

template <typename T, bool ALIBI>
__global__ void __launch_bounds__(kP128Threads, 1)
    attn_pair128_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
    constexpr int kStages = Cfg::kStages;
    // With ALiBi the key tiles are walked from the diagonal down: the bias
    // +slope*j is largest there, so the row max is set by the first tile and
    // the O rescale (max grown past 2^8) stays rare; walked upwards, the max
    // rises by slope*128*log2(e) per tile, past 2^8 on most tiles for
    // slopes above 1/23.
    constexpr bool kRev = ALIBI;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const uint32_t sQ = smem_u32(smem);     // Q_x at x tiles
    const uint32_t sKV = sQ + Cfg::kOffKV;  // stage s: K at 2s, V at 2s + 1 tiles
    const uint32_t bar0 = sQ + Cfg::kOffBar;
    auto s_full = [&](int x) { return bar0 + 8u * x; };
    const uint32_t s_free = bar0 + 96u + 32u * kStages;  // the shared S buffer was read
    auto p_full = [&](int x) { return bar0 + 16u + 8u * x; };
    auto pv_done = [&](int x) { return bar0 + 32u + 8u * x; };
    auto o_free = [&](int x) { return bar0 + 48u + 8u * x; };
    auto q_full = [&](int x) { return bar0 + 64u + 8u * x; };
    auto q_empty = [&](int x) { return bar0 + 80u + 8u * x; };
    auto k_full = [&](int i) { return bar0 + 96u + 8u * i; };
    auto v_full = [&](int i) { return bar0 + 96u + 8u * (kStages + i); };
    auto k_empty = [&](int i) { return bar0 + 96u + 8u * (2 * kStages + i); };
    auto v_empty = [&](int i) { return bar0 + 96u + 8u * (3 * kStages + i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffBar + 104 + 32 * kStages);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int nq = (a.S + kTQ - 1) / kTQ;
    const int np = (nq + 1) / 2;
    const int n_items = np * a.B * a.H;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(p_full(x), 4);
            mbar_init(pv_done(x), 1);
            mbar_init(o_free(x), 4);
            mbar_init(q_full(x), 1);
            mbar_init(q_empty(x), 1);
        }
        if (ALIBI)
            for (int x = 0; x < 2; ++x) mbar_init(sQ + Cfg::kOffTabBar + 8u * x, 4);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(v_full(i), 1);
            mbar_init(k_empty(i), 1);
            mbar_init(v_empty(i), 1);
        }
        mbar_init(s_free, 4);
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
    if (a.pdl) {  // launched for programmatic dependent launch
        pdl_wait();  // inputs written by the previous kernel are visible from here on
        pdl_launch_dependents();
    }
    static_assert(4 * kRegsControl + 8 * kRegsSoftmax <= 12 * kLaunchRegs,
                  "register split exceeds the launch's registers");
    if (warp < 4) {
        setmaxnreg_dec<kRegsControl>();
        if (warp == 0 && lane == 0) {
            const uint64_t pol_kv = l2_evict_last_policy(), pol_q = l2_evict_first_policy();
            PairCursor c;
            c.start(a, nq, np, n_items);
            int gkv = 0;
            int itq[2] = {0, 0};  // Q fills per query tile
            bool ok = true;
            while (ok && c.valid) {
                for (int x = 0; x < (c.nB ? 2 : 1) && ok; ++x) {
                    if (!mbar_wait_inl(q_empty(x), (itq[x] & 1) ^ 1u, a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(q_full(x), Cfg::kQBytes);
#pragma unroll
                    for (int sub = 0; sub < Cfg::kSub; ++sub)
                        tma_load_3d_hint(sQ + x * Cfg::kQBytes + sub * kTQ * 128, &tmQ, q_full(x),
                                    sub * 64, (2 * c.i + x) * kTQ, c.b * a.H + c.h, pol_q);
                    ++itq[x];
                }
                const int nkv = c.n_kv();
                for (int j = 0; j < nkv && ok; ++j, ++gkv) {
                    const int kt = kRev ? nkv - 1 - j : j;  // key tile of shared step j
                    const int st = gkv % kStages;
                    const uint32_t ph = (gkv / kStages) & 1;
                    const uint32_t sK = sKV + (2 * st) * Cfg::kKVBytes;
                    if (!mbar_wait_inl(k_empty(st), ph ^ 1u, a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(k_full(st), Cfg::kKVBytes);
#pragma unroll
                    for (int sub = 0; sub < Cfg::kSub; ++sub)
                        tma_load_3d_hint(sK + sub * kTK * 128, &tmK, k_full(st), sub * 64, kt * kTK,
                                    c.b * a.Hk + c.g, pol_kv);
                    if (!mbar_wait_inl(v_empty(st), ph ^ 1u, a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(v_full(st), Cfg::kKVBytes);
#pragma unroll
                    for (int sub = 0; sub < Cfg::kSub; ++sub)
                        tma_load_3d_hint(sK + Cfg::kKVBytes + sub * kTK * 128, &tmV, v_full(st),
                                    sub * 64, kt * kTK, c.b * a.Hk + c.g, pol_kv);
                }
                c.next(a, nq, np, n_items);
            }
        } else if (warp == 1 && lane == 0) {
            constexpr uint32_t fmt = dt_traits<T>::mma_fmt;
            constexpr uint32_t idesc_s = make_idesc_f16(fmt, kTQ, kTK, false);
            constexpr uint32_t idesc_o = make_idesc_f16(fmt, kTQ, D, true);
            constexpr uint64_t kStageStep = (2 * Cfg::kKVBytes) >> 4;
            constexpr uint64_t kAtom = (kTQ * 128) >> 4;
            constexpr uint64_t kQStep = Cfg::kQBytes >> 4;
            const uint64_t dq0 = make_sdesc_sw128(sQ, 16, 1024);
            const uint64_t dk0 = make_sdesc_sw128(sKV, 16, 1024);
            const uint64_t dv0 = make_sdesc_sw128(sKV + Cfg::kKVBytes, kTK * 128, 1024);
            int ns = 0;                 // S products issued (the shared buffer's fills)
            int gp[2] = {0, 0};         // PV products issued per query tile
            int itx[2] = {0, 0};        // items started per query tile
            // S_x = Q_x K^T into the shared buffer once the previous S has been read
            auto issue_s = [&](int x, int st) -> bool {
                if (ns > 0 && !mbar_wait_inl(s_free, (ns - 1) & 1, a.err)) return false;
                tc_fence_after();
                const uint64_t dq = dq0 + x * kQStep, dk = dk0 + st * kStageStep;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t off = (ks / 4) * kAtom + (ks % 4) * 2;
                    tc_mma_ss(tmem_base, dq + off, dk + off, idesc_s, ks > 0 ? 1u : 0u);
                }
                tc_commit(s_full(x));
                ++ns;
                return true;
            };
            // O_x += P_x V once the softmax has written P_x (the first PV of an
            // item overwrites O_x, so it also waits for the previous read-out)
            auto issue_pv = [&](int x, int st, bool first) -> bool {
                if (!mbar_wait_inl(p_full(x), gp[x] & 1, a.err)) return false;
                if (first) {
                    if (itx[x] > 0 && !mbar_wait_inl(o_free(x), (itx[x] - 1) & 1, a.err))
                        return false;
                    ++itx[x];
                }
                tc_fence_after();
                const uint32_t tP = tmem_base + Cfg::kColP + 64u * x;
                const uint32_t tO = tmem_base + Cfg::kColO + D * x;
                const uint64_t dv = dv0 + st * kStageStep;
#pragma unroll
                for (int ks = 0; ks < kTK / 16; ++ks)
                    tc_mma_ts(tO, tP + ks * 8, dv + ks * ((16 * 128) >> 4), idesc_o,
                              (!first || ks > 0) ? 1u : 0u);
                tc_commit(pv_done(x));
                ++gp[x];
                return true;
            };
            PairCursor c;
            c.start(a, nq, np, n_items);
            int gkv = 0;
            int itq[2] = {0, 0};
            bool ok = true;
            auto s_step = [&](int x, int j, int lo, int hi, int gj) -> bool {
                // QK^T of shared step j for query tile x, whose steps are
                // [lo, hi) (K slot gj already waited)
                if (j < lo || j >= hi) return true;
                if (j == lo && !mbar_wait_inl(q_full(x), itq[x] & 1, a.err)) return false;
                if (!issue_s(x, gj % kStages)) return false;
                if (j == hi - 1) {
                    tc_commit(q_empty(x));
                    ++itq[x];
                }
                return true;
            };
            while (ok && c.valid) {
                const int nA = c.nA, nB = c.nB, nkv = c.n_kv();
                // each tile's shared steps: its first n key tiles in key order,
                // its last n when the walk runs down from the diagonal
                const int loA = kRev ? nkv - nA : 0, hiA = kRev ? nkv : nA;
                const int loB = kRev ? nkv - nB : 0, hiB = kRev ? nkv : nB;
                // step 0: S_A(0), S_B(0) (where the tiles take part)
                if (!mbar_wait_inl(k_full(gkv % kStages), (gkv / kStages) & 1, a.err)) break;
                if (!s_step(0, 0, loA, hiA, gkv) || !s_step(1, 0, loB, hiB, gkv)) break;
                tc_commit(k_empty(gkv % kStages));
                for (int j = 0; j < nkv; ++j) {
                    const int gj = gkv + j;
                    const int stj = gj % kStages;
                    const bool more = j + 1 < nkv;
                    if (!mbar_wait_inl(v_full(stj), (gj / kStages) & 1, a.err)) {
                        ok = false;
                        break;
                    }
                    if (more && !mbar_wait_inl(k_full((gj + 1) % kStages),
                                               ((gj + 1) / kStages) & 1, a.err)) {
                        ok = false;
                        break;
                    }
                    // PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
                    if (j >= loA && j < hiA && !issue_pv(0, stj, j == loA)) {
                        ok = false;
                        break;
                    }
                    if (more && !s_step(0, j + 1, loA, hiA, gj + 1)) {
                        ok = false;
                        break;
                    }
                    if (j >= loB && j < hiB && !issue_pv(1, stj, j == loB)) {
                        ok = false;
                        break;
                    }
                    if (more && !s_step(1, j + 1, loB, hiB, gj + 1)) {
                        ok = false;
                        break;
                    }
                    tc_commit(v_empty(stj));
                    if (more) tc_commit(k_empty((gj + 1) % kStages));
                }
                gkv += nkv;
                c.next(a, nq, np, n_items);
            }
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        const int x = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem_base;  // shared by both query tiles
        const uint32_t tP = tmem_base + Cfg::kColP + 64u * x;
        const uint32_t tO = tmem_base + Cfg::kColO + D * x;
        const float scale_l2 = a.scale * kLog2e;
        PairCursor c;
        c.start(a, nq, np, n_items);
        int g = 0;
        bool ok = true;
        bool pend = false;
        float pend_l = 0.f;
        int64_t pend_row = -1;
        int n_done = 0;  // items this warpgroup has started (ALiBi table parity)
        // O / l of the previous item, 32 columns at a time, once its last PV
        // has completed
        auto flush = [&]() {
            const float inv_l = 1.0f / pend_l;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32(tO + lane_off + cc * 32, o);
                if (pend_row >= 0) {
                    T* dst = static_cast<T*>(a.o) + pend_row * static_cast<int64_t>(D) + cc * 32;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[v * 8 + e]) * inv_l;
                        store8(dst + v * 8, f);
                    }
                }
            }
        };
        while (ok && c.valid) {
            const int nx = x ? c.nB : c.nA;
            if (nx == 0) {
                c.next(a, nq, np, n_items);
                continue;
            }
            const int qt = 2 * c.i + x;
            const int qpos = qt * kTQ + row;
            float m_used = -INFINITY;
            float l = 0.f;
            float slope_l2 = 0.f;
            uint32_t bias_tab = 0;
            if constexpr (ALIBI) {
                const float slope = a.slopes ? a.slopes[c.h]
                                             : exp2f(-8.0f * static_cast<float>(c.h + 1) /
                                                     static_cast<float>(a.H));
                slope_l2 = slope * kLog2e;
                // the item's column bias table, in the buffer the warpgroup's
                // previous item did not use (its last readers may still be on
                // that item); each warp's arrival publishes its 32 entries,
                // and no warp reads before all four have arrived
                const int off = Cfg::kOffBias + (2 * x + (n_done & 1)) * kTK * 4;
                reinterpret_cast<float*>(smem + off)[row] = slope_l2 * static_cast<float>(row);
                bias_tab = sQ + off;
                const uint32_t tab_bar = sQ + Cfg::kOffTabBar + 8u * x;
                __syncwarp();
                if (lane == 0) mbar_arrive(tab_bar);
                if (!mbar_wait_inl(tab_bar, n_done & 1, a.err)) {
                    ok = false;
                    break;
                }
            }
            ++n_done;
            for (int j = 0; j < nx; ++j, ++g) {
                if (!mbar_wait_inl(s_full(x), g & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t r[kTK];
                tmem_ld128(tS + lane_off, r);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free);
                const int kt = kRev ? nx - 1 - j : j;  // key tile of this step
                const int kbase = kt * kTK;
                // ALiBi: u = s*scale*log2(e) + slope*log2(e)*i, one paired FMA
                // per two scores from the column table; the tile's uniform
                // part slope*log2(e)*kbase joins the max and the exponent
                // (entry 1 of the table is slope*log2(e) itself: read back, so
                // that the slope holds no register across the tile loop)
                const float sk =
                    ALIBI ? ld_shared_f32(bias_tab + 4) * static_cast<float>(kbase) : 0.f;
                if constexpr (ALIBI) {
                    const uint64_t sc2 = f2_pack(scale_l2, scale_l2);
#pragma unroll
                    for (int i = 0; i < kTK; i += 4) {
                        uint64_t c01, c23;
                        ld_shared_v2_u64(bias_tab + i * 4, c01, c23);
                        float u0, u1, u2, u3;
                        ffma2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), sc2, c01, u0, u1);
                        ffma2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]), sc2, c23, u2,
                              u3);
                        r[i] = __float_as_uint(u0);
                        r[i + 1] = __float_as_uint(u1);
                        r[i + 2] = __float_as_uint(u2);
                        r[i + 3] = __float_as_uint(u3);
                    }
                }
                if (kt == qt || kbase + kTK > a.S) {
                    const int lim = min(qpos, a.S - 1) - kbase;
#pragma unroll
                    for (int i = 0; i < kTK; ++i)
                        if (i > lim) r[i] = __float_as_uint(-INFINITY);
                }
                float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
                for (int i = 0; i < kTK; i += 8) {
                    m0 = fmax3f(m0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                    m1 = fmax3f(m1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                    m2 = fmax3f(m2, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
                    m3 = fmax3f(m3, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
                }
                float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
                if constexpr (!ALIBI) mx *= scale_l2;
                if constexpr (ALIBI) mx += sk;
                float corr = 1.f;
                if (mx > m_used + kRescaleThreshold) {
                    corr = ex2_approx(m_used - mx);
                    m_used = mx;
                }
                const uint64_t mul2 = f2_pack(ALIBI ? 1.f : scale_l2, ALIBI ? 1.f : scale_l2);
                const float off = ALIBI ? sk - m_used : -m_used;
                const uint64_t neg2 = f2_pack(off, off);
                uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
                uint32_t pk[kTK / 2];
#pragma unroll
                for (int k = 0; k < kTK; k += 4) {
                    float e0, e1, e2, e3;
                    ffma2(__uint_as_float(r[k]), __uint_as_float(r[k + 1]), mul2, neg2, e0, e1);
                    ffma2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3]), mul2, neg2, e2,
                          e3);
                    const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
                    const float p2 = ex2_approx(e2), p3 = ex2_approx(e3);
                    fadd2_acc(acc0, p0, p1);
                    fadd2_acc(acc1, p2, p3);
                    pk[k / 2] = dt_traits<T>::pack2(p0, p1);
                    pk[k / 2 + 1] = dt_traits<T>::pack2(p2, p3);
                }
                // the previous PV has read P_x and O_x is settled: read out the
                // previous item's O if pending, publish P_x, rescale O if the
                // max moved (before this tile's PV)
                if (j > 0 || pend) {
                    if (!mbar_wait_inl(pv_done(x), (g - 1) & 1, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                if (j == 0 && pend) {
                    flush();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(o_free(x));
                    pend = false;
                }
                tmem_st64_nowait(tP + lane_off, pk);
                if (j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                    for (int cc = 0; cc < D / 16; ++cc) {
                        uint32_t o[16];
                        const uint32_t col = tO + lane_off + cc * 16;
                        tmem_ld16(col, o);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                        tmem_st16_nowait(col, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(x));
                float s0, s1, s2, s3;
                f2_unpack(acc0, s0, s1);
                f2_unpack(acc1, s2, s3);
                l = l * corr + ((s0 + s1) + (s2 + s3));
            }
            if (!ok) break;
            pend = true;
            pend_l = l;
            pend_row = qpos < a.S ? (static_cast<int64_t>(c.b) * a.S + qpos) * a.H + c.h : -1;
            c.next(a, nq, np, n_items);
        }
        // the last item's O
        if (ok && pend) {
            if (mbar_wait_inl(pv_done(x), (g - 1) & 1, a.err)) {
                tc_fence_after();
                flush();
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

template <typename T, bool ALIBI>
cudaError_t launch_pair128_t(DType dt, const AttnArgs& a, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    if (!make_tmap_3d(&tq, dt, a.q, static_cast<uint64_t>(a.B) * a.H, a.S, D, kTQ) ||
        !make_tmap_3d(&tk, dt, a.k, static_cast<uint64_t>(a.B) * a.Hk, a.S, D, kTK) ||
        !make_tmap_3d(&tv, dt, a.v, static_cast<uint64_t>(a.B) * a.Hk, a.S, D, kTK))
        return cudaErrorInvalidValue;
    auto kern = attn_pair128_kernel<T, ALIBI>;
    {
        const cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), Cfg::kSmem);
        if (e != cudaSuccess) return e;
    }
    const int64_t nq = (a.S + kTQ - 1) / kTQ;
    const int64_t items = (nq + 1) / 2 * a.B * a.H;
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    const int64_t grid = items < a.num_sms ? items : a.num_sms;
    AttnArgs ap = a;
    ap.pdl = pdl_allowed(s);
    (void)launch_pdl(ap.pdl != 0, kern, dim3(static_cast<unsigned>(grid)), dim3(kP128Threads), Cfg::kSmem, s,
                     tq, tk, tv, ap);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_pair128(DType dt, const AttnArgs& a, cudaStream_t s) {
    if (a.d != 128) return cudaErrorInvalidValue;
    if (dt == DType::F16)
        return a.alibi ? launch_pair128_t<__half, true>(dt, a, s)
                       : launch_pair128_t<__half, false>(dt, a, s);
    return a.alibi ? launch_pair128_t<__nv_bfloat16, true>(dt, a, s)
                   : launch_pair128_t<__nv_bfloat16, false>(dt, a, s);
}

}  // namespace blk
