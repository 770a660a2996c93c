// K3: causal softmax attention, flash-style, on tcgen05 tensor cores: the
// single-query-tile kernel, which serves head_dim 160 (head_dim 64 and 128
// run the paired-query-tile kernels of attn_pair.cu and attn_pair128.cu; at
// 160 two query tiles' O no longer leave TMEM room for S and P), and the
// dispatch by head_dim.
//
// Persistent: each CTA walks (128-query tile, batch, head) items, heaviest
// (latest) query tiles first, keeping its TMEM and barriers; the next item's
// Q loads into a second buffer and its first QK^T overlaps the current item's
// last tile. 10 warps:
//   warp 0      TMA: the Q tile once, then K and V tiles of 128 keys into a
//               STAGES-deep ring (128-byte swizzle, 64-column boxes). A K
//               slot is refilled once its QK^T has completed and a V slot once
//               its PV has, so S_{j+1} never waits on PV_j (even with one stage).
//   warp 1      TMEM allocator and single-thread MMA issuer:
//                 S  = Q K^T  (M=128, N=128, K=d; Q and K K-major in smem)  -> TMEM S
//                 O += P V    (M=128, N=d, K=128; P read from TMEM,
//                              V MN-major in smem)                          -> TMEM O
//               S_{j+1} is issued as soon as the softmax warps have read S_j,
//               so the next QK^T overlaps the exponentials of this tile; the
//               first PV of an item waits until the previous O was read out.
//   warps 2..9  softmax, two threads per query row (warps w and w+4 share a
//               TMEM lane quarter and split each 128-key tile into halves; the
//               halves' row maxima meet through shared memory, their row
//               sums at the end): one tcgen05.ld of the thread's 64 scores
//               (S is released at once), the causal
//               mask on the diagonal (and ragged last) tile only, the row max
//               on the raw scores (3-input max), one paired (f32x2) FMA per two
//               scores into ex2 (scale log2(e)/sqrt(d) folded in; for ALiBi the
//               bias -slope*(i-j), "Bloom in a sovereign engine",
//               Contribution, enters as +slope*j, the -slope*i part being
//               constant along the row), P rounded to the storage type and
//               written to TMEM (32 keys at a time) as the A operand of PV,
//               after PV_{j-1} has finished reading the previous P. O is rescaled in TMEM
//               only when the running max grows by more than 2^8. At the end
//               of an item O / l is read out of TMEM and written as [B, S, H, d].
// TMEM columns: S [0, 128), P [128, 192) (two 16-bit values per column),
// O [192, 192 + d).
// Query scale head_dim^-0.5 and GQA (kv head = h / (H/Hk)) follow nnterp
// "stablelm" 03 Notes.
#include "internal.h"

namespace blk {

namespace {

constexpr int kAttnThreads = 320;
constexpr int kBQ = 128;
constexpr int kBKV = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest unnormalised p
constexpr int kHalfKV = kBKV / 2;  // keys per softmax warp per tile
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;

template <int D>
struct AttnCfg {
    static constexpr int kSub = (D + 63) / 64;          // 64-column boxes per row
    static constexpr int kTileBytes = kSub * kBQ * 128;  // 128 rows x kSub x 128 B
    static constexpr int kStages = D > 128 ? 1 : 2;      // K/V ring depth
    static constexpr int kQBufs = 2;                     // next item's Q loads early
    static constexpr int kBarBytes = 256;
    static constexpr int kXchgBytes = 2 * 2 * kBQ * 4;  // [parity][half][row] floats
    static constexpr int kSmem =
        kTileBytes * (kQBufs + 2 * kStages) + 1024 + kBarBytes + kXchgBytes;
    static constexpr uint32_t kTmemCols = (kColO + D) <= 256 ? 256 : 512;
    static constexpr int kMinBlocks = kTmemCols == 256 ? 2 : 1;
};

// Walks this CTA's share of the (query tile, batch, head) items one 128-key
// tile at a time. Items are ordered heaviest (latest query tile) first and
// dealt to the CTAs in alternating directions (round r gives item
// r*G + blockIdx on even rounds, r*G + G-1-blockIdx on odd ones), which
// evens out the work per CTA.
struct TileCursor {
    int item, it, j, nkv, qt, b, h, g;
    bool valid;
    __device__ __forceinline__ int item_of(int round) const {
        const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
        return round * G + ((round & 1) ? G - 1 - c : c);
    }
    __device__ __forceinline__ void decode(const AttnArgs& a, int nq) {
        const int bh_count = a.B * a.H;
        qt = nq - 1 - item / bh_count;
        const int bh = item % bh_count;
        b = bh / a.H;
        h = bh - b * a.H;
        g = h / (a.H / a.Hk);
        nkv = qt + 1;
    }
    __device__ __forceinline__ void start(const AttnArgs& a, int nq, int n_items) {
        it = 0;
        item = item_of(0);
        j = 0;
        valid = item < n_items;
        if (valid) decode(a, nq);
    }
    __device__ __forceinline__ void advance(const AttnArgs& a, int nq, int n_items) {
        if (++j < nkv) return;
        j = 0;
        ++it;
        item = item_of(it);
        valid = item < n_items;
        if (valid) decode(a, nq);
    }
};

template <typename T, int D, bool ALIBI>
__global__ void __launch_bounds__(kAttnThreads, AttnCfg<D>::kMinBlocks)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
    using Cfg = AttnCfg<D>;
    constexpr int kStages = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const uint32_t sQ = smem_u32(smem);                    // Q buffer i at + i tiles
    const uint32_t sKV = sQ + Cfg::kQBufs * Cfg::kTileBytes;  // stage i: K at +2i, V at +2i+1
    uint64_t* bars = reinterpret_cast<uint64_t*>(
        smem + (Cfg::kQBufs + 2 * kStages) * Cfg::kTileBytes);
    float* xchg = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + Cfg::kBarBytes);
    const uint32_t bar0 = smem_u32(bars);
    // barrier map (8 bytes each)
    const uint32_t s_full = bar0 + 0;
    const uint32_t s_free = bar0 + 8;
    const uint32_t p_full = bar0 + 16;
    const uint32_t o_done = bar0 + 24;
    const uint32_t o_free = bar0 + 32;
    auto q_full = [&](int i) { return bar0 + 40u + 8u * i; };
    auto q_empty = [&](int i) { return bar0 + 56u + 8u * i; };
    auto x_bar = [&](int i) { return bar0 + 72u + 8u * i; };  // per lane quarter
    auto k_full = [&](int i) { return bar0 + 104u + 8u * i; };
    auto v_full = [&](int i) { return bar0 + 104u + 8u * (kStages + i); };
    auto k_empty = [&](int i) { return bar0 + 104u + 8u * (2 * kStages + i); };
    auto v_empty = [&](int i) { return bar0 + 104u + 8u * (3 * kStages + i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13 + 4 * kStages);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int nq = (a.S + kBQ - 1) / kBQ;
    const int n_items = nq * a.B * a.H;

    if (threadIdx.x == 0) {
        mbar_init(s_full, 1);
        mbar_init(s_free, 8);
        mbar_init(p_full, 8);
        mbar_init(o_done, 1);
        mbar_init(o_free, 8);
        for (int i = 0; i < 2; ++i) {
            mbar_init(q_full(i), 1);
            mbar_init(q_empty(i), 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(x_bar(i), 2);
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
            // producer: Q of each item, then its K/V tiles; the ring index is
            // this CTA's running tile count
            TileCursor c;
            c.start(a, nq, n_items);
            int gt = 0;
            bool ok = true;
            while (c.valid && ok) {
                if (c.j == 0) {
                    const int qb = c.it & 1;
                    if (!mbar_wait(q_empty(qb), ((c.it >> 1) & 1) ^ 1u, a.err)) break;
                    mbar_expect_tx(q_full(qb), Cfg::kTileBytes);
#pragma unroll
                    for (int sub = 0; sub < Cfg::kSub; ++sub)
                        tma_load_3d(sQ + qb * Cfg::kTileBytes + sub * kBQ * 128, &tmQ, q_full(qb),
                                    sub * 64, c.qt * kBQ, c.b * a.H + c.h);
                }
                const int st = gt % kStages;
                const uint32_t ph = (gt / kStages) & 1;
                const uint32_t sK = sKV + (2 * st) * Cfg::kTileBytes;
                const uint32_t sV = sK + Cfg::kTileBytes;
                if (!mbar_wait(k_empty(st), ph ^ 1u, a.err)) break;
                mbar_expect_tx(k_full(st), Cfg::kTileBytes);
#pragma unroll
                for (int sub = 0; sub < Cfg::kSub; ++sub)
                    tma_load_3d(sK + sub * kBKV * 128, &tmK, k_full(st), sub * 64, c.j * kBKV,
                                c.b * a.Hk + c.g);
                if (!mbar_wait(v_empty(st), ph ^ 1u, a.err)) break;
                mbar_expect_tx(v_full(st), Cfg::kTileBytes);
#pragma unroll
                for (int sub = 0; sub < Cfg::kSub; ++sub)
                    tma_load_3d(sV + sub * kBKV * 128, &tmV, v_full(st), sub * 64, c.j * kBKV,
                                c.b * a.Hk + c.g);
                c.advance(a, nq, n_items);
                ++gt;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer: the S cursor runs one tile ahead of the PV cursor, also
            // across item boundaries
            constexpr uint32_t fmt = dt_traits<T>::mma_fmt;
            constexpr uint32_t idesc_s = make_idesc_f16(fmt, kBQ, kBKV, false);
            constexpr uint32_t idesc_o = make_idesc_f16(fmt, kBQ, D, true);
            constexpr uint64_t kStageStep = (2 * Cfg::kTileBytes) >> 4;
            constexpr uint64_t kQStep = Cfg::kTileBytes >> 4;
            const uint64_t dq0 = make_sdesc_sw128(sQ, 16, 1024);
            const uint64_t dk0 = make_sdesc_sw128(sKV, 16, 1024);
            const uint64_t dv0 = make_sdesc_sw128(sKV + Cfg::kTileBytes, kBKV * 128, 1024);
            TileCursor cs, cp;
            cs.start(a, nq, n_items);
            cp.start(a, nq, n_items);
            int gs = 0, gp = 0;
            auto issue_s = [&]() -> bool {
                const int qb = cs.it & 1;
                if (cs.j == 0 && !mbar_wait(q_full(qb), (cs.it >> 1) & 1, a.err)) return false;
                const int st = gs % kStages;
                if (!mbar_wait(k_full(st), (gs / kStages) & 1, a.err)) return false;
                tc_fence_after();
                const uint64_t dq = dq0 + qb * kQStep;
                const uint64_t dk = dk0 + st * kStageStep;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    constexpr uint32_t kSubStep = (kBQ * 128) >> 4;
                    const uint64_t off = (ks / 4) * kSubStep + (ks % 4) * 2;
                    tc_mma_ss(tS, dq + off, dk + off, idesc_s, ks > 0 ? 1u : 0u);
                }
                tc_commit(s_full);
                tc_commit(k_empty(st));
                if (cs.j == cs.nkv - 1) tc_commit(q_empty(qb));
                cs.advance(a, nq, n_items);
                ++gs;
                return true;
            };
            bool ok = !cs.valid || issue_s();
            while (ok && cp.valid) {
                if (cs.valid) {
                    if (!mbar_wait(s_free, gp & 1, a.err)) break;
                    tc_fence_after();
                    if (!issue_s()) break;
                }
                const int st = gp % kStages;
                if (!mbar_wait(p_full, gp & 1, a.err)) break;
                if (!mbar_wait(v_full(st), (gp / kStages) & 1, a.err)) break;
                // the first PV of an item overwrites O: the previous item's O
                // must have been read out
                if (cp.j == 0 && cp.it > 0 && !mbar_wait(o_free, (cp.it - 1) & 1, a.err)) break;
                tc_fence_after();
                const uint64_t dv = dv0 + st * kStageStep;
#pragma unroll
                for (int ks = 0; ks < kBKV / 16; ++ks) {
                    tc_mma_ts(tO, tP + ks * 8, dv + ks * ((16 * 128) >> 4), idesc_o,
                              (cp.j > 0 || ks > 0) ? 1u : 0u);
                }
                tc_commit(o_done);
                tc_commit(v_empty(st));
                cp.advance(a, nq, n_items);
                ++gp;
            }
        }
    } else {
        // softmax warps 2..9: warps w and w + 4 share TMEM lane quarter w % 4
        // (rows quarter*32 .. +31); the first takes keys 0..63 of each tile,
        // the second keys 64..127 (and O columns [0, d/2) / [d/2, d)).
        const int quarter = warp & 3;
        const int half = (warp - 2) / 4;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t xbar = x_bar(quarter);
        float* xmax = xchg + row;  // [parity][half][128 rows]
        const float scale_l2 = a.scale * kLog2e;
        uint32_t xphase = 0;       // phases of this lane quarter's exchange barrier
        // the two halves swap one float per row through shared memory
        auto exchange = [&](float v) -> float {
            const int par = static_cast<int>(xphase);
            xmax[(par * 2 + half) * kBQ] = v;
            __syncwarp();
            if (lane == 0) mbar_arrive(xbar);
            if (!mbar_wait(xbar, xphase, a.err)) return NAN;
            xphase ^= 1u;
            return xmax[(par * 2 + (half ^ 1)) * kBQ];
        };
        TileCursor c;
        c.start(a, nq, n_items);
        int gt = 0;
        float m_used = -INFINITY;  // running max, log2 domain (scores * scale * log2 e)
        float l = 0.f;             // this warp's part of the row sum
        float slope_l2 = 0.f;
        bool ok = true;
        while (c.valid) {
            const int qpos = c.qt * kBQ + row;
            if (c.j == 0) {
                m_used = -INFINITY;
                l = 0.f;
                if constexpr (ALIBI) {
                    const float slope = a.slopes ? a.slopes[c.h]
                                                 : exp2f(-8.0f * static_cast<float>(c.h + 1) /
                                                         static_cast<float>(a.H));
                    slope_l2 = slope * kLog2e;
                }
            }
            if (!mbar_wait(s_full, gt & 1, a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int kbase = c.j * kBKV + half * kHalfKV;
            const bool masked = c.j == c.qt || c.j * kBKV + kBKV > a.S;
            const int lim = min(qpos, a.S - 1) - kbase;  // keys <= lim are visible
            uint32_t r[kHalfKV];
            tmem_ld64(tS + lane_off + half * kHalfKV, r);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            if constexpr (ALIBI) {
                // s * scale + slope * key_pos (the -slope * query_pos part is
                // constant along the row and cancels in the softmax)
                const float sk = slope_l2 * static_cast<float>(kbase);
#pragma unroll
                for (int i = 0; i < kHalfKV; ++i)
                    r[i] = __float_as_uint(fmaf(__uint_as_float(r[i]), scale_l2,
                                                fmaf(slope_l2, static_cast<float>(i), sk)));
            }
            if (masked) {
#pragma unroll
                for (int i = 0; i < kHalfKV; ++i)
                    if (i > lim) r[i] = __float_as_uint(-INFINITY);
            }
            float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
            for (int i = 0; i < kHalfKV; i += 4) {
                m0 = fmax3f(m0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                m1 = fmax3f(m1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
            }
            float mx = fmaxf(m0, m1);
            const float other = exchange(mx);
            if (isnan(other)) {
                ok = false;
                break;
            }
            mx = fmaxf(mx, other);
            if constexpr (!ALIBI) mx *= scale_l2;  // scale > 0: max commutes with it
            float corr = 1.f;
            if (mx > m_used + kRescaleThreshold) {
                corr = ex2_approx(m_used - mx);
                m_used = mx;
            }
            // PV of the previous tile must be done before O is rescaled and
            // before P is overwritten (the first tile of an item follows an
            // epilogue that waited for it)
            if (c.j > 0) {
                if (!mbar_wait(o_done, (gt - 1) & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[16];
                        const uint32_t col = tO + lane_off + half * (D / 2) + cc * 16;
                        tmem_ld16(col, o);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                        tmem_st16_nowait(col, o);
                    }
                }
            }
            // p = 2^(logit - m), this warp's row sum, P (storage type) into TMEM
            const uint64_t mul2 = f2_pack(ALIBI ? 1.f : scale_l2, ALIBI ? 1.f : scale_l2);
            const uint64_t neg2 = f2_pack(-m_used, -m_used);
            uint64_t acc2 = f2_pack(0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < kHalfKV / 32; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float e0, e1;
                    ffma2(__uint_as_float(r[cc * 32 + i]), __uint_as_float(r[cc * 32 + i + 1]),
                          mul2, neg2, e0, e1);
                    const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
                    fadd2_acc(acc2, p0, p1);
                    pk[i / 2] = dt_traits<T>::pack2(p0, p1);
                }
                tmem_st16_nowait(tP + lane_off + half * (kHalfKV / 2) + cc * 16, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            float sum0, sum1;
            f2_unpack(acc2, sum0, sum1);
            l = l * corr + (sum0 + sum1);

            if (c.j == c.nkv - 1) {
                // epilogue of the item: the row sum is the two halves' sums
                const float other_l = exchange(l);
                if (isnan(other_l) || !mbar_wait(o_done, gt & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float inv_l = 1.0f / (l + other_l);
                uint32_t o[D / 2];
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t(&oc)[16] = *reinterpret_cast<uint32_t(*)[16]>(&o[cc * 16]);
                    tmem_ld16(tO + lane_off + half * (D / 2) + cc * 16, oc);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free);
                if (qpos < a.S) {
                    T* dst = static_cast<T*>(a.o) +
                             ((static_cast<int64_t>(c.b) * a.S + qpos) * a.H + c.h) *
                                 static_cast<int64_t>(D) +
                             half * (D / 2);
#pragma unroll
                    for (int v = 0; v < D / 16; ++v) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[v * 8 + e]) * inv_l;
                        store8(dst + v * 8, f);
                    }
                }
            }
            c.advance(a, nq, n_items);
            ++gt;
        }
        (void)ok;
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
    {
        const cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), Cfg::kSmem);
        if (e != cudaSuccess) return e;
    }
    const int64_t items = static_cast<int64_t>((a.S + kBQ - 1) / kBQ) * a.B * a.H;
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    const int64_t slots = static_cast<int64_t>(Cfg::kMinBlocks) * a.num_sms;
    const int64_t grid = items < slots ? items : slots;
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
        case 64: return launch_attention_pair64(dt, a, s);
        case 128: return launch_attention_pair128(dt, a, s);
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
