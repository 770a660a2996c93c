// K3 for grouped-query attention at head_dim 128 and 160: the query heads
// that share one key/value head are packed into the rows of one 128-row
// query tile, so every K/V tile a CTA loads serves the whole group.
//
// GQA (nnterp "stablelm", 03 Notes: on the 12B model kv head j serves query
// heads 4j .. 4j+3; kv head = h / (H/Hk)). With G = H/Hk query heads per kv
// head, a tile holds Gt = min(G, 16) of them (all G unless G > 16; a larger
// group is split into chunks of Gt heads) and R = 128/Gt consecutive
// positions (rounded down to a multiple of 8) of each: row r is head
// g*G + chunk*Gt + r/R at position p0 + r%R. MHA (G = 1) is the plain
// 128-position tile. The scores S = Q K^T of one 128-key tile are then one
// M=128, N=128 product for all G heads at once, and one PV product
// (M=128, N=d) follows it; both run at the tensor core's full-size shapes
// (K=d for S, N=d for PV), with each K/V tile read from L2 once per group
// and position block instead of once per head. Work items are
// (position block, batch, kv head, head chunk), latest (heaviest) blocks
// first, dealt to the persistent CTAs in alternating directions.
//
// 6 warps, one CTA per SM:
//   warp 0      TMA: the item's Q tile (G boxes of R rows per 64-column
//               slice), then K tiles one ahead of V tiles (each 128 keys,
//               128-byte swizzle, zero fill past S), K and V in rings of
//               their own; K and V load with an evict-last L2 policy (other
//               position blocks of the group read the same key prefix), Q
//               evict-first
//   warp 1      TMEM allocator and single-thread MMA issuer, in the order
//               S(0), S(1), PV(0), S(2), PV(1), ...: S is double-buffered in
//               TMEM, so the next tile's scores are computed while the
//               softmax works on this one
//   warps 2..5  softmax, one thread per query row (TMEM lane; a warp reaches
//               the lane quarter of its index mod 4): one tcgen05.ld of the
//               row's 128 scores (the S buffer is released at once), the
//               causal mask on the key tiles past the block's first
//               position, the row max (3-input max), one paired (f32x2) FMA
//               per two scores into ex2 (scale log2(e)/sqrt(d) folded in;
//               ALiBi, "Bloom in a sovereign engine", Contribution, enters as
//               +slope*key with the row's own head slope), P packed to the
//               storage type in registers and stored to TMEM once the
//               previous PV has read the old P. O is rescaled in TMEM only
//               when the running max grows by more than 2^8. An item's O / l
//               is read out and written as [B, S, H, d] during the first
//               tile of the next item, so no softmax waits on a last PV.
// TMEM columns: S0 [0, 128), S1 [128, 256), P [256, 320) (two 16-bit values
// per column), O [320, 320 + d).
// Query scale head_dim^-0.5 follows nnterp "stablelm" 03 Notes.
#include "internal.h"

namespace blk {

namespace {

constexpr int kGqaThreads = 192;
constexpr int kTQ = 128;  // query rows per tile (G heads x R positions)
constexpr int kTK = 128;  // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest unnormalised p
constexpr uint32_t kColP = 256, kColO = 320;

template <int D>
struct GqaCfg {
    static_assert(D == 128 || D == 160, "GQA-packed attention is built for head_dim 128 and 160");
    static constexpr int kSub = (D + 63) / 64;          // 64-column slices per row
    static constexpr int kTileBytes = kSub * 128 * 128;  // 128 rows x kSub x 128 B
    static constexpr int kQBufs = D > 128 ? 1 : 2;
    static constexpr int kKStages = 2;
    static constexpr int kVStages = D > 128 ? 1 : 2;
    static constexpr int kOffK = kQBufs * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
    static constexpr int kSmem = kOffBar + 256 + 1024;   // + barriers + alignment slack
    static constexpr uint32_t kTmemCols = 512;
};

// Packing of a group's query heads into 128-row tiles.
struct GqaPack {
    int G;     // query heads per kv head
    int Gt;    // query heads per tile
    int R;     // positions per head in a tile (multiple of 8)
    int nhc;   // head chunks per group
};

// This CTA's items: (position block pb, batch b, kv head g, head chunk hc).
// Round r gives item r*Gd + blockIdx on even rounds and r*Gd + Gd-1-blockIdx
// on odd ones (Gd = grid size); items are numbered latest block first.
struct GqaCursor {
    int item, it, pb, b, g, hc, p0, nkv;
    bool valid;
    __device__ __forceinline__ int item_of(int round) const {
        const int Gd = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
        return round * Gd + ((round & 1) ? Gd - 1 - c : c);
    }
    __device__ __forceinline__ void decode(const AttnArgs& a, const GqaPack& pk, int nblk) {
        const int per_block = a.B * a.Hk * pk.nhc;
        pb = nblk - 1 - item / per_block;
        int rest = item % per_block;
        hc = rest % pk.nhc;
        rest /= pk.nhc;
        b = rest / a.Hk;
        g = rest - b * a.Hk;
        p0 = pb * pk.R;
        const int last = min(p0 + pk.R, a.S);  // one past the block's last position
        nkv = (last + kTK - 1) / kTK;
    }
    __device__ __forceinline__ void start(const AttnArgs& a, const GqaPack& pk, int nblk,
                                          int n_items) {
        it = 0;
        item = item_of(0);
        valid = item < n_items;
        if (valid) decode(a, pk, nblk);
    }
    __device__ __forceinline__ void next(const AttnArgs& a, const GqaPack& pk, int nblk,
                                         int n_items) {
        ++it;
        item = item_of(it);
        valid = item < n_items;
        if (valid) decode(a, pk, nblk);
    }
};

template <typename T, int D, bool ALIBI>
__global__ void __launch_bounds__(kGqaThreads, 1)
    attn_gqa_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnArgs a,
                    const GqaPack pk) {
    using Cfg = GqaCfg<D>;
    constexpr int kQB = Cfg::kQBufs, kKS = Cfg::kKStages, kVS = Cfg::kVStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + Cfg::kOffK;
    const uint32_t sV = sQ + Cfg::kOffV;
    const uint32_t bar0 = sQ + Cfg::kOffBar;
    // barriers (8 bytes each)
    auto s_full = [&](int i) { return bar0 + 8u * i; };
    auto s_free = [&](int i) { return bar0 + 16u + 8u * i; };
    const uint32_t p_full = bar0 + 32u;
    const uint32_t pv_done = bar0 + 40u;
    const uint32_t o_free = bar0 + 48u;
    auto q_full = [&](int i) { return bar0 + 56u + 8u * i; };
    auto q_empty = [&](int i) { return bar0 + 72u + 8u * i; };
    auto k_full = [&](int i) { return bar0 + 88u + 8u * i; };
    auto k_empty = [&](int i) { return bar0 + 104u + 8u * i; };
    auto v_full = [&](int i) { return bar0 + 120u + 8u * i; };
    auto v_empty = [&](int i) { return bar0 + 136u + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffBar + 152);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int G = pk.G, R = pk.R;
    const int nblk = (a.S + R - 1) / R;
    const int n_items = nblk * a.B * a.Hk * pk.nhc;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(s_free(x), 4);
            mbar_init(q_full(x), 1);
            mbar_init(q_empty(x), 1);
            mbar_init(k_full(x), 1);
            mbar_init(k_empty(x), 1);
            mbar_init(v_full(x), 1);
            mbar_init(v_empty(x), 1);
        }
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(o_free, 4);
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

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_kv = l2_evict_last_policy(), pol_q = l2_evict_first_policy();
            GqaCursor c;
            c.start(a, pk, nblk, n_items);
            int gk = 0, gv = 0;  // K and V tiles loaded so far (ring positions)
            bool ok = true;
            auto load_k = [&](int j) -> bool {
                const int st = gk % kKS;
                if (!mbar_wait(k_empty(st), ((gk / kKS) & 1) ^ 1u, a.err)) return false;
                mbar_expect_tx(k_full(st), Cfg::kTileBytes);
#pragma unroll
                for (int sub = 0; sub < Cfg::kSub; ++sub)
                    tma_load_3d_hint(sK + st * Cfg::kTileBytes + sub * kTK * 128, &tmK, k_full(st),
                                sub * 64, j * kTK, c.b * a.Hk + c.g, pol_kv);
                ++gk;
                return true;
            };
            auto load_v = [&](int j) -> bool {
                const int st = gv % kVS;
                if (!mbar_wait(v_empty(st), ((gv / kVS) & 1) ^ 1u, a.err)) return false;
                mbar_expect_tx(v_full(st), Cfg::kTileBytes);
#pragma unroll
                for (int sub = 0; sub < Cfg::kSub; ++sub)
                    tma_load_3d_hint(sV + st * Cfg::kTileBytes + sub * kTK * 128, &tmV, v_full(st),
                                sub * 64, j * kTK, c.b * a.Hk + c.g, pol_kv);
                ++gv;
                return true;
            };
            while (ok && c.valid) {
                const int qb = c.it % kQB;
                if (!mbar_wait(q_empty(qb), ((c.it / kQB) & 1) ^ 1u, a.err)) break;
                // one box of R rows per head of the chunk and 64-column
                // slice; rows past the chunk's heads keep stale values and are
                // never written out
                const int nh = min(pk.Gt, G - c.hc * pk.Gt);
                mbar_expect_tx(q_full(qb), static_cast<uint32_t>(Cfg::kSub * nh * R * 128));
                for (int i = 0; i < nh; ++i) {
#pragma unroll
                    for (int sub = 0; sub < Cfg::kSub; ++sub)
                        tma_load_3d_hint(sQ + qb * Cfg::kTileBytes + sub * kTQ * 128 + i * R * 128,
                                    &tmQ, q_full(qb), sub * 64, c.p0,
                                    c.b * a.H + c.g * G + c.hc * pk.Gt + i, pol_q);
                }
                // consumption order: K(0), then K(j+1) ahead of V(j)
                ok = load_k(0);
                for (int j = 0; ok && j < c.nkv; ++j) {
                    if (j + 1 < c.nkv) ok = load_k(j + 1);
                    if (ok) ok = load_v(j);
                }
                c.next(a, pk, nblk, n_items);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t fmt = dt_traits<T>::mma_fmt;
            constexpr uint32_t idesc_s = make_idesc_f16(fmt, kTQ, kTK, false);
            constexpr uint32_t idesc_o = make_idesc_f16(fmt, kTQ, D, true);
            constexpr uint64_t kTileStep = Cfg::kTileBytes >> 4;
            constexpr uint64_t kSubStep = (kTQ * 128) >> 4;  // next 64-column slice
            const uint64_t dq0 = make_sdesc_sw128(sQ, 16, 1024);
            const uint64_t dk0 = make_sdesc_sw128(sK, 16, 1024);
            const uint64_t dv0 = make_sdesc_sw128(sV, kTK * 128, 1024);
            const uint32_t tP = tmem_base + kColP;
            const uint32_t tO = tmem_base + kColO;
            int gk = 0, gv = 0, gs = 0, gp = 0, itx = 0;
            // S(buffer gs % 2) = Q K^T, once the softmax has read that buffer's
            // previous scores
            auto issue_s = [&](uint64_t dq) -> bool {
                const int st = gk % kKS;
                const int sb = gs & 1;
                if (!mbar_wait(k_full(st), (gk / kKS) & 1, a.err)) return false;
                if (gs >= 2 && !mbar_wait(s_free(sb), ((gs >> 1) - 1) & 1, a.err)) return false;
                tc_fence_after();
                const uint64_t dk = dk0 + st * kTileStep;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t off = (ks / 4) * kSubStep + (ks % 4) * 2;
                    tc_mma_ss(tmem_base + 128u * sb, dq + off, dk + off, idesc_s, ks > 0 ? 1u : 0u);
                }
                tc_commit(s_full(sb));
                tc_commit(k_empty(st));
                ++gk;
                ++gs;
                return true;
            };
            // O += P V once the softmax has written P (the first PV of an item
            // overwrites O, so it also waits for the previous item's read-out)
            auto issue_pv = [&](bool first) -> bool {
                const int st = gv % kVS;
                if (!mbar_wait(v_full(st), (gv / kVS) & 1, a.err)) return false;
                if (!mbar_wait(p_full, gp & 1, a.err)) return false;
                if (first && itx > 0 && !mbar_wait(o_free, (itx - 1) & 1, a.err)) return false;
                tc_fence_after();
                const uint64_t dv = dv0 + st * kTileStep;
#pragma unroll
                for (int ks = 0; ks < kTK / 16; ++ks)
                    tc_mma_ts(tO, tP + ks * 8, dv + ks * ((16 * 128) >> 4), idesc_o,
                              (!first || ks > 0) ? 1u : 0u);
                tc_commit(pv_done);
                tc_commit(v_empty(st));
                ++gv;
                ++gp;
                return true;
            };
            GqaCursor c;
            c.start(a, pk, nblk, n_items);
            bool ok = true;
            while (ok && c.valid) {
                const int qb = c.it % kQB;
                if (!mbar_wait(q_full(qb), (c.it / kQB) & 1, a.err)) break;
                const uint64_t dq = dq0 + qb * kTileStep;
                ok = issue_s(dq);
                if (ok && c.nkv == 1) tc_commit(q_empty(qb));
                for (int j = 0; ok && j < c.nkv; ++j) {
                    if (j + 1 < c.nkv) {
                        ok = issue_s(dq);
                        if (ok && j + 2 == c.nkv) tc_commit(q_empty(qb));
                    }
                    if (ok) ok = issue_pv(j == 0);
                }
                ++itx;
                c.next(a, pk, nblk, n_items);
            }
        }
    } else {
        // softmax: warp w reads TMEM lanes 32 (w % 4) .. +31, one query row
        // per thread
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tO = tmem_base + kColO;
        const uint32_t tP = tmem_base + kColP;
        const float scale_l2 = a.scale * kLog2e;
        const int hl = row / R;          // head of this row within the tile
        const int rpos = row - hl * R;   // position offset within the block
        float slope_l2 = 0.f;
        GqaCursor c;
        c.start(a, pk, nblk, n_items);
        int g = 0;  // key tiles processed (across items)
        bool ok = true;
        bool pend = false;      // an item's O is still in TMEM
        float pend_l = 0.f;
        int64_t pend_row = -1;  // output row (b * S + pos) * H + h, or -1
        while (ok && c.valid) {
            const int pos = c.p0 + rpos;
            // rows past the chunk's heads are padding
            const bool in_group = hl < pk.Gt && c.hc * pk.Gt + hl < G;
            const int h = c.g * G + (in_group ? c.hc * pk.Gt + hl : 0);
            if constexpr (ALIBI) {
                const float slope = a.slopes ? a.slopes[h]
                                             : exp2f(-8.0f * static_cast<float>(h + 1) /
                                                     static_cast<float>(a.H));
                slope_l2 = slope * kLog2e;
            }
            const int lim_abs = min(pos, a.S - 1);  // keys <= lim_abs are visible
            float m_used = -INFINITY;  // running max, log2 domain
            float l = 0.f;
            for (int j = 0; j < c.nkv; ++j, ++g) {
                const int sb = g & 1;
                if (!mbar_wait(s_full(sb), (g >> 1) & 1, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t r[kTK];
                tmem_ld128(tmem_base + 128u * sb + lane_off, r);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free(sb));
                const int kbase = j * kTK;
                if constexpr (ALIBI) {
                    const float sk = slope_l2 * static_cast<float>(kbase);
#pragma unroll
                    for (int i = 0; i < kTK; ++i)
                        r[i] = __float_as_uint(fmaf(__uint_as_float(r[i]), scale_l2,
                                                    fmaf(slope_l2, static_cast<float>(i), sk)));
                }
                if (kbase + kTK - 1 > c.p0 || kbase + kTK > a.S) {
                    const int lim = lim_abs - kbase;
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
                if constexpr (!ALIBI) mx *= scale_l2;  // scale > 0: max commutes with it
                float corr = 1.f;
                if (mx > m_used + kRescaleThreshold) {
                    corr = ex2_approx(m_used - mx);
                    m_used = mx;
                }
                // a row with no visible key in this tile and none before it
                // (possible only for padding rows) keeps m = -inf: use 0
                const float m_eff = m_used == -INFINITY ? 0.f : m_used;
                const uint64_t mul2 = f2_pack(ALIBI ? 1.f : scale_l2, ALIBI ? 1.f : scale_l2);
                const uint64_t neg2 = f2_pack(-m_eff, -m_eff);
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
                // the previous PV has read P and O is settled: read out the
                // previous item's O if pending, publish P, rescale O if the
                // max moved (before this tile's PV)
                if (j > 0 || pend) {
                    if (!mbar_wait(pv_done, (g - 1) & 1, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                if (j == 0 && pend) {
                    float inv_l = pend_l > 0.f ? 1.0f / pend_l : 0.f;
                    T* dst = pend_row >= 0 ? static_cast<T*>(a.o) + pend_row * static_cast<int64_t>(D)
                                           : nullptr;
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + lane_off + cc * 32, o);
                        if (dst) {
                            float f[32];
#pragma unroll
                            for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(o[e]) * inv_l;
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                store8(dst + cc * 32 + v * 8,
                                       *reinterpret_cast<const float(*)[8]>(&f[v * 8]));
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(o_free);
                    pend = false;
                }
                tmem_st64_nowait(tP + lane_off, *reinterpret_cast<const uint32_t(*)[64]>(pk));
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
                if (lane == 0) mbar_arrive(p_full);
                float s0, s1, s2, s3;
                f2_unpack(acc0, s0, s1);
                f2_unpack(acc1, s2, s3);
                l = l * corr + ((s0 + s1) + (s2 + s3));
            }
            if (!ok) break;
            pend = true;
            pend_l = l;
            pend_row = (in_group && pos < a.S) ? (static_cast<int64_t>(c.b) * a.S + pos) * a.H + h
                                               : -1;
            c.next(a, pk, nblk, n_items);
        }
        // the last item's O
        if (ok && pend && mbar_wait(pv_done, (g - 1) & 1, a.err)) {
            tc_fence_after();
            const float inv_l = pend_l > 0.f ? 1.0f / pend_l : 0.f;
            T* dst = pend_row >= 0 ? static_cast<T*>(a.o) + pend_row * static_cast<int64_t>(D)
                                   : nullptr;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32(tO + lane_off + cc * 32, o);
                if (dst) {
                    float f[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(o[e]) * inv_l;
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        store8(dst + cc * 32 + v * 8, *reinterpret_cast<const float(*)[8]>(&f[v * 8]));
                }
            }
            tc_fence_before();
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

template <typename T, int D, bool ALIBI>
cudaError_t launch_gqa_d(DType dt, const AttnArgs& a, const GqaPack& pk, cudaStream_t s) {
    const int R = pk.R;
    using Cfg = GqaCfg<D>;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_3d(&tq, dt, a.q, static_cast<uint64_t>(a.B) * a.H, a.S, D, R) ||
        !make_tmap_3d(&tk, dt, a.k, static_cast<uint64_t>(a.B) * a.Hk, a.S, D, kTK) ||
        !make_tmap_3d(&tv, dt, a.v, static_cast<uint64_t>(a.B) * a.Hk, a.S, D, kTK))
        return cudaErrorInvalidValue;
    auto kern = attn_gqa_kernel<T, D, ALIBI>;
    {
        const cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), Cfg::kSmem);
        if (e != cudaSuccess) return e;
    }
    const int64_t items = static_cast<int64_t>((a.S + R - 1) / R) * a.B * a.Hk * pk.nhc;
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    const int64_t grid = items < a.num_sms ? items : a.num_sms;
    AttnArgs ap = a;
    ap.pdl = pdl_allowed(s);
    (void)launch_pdl(ap.pdl != 0, kern, dim3(static_cast<unsigned>(grid)), dim3(kGqaThreads), Cfg::kSmem, s,
                     tq, tk, tv, ap, pk);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_gqa_a(DType dt, const AttnArgs& a, const GqaPack& pk, cudaStream_t s) {
    return a.alibi ? launch_gqa_d<T, D, true>(dt, a, pk, s)
                   : launch_gqa_d<T, D, false>(dt, a, pk, s);
}

}  // namespace

cudaError_t launch_attention_gqa(DType dt, const AttnArgs& a, cudaStream_t s) {
    if (a.Hk <= 0 || a.H % a.Hk || (a.d != 128 && a.d != 160)) return cudaErrorInvalidValue;
    if (a.B == 0 || a.S == 0) return cudaSuccess;
    GqaPack pk;
    pk.G = a.H / a.Hk;
    pk.Gt = pk.G < 16 ? pk.G : 16;
    pk.R = (kTQ / pk.Gt) / 8 * 8;
    pk.nhc = (pk.G + pk.Gt - 1) / pk.Gt;
    if (dt == DType::F16)
        return a.d == 128 ? launch_gqa_a<__half, 128>(dt, a, pk, s)
                          : launch_gqa_a<__half, 160>(dt, a, pk, s);
    return a.d == 128 ? launch_gqa_a<__nv_bfloat16, 128>(dt, a, pk, s)
                      : launch_gqa_a<__nv_bfloat16, 160>(dt, a, pk, s);
}

}  // namespace blk
