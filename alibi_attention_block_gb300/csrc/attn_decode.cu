// K6: one decode step of causal attention over a KV cache (split-KV).
//
// Each sequence b has lens[b] tokens in the cache k/v [B, Hk, S_max, d]; its
// newest token's query q [B, H, d] (position lens[b] - 1) attends to all of
// them (the attention of nnterp "stablelm" 03 Notes; ALiBi as in "Bloom in
// a sovereign engine", Contribution: -slope * (i - j)). The work is a pass
// over the cache: 4 d bytes of K and V per key against 4 d flops per query
// head, so it is HBM bound and runs on the CUDA cores, not the tensor cores.
//
// Pass 1 (decode_partial_kernel): one warp per (b, kv head, part). A part is
// a contiguous range of keys; the warp keeps, for each of the kv head's
// query heads, the running max, the running sum and the unnormalised output
// (lane c owns output columns c*d/32 ..), and walks its range 32 keys at a
// time through its own three-stage shared-memory ring filled by cp.async
// (blocks i+1 and i+2 are in flight while block i is used, and in-flight
// data costs no registers): lane l scores key l against the queries
// (shared memory, broadcast), the warp takes the max and sum by shuffles
// and accumulates p * V reading one V row per key. Each part writes (max,
// sum, output) to the workspace.
// Pass 2 (decode_combine_kernel): one warp per (b, query head) merges the
// parts: o = sum_i e^{m_i - m} O_i / sum_i e^{m_i - m} l_i.
#include <type_traits>

#include "internal.h"

namespace blk {

namespace {

constexpr int kDecThreads = 128;  // combine kernel: 4 warps per block
constexpr float kLog2eDec = 1.4426950408889634f;

// Ring depth and warps per block: at head_dim 64 a three-stage ring is 24 KB
// a warp (eight warps per SM); at 128 a three-stage ring would be 48 KB and
// leave four warps per SM, one per scheduler, with nothing to hide the
// latencies of its shared-memory loads and shuffles, so there a two-stage
// ring in two-warp blocks gives six.
template <int D>
struct DecCfg {
    static constexpr int kStages = D > 64 ? 2 : 3;       // key blocks in flight per warp
    static constexpr int kWarps = D > 64 ? 2 : 4;        // warps per block
    static constexpr int kBlockBytes = 32 * D * 2;       // 32 K (or V) rows
    static constexpr int kStageBytes = 2 * kBlockBytes;  // K then V
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kSmem = kWarps * kWarpBytes;
};

// HS > 1 (head_dim 128, G >= 2): a block of HS warps shares one item and
// its ring, each warp taking G / HS of the kv head's query heads, so each
// warp does that share of the per-key work and an SM holds HS times the
// warps for the same ring space (the kernel is bound by the latency of its
// dependent work there, not by the bytes in flight).
template <typename T, int D, int G, int HS>
__global__ void __launch_bounds__(HS == 1 ? 32 * DecCfg<D>::kWarps : 32 * HS)
    decode_partial_kernel(DecodeArgs a) {
    using Cfg = DecCfg<D>;
    static_assert(HS == 1 || G % HS == 0, "head split: whole heads per warp");
    constexpr int kQW = HS == 1 ? Cfg::kWarps : HS;  // warps of the block
    constexpr int GW = G / HS;     // query heads of this warp
    constexpr int kCols = D / 32;  // output columns per lane
    constexpr int kChunks = D / 8; // 16-byte pieces per row
    __shared__ __align__(16) float qs[kQW][GW][D];  // each warp's queries, pre-scaled (log2)
    extern __shared__ __align__(128) uint8_t dsm[];
    const int lane = threadIdx.x & 31;
    const int wl = threadIdx.x / 32;
    const int64_t wid = HS == 1 ? static_cast<int64_t>(blockIdx.x) * Cfg::kWarps + wl
                                : static_cast<int64_t>(blockIdx.x);
    const int64_t total = static_cast<int64_t>(a.B) * a.Hk * a.parts;
    if (wid >= total) return;  // whole warps (for HS = 2 the whole block) exit together
    const uint32_t ring = smem_u32(dsm) + (HS == 1 ? wl * Cfg::kWarpBytes : 0);
    const int h0 = HS == 1 ? 0 : wl * GW;  // this warp's first query head of the group
    const int part = static_cast<int>(wid % a.parts);
    const int bg = static_cast<int>(wid / a.parts);
    const int b = bg / a.Hk;
    const int g = bg - b * a.Hk;
    // lengths live in device memory: clamp to [0, S_max] so that a bad one
    // reads nothing outside the cache (a sequence of length 0 gets zeros)
    const int n = min(max(a.lens[b], 0), a.S_max);
    const int per = (a.S_max + a.parts - 1) / a.parts;
    const int j0 = part * per;
    const int j1 = min(n, j0 + per);
    const int nblk = j1 > j0 ? (j1 - j0 + 31) / 32 : 0;
    const float qscale = a.scale * kLog2eDec;
    const T* qp = static_cast<const T*>(a.q) + (static_cast<int64_t>(b) * a.H + g * G + h0) * D;
    for (int i = lane; i < GW * D / 8; i += 32) {
        float f[8];
        load8(qp + i * 8, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) qs[wl][(i * 8) / D][(i * 8) % D + e] = f[e] * qscale;
    }
    float slope[GW];
#pragma unroll
    for (int h = 0; h < GW; ++h) {
        slope[h] = 0.f;
        if (a.alibi) {
            const int hq = g * G + h0 + h;
            const float sl = a.slopes ? a.slopes[hq]
                                      : exp2f(-8.0f * static_cast<float>(hq + 1) /
                                              static_cast<float>(a.H));
            slope[h] = sl * kLog2eDec;
        }
    }
    const int64_t kv_base = (static_cast<int64_t>(b) * a.Hk + g) * a.S_max;
    const T* kp = static_cast<const T*>(a.k) + kv_base * D;
    const T* vp = static_cast<const T*>(a.v) + kv_base * D;
    // copy key block i into its stage: K rows with their 16-byte pieces
    // XOR-swizzled by row (conflict-free when lane l reads row l), V rows
    // plain (lanes read one row together); rows past the range are zeros
    // (HS = 2: the block's 64 threads share the copies)
    auto issue = [&](int i) {
        if (i < nblk) {
            const int jb = j0 + i * 32;
            const uint32_t st = ring + (i % Cfg::kStages) * Cfg::kStageBytes;
#pragma unroll
            for (int q = HS == 1 ? lane : static_cast<int>(threadIdx.x); q < 32 * kChunks;
                 q += 32 * HS) {
                const int r = q / kChunks, c = q % kChunks;
                const bool ok = jb + r < j1;
                const int64_t src = static_cast<int64_t>(ok ? jb + r : j0) * D + c * 8;
                cp_async16(st + r * (D * 2) + ((c ^ (r & 7)) << 4), kp + src, ok ? 16u : 0u);
                cp_async16(st + Cfg::kBlockBytes + r * (D * 2) + (c << 4), vp + src, ok ? 16u : 0u);
            }
        }
        cp_async_commit();  // one group per block index, empty past the end
    };
    float m[GW], l[GW], acc[GW][kCols];
#pragma unroll
    for (int h = 0; h < GW; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int c = 0; c < kCols; ++c) acc[h][c] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < Cfg::kStages - 1; ++i) issue(i);
    if (HS == 1) __syncwarp();
    else __syncthreads();  // the queries of both warps are in place
    const float qpos = static_cast<float>(n - 1);
    const uint32_t qs_addr = smem_u32(&qs[wl][0][0]);
    for (int i = 0; i < nblk; ++i) {
        issue(i + Cfg::kStages - 1);
        cp_async_wait<Cfg::kStages - 1>();  // block i has landed (this thread's copies)
        if (HS == 1) __syncwarp();          // ... and every lane's
        else __syncthreads();               // ... and every thread's of the block
        const uint32_t st = ring + (i % Cfg::kStages) * Cfg::kStageBytes;
        const int jb = j0 + i * 32;
        const int j = jb + lane;
        const bool valid = j < j1;
        // scores of key j against the G queries (log2 domain): paired
        // (f32x2) FMAs over even and odd dims, the queries read 16 bytes at
        // a time (the same address in every lane: a broadcast)
        uint64_t sc2[GW];
#pragma unroll
        for (int h = 0; h < GW; ++h) sc2[h] = f2_pack(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            const uint4 kv = ld_shared_u4(st + lane * (D * 2) + ((c ^ (lane & 7)) << 4));
            const uint32_t w4[4] = {kv.x, kv.y, kv.z, kv.w};
            uint64_t k2[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const float2 kf = dt_traits<T>::unpack2(w4[e2]);
                k2[e2] = f2_pack(kf.x, kf.y);
            }
#pragma unroll
            for (int h = 0; h < GW; ++h) {
                uint64_t q0, q1, q2, q3;
                ld_shared_v2_u64(qs_addr + (h * D + c * 8) * 4, q0, q1);
                ld_shared_v2_u64(qs_addr + (h * D + c * 8 + 4) * 4, q2, q3);
                ffma2_acc(sc2[h], q0, k2[0]);
                ffma2_acc(sc2[h], q1, k2[1]);
                ffma2_acc(sc2[h], q2, k2[2]);
                ffma2_acc(sc2[h], q3, k2[3]);
            }
        }
        float sc[GW];
#pragma unroll
        for (int h = 0; h < GW; ++h) {
            float lo, hi;
            f2_unpack(sc2[h], lo, hi);
            sc[h] = lo + hi;
        }
#pragma unroll
        for (int h = 0; h < GW; ++h) {
            float s = valid ? sc[h] - slope[h] * (qpos - static_cast<float>(j)) : -INFINITY;
            float mb = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
            const float mn = fmaxf(m[h], mb);  // finite: key jb is valid
            const float corr = exp2f(m[h] - mn);
            const float p = exp2f(s - mn);
            float ps = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            l[h] = l[h] * corr + ps;
            m[h] = mn;
#pragma unroll
            for (int c = 0; c < kCols; ++c) acc[h][c] *= corr;
            sc[h] = p;  // 0 for keys past the range (their V rows are zeros)
        }
        // O += p V over the block's keys
        const uint32_t vrow0 = st + Cfg::kBlockBytes + lane * (kCols * 2);
#pragma unroll 8
        for (int t = 0; t < 32; ++t) {
            float vf[kCols];
            if constexpr (kCols == 2) {
                uint32_t u;
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(u) : "r"(vrow0 + t * (D * 2)));
                const float2 f = dt_traits<T>::unpack2(u);
                vf[0] = f.x;
                vf[1] = f.y;
            } else {
                uint32_t u0, u1;
                asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                             : "=r"(u0), "=r"(u1)
                             : "r"(vrow0 + t * (D * 2)));
                const float2 f0 = dt_traits<T>::unpack2(u0), f1 = dt_traits<T>::unpack2(u1);
                vf[0] = f0.x;
                vf[1] = f0.y;
                vf[2] = f1.x;
                vf[3] = f1.y;
            }
#pragma unroll
            for (int h = 0; h < GW; ++h) {
                const float pt = __shfl_sync(0xffffffffu, sc[h], t);
#pragma unroll
                for (int c = 0; c < kCols; ++c) acc[h][c] = fmaf(pt, vf[c], acc[h][c]);
            }
        }
        if (HS == 1) __syncwarp();  // the stage is refilled by the next issue
        else __syncthreads();      // (both warps done with it)
    }
    cp_async_wait<0>();
    // (max, sum, output) of this part for each query head; an empty part
    // (j0 >= n) writes max = -inf, sum = 0
    float* rec = a.ws + (static_cast<int64_t>(b) * a.H + g * G + h0) * a.parts * (D + 2);
#pragma unroll
    for (int h = 0; h < GW; ++h) {
        float* r = rec + (static_cast<int64_t>(h) * a.parts + part) * (D + 2);
        if (lane == 0) {
            r[0] = m[h];
            r[1] = l[h];
        }
#pragma unroll
        for (int c = 0; c < kCols; ++c) r[2 + lane * kCols + c] = acc[h][c];
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kDecThreads) decode_combine_kernel(DecodeArgs a) {
    constexpr int kCols = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * 4 + threadIdx.x / 32;
    if (wid >= static_cast<int64_t>(a.B) * a.H) return;
    const float* rec = a.ws + wid * a.parts * (D + 2);
    float mx = -INFINITY;
    for (int p = 0; p < a.parts; ++p) mx = fmaxf(mx, rec[p * (D + 2)]);
    float lsum = 0.f, o[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) o[c] = 0.f;
    for (int p = 0; p < a.parts; ++p) {
        const float* r = rec + p * (D + 2);
        const float w = r[0] == -INFINITY ? 0.f : exp2f(r[0] - mx);  // 0 for an empty part
        lsum = fmaf(w, r[1], lsum);
#pragma unroll
        for (int c = 0; c < kCols; ++c) o[c] = fmaf(w, r[2 + lane * kCols + c], o[c]);
    }
    const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
    T* dst = static_cast<T*>(a.o) + wid * D + lane * kCols;
#pragma unroll
    for (int c = 0; c < kCols; c += 2)
        *reinterpret_cast<uint32_t*>(dst + c) = dt_traits<T>::pack2(o[c] * inv, o[c + 1] * inv);
}

template <typename T, int D, int G>
cudaError_t launch_g(const DecodeArgs& a, cudaStream_t s) {
    const int64_t items = static_cast<int64_t>(a.B) * a.Hk * a.parts;
    constexpr int kW = DecCfg<D>::kWarps;
    // head_dim 128 with G >= 2: a block of two warps per item sharing one
    // ring (four, each with a quarter of the heads, measured slower: every
    // warp reads all of the block's K rows from shared memory)
    constexpr int HS = (D == 128 && G >= 2) ? 2 : 1;
    constexpr int kSmem = HS == 1 ? DecCfg<D>::kSmem : DecCfg<D>::kWarpBytes;
    auto kern = decode_partial_kernel<T, D, G, HS>;
    {
        const cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), kSmem);
        if (e != cudaSuccess) return e;
    }
    const int64_t blocks = HS == 1 ? (items + kW - 1) / kW : items;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    kern<<<static_cast<unsigned>(blocks), HS == 1 ? 32 * kW : 32 * HS, kSmem, s>>>(a);
    const int64_t cw = static_cast<int64_t>(a.B) * a.H;
    decode_combine_kernel<T, D><<<static_cast<unsigned>((cw + 3) / 4), kDecThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
    switch (a.H / a.Hk) {
        case 1: return launch_g<T, D, 1>(a, s);
        case 2: return launch_g<T, D, 2>(a, s);
        case 4: return launch_g<T, D, 4>(a, s);
        case 8: return launch_g<T, D, 8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t s) {
    switch (a.d) {
        case 64: return launch_d<T, 64>(a, s);
        case 128: return launch_d<T, 128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int decode_parts_max(int64_t S_max) {
    const int64_t most = (S_max + 63) / 64;
    return static_cast<int>(most < 256 ? most : 256);
}

int decode_parts(int64_t B, int64_t Hk, int64_t S_max, int64_t head_dim, int num_sms) {
    // at least 64 keys per part; head_dim 64: about 16 warps per SM in all
    // (two rounds of the eight resident); head_dim 128: one round of the six
    // resident warps, each with a longer range, so its two-stage ring stays
    // full and no partial round is left
    const int64_t want = head_dim > 64 ? (6LL * num_sms) / (B * Hk)
                                       : (16LL * num_sms + B * Hk - 1) / (B * Hk);
    const int64_t most = decode_parts_max(S_max);
    int64_t p = want < most ? want : most;
    if (p < 1) p = 1;
    if (p > 256) p = 256;
    return static_cast<int>(p);
}

cudaError_t launch_attention_decode(DType dt, const DecodeArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    if (dt == DType::F16) return launch_t<__half>(a, s);
    return launch_t<__nv_bfloat16>(a, s);
}

}  // namespace blk
