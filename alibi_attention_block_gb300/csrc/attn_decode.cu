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
// time: lane l takes key l, computes its scores from 16-byte loads of its K
// row against the queries (shared memory, broadcast), then the warp takes
// the max and sum by shuffles and accumulates p * V with one coalesced load
// of each V row. Each part writes (max, sum, output) to the workspace.
// Pass 2 (decode_combine_kernel): one warp per (b, query head) merges the
// parts: o = sum_i e^{m_i - m} O_i / sum_i e^{m_i - m} l_i.
#include "internal.h"

namespace blk {

namespace {

constexpr int kDecThreads = 128;  // 4 warps per block, one part each
constexpr float kLog2eDec = 1.4426950408889634f;

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecThreads) decode_partial_kernel(DecodeArgs a) {
    constexpr int kCols = D / 32;  // output columns per lane
    __shared__ float qs[4][G][D];  // this warp's queries, pre-scaled (log2 domain)
    const int lane = threadIdx.x & 31;
    const int wl = threadIdx.x / 32;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * 4 + wl;
    const int64_t total = static_cast<int64_t>(a.B) * a.Hk * a.parts;
    if (wid >= total) return;  // whole warps exit together
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
    const float qscale = a.scale * kLog2eDec;
    const T* qp = static_cast<const T*>(a.q) + (static_cast<int64_t>(b) * a.H + g * G) * D;
    for (int i = lane; i < G * D / 8; i += 32) {
        float f[8];
        load8(qp + i * 8, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) qs[wl][(i * 8) / D][(i * 8) % D + e] = f[e] * qscale;
    }
    __syncwarp();
    float slope[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        slope[h] = 0.f;
        if (a.alibi) {
            const int hq = g * G + h;
            const float sl = a.slopes ? a.slopes[hq]
                                      : exp2f(-8.0f * static_cast<float>(hq + 1) /
                                              static_cast<float>(a.H));
            slope[h] = sl * kLog2eDec;
        }
    }
    float m[G], l[G], acc[G][kCols];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int c = 0; c < kCols; ++c) acc[h][c] = 0.f;
    }
    const int64_t kv_base = (static_cast<int64_t>(b) * a.Hk + g) * a.S_max;
    const T* kp = static_cast<const T*>(a.k) + kv_base * D;
    const T* vp = static_cast<const T*>(a.v) + kv_base * D;
    const float qpos = static_cast<float>(n - 1);
    for (int jb = j0; jb < j1; jb += 32) {
        const int j = jb + lane;
        const bool valid = j < j1;
        // scores of key j against the G queries (log2 domain)
        float sc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] = 0.f;
        if (valid) {
            const T* krow = kp + static_cast<int64_t>(j) * D;
#pragma unroll 4
            for (int c = 0; c < D / 8; ++c) {
                float kf[8];
                load8(krow + c * 8, kf);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) sc[h] = fmaf(qs[wl][h][c * 8 + e], kf[e], sc[h]);
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
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
            sc[h] = p;
        }
        // O += p V over this block's keys, one coalesced row load per key
        const int nk = min(32, j1 - jb);
        for (int t = 0; t < nk; ++t) {
            const T* vrow = vp + static_cast<int64_t>(jb + t) * D + lane * kCols;
            float vf[kCols];
            if constexpr (kCols == 2) {
                const float2 u = dt_traits<T>::unpack2(*reinterpret_cast<const uint32_t*>(vrow));
                vf[0] = u.x;
                vf[1] = u.y;
            } else {
                const uint2 u = *reinterpret_cast<const uint2*>(vrow);
                const float2 u0 = dt_traits<T>::unpack2(u.x), u1 = dt_traits<T>::unpack2(u.y);
                vf[0] = u0.x;
                vf[1] = u0.y;
                vf[2] = u1.x;
                vf[3] = u1.y;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pt = __shfl_sync(0xffffffffu, sc[h], t);
#pragma unroll
                for (int c = 0; c < kCols; ++c) acc[h][c] = fmaf(pt, vf[c], acc[h][c]);
            }
        }
    }
    // (max, sum, output) of this part for each query head; an empty part
    // (j0 >= n) writes max = -inf, sum = 0
    float* rec = a.ws + (static_cast<int64_t>(b) * a.H + g * G) * a.parts * (D + 2);
#pragma unroll
    for (int h = 0; h < G; ++h) {
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
    const int64_t warps = static_cast<int64_t>(a.B) * a.Hk * a.parts;
    decode_partial_kernel<T, D, G><<<static_cast<unsigned>((warps + 3) / 4), kDecThreads, 0, s>>>(a);
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

int decode_parts(int64_t B, int64_t Hk, int64_t S_max, int num_sms) {
    // about 16 warps per SM in flight, and at least 64 keys per part
    const int64_t want = (16LL * num_sms + B * Hk - 1) / (B * Hk);
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
