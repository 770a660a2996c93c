// K4/K5: in-place qk-norm and partial NeoX split-half rotary on head-split
// q [B, H, S, d] and k [B, Hk, S, d].
//
// Per token (b, s) one CTA stages the token's q heads and k heads in shared
// memory as fp32 (16-byte loads per head row), then:
//   1. adds the q/k bias (the projection bias comes before the rotary:
//      nnterp "stablelm" 03 Notes, "Biased queries, keys and values"),
//   2. QKN_RMS_FULL: one RMSNorm over the whole H*d (and Hk*d) row ("OLMo-2:
//      reordered (post) normalization", section 1: full-width, not per head);
//      QKN_LN_PER_HEAD: one bias-free LayerNorm per head (nnterp "stablelm"
//      03 Notes, "Per-head LayerNorms on queries and keys on 12B"),
//   3. rotates pairs (j, j + r/2), j < r/2, of each head by p * theta_j
//      ("StableLM-2: partial RoPE ...", section 1); dims >= r pass through,
//   4. writes the rows back with 16-byte stores.
// HBM-bound: every element of q and k is read and written once.
#include "internal.h"

namespace blk {

namespace {

constexpr int kRopeThreads = 128;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kRopeThreads / 32; ++w) t += red[w];
    return t;
}

template <typename T>
__global__ void __launch_bounds__(kRopeThreads) qk_norm_rope_kernel(QkNormRopeArgs a,
                                                                    RopeParams rp) {
    extern __shared__ float buf[];  // (H + Hk) * d floats
    __shared__ float red[kRopeThreads / 32];
    const int token = blockIdx.x;
    const int b = token / a.S;
    const int s = token % a.S;
    const int d = a.d;
    const int nh = a.H + a.Hk;
    const int nvec = nh * d / 8;
    const int vpr = d / 8;  // vectors per head row

    auto row_ptr = [&](int head) -> T* {
        if (head < a.H)
            return static_cast<T*>(a.q) + ((static_cast<int64_t>(b) * a.H + head) * a.S + s) * d;
        return static_cast<T*>(a.k) +
               ((static_cast<int64_t>(b) * a.Hk + (head - a.H)) * a.S + s) * d;
    };

    // 1. load (+ bias)
    for (int i = threadIdx.x; i < nvec; i += kRopeThreads) {
        const int head = i / vpr;
        const int c = (i % vpr) * 8;
        float f[8];
        load8(row_ptr(head) + c, f);
        const T* bias = head < a.H ? static_cast<const T*>(a.q_bias) : static_cast<const T*>(a.k_bias);
        if (bias) {
            float bb[8];
            load8(bias + (head < a.H ? head : head - a.H) * d + c, bb);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] += bb[e];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) buf[head * d + c + e] = f[e];
    }
    __syncthreads();

    // 2. qk-norm
    if (a.mode == QKN_RMS_FULL) {
        for (int part = 0; part < 2; ++part) {
            const int h0 = part == 0 ? 0 : a.H;
            const int n = (part == 0 ? a.H : a.Hk) * d;
            if (n == 0) continue;
            float sq = 0.f;
            for (int i = threadIdx.x; i < n; i += kRopeThreads) {
                const float t = buf[h0 * d + i];
                sq += t * t;
            }
            const float rstd = rsqrtf(block_sum(sq, red) / static_cast<float>(n) + a.eps);
            const T* w = static_cast<const T*>(part == 0 ? a.q_w : a.k_w);
            for (int i = threadIdx.x; i < n; i += kRopeThreads)
                buf[h0 * d + i] *= rstd * dt_traits<T>::to_f(w[i]);
        }
        __syncthreads();
    } else if (a.mode == QKN_LN_PER_HEAD) {
        const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
        for (int head = warp; head < nh; head += kRopeThreads / 32) {
            float* r = buf + head * d;
            float sum = 0.f;
            for (int i = lane; i < d; i += 32) sum += r[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            const float mean = sum / static_cast<float>(d);
            float sq = 0.f;
            for (int i = lane; i < d; i += 32) {
                const float c = r[i] - mean;
                sq += c * c;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
            const float rstd = rsqrtf(sq / static_cast<float>(d) + a.eps);
            const T* g = head < a.H ? static_cast<const T*>(a.q_w) + head * d
                                    : static_cast<const T*>(a.k_w) + (head - a.H) * d;
            for (int i = lane; i < d; i += 32) r[i] = (r[i] - mean) * rstd * dt_traits<T>::to_f(g[i]);
        }
        __syncthreads();
    }

    // 3. rotary over the first rp.span dims of every q and k head
    const int half = rp.span / 2;
    if (half > 0) {
        for (int i = threadIdx.x; i < nh * half; i += kRopeThreads) {
            const int head = i / half;
            const int j = i % half;
            float c, sn;
            rope_cos_sin(rp, s, j, c, sn);
            float* r = buf + head * d;
            const float x1 = r[j], x2 = r[j + half];
            r[j] = x1 * c - x2 * sn;
            r[j + half] = x2 * c + x1 * sn;
        }
        __syncthreads();
    }

    // 4. store
    for (int i = threadIdx.x; i < nvec; i += kRopeThreads) {
        const int head = i / vpr;
        const int c = (i % vpr) * 8;
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = buf[head * d + c + e];
        store8(row_ptr(head) + c, f);
    }
}

// Fast path: one warp per (token, q or k). Lane l holds the 16-byte vectors
// V = l + 32 i of the token's heads laid end to end (head = V / vph,
// vph = d / 8 vectors per head, vph dividing 32 so a head is a fixed group of
// lanes); all loads are issued first. The full-width RMS sum is a warp
// reduction, the per-head LayerNorm a reduction over the head's lane group,
// and the rotary partner (dims j and j + r/2) is the same vector slot of the
// lane r/16 away, fetched with a shuffle. Cosines and sines depend only on
// the lane's vector slot within the head, so each lane evaluates them once.
template <typename T, int NV>
__global__ void __launch_bounds__(128) qk_warp_kernel(QkNormRopeArgs a, RopeParams rp) {
    const int lane = threadIdx.x & 31;
    const int wid = blockIdx.x * 4 + threadIdx.x / 32;
    const int parts = a.Hk > 0 ? 2 : 1;
    const int64_t tokens = static_cast<int64_t>(a.B) * a.S;
    if (wid >= tokens * parts) return;  // whole warps exit together
    const int part = wid % parts;
    const int64_t token = wid / parts;
    const int b = static_cast<int>(token / a.S);
    const int s = static_cast<int>(token % a.S);
    const int nh = part == 0 ? a.H : a.Hk;
    T* base = static_cast<T*>(part == 0 ? a.q : a.k);
    const T* bias = static_cast<const T*>(part == 0 ? a.q_bias : a.k_bias);
    const T* w = static_cast<const T*>(part == 0 ? a.q_w : a.k_w);
    const int d = a.d;
    const int vph = d / 8;
    const int nvec = nh * vph;
    const int vin = lane % vph;  // same for every i because vph divides 32

    float v[NV][8];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int V = lane + 32 * i;
        if (V < nvec) {
            const int head = V / vph;
            load8(base + ((static_cast<int64_t>(b) * nh + head) * a.S + s) * d + vin * 8, v[i]);
            if (bias) {
                float bb[8];
                load8(bias + V * 8, bb);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] += bb[e];
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[i][e] = 0.f;
        }
    }
    if (a.mode == QKN_RMS_FULL) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(v[i][e], v[i][e], acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        const float rstd = rsqrtf(acc / static_cast<float>(nh * d) + a.eps);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int V = lane + 32 * i;
            if (V < nvec) {
                float g[8];
                load8(w + V * 8, g);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] *= rstd * g[e];
            }
        }
    } else if (a.mode == QKN_LN_PER_HEAD) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) sum += v[i][e];
            for (int o = vph / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            const float mean = sum / static_cast<float>(d);
            float sq = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float c = v[i][e] - mean;
                sq = fmaf(c, c, sq);
            }
            for (int o = vph / 2; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
            const float rstd = rsqrtf(sq / static_cast<float>(d) + a.eps);
            const int V = lane + 32 * i;
            if (V < nvec) {
                float g[8];
                load8(w + V * 8, g);  // gamma [nh, d] read at head * d + vin * 8 = V * 8
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] = (v[i][e] - mean) * rstd * g[e];
            }
        }
    }
    const int hv = rp.span / 16;  // vectors in each rotated half
    if (hv > 0) {
        const bool lo = vin < hv;
        const bool rot = vin < 2 * hv;
        const int partner = lo ? lane + hv : lane - hv;
        float c[8], sn[8];
        if (rot) {
            const int j0 = (lo ? vin : vin - hv) * 8;
#pragma unroll
            for (int e = 0; e < 8; ++e) rope_cos_sin(rp, s, j0 + e, c[e], sn[e]);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float other = __shfl_sync(0xffffffffu, v[i][e], rot ? partner : lane);
                if (rot) v[i][e] = lo ? v[i][e] * c[e] - other * sn[e] : v[i][e] * c[e] + other * sn[e];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int V = lane + 32 * i;
        if (V < nvec)
            store8(base + ((static_cast<int64_t>(b) * nh + V / vph) * a.S + s) * d + vin * 8, v[i]);
    }
}

// Unit path, head_dim D of 64 or 128 and rotary spans r with r/2 a multiple
// of 8: a warp per (token, q|k) item as above, but each lane owns units of
// two 16-byte vectors of one head, chosen so that no data crosses lanes for
// the rotation: unit u < r/16 holds vectors u and u + r/16 (dims 8u..8u+7
// and their partners 8u+r/2..), the other units hold two neighbouring
// vectors of the unrotated tail. The head index and the lane's unit are
// compile-time shifts of the lane id, the full-width RMS is one warp
// reduction, the per-head LayerNorm a reduction over the head's D/16 lanes.
// Persistent warps walk their items with a three-stage cp.async ring in
// shared memory, so the next two items' bytes are in flight (without
// holding registers) while one is computed.
template <int NU>
struct UnitCfg {
    static constexpr int kStages = 3;                 // tokens in flight per warp
    static constexpr int kStageBytes = NU * 2 * 512;  // [slot][vector a|b][lane] x 16 B
    static constexpr int kSmem = 4 * kStages * kStageBytes;
};

template <typename T, int D, int NU>
__global__ void __launch_bounds__(128) qk_unit_kernel(QkNormRopeArgs a, RopeParams rp) {
    using Cfg = UnitCfg<NU>;
    constexpr int kLph = D / 16;  // lanes per head
    extern __shared__ __align__(128) uint8_t usm[];
    const int lane = threadIdx.x & 31;
    const int parts = a.Hk > 0 ? 2 : 1;
    const int total = a.B * a.S * parts;
    const int nwarps = static_cast<int>(gridDim.x) * 4;
    const int w0 = blockIdx.x * 4 + threadIdx.x / 32;
    const uint32_t ring = smem_u32(usm) + (threadIdx.x / 32) * Cfg::kStages * Cfg::kStageBytes;
    const int hv = rp.span / 16;  // rotated vectors in each half
    const int u = lane % kLph;    // this lane's unit within its head (every slot)
    const bool rot = u < hv;
    const int va = rot ? u : 2 * hv + 2 * (u - hv);
    const int vb = rot ? u + hv : va + 1;
    // this warp's k-th item: (token, q|k)
    auto item = [&](int k, int& part, int& b, int& s) {
        const int w = w0 + k * nwarps;
        part = w % parts;
        const int token = w / parts;
        b = token / a.S;
        s = token - b * a.S;
    };
    // cp.async of the k-th item's units into its stage (lane-private slots)
    auto issue = [&](int k) {
        if (w0 + k * nwarps < total) {
            int part, b, s;
            item(k, part, b, s);
            const int nh = part == 0 ? a.H : a.Hk;
            const T* base = static_cast<const T*>(part == 0 ? a.q : a.k);
            const uint32_t st = ring + (k % Cfg::kStages) * Cfg::kStageBytes;
#pragma unroll
            for (int i = 0; i < NU; ++i) {
                const int U = lane + 32 * i;
                if (U < nh * kLph) {
                    const T* row = base + ((static_cast<int64_t>(b) * nh + U / kLph) * a.S + s) * D;
                    cp_async16(st + ((2 * i) * 32 + lane) * 16, row + va * 8, 16u);
                    cp_async16(st + ((2 * i + 1) * 32 + lane) * 16, row + vb * 8, 16u);
                }
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < Cfg::kStages - 1; ++k) issue(k);
    for (int k = 0; w0 + k * nwarps < total; ++k) {
        issue(k + Cfg::kStages - 1);
        cp_async_wait<Cfg::kStages - 1>();  // this lane's copies of item k landed
        int part, b, s;
        item(k, part, b, s);
        const int nh = part == 0 ? a.H : a.Hk;
        T* base = static_cast<T*>(part == 0 ? a.q : a.k);
        const T* bias = static_cast<const T*>(part == 0 ? a.q_bias : a.k_bias);
        const T* w = static_cast<const T*>(part == 0 ? a.q_w : a.k_w);
        const int nunits = nh * kLph;
        const uint32_t st = ring + (k % Cfg::kStages) * Cfg::kStageBytes;
        float x[NU][16];
#pragma unroll
        for (int i = 0; i < NU; ++i) {
            const int U = lane + 32 * i;
            if (U < nunits) {
                const uint4 r0 = ld_shared_u4(st + ((2 * i) * 32 + lane) * 16);
                const uint4 r1 = ld_shared_u4(st + ((2 * i + 1) * 32 + lane) * 16);
                const uint32_t w8[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 f = dt_traits<T>::unpack2(w8[e]);
                    x[i][(e / 4) * 8 + (e % 4) * 2] = f.x;
                    x[i][(e / 4) * 8 + (e % 4) * 2 + 1] = f.y;
                }
                if (bias) {
                    const int head = U / kLph;
                    float b0[8], b1[8];
                    load8(bias + head * D + va * 8, b0);
                    load8(bias + head * D + vb * 8, b1);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        x[i][e] += b0[e];
                        x[i][8 + e] += b1[e];
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) x[i][e] = 0.f;
            }
        }
        if (a.mode == QKN_RMS_FULL) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < NU; ++i)
#pragma unroll
                for (int e = 0; e < 16; ++e) acc = fmaf(x[i][e], x[i][e], acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            const float rstd = rsqrtf(acc / static_cast<float>(nh * D) + a.eps);
#pragma unroll
            for (int i = 0; i < NU; ++i) {
                const int U = lane + 32 * i;
                if (U < nunits) {
                    const int head = U / kLph;
                    float g0[8], g1[8];
                    load8(w + head * D + va * 8, g0);
                    load8(w + head * D + vb * 8, g1);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        x[i][e] *= rstd * g0[e];
                        x[i][8 + e] *= rstd * g1[e];
                    }
                }
            }
        } else if (a.mode == QKN_LN_PER_HEAD) {
#pragma unroll
            for (int i = 0; i < NU; ++i) {
                float sum = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) sum += x[i][e];
#pragma unroll
                for (int o = kLph / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                const float mean = sum / static_cast<float>(D);
                float sq = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float c = x[i][e] - mean;
                    sq = fmaf(c, c, sq);
                }
#pragma unroll
                for (int o = kLph / 2; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
                const float rstd = rsqrtf(sq / static_cast<float>(D) + a.eps);
                const int U = lane + 32 * i;
                if (U < nunits) {
                    const int head = U / kLph;
                    float g0[8], g1[8];
                    load8(w + head * D + va * 8, g0);  // gamma [nh, D]
                    load8(w + head * D + vb * 8, g1);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        x[i][e] = (x[i][e] - mean) * rstd * g0[e];
                        x[i][8 + e] = (x[i][8 + e] - mean) * rstd * g1[e];
                    }
                }
            }
        }
        if (rot) {
            float c[8], sn[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) rope_cos_sin(rp, s, u * 8 + e, c[e], sn[e]);
#pragma unroll
            for (int i = 0; i < NU; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x0 = x[i][e], x1 = x[i][8 + e];
                    x[i][e] = x0 * c[e] - x1 * sn[e];
                    x[i][8 + e] = x1 * c[e] + x0 * sn[e];
                }
        }
#pragma unroll
        for (int i = 0; i < NU; ++i) {
            const int U = lane + 32 * i;
            if (U < nunits) {
                T* row = base + ((static_cast<int64_t>(b) * nh + U / kLph) * a.S + s) * D;
                store8(row + va * 8, *reinterpret_cast<const float(*)[8]>(&x[i][0]));
                store8(row + vb * 8, *reinterpret_cast<const float(*)[8]>(&x[i][8]));
            }
        }
    }
    cp_async_wait<0>();
}

template <typename T, int D, int NU>
void launch_unit(const QkNormRopeArgs& a, const RopeParams& rp, cudaStream_t s, int64_t warps) {
    using Cfg = UnitCfg<NU>;
    auto kern = qk_unit_kernel<T, D, NU>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
        attr_set = true;
    }
    // persistent: as many 4-warp blocks as fit (shared memory bound) on every SM
    const int per_sm = (200 * 1024) / Cfg::kSmem > 0 ? (200 * 1024) / Cfg::kSmem : 1;
    int64_t blocks = (warps + 3) / 4;
    const int64_t cap = static_cast<int64_t>(per_sm < 8 ? per_sm : 8) * a.num_sms;
    if (blocks > cap) blocks = cap;
    kern<<<static_cast<unsigned>(blocks), 128, Cfg::kSmem, s>>>(a, rp);
}

template <typename T, int D>
bool launch_unit_d(const QkNormRopeArgs& a, const RopeParams& rp, cudaStream_t s) {
    const int nunits = (a.H > a.Hk ? a.H : a.Hk) * (D / 16);
    const int64_t warps = static_cast<int64_t>(a.B) * a.S * (a.Hk > 0 ? 2 : 1);
    if (nunits > 256 || warps > 0x7fffffff || a.num_sms <= 0) return false;
    if (nunits <= 32) launch_unit<T, D, 1>(a, rp, s, warps);
    else if (nunits <= 64) launch_unit<T, D, 2>(a, rp, s, warps);
    else if (nunits <= 128) launch_unit<T, D, 4>(a, rp, s, warps);
    else launch_unit<T, D, 8>(a, rp, s, warps);
    return true;
}

template <typename T>
bool launch_unit_path(const QkNormRopeArgs& a, const RopeParams& rp, cudaStream_t s) {
    if ((rp.span / 2) % 8 != 0) return false;
    if (a.d == 64) return launch_unit_d<T, 64>(a, rp, s);
    if (a.d == 128) return launch_unit_d<T, 128>(a, rp, s);
    return false;
}

template <typename T>
bool launch_warp_path(const QkNormRopeArgs& a, const RopeParams& rp, cudaStream_t s) {
    const int vph = a.d / 8;
    const int maxh = a.H > a.Hk ? a.H : a.Hk;
    const int nvec = maxh * vph;
    if (a.d % 8 || vph > 32 || 32 % vph || (rp.span / 2) % 8 || nvec > 256) return false;
    const int64_t warps = static_cast<int64_t>(a.B) * a.S * (a.Hk > 0 ? 2 : 1);
    const int64_t blocks = (warps + 3) / 4;
    if (blocks > 0x7fffffff) return false;
    const unsigned g = static_cast<unsigned>(blocks);
    if (nvec <= 32) qk_warp_kernel<T, 1><<<g, 128, 0, s>>>(a, rp);
    else if (nvec <= 64) qk_warp_kernel<T, 2><<<g, 128, 0, s>>>(a, rp);
    else if (nvec <= 128) qk_warp_kernel<T, 4><<<g, 128, 0, s>>>(a, rp);
    else qk_warp_kernel<T, 8><<<g, 128, 0, s>>>(a, rp);
    return true;
}

}  // namespace

cudaError_t launch_qk_norm_rope(DType dt, const QkNormRopeArgs& a, const RopeParams& rp,
                                cudaStream_t s) {
    const int64_t tokens = static_cast<int64_t>(a.B) * a.S;
    if (tokens == 0) return cudaSuccess;
    if (dt == DType::F16 ? launch_unit_path<__half>(a, rp, s)
                         : launch_unit_path<__nv_bfloat16>(a, rp, s))
        return cudaGetLastError();
    if (dt == DType::F16 ? launch_warp_path<__half>(a, rp, s)
                         : launch_warp_path<__nv_bfloat16>(a, rp, s))
        return cudaGetLastError();
    // general path (e.g. head_dim 160 or spans not a multiple of 16)
    const size_t smem = static_cast<size_t>(a.H + a.Hk) * a.d * sizeof(float);
    if (dt == DType::F16) {
        auto k = qk_norm_rope_kernel<__half>;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        k<<<static_cast<unsigned>(tokens), kRopeThreads, smem, s>>>(a, rp);
    } else {
        auto k = qk_norm_rope_kernel<__nv_bfloat16>;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        k<<<static_cast<unsigned>(tokens), kRopeThreads, smem, s>>>(a, rp);
    }
    return cudaGetLastError();
}

}  // namespace blk
