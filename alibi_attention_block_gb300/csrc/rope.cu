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
constexpr int kRopeBatch = 8;  // 16-byte loads in flight per thread and round

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
__global__ void __launch_bounds__(kRopeThreads, 5) qk_norm_rope_kernel(QkNormRopeArgs a,
                                                                       RopeParams rp) {
    if (a.pdl) {  // launched for programmatic dependent launch
        pdl_wait();
        pdl_launch_dependents();
    }
    extern __shared__ float buf[];  // (H + Hk) * d floats, then cos[r/2], sin[r/2]
    __shared__ float red[kRopeThreads / 32];
    const int token = blockIdx.x;
    const int b = token / a.S;
    const int s = token % a.S;
    const int d = a.d;
    const int nh = a.H + a.Hk;
    const int nvec = nh * d / 8;
    const int vpr = d / 8;  // vectors per head row
    const int half = rp.span / 2;
    float* cs_tab = buf + nh * d;

    auto row_ptr = [&](int head) -> T* {
        if (head < a.H)
            return static_cast<T*>(a.q) + ((static_cast<int64_t>(b) * a.H + head) * a.S + s) * d;
        return static_cast<T*>(a.k) +
               ((static_cast<int64_t>(b) * a.Hk + (head - a.H)) * a.S + s) * d;
    };

    // 0. cos / sin of this token's position, shared by every head
    for (int j = threadIdx.x; j < half; j += kRopeThreads)
        rope_cos_sin(rp, s, j, cs_tab[j], cs_tab[half + j]);

    // 1. load (+ bias): in rounds of kRopeBatch 16-byte vectors per thread,
    // every load of a round (and its bias vector) issued before any is used,
    // so a token's rows cost one memory latency, not one per vector
    const T* q_bias = static_cast<const T*>(a.q_bias);
    const T* k_bias = static_cast<const T*>(a.k_bias);
    for (int base = 0; base < nvec; base += kRopeThreads * kRopeBatch) {
        uint4 raw[kRopeBatch], rb[kRopeBatch];
#pragma unroll
        for (int t = 0; t < kRopeBatch; ++t) {
            const int i = base + t * kRopeThreads + static_cast<int>(threadIdx.x);
            raw[t] = make_uint4(0u, 0u, 0u, 0u);
            rb[t] = raw[t];
            if (i < nvec) {
                const int head = i / vpr;
                const int c = (i - head * vpr) * 8;
                raw[t] = *reinterpret_cast<const uint4*>(row_ptr(head) + c);
                const T* bias = head < a.H ? q_bias : k_bias;
                if (bias)
                    rb[t] = *reinterpret_cast<const uint4*>(
                        bias + (head < a.H ? head : head - a.H) * d + c);
            }
        }
#pragma unroll
        for (int t = 0; t < kRopeBatch; ++t) {
            const int i = base + t * kRopeThreads + static_cast<int>(threadIdx.x);
            if (i < nvec) {
                const uint32_t w[4] = {raw[t].x, raw[t].y, raw[t].z, raw[t].w};
                const uint32_t wb[4] = {rb[t].x, rb[t].y, rb[t].z, rb[t].w};
                float f[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 v = dt_traits<T>::unpack2(w[e]);
                    const float2 vb = dt_traits<T>::unpack2(wb[e]);
                    f[2 * e] = v.x + vb.x;
                    f[2 * e + 1] = v.y + vb.y;
                }
                float4* dst = reinterpret_cast<float4*>(buf + i * 8);  // = head * d + c
                dst[0] = make_float4(f[0], f[1], f[2], f[3]);
                dst[1] = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
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
    if (half > 0) {
        for (int i = threadIdx.x; i < nh * half; i += kRopeThreads) {
            const int head = i / half;
            const int j = i - head * half;
            const float c = cs_tab[j], sn = cs_tab[half + j];
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
    if (a.pdl) {  // launched for programmatic dependent launch
        pdl_wait();
        pdl_launch_dependents();
    }
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
    if (a.pdl) {  // launched for programmatic dependent launch
        pdl_wait();
        pdl_launch_dependents();
    }
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
    // a failure here stays the runtime's last error, which the caller returns
    if (set_smem_attr_once(reinterpret_cast<const void*>(kern), Cfg::kSmem) != cudaSuccess) return;
    // persistent: as many 4-warp blocks as fit (shared memory bound) on every SM
    const int per_sm = (200 * 1024) / Cfg::kSmem > 0 ? (200 * 1024) / Cfg::kSmem : 1;
    int64_t blocks = (warps + 3) / 4;
    const int64_t cap = static_cast<int64_t>(per_sm < 8 ? per_sm : 8) * a.num_sms;
    if (blocks > cap) blocks = cap;
    (void)launch_pdl(a.pdl != 0, kern, dim3(static_cast<unsigned>(blocks)), dim3(128), Cfg::kSmem, s, a, rp);
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

// Head-row path (any head_dim d <= 256 with d % 8 == 0; per-head LayerNorm
// or none): a CTA per token. Its q and k rows are first copied into shared
// memory with cp.async by all threads (one memory latency per token, no
// registers held for data in flight); then each warp takes head rows warp,
// warp + 8, ... (q heads, then k heads), lane l holding the row's 16-byte
// vector l (dims 8l .. 8l + 7), so the per-head LayerNorm is a warp
// reduction. The rotary partner of dim g (g + r/2 for g < r/2, g - r/2 for
// r/2 <= g < r) lies (g +- r/2) / 8 lanes away at slot (g +- r/2) mod 8: with
// HM = (r/2) mod 8 a template parameter the slot is a compile-time register
// and only the lane offset is computed. cos / sin of the token's position
// come from a shared table filled once per token.
constexpr int kHeadWarps = 8;

template <typename T, int HM>
__global__ void __launch_bounds__(kHeadWarps * 32) qk_head_kernel(QkNormRopeArgs a,
                                                                  RopeParams rp) {
    if (a.pdl) {  // launched for programmatic dependent launch
        pdl_wait();
        pdl_launch_dependents();
    }
    __shared__ float cs_tab[2 * kMaxRotaryPairs];  // cos[r/2], then sin[r/2]
    extern __shared__ __align__(16) uint8_t rows[];  // (H + Hk) rows of d values
    const int token = blockIdx.x;
    const int b = token / a.S;
    const int s = token - b * a.S;
    const int d = a.d;
    const int nv = d / 8;
    const int nh = a.H + a.Hk;
    const int half = rp.span / 2;
    const int hq = half >> 3;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool active = lane < nv;
    const bool ln = a.mode == QKN_LN_PER_HEAD;
    auto row_ptr = [&](int head) -> T* {
        if (head < a.H)
            return static_cast<T*>(a.q) + ((static_cast<int64_t>(b) * a.H + head) * a.S + s) * d;
        return static_cast<T*>(a.k) +
               ((static_cast<int64_t>(b) * a.Hk + (head - a.H)) * a.S + s) * d;
    };
    const uint32_t srow = smem_u32(rows);
    if (active)
        for (int head = warp; head < nh; head += kHeadWarps)
            cp_async16(srow + (head * nv + lane) * 16, row_ptr(head) + lane * 8, 16u);
    cp_async_commit();
    for (int j = threadIdx.x; j < half; j += kHeadWarps * 32)
        rope_cos_sin(rp, s, j, cs_tab[j], cs_tab[kMaxRotaryPairs + j]);
    __syncthreads();
    // this lane's rotary coefficients, the same for every head of the token:
    // x'_g = x_g c_g + x_{g+r/2} f_g + x_{g-r/2} b_g, with f = -sin for
    // g < r/2, b = +sin for r/2 <= g < r, zero otherwise (the direction is
    // data, not a predicate kept live across the head loop). With (r/2) mod 8
    // = 0 or 4 both partners sit in the same slot: one shuffle from the lane
    // src_l serves either direction.
    float rot_c[8], rot_f[8], rot_b[8];
    int src_l[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int g = lane * 8 + e;
        rot_c[e] = 1.f;
        rot_f[e] = 0.f;
        rot_b[e] = 0.f;
        src_l[e] = lane - hq - (e < HM ? 1 : 0);
        if (g < half) {
            rot_c[e] = cs_tab[g];
            rot_f[e] = -cs_tab[kMaxRotaryPairs + g];
            src_l[e] = lane + hq + ((e + HM) >> 3);
        } else if (g < 2 * half) {
            rot_c[e] = cs_tab[g - half];
            rot_b[e] = cs_tab[kMaxRotaryPairs + g - half];
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    for (int head = warp; head < nh; head += kHeadWarps) {
        const bool isq = head < a.H;
        const int hh = isq ? head : head - a.H;
        const T* bias = static_cast<const T*>(isq ? a.q_bias : a.k_bias);
        uint4 rb = make_uint4(0u, 0u, 0u, 0u), rg = rb, raw = rb;
        if (active) {
            if (bias) rb = *reinterpret_cast<const uint4*>(bias + hh * d + lane * 8);
            if (ln)
                rg = *reinterpret_cast<const uint4*>(static_cast<const T*>(isq ? a.q_w : a.k_w) +
                                                     hh * d + lane * 8);
            raw = ld_shared_u4(srow + (head * nv + lane) * 16);
        }
        float x[8];
        {
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            const uint32_t wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 v = dt_traits<T>::unpack2(w[e]);
                const float2 vb = dt_traits<T>::unpack2(wb[e]);
                x[2 * e] = v.x + vb.x;
                x[2 * e + 1] = v.y + vb.y;
            }
        }
        if (ln) {
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) sum += x[e];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            const float mean = sum / static_cast<float>(d);
            float sq = 0.f;
            if (active) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float c = x[e] - mean;
                    sq = fmaf(c, c, sq);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
            const float rstd = rsqrtf(sq / static_cast<float>(d) + a.eps);
            const uint32_t wg[4] = {rg.x, rg.y, rg.z, rg.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 g = dt_traits<T>::unpack2(wg[e]);
                x[2 * e] = (x[2 * e] - mean) * rstd * g.x;
                x[2 * e + 1] = (x[2 * e + 1] - mean) * rstd * g.y;
            }
        }
        if (half > 0) {
            // every lane takes part in the shuffles; past r the coefficients
            // are (1, 0). With (r/2) mod 8 = 0 or 4 both partners sit in the
            // same slot, so one shuffle per slot serves both directions.
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if constexpr ((HM & 3) == 0) {
                    const float p = __shfl_sync(0xffffffffu, x[(e + HM) & 7], src_l[e]);
                    y[e] = fmaf(p, rot_f[e] + rot_b[e], x[e] * rot_c[e]);
                } else {
                    const float pf = __shfl_sync(0xffffffffu, x[(e + HM) & 7],
                                                 lane + hq + ((e + HM) >> 3));
                    const float pb = __shfl_sync(0xffffffffu, x[(e + 8 - HM) & 7],
                                                 lane - hq - (e < HM ? 1 : 0));
                    y[e] = fmaf(pb, rot_b[e], fmaf(pf, rot_f[e], x[e] * rot_c[e]));
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = y[e];
        }
        if (active) store8(row_ptr(head) + lane * 8, x);
    }
}

template <typename T, int HM>
void launch_head(unsigned grid, size_t smem, const QkNormRopeArgs& a, const RopeParams& rp,
                 cudaStream_t s) {
    auto kern = qk_head_kernel<T, HM>;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    (void)launch_pdl(a.pdl != 0, kern, dim3(grid), dim3(kHeadWarps * 32), smem, s, a, rp);
}

template <typename T>
bool launch_head_path(const QkNormRopeArgs& a, const RopeParams& rp, cudaStream_t s) {
    if (a.mode == QKN_RMS_FULL || a.d % 8 || a.d > 256) return false;
    const int64_t tokens = static_cast<int64_t>(a.B) * a.S;
    if (tokens > 0x7fffffff) return false;
    const unsigned g = static_cast<unsigned>(tokens);
    const size_t smem = static_cast<size_t>(a.H + a.Hk) * a.d * sizeof(T);
    if (smem > 200 * 1024) return false;
    switch ((rp.span / 2) & 7) {
        case 0: launch_head<T, 0>(g, smem, a, rp, s); break;
        case 1: launch_head<T, 1>(g, smem, a, rp, s); break;
        case 2: launch_head<T, 2>(g, smem, a, rp, s); break;
        case 3: launch_head<T, 3>(g, smem, a, rp, s); break;
        case 4: launch_head<T, 4>(g, smem, a, rp, s); break;
        case 5: launch_head<T, 5>(g, smem, a, rp, s); break;
        case 6: launch_head<T, 6>(g, smem, a, rp, s); break;
        default: launch_head<T, 7>(g, smem, a, rp, s); break;
    }
    return true;
}

// Row-group path at head_dim D = 64, 128 or 160 (StableLM-2-12B's 160, the
// attention sweep's 64): bias, per-head LayerNorm (or none) and rotary over
// the first ROT <= D/4 dims, in place. A plane (b, head) of q or k is [S, D]
// contiguous, so 8 consecutive rows are 16 D contiguous bytes: one warp takes
// them, 4 lanes per row and D/4 elements (D/32 16-byte vectors) per lane.
// The row statistics are two shuffle steps over a row's 4 lanes. The rotary
// span lies within each row's first lane: the row's 4 lanes compute every
// 4th of its ROT/2 (cos, sin) pairs and hand them to the first lane by
// shuffle. Persistent warps over blocks, the next block's rows loaded before
// this one is computed.
constexpr int kRgWarps = 8;
template <typename T, int D, int ROT>
__global__ void __launch_bounds__(kRgWarps * 32) qk_rowgroup_kernel(QkNormRopeArgs a,
                                                                    RopeParams rp) {
    if (a.pdl) {  // launched for programmatic dependent launch
        pdl_wait();
        pdl_launch_dependents();
    }
    constexpr int VL = D / 32;  // 16-byte vectors per lane
    constexpr int kPairs = ROT / 2;
    static_assert(ROT % 2 == 0 && ROT <= 8 * VL, "the rotary span must lie in a row's first lane");
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2;    // row of the block
    const int sub = lane & 3;   // which 40 dims of the row
    const int rblocks = (a.S + 7) / 8;
    const int64_t q_items = static_cast<int64_t>(a.B) * a.H * rblocks;
    const int64_t items = q_items + static_cast<int64_t>(a.B) * a.Hk * rblocks;
    const int64_t wstep = static_cast<int64_t>(gridDim.x) * kRgWarps;
    const bool ln = a.mode == QKN_LN_PER_HEAD;
    auto locate = [&](int64_t it, T*& row, int& head, bool& isq, int& pos) {
        isq = it < q_items;
        const int64_t local = isq ? it : it - q_items;
        const int64_t plane = local / rblocks;
        const int rb = static_cast<int>(local - plane * rblocks);
        const int nh = isq ? a.H : a.Hk;
        head = static_cast<int>(plane % nh);
        pos = rb * 8 + r;
        row = static_cast<T*>(isq ? a.q : a.k) + (plane * a.S + pos) * D + sub * 8 * VL;
    };
    int64_t it = static_cast<int64_t>(blockIdx.x) * kRgWarps + (threadIdx.x >> 5);
    uint4 nxt[VL];
    T* nrow = nullptr;
    int nhead = 0, npos = 0;
    bool nisq = true;
    if (it < items) {
        locate(it, nrow, nhead, nisq, npos);
#pragma unroll
        for (int v = 0; v < VL; ++v)
            nxt[v] = npos < a.S ? reinterpret_cast<const uint4*>(nrow)[v] : make_uint4(0, 0, 0, 0);
    }
    for (; it < items; it += wstep) {
        uint4 cur[VL];
#pragma unroll
        for (int v = 0; v < VL; ++v) cur[v] = nxt[v];
        T* row = nrow;
        const int head = nhead, pos = npos;
        const bool isq = nisq;
        if (it + wstep < items) {
            locate(it + wstep, nrow, nhead, nisq, npos);
#pragma unroll
            for (int v = 0; v < VL; ++v)
                nxt[v] = npos < a.S ? reinterpret_cast<const uint4*>(nrow)[v]
                                    : make_uint4(0, 0, 0, 0);
        }
        float x[8 * VL];
#pragma unroll
        for (int v = 0; v < VL; ++v) {
            const uint32_t w[4] = {cur[v].x, cur[v].y, cur[v].z, cur[v].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = dt_traits<T>::unpack2(w[e]);
                x[v * 8 + 2 * e] = f.x;
                x[v * 8 + 2 * e + 1] = f.y;
            }
        }
        const int col0 = sub * 8 * VL;
        const T* bias = static_cast<const T*>(isq ? a.q_bias : a.k_bias);
        if (bias) {
#pragma unroll
            for (int v = 0; v < VL; ++v) {
                float b[8];
                load8(bias + head * D + col0 + v * 8, b);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[v * 8 + e] += b[e];
            }
        }
        if (ln) {
            float s1 = 0.f;
#pragma unroll
            for (int e = 0; e < 8 * VL; ++e) s1 += x[e];
            s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
            const float mean = s1 * (1.0f / D);
            float s2 = 0.f;
#pragma unroll
            for (int e = 0; e < 8 * VL; ++e) {
                const float c = x[e] - mean;
                s2 = fmaf(c, c, s2);
            }
            s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
            s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
            const float rstd = rsqrtf(s2 * (1.0f / D) + a.eps);
            const T* gam = static_cast<const T*>(isq ? a.q_w : a.k_w) + head * D + col0;
#pragma unroll
            for (int v = 0; v < VL; ++v) {
                float gv[8];
                load8(gam + v * 8, gv);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[v * 8 + e] = (x[v * 8 + e] - mean) * rstd * gv[e];
            }
        }
        if constexpr (kPairs > 0) {
            // the row's lanes each compute every 4th (cos, sin) pair
            constexpr int kPer = (kPairs + 3) / 4;
            float cs[kPer], sn[kPer];
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int j = i * 4 + sub;
                cs[i] = 1.f;
                sn[i] = 0.f;
                if (j < kPairs) rope_cos_sin(rp, pos, j, cs[i], sn[i]);
            }
#pragma unroll
            for (int j = 0; j < kPairs; ++j) {
                const int src = (lane & ~3) | (j & 3);
                const float c = __shfl_sync(0xffffffffu, cs[j >> 2], src);
                const float sv = __shfl_sync(0xffffffffu, sn[j >> 2], src);
                if (sub == 0) {
                    const float x1 = x[j], x2 = x[j + kPairs];
                    x[j] = x1 * c - x2 * sv;
                    x[j + kPairs] = x2 * c + x1 * sv;
                }
            }
        }
        if (pos < a.S) {
#pragma unroll
            for (int v = 0; v < VL; ++v)
                store8(row + v * 8, *reinterpret_cast<const float(*)[8]>(&x[v * 8]));
        }
    }
}

template <typename T>
bool launch_rowgroup_path(const QkNormRopeArgs& a, const RopeParams& rp, cudaStream_t s) {
    if (a.mode == QKN_RMS_FULL || a.num_sms <= 0) return false;
    const int64_t items = static_cast<int64_t>(a.B) * (a.H + a.Hk) * ((a.S + 7) / 8);
    if (items > (static_cast<int64_t>(1) << 40)) return false;
    using K = void (*)(QkNormRopeArgs, RopeParams);
    K kern = nullptr;
    if (a.d == 64) {
        kern = rp.span == 0 ? qk_rowgroup_kernel<T, 64, 0>
             : rp.span == 16 ? qk_rowgroup_kernel<T, 64, 16> : nullptr;
    } else if (a.d == 128) {
        kern = rp.span == 0 ? qk_rowgroup_kernel<T, 128, 0>
             : rp.span == 16 ? qk_rowgroup_kernel<T, 128, 16>
             : rp.span == 32 ? qk_rowgroup_kernel<T, 128, 32> : nullptr;
    } else if (a.d == 160) {
        kern = rp.span == 0 ? qk_rowgroup_kernel<T, 160, 0>
             : rp.span == 16 ? qk_rowgroup_kernel<T, 160, 16>
             : rp.span == 32 ? qk_rowgroup_kernel<T, 160, 32>
             : rp.span == 40 ? qk_rowgroup_kernel<T, 160, 40> : nullptr;
    }
    if (!kern) return false;
    // persistent: as many blocks as are resident at once
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRgWarps * 32, 0) !=
            cudaSuccess || per_sm <= 0)
        per_sm = 1;
    int64_t blocks = (items + kRgWarps - 1) / kRgWarps;
    const int64_t cap = static_cast<int64_t>(per_sm) * a.num_sms;
    if (blocks > cap) blocks = cap;
    (void)launch_pdl(a.pdl != 0, kern, dim3(static_cast<unsigned>(blocks)), dim3(kRgWarps * 32), 0, s, a, rp);
    return true;
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
    if (nvec <= 32) (void)launch_pdl(a.pdl != 0, qk_warp_kernel<T, 1>, dim3(g), dim3(128), 0, s, a, rp);
    else if (nvec <= 64) (void)launch_pdl(a.pdl != 0, qk_warp_kernel<T, 2>, dim3(g), dim3(128), 0, s, a, rp);
    else if (nvec <= 128) (void)launch_pdl(a.pdl != 0, qk_warp_kernel<T, 4>, dim3(g), dim3(128), 0, s, a, rp);
    else (void)launch_pdl(a.pdl != 0, qk_warp_kernel<T, 8>, dim3(g), dim3(128), 0, s, a, rp);
    return true;
}

}  // namespace

cudaError_t launch_qk_norm_rope(DType dt, const QkNormRopeArgs& args, const RopeParams& rp,
                                cudaStream_t s) {
    QkNormRopeArgs a = args;
    a.pdl = pdl_allowed(s);
    const int64_t tokens = static_cast<int64_t>(a.B) * a.S;
    if (tokens == 0) return cudaSuccess;
    if (dt == DType::F16 ? launch_rowgroup_path<__half>(a, rp, s)
                         : launch_rowgroup_path<__nv_bfloat16>(a, rp, s))
        return cudaGetLastError();
    if (dt == DType::F16 ? launch_unit_path<__half>(a, rp, s)
                         : launch_unit_path<__nv_bfloat16>(a, rp, s))
        return cudaGetLastError();
    if (dt == DType::F16 ? launch_warp_path<__half>(a, rp, s)
                         : launch_warp_path<__nv_bfloat16>(a, rp, s))
        return cudaGetLastError();
    if (dt == DType::F16 ? launch_head_path<__half>(a, rp, s)
                         : launch_head_path<__nv_bfloat16>(a, rp, s))
        return cudaGetLastError();
    // general path (full-width RMSNorm at other head sizes or spans)
    const size_t smem =
        (static_cast<size_t>(a.H + a.Hk) * a.d + 2 * static_cast<size_t>(rp.span / 2)) * sizeof(float);
    if (dt == DType::F16) {
        auto k = qk_norm_rope_kernel<__half>;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        (void)launch_pdl(a.pdl != 0, k, dim3(static_cast<unsigned>(tokens)), dim3(kRopeThreads), smem, s, a, rp);
    } else {
        auto k = qk_norm_rope_kernel<__nv_bfloat16>;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        (void)launch_pdl(a.pdl != 0, k, dim3(static_cast<unsigned>(tokens)), dim3(kRopeThreads), smem, s, a, rp);
    }
    return cudaGetLastError();
}

}  // namespace blk
