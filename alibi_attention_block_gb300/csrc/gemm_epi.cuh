// The GEMM kernels' shared pieces (gemm.cu, gemm_q8.cu): tile constants,
// the persistent work-unit decode with its split last round, and the fused
// epilogues run on one accumulator tile read from TMEM.
#pragma once

#include "internal.h"

namespace blk {
namespace gemm {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each with half of the columns
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr int kSplitMinKb = 32;  // k-blocks per segment of a split unit, at least

// Work unit v of the persistent loop: unit u over k-blocks [kb0, kb1). Units
// before split_base run whole; each unit of the last, partial round is
// split into split_s segments along K, run by otherwise idle CTAs.
struct Unit {
    int u, q, kb0, kb1;
};
template <bool SPLIT>
__device__ __forceinline__ Unit decode_unit(const GemmArgs& g, int v, int kb_count) {
    if (!SPLIT || v < g.split_base) return {v, 0, 0, kb_count};
    const int t = (v - g.split_base) / g.split_s;
    const int q = v - g.split_base - t * g.split_s;
    return {g.split_base + t, q, q * kb_count / g.split_s, (q + 1) * kb_count / g.split_s};
}

// Sum of a split unit's partial tiles for 32 columns of this thread's row, in
// segment order (the same order whichever segment finishes last): its own
// segment's values come from o, the others' from their [column][row]
// partials.
template <int BN>
__device__ __forceinline__ void add_partials(float (&o)[32], const float* part, int part_s,
                                             int self, int col0, int trow) {
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    for (int q = 0; q < part_s; ++q) {
        if (q == self) {
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] += o[i];
        } else {
            const float* p = part + static_cast<size_t>(q) * (kBM * BN) +
                             static_cast<size_t>(col0) * kBM + trow;
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] += __ldcg(p + i * kBM);
        }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = acc[i];
}

template <typename T>
__device__ __forceinline__ void store_row32(T* dst, const float (&o)[32], int valid) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        if (v * 8 < valid) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = o[v * 8 + e];
            store8(dst + v * 8, f);
        }
    }
}

template <typename T>
__device__ __forceinline__ void add_row32(const T* src, float (&o)[32], int valid) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        if (v * 8 < valid) {
            float f[8];
            load8(src + v * 8, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[v * 8 + e] += f[e];
        }
    }
}

// fp32 write-out of a warp's 32 output rows x 32 columns, held one row per
// thread (the TMEM lane layout): staged through the warp's 4 KB of shared
// memory (16-byte chunks XOR-swizzled by row, conflict-free both ways), then
// stored 4 rows x 128 bytes per instruction, whole lines instead of 16 bytes
// of each of 32 rows (half-sector writes). Storage-type rows (64 bytes per
// chunk) are stored directly: there the staging only lengthens the epilogue.
__device__ __forceinline__ void store_chunk_f32(const GemmArgs& g, uint32_t stg, int lane,
                                                int m_base, int n0, const float (&o)[32]) {
#pragma unroll
    for (int v = 0; v < 8; ++v)
        st_shared_v4(stg + lane * 128 + ((v ^ (lane & 7)) << 4), __float_as_uint(o[4 * v]),
                     __float_as_uint(o[4 * v + 1]), __float_as_uint(o[4 * v + 2]),
                     __float_as_uint(o[4 * v + 3]));
    __syncwarp();
    const int cq = lane & 7;       // columns 4 cq .. 4 cq + 3 of the chunk
    const int gcol = n0 + cq * 4;  // N % 8 == 0: four columns are all valid or none
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const int rr = p * 4 + (lane >> 3);
        const float4 v = ld_shared_v4(stg + rr * 128 + ((cq ^ (rr & 7)) << 4));
        const int grow = m_base + rr;
        if (grow < g.M && gcol < g.N)
            *reinterpret_cast<float4*>(static_cast<float*>(g.out) +
                                       static_cast<int64_t>(grow) * g.N + gcol) = v;
    }
    __syncwarp();
}

// One thread's 32 output values of one row into its warp's staging box of
// 32 rows x 128 bytes, laid out for a TMA store with the 128-byte swizzle
// (16-byte piece p of row r at r * 128 + ((p ^ (r & 7)) << 4), the box
// 1024-byte aligned): 16-bit values as pieces p0 .. p0 + 3 (half a box row),
// fp32 values as all eight pieces.
template <typename T>
__device__ __forceinline__ void stage_row(uint32_t stg, int r, int p0, bool f32,
                                          const float (&o)[32]) {
    const uint32_t row = stg + r * 128;
    if (f32) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
            st_shared_v4(row + ((v ^ (r & 7)) << 4), __float_as_uint(o[4 * v]),
                         __float_as_uint(o[4 * v + 1]), __float_as_uint(o[4 * v + 2]),
                         __float_as_uint(o[4 * v + 3]));
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v)
            st_shared_v4(row + (((p0 + v) ^ (r & 7)) << 4),
                         dt_traits<T>::pack2(o[8 * v], o[8 * v + 1]),
                         dt_traits<T>::pack2(o[8 * v + 2], o[8 * v + 3]),
                         dt_traits<T>::pack2(o[8 * v + 4], o[8 * v + 5]),
                         dt_traits<T>::pack2(o[8 * v + 6], o[8 * v + 7]));
    }
}

// One thread's 32 16-bit values as one 64-byte row of a 32 x 64-byte staging
// box laid out for a TMA store with the 64-byte swizzle (16-byte piece p of
// row r at r * 64 + ((p ^ ((r >> 1) & 3)) << 4), the box 512-byte aligned).
template <typename T>
__device__ __forceinline__ void stage_row64(uint32_t stg, int r, const float (&o)[32]) {
    const uint32_t row = stg + r * 64;
#pragma unroll
    for (int v = 0; v < 4; ++v)
        st_shared_v4(row + ((v ^ ((r >> 1) & 3)) << 4), dt_traits<T>::pack2(o[8 * v], o[8 * v + 1]),
                     dt_traits<T>::pack2(o[8 * v + 2], o[8 * v + 3]),
                     dt_traits<T>::pack2(o[8 * v + 4], o[8 * v + 5]),
                     dt_traits<T>::pack2(o[8 * v + 6], o[8 * v + 7]));
}

// Around one staged box: before its first chunk is written, the previous
// box's store has read the staging buffer; after its last, the writes are
// made visible to the TMA and one lane stores the box (x, y: its first
// column and row; a box wholly past N or M is skipped, a partial one is
// clipped by the TMA).
__device__ __forceinline__ void stage_begin(int lane) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
}
__device__ __forceinline__ void stage_store(const CUtensorMap* tmo, uint32_t stg, int lane, int x,
                                            int y, const GemmArgs& g) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && x < g.N && y < g.M) {
        tma_store_2d(tmo, stg, x, y);
        bulk_commit();
    }
}

// A tile's accumulator started as its bias row, for this thread's lane of
// TMEM and its half of the tile's 32-column chunks (columns past N start at
// zero), before the tile's MMAs accumulate onto it. Every lane reads the
// same bias words (one transaction per warp each), two chunks' words in
// flight at a time.
template <typename T, int NB>
__device__ __forceinline__ void preload_bias_batch(const GemmArgs& g, uint32_t tbase, int n00,
                                                   int c0) {
    const T* bp = static_cast<const T*>(g.bias);
    uint4 w[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int n0 = n00 + (c0 + b) * 32;
        const int valid = g.N - n0;
        const uint4* p = reinterpret_cast<const uint4*>(bp + n0);
#pragma unroll
        for (int v = 0; v < 4; ++v) w[b][v] = v * 8 < valid ? p[v] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint32_t u[4] = {w[b][v].x, w[b][v].y, w[b][v].z, w[b][v].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = dt_traits<T>::unpack2(u[e]);
                r[8 * v + 2 * e] = __float_as_uint(f.x);
                r[8 * v + 2 * e + 1] = __float_as_uint(f.y);
            }
        }
        tmem_st32_nowait(tbase + (c0 + b) * 32, r);
    }
}
template <typename T, int BN>
__device__ __forceinline__ void preload_bias(const GemmArgs& g, uint32_t tbase, int nt, int half) {
    constexpr int kC = BN / 64;  // this warp's chunks, two at a time
    const int c0 = half * kC;
#pragma unroll 1
    for (int b = 0; b < kC; b += 2) preload_bias_batch<T, 2>(g, tbase, nt * BN, c0 + b);
    tmem_st_wait();
}

// (a0 b0, a1 b1) in one instruction.
__device__ __forceinline__ void fmul2(float a0, float a1, float b0, float b1, float& d0, float& d1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// silu(g) u for two elements: g u / (1 + 2^(-g log2(e))), in paired f32x2
// arithmetic with ex2.approx and an approximate reciprocal (g -> -inf: the
// denominator overflows, its reciprocal is 0, and so is the result).
__device__ __forceinline__ void swiglu2(float g0, float g1, float u0, float u1, float& o0,
                                        float& o1) {
    constexpr float kNegL2e = -1.4426950408889634f;
    const uint64_t one2 = f2_pack(1.0f, 1.0f);
    float t0, t1, d0, d1, p0, p1;
    fmul2(g0, g1, kNegL2e, kNegL2e, t0, t1);
    ffma2(ex2_approx(t0), ex2_approx(t1), one2, one2, d0, d1);
    fmul2(g0, g1, u0, u1, p0, p1);
    fmul2(p0, p1, rcp_approx(d0), rcp_approx(d1), o0, o1);
}

// GELU, tanh form, for two elements: 0.5 z (1 + tanh(u)) with u = sqrt(2/pi)
// (z + 0.044715 z^3). Since 0.5 (1 + tanh(u)) = 1 / (1 + e^(-2u)), it is
// z / (1 + 2^t), t = -2 sqrt(2/pi) log2(e) z (1 + 0.044715 z^2): one
// ex2.approx and one approximate reciprocal per element instead of a tanh,
// the rest in paired f32x2 arithmetic (z -> -inf: the result goes to 0).
__device__ __forceinline__ void gelu2(float z0, float z1, float& o0, float& o1) {
    constexpr float kT = -2.0f * 0.7978845608028654f * 1.4426950408889634f;
    const uint64_t one2 = f2_pack(1.0f, 1.0f);
    float q0, q1, w0, w1, t0, t1, d0, d1;
    fmul2(z0, z1, z0, z1, q0, q1);
    ffma2(q0, q1, f2_pack(0.044715f, 0.044715f), one2, q0, q1);
    fmul2(z0, z1, kT, kT, w0, w1);
    fmul2(w0, w1, q0, q1, t0, t1);
    ffma2(ex2_approx(t0), ex2_approx(t1), one2, one2, d0, d1);
    fmul2(z0, z1, rcp_approx(d0), rcp_approx(d1), o0, o1);
}

// tmo: the output's tensor map for TMA stores of staged boxes (16-bit
// outputs of LINEAR, GELU, SWIGLU: [M, N]; QKV: q, with tmo_k and tmo_v, each
// [B * heads, S, d]; stg then a 1024-byte-aligned 4 KB staging box), or
// nullptr for per-thread stores.
template <typename T, int BN, int EPI, int ROT, bool SPLIT>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& g, const RopeParams& rp,
                                              uint32_t tbase, int m, int nt, uint32_t stg,
                                              int lane, int m_base, const float* part, int self,
                                              int trow, int half,
                                              const CUtensorMap* tmo = nullptr,
                                              const CUtensorMap* tmo_k = nullptr,
                                              const CUtensorMap* tmo_v = nullptr,
                                              bool bias_in_acc = false) {
    // this warp's half of the tile's 32-column chunks
    constexpr int kChunks = (EPI == EPI_SWIGLU ? BN / 2 : BN) / 32;
    const int c_begin = half * (kChunks / 2), c_end = c_begin + kChunks / 2;
    const bool row_ok = m < g.M;
    if constexpr (EPI == EPI_SWIGLU) {
        constexpr int kHalf = BN / 2;
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
            uint32_t gr[32], ur[32];
            tmem_ld32(tbase + c * 32, gr);
            tmem_ld32(tbase + kHalf + c * 32, ur);
            const int n0 = nt * kHalf + c * 32;
            if (tmo) {
                // two chunks per box (64 columns of 16-bit values)
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                    swiglu2(__uint_as_float(gr[i]), __uint_as_float(gr[i + 1]), __uint_as_float(ur[i]),
                            __uint_as_float(ur[i + 1]), o[i], o[i + 1]);
                const int k = c - c_begin;
                if ((k & 1) == 0) stage_begin(lane);
                stage_row<T>(stg, lane, (k & 1) * 4, false, o);
                if ((k & 1) == 1 || c + 1 == c_end)
                    stage_store(tmo, stg, lane, nt * kHalf + (c_begin + (k & ~1)) * 32, m_base, g);
                continue;
            }
            if (!row_ok || n0 >= g.N) continue;
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; i += 2)
                swiglu2(__uint_as_float(gr[i]), __uint_as_float(gr[i + 1]), __uint_as_float(ur[i]),
                        __uint_as_float(ur[i + 1]), o[i], o[i + 1]);
            store_row32(static_cast<T*>(g.out) + static_cast<int64_t>(m) * g.N + n0, o, g.N - n0);
        }
    } else if constexpr (EPI == EPI_QKV) {
        const int d = g.d;
        const int b = m / g.S;
        const int s = m - b * g.S;
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
            uint32_t r[32];
            tmem_ld32(tbase + c * 32, r);
            const int n0 = nt * BN + c * 32;
            if (!row_ok || n0 >= g.N) continue;
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
            if constexpr (SPLIT)
                if (part) add_partials<BN>(o, part, g.split_s, self, c * 32, trow);
            if (g.bias && !bias_in_acc) add_row32(static_cast<const T*>(g.bias) + n0, o, 32);
            int which, head, dd0;
            if (g.interleaved) {
                head = n0 / (3 * d);
                const int w = n0 - head * 3 * d;
                which = w / d;
                dd0 = w - which * d;
            } else {
                const int hd = g.H * d, kd = g.Hk * d;
                which = n0 < hd ? 0 : (n0 < hd + kd ? 1 : 2);
                const int off = which == 0 ? 0 : (which == 1 ? hd : hd + kd);
                head = (n0 - off) / d;
                dd0 = n0 - off - head * d;
            }
            if constexpr (ROT > 0) {
                // the span is a compile-time constant so o[] stays in registers
                if (which < 2 && dd0 == 0) {
                    constexpr int kHalf = ROT / 2;
#pragma unroll
                    for (int j = 0; j < kHalf; ++j) {
                        float cs, sn;
                        rope_cos_sin(rp, s, j, cs, sn);
                        const float x1 = o[j], x2 = o[j + kHalf];
                        o[j] = x1 * cs - x2 * sn;
                        o[j + kHalf] = x2 * cs + x1 * sn;
                    }
                }
            }
            const int nheads = which == 0 ? g.H : g.Hk;
            if (tmo) {
                // one chunk (32 columns of one head) per box of the warp's 32
                // positions (S % 32 == 0: one sequence), two 2 KB boxes of
                // the warp's staging area in turn, so a box is staged while
                // the previous one's store still reads
                const uint32_t sb = stg + ((c - c_begin) & 1) * 2048;
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
                stage_row64<T>(sb, lane, o);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && m_base < g.M) {
                    const int b0 = m_base / g.S;
                    tma_store_3d(which == 0 ? tmo : (which == 1 ? tmo_k : tmo_v), sb, dd0,
                                 m_base - b0 * g.S, b0 * nheads + head);
                    bulk_commit();
                }
                continue;
            }
            T* base = static_cast<T*>(which == 0 ? g.q : (which == 1 ? g.k : g.v));
            T* dst = base + ((static_cast<int64_t>(b) * nheads + head) * g.S + s) * d + dd0;
            store_row32(dst, o, 32);
        }
    } else if (tmo) {
        // TMA stores of staged boxes: fp32 output one chunk per box (32
        // columns), 16-bit output two (64 columns); a chunk past N is staged
        // as it is and clipped by the store
        const bool f32 = EPI == EPI_LINEAR && g.out_f32;
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
            uint32_t r[32];
            tmem_ld32(tbase + c * 32, r);
            const int n0 = nt * BN + c * 32;
            const int valid = g.N - n0;
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
            if (valid > 0) {
                if constexpr (SPLIT)
                    if (part) add_partials<BN>(o, part, g.split_s, self, c * 32, trow);
                if (g.bias && !bias_in_acc) add_row32(static_cast<const T*>(g.bias) + n0, o, valid);
                if constexpr (EPI == EPI_GELU) {
#pragma unroll
                    for (int i = 0; i < 32; i += 2) gelu2(o[i], o[i + 1], o[i], o[i + 1]);
                }
                const int64_t off = static_cast<int64_t>(m) * g.N + n0;
                if (row_ok && g.res1) {
                    if (g.res1_f32) add_row32(static_cast<const float*>(g.res1) + off, o, valid);
                    else add_row32(static_cast<const T*>(g.res1) + off, o, valid);
                }
                if (row_ok && g.res2) {
                    if (g.res2_f32) add_row32(static_cast<const float*>(g.res2) + off, o, valid);
                    else add_row32(static_cast<const T*>(g.res2) + off, o, valid);
                }
            }
            const int k = c - c_begin;
            const bool first = f32 || (k & 1) == 0;
            const bool last = f32 || (k & 1) == 1 || c + 1 == c_end;
            if (first) stage_begin(lane);
            stage_row<T>(stg, lane, f32 ? 0 : (k & 1) * 4, f32, o);
            if (last)
                stage_store(tmo, stg, lane, f32 ? n0 : nt * BN + (c_begin + (k & ~1)) * 32,
                            m_base, g);
        }
    } else {
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
            uint32_t r[32];
            tmem_ld32(tbase + c * 32, r);
            const int n0 = nt * BN + c * 32;
            if (n0 >= g.N) continue;  // uniform across the warp
            const int valid = g.N - n0;
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
            if constexpr (SPLIT)
                if (part) add_partials<BN>(o, part, g.split_s, self, c * 32, trow);
            if (g.bias && !bias_in_acc) add_row32(static_cast<const T*>(g.bias) + n0, o, valid);
            if constexpr (EPI == EPI_GELU) {
#pragma unroll
                for (int i = 0; i < 32; i += 2) gelu2(o[i], o[i + 1], o[i], o[i + 1]);
            }
            const int64_t off = static_cast<int64_t>(m) * g.N + n0;
            if (row_ok && g.res1) {
                if (g.res1_f32) add_row32(static_cast<const float*>(g.res1) + off, o, valid);
                else add_row32(static_cast<const T*>(g.res1) + off, o, valid);
            }
            if (row_ok && g.res2) {
                if (g.res2_f32) add_row32(static_cast<const float*>(g.res2) + off, o, valid);
                else add_row32(static_cast<const T*>(g.res2) + off, o, valid);
            }
            // fp32 output (LINEAR only: the other epilogues' kernels keep no
            // staging room in shared memory)
            if (EPI == EPI_LINEAR && g.out_f32)
                store_chunk_f32(g, stg, lane, m_base, n0, o);  // all lanes (rows checked inside)
            else if (row_ok)
                store_row32(static_cast<T*>(g.out) + off, o, valid);
        }
    }
}


}  // namespace gemm
}  // namespace blk
