// Host-side launch interface between the C-ABI layer (api.cu) and the
// kernel translation units. Launchers assume validated arguments.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "blk.h"
#include "common.cuh"

namespace blk {

enum class DType { F16 = 0, BF16 = 1 };

// ---- K1: row norms (norm.cu)
// x, res and y are in the storage dtype unless the matching *_f32 flag is set
// (fp32 row-major); y32 (nullable) receives an fp32 copy of y. Supported
// combinations: any of x and res in fp32.
struct NormIO {
    const void* x;
    bool x_f32;
    const void* res;
    bool res_f32;
    void* y;
    float* y32;
    unsigned* err;  // device error word (bounded waits)
    int sms;        // SM count (persistent grid)
};
cudaError_t launch_norm(DType dt, bool rms, const NormIO& io, const void* gamma, const void* beta,
                        int64_t rows, int cols, float eps, cudaStream_t s);

// ---- K4/K5: qk-norm + rotary on head-split q/k, in place (rope.cu)
enum QkNormMode { QKN_NONE = 0, QKN_RMS_FULL = 1, QKN_LN_PER_HEAD = 2 };
struct QkNormRopeArgs {
    int pdl;            // launched with programmatic stream serialization (set by the launcher)
    void* q;            // [B, H, S, d]
    void* k;            // [B, Hk, S, d] or nullptr (then Hk must be 0)
    const void* q_w;    // norm weights (mode-dependent layout) or nullptr
    const void* k_w;
    const void* q_bias; // [H*d] or nullptr (added first)
    const void* k_bias; // [Hk*d] or nullptr
    int B, S, H, Hk, d;
    int mode;           // QkNormMode
    float eps;
    int num_sms;        // persistent grid size for the unit path
};
cudaError_t launch_qk_norm_rope(DType dt, const QkNormRopeArgs& a, const RopeParams& rp,
                                cudaStream_t s);

// ---- K2: tcgen05 GEMM with fused epilogues (gemm.cu)
enum GemmEpi { EPI_LINEAR = 0, EPI_SWIGLU = 1, EPI_GELU = 2, EPI_QKV = 3 };
struct GemmArgs {
    int pdl;              // launched with programmatic stream serialization (set by the launcher)
    int M, N, K;          // out is [M, N]; for SWIGLU N = intermediate (gate/up rows each)
    void* out;            // LINEAR / SWIGLU / GELU output, row stride N
    const void* bias;     // [N] or nullptr
    const void* res1;     // [M, N] or nullptr
    const void* res2;
    int out_f32;          // LINEAR: out is fp32
    int res1_f32;         // LINEAR: res1 / res2 are fp32
    int res2_f32;
    // EPI_QKV: scatter of [M, (H+2Hk)d] into head-split q/k/v
    void* q;
    void* k;
    void* v;
    int S, H, Hk, d, interleaved;
    unsigned* err;
    int n_fastest;        // work-unit order (set by launch_gemm)
    // split of the last, partial round of work units along K (LINEAR, GELU,
    // QKV; only with scratch): fp32 partial tiles and per-warp arrival
    // counters (zero before the launch, left zero after it)
    float* split_ws;
    unsigned* split_cnt;
    int split_s;          // segments per split unit (set by launch_gemm; 1 = none)
    int split_base;       // first split unit
    // pair GEMM: the output goes out by TMA stores (set by its launcher): 1
    // in boxes of 64 columns, 2 (QKV) of 32
    int tma_out;
};
// scratch of a split GEMM: kGemmSplitSlots partial 128 x 256 fp32 tiles, then
// kGemmSplitCounters counters
constexpr int kGemmSplitSlots = 256;
constexpr int kGemmSplitCounters = 1024;
constexpr size_t kGemmSplitBytes =
    static_cast<size_t>(kGemmSplitSlots) * 128 * 256 * 4 + kGemmSplitCounters * 4;
// a: [M, K]; b: [N(or N rows of gate), K]; b2: up weights for SWIGLU.
cudaError_t launch_gemm(DType dt, int epi, const void* a, const void* b, const void* b2,
                        const GemmArgs& args, const RopeParams& rp, int num_sms, cudaStream_t s);

// the same GEMM on CTA pairs (gemm2.cu): 256-row tiles, one tcgen05 MMA of
// M = 256 per pair of SMs; launch_gemm takes it whenever M > 128
cudaError_t launch_gemm_pair(DType dt, int epi, const void* a, const void* b, const void* b2,
                             const GemmArgs& g, const RopeParams& rp, int num_sms,
                             cudaStream_t s);

// ---- K2q: Q8_0 weights (gemm_q8.cu): codes q int8 [N, K], scales fp16
// d [K/32, N]; for SWIGLU q/d are the gate weight and q2/d2 the up weight.
// No split of the last round (the args' split fields are ignored).
cudaError_t launch_gemm_q8(DType dt, int epi, const void* a, const int8_t* q, const void* d,
                           const int8_t* q2, const void* d2, const GemmArgs& args,
                           const RopeParams& rp, int num_sms, cudaStream_t s);
// w [rows, cols] (storage dtype, cols % 32 == 0) -> codes q [rows, cols],
// scales d [cols/32, rows] (fp16)
// W = q * d in the storage type (see q8_dequant_kernel), for up to
// kQ8DequantMaxJobs matrices in one launch: codes q [rows, cols], fp16
// scales d [cols/32, rows], output w [rows, cols]; cols % 32 == 0, every
// pointer 16-byte aligned.
constexpr int kQ8DequantMaxJobs = 5;
struct Q8DequantJob {
    const int8_t* q;
    const void* d;
    void* w;
    int64_t rows, cols;
};
cudaError_t launch_q8_dequant(DType dt, const Q8DequantJob* jobs, int n_jobs, cudaStream_t s);
cudaError_t launch_q8_quantize(DType dt, const void* w, int64_t rows, int64_t cols, int8_t* q,
                               void* d, cudaStream_t s);

// ---- K3: tcgen05 flash attention (dispatch in attn.cu)
struct AttnArgs {
    int pdl;  // launched with programmatic stream serialization (set by the launcher)
    const void* q;
    const void* k;
    const void* v;
    void* o;
    int B, S, H, Hk, d;
    float scale;
    int alibi;
    const float* slopes;  // device [H] or nullptr (standard slopes)
    unsigned* err;
    int num_sms;          // persistent grid size
};
cudaError_t launch_attention(DType dt, const AttnArgs& a, cudaStream_t s);
// head_dim 64 / 128: the paired-query-tile kernels (attn_pair.cu, attn_pair128.cu)
cudaError_t launch_attention_pair64(DType dt, const AttnArgs& a, cudaStream_t s);
cudaError_t launch_attention_pair128(DType dt, const AttnArgs& a, cudaStream_t s);
// head_dim 128 / 160: a group's query heads packed into one tile (attn_gqa.cu)
cudaError_t launch_attention_gqa(DType dt, const AttnArgs& a, cudaStream_t s);

// ---- K6: decode-step attention over a KV cache (attn_decode.cu)
struct DecodeArgs {
    const void* q;        // [B, H, d]
    const void* k;        // [B, Hk, S_max, d]
    const void* v;
    void* o;              // [B, H, d]
    const int32_t* lens;  // device [B]
    const float* slopes;  // device [H] or nullptr (standard slopes)
    float* ws;            // [B, H, parts, d + 2] partial results
    int B, H, Hk, d, S_max, parts;
    float scale;
    int alibi;
};
cudaError_t launch_attention_decode(DType dt, const DecodeArgs& a, cudaStream_t s);
// number of key ranges per (batch, kv head), and its device-independent bound
int decode_parts(int64_t B, int64_t Hk, int64_t S_max, int64_t head_dim, int num_sms);
int decode_parts_max(int64_t S_max);

// ---- per-device state and error reporting shared with other entry points (api.cu)
// SM count and device error word of the current device (set up on first use).
blk_status current_device_info(int* sms, unsigned** err);
// Set a kernel's maximum dynamic shared memory on the current device, once
// per (kernel, device): the attribute belongs to the device's context, so a
// process that drives several GPUs sets it on each. Thread-safe.
cudaError_t set_smem_attr_once(const void* func, int smem_bytes);
// Whether launches on `s` take programmatic stream serialization: yes for
// direct launches, which it spares most of the launch latency (whole-block
// forwards 2-5% faster); no while `s` is being captured into a CUDA graph,
// whose replay already hides that latency and where the next kernel's blocks,
// placed early, slowed the OLMo-2 block by 1.2%.
bool pdl_allowed(cudaStream_t s);
// Launch a hot-path kernel, with programmatic stream serialization when
// `pdl` (from pdl_allowed(s)): it may then begin (set-up only) while the
// previous kernel on `s` drains. The kernel is told the same through its
// arguments and then calls pdl_wait() before any global memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}
// Record a printf-style message for blk_last_error() and return `st`.
blk_status report_error_status(blk_status st, const char* fmt, ...);

// ---- tensor maps (api.cu)
// 2D row-major [rows, cols] map with a {64, box_rows} box and 128B swizzle.
bool make_tmap_2d(CUtensorMap* m, DType dt, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t box_rows);
// 2D row-major [rows, cols] map of any element type with a {box_cols,
// box_rows} box: no swizzle, or the 128-byte swizzle (box rows of 128 bytes,
// shared-memory side 1024-byte aligned).
bool make_tmap_2d_plain(CUtensorMap* m, CUtensorMapDataType type, uint32_t elem_bytes,
                        const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                        uint32_t box_rows, bool swizzle128 = false);
// 3D [planes, rows, cols] map of 16-bit values with a {box_cols, box_rows, 1}
// box: 64 columns (128-byte rows) with the 128-byte swizzle, or 32 columns
// (64-byte rows) with the 64-byte swizzle.
bool make_tmap_3d(CUtensorMap* m, DType dt, const void* base, uint64_t planes, uint64_t rows,
                  uint64_t cols, uint32_t box_rows, uint32_t box_cols = 64);

}  // namespace blk
