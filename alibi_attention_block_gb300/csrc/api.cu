// C ABI of the block library (include/blk.h): argument validation (before any
// CUDA call, so a rejected call has no side effects), TMA descriptor set-up,
// kernel dispatch and the blk_forward step sequence.
#include <algorithm>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <utility>
#include <string>

#include "blk.h"
#include "internal.h"
#include "model.h"

namespace blk {

// Device error word, set by kernels whose bounded waits give up.
__device__ unsigned int g_dev_err;

// Self-test of the bounded-wait path: one thread waits on an mbarrier that
// nothing arrives at; the wait gives up after limit_ns and sets the error word.
__global__ void bounded_wait_selftest_kernel(unsigned* err, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_barrier_init();
    if (!mbar_try_wait(b, 0)) mbar_wait_slow(b, 0, err, limit_ns);
}

namespace {

thread_local std::string t_last_error;

blk_status fail(blk_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

blk_status cuda_fail(cudaError_t e, const char* what) {
    return fail(BLK_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxHostChunks = 16;
struct DevState {
    bool init = false;
    int sms = 0;
    unsigned* err = nullptr;
    // copy streams and events of blk_forward_host (created on its first use)
    bool pipe_init = false;
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_in[kMaxHostChunks] = {}, ev_out[kMaxHostChunks] = {},
                ev_done = nullptr;
};
constexpr int kMaxDevices = 64;
DevState g_dev[kMaxDevices];
std::mutex g_mu;

blk_status dev_state(DevState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(BLK_EUNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DevState& d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(BLK_EUNSUPPORTED, "kernels are built for sm_103a; device is sm_%d%d", major,
                        minor);
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dev_err);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
        d.err = static_cast<unsigned*>(p);
        d.init = true;
    }
    *out = &d;
    return BLK_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dt(blk_dtype dt) { return dt == BLK_F16 || dt == BLK_BF16; }

DType to_dt(blk_dtype dt) { return dt == BLK_F16 ? DType::F16 : DType::BF16; }

RopeParams make_rope(int span, float base) {
    RopeParams rp;
    std::memset(&rp, 0, sizeof(rp));
    rp.span = span;
    const double two_pi = 6.283185307179586476925286766559;
    rp.c1 = 6.28125f;  // 201/32: 8 significant bits, so k * c1 is exact for k < 2^16
    const double r1 = two_pi - 6.28125;
    rp.c2 = static_cast<float>(r1);
    rp.c3 = static_cast<float>(r1 - static_cast<double>(rp.c2));
    rp.inv_2pi = static_cast<float>(1.0 / two_pi);
    for (int j = 0; j < span / 2; ++j) {
        const double th = std::pow(static_cast<double>(base), -2.0 * j / span);
        const float hi = static_cast<float>(th);
        rp.theta_hi[j] = hi;
        rp.theta_lo[j] = static_cast<float>(th - static_cast<double>(hi));
    }
    return rp;
}

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

constexpr int64_t kI32 = 0x7fffffff;

}  // namespace

blk_status current_device_info(int* sms, unsigned** err) {
    DevState* ds = nullptr;
    const blk_status st = dev_state(&ds);
    if (st != BLK_OK) return st;
    *sms = ds->sms;
    *err = ds->err;
    return BLK_OK;
}

cudaError_t set_smem_attr_once(const void* func, int smem_bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({func, dev})) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess) done.insert({func, dev});
    return e;
}

blk_status report_error_status(blk_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

bool pdl_allowed(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        (void)cudaGetLastError();  // not the launch's error: launch plainly
        return false;
    }
    return st == cudaStreamCaptureStatusNone;
}

bool make_tmap_2d(CUtensorMap* m, DType dt, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, dt == DType::F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_2d_plain(CUtensorMap* m, CUtensorMapDataType type, uint32_t elem_bytes,
                        const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                        uint32_t box_rows, bool swizzle128) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * elem_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap* m, DType dt, const void* base, uint64_t planes, uint64_t rows,
                  uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {cols, rows, planes};
    const cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
    const cuuint32_t box[3] = {box_cols, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, dt == DType::F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace blk

using namespace blk;

// ------------------------------------------------------------ validation --
namespace {

#define BLK_REQUIRE(cond, ...)                              \
    do {                                                    \
        if (!(cond)) return fail(BLK_EINVAL, __VA_ARGS__);  \
    } while (0)

blk_status check_ptr(const void* p, const char* name, bool required) {
    if (!p) return required ? fail(BLK_EINVAL, "%s is NULL", name) : BLK_OK;
    if (!aligned16(p)) return fail(BLK_EINVAL, "%s is not 16-byte aligned", name);
    return BLK_OK;
}

#define BLK_CHECK_PTR(p, required)                                     \
    do {                                                               \
        blk_status st_ = check_ptr((p), #p, (required));               \
        if (st_ != BLK_OK) return st_;                                 \
    } while (0)

blk_status validate_norm(const void* x, const void* res, const void* g, const void* b,
                         const void* y, int64_t rows, int64_t cols, float eps, blk_dtype dt) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    BLK_REQUIRE(rows >= 0 && rows <= kI32 * 16, "rows out of range");
    BLK_REQUIRE(cols >= 8 && cols % 8 == 0 && cols <= 16384, "cols must be a multiple of 8 in [8, 16384]");
    BLK_REQUIRE(std::isfinite(eps) && eps >= 0.f, "eps must be finite and >= 0");
    BLK_CHECK_PTR(x, true);
    BLK_CHECK_PTR(res, false);
    BLK_CHECK_PTR(g, true);
    BLK_CHECK_PTR(b, false);
    BLK_CHECK_PTR(y, true);
    return BLK_OK;
}

blk_status validate_qkv_desc(const blk_qkv_desc* d) {
    BLK_REQUIRE(d, "descriptor is NULL");
    BLK_REQUIRE(d->batch >= 1 && d->seq >= 1 && d->batch * d->seq <= kI32, "batch*seq out of range");
    BLK_REQUIRE(d->hidden >= 8 && d->hidden % 8 == 0 && d->hidden <= kI32, "hidden must be a positive multiple of 8");
    BLK_REQUIRE(d->n_heads >= 1 && d->n_kv_heads >= 1 && d->n_heads % d->n_kv_heads == 0,
                "n_heads must be a positive multiple of n_kv_heads");
    BLK_REQUIRE(d->head_dim >= 32 && d->head_dim % 32 == 0 && d->head_dim <= 256,
                "head_dim must be a multiple of 32 in [32, 256]");
    BLK_REQUIRE(d->qkv_layout == BLK_QKV_STACKED || d->qkv_layout == BLK_QKV_HEAD_INTERLEAVED,
                "unknown qkv_layout");
    BLK_REQUIRE(d->qkv_layout == BLK_QKV_STACKED || d->n_heads == d->n_kv_heads,
                "head-interleaved QKV needs n_heads == n_kv_heads");
    BLK_REQUIRE(d->qk_norm >= BLK_QKNORM_NONE && d->qk_norm <= BLK_QKNORM_LN_PER_HEAD,
                "unknown qk_norm");
    BLK_REQUIRE(std::isfinite(d->qk_norm_eps) && d->qk_norm_eps >= 0.f, "qk_norm_eps must be >= 0");
    BLK_REQUIRE(d->rotary_span >= 0 && d->rotary_span % 2 == 0 && d->rotary_span <= d->head_dim &&
                    d->rotary_span / 2 <= kMaxRotaryPairs,
                "rotary_span must be even and in [0, head_dim]");
    BLK_REQUIRE(d->rotary_span == 0 || (std::isfinite(d->rope_base) && d->rope_base > 1.f),
                "rope_base must be > 1 when rotary is on");
    BLK_REQUIRE((d->n_heads + d->n_kv_heads) * d->head_dim * 4 <= 200 * 1024,
                "(n_heads + n_kv_heads) * head_dim too large for the qk-norm kernel");
    return BLK_OK;
}

blk_status validate_attn_desc(const blk_attn_desc* d) {
    BLK_REQUIRE(d, "descriptor is NULL");
    BLK_REQUIRE(d->batch >= 1 && d->seq >= 1 && d->batch * d->seq <= kI32, "batch*seq out of range");
    BLK_REQUIRE(d->n_heads >= 1 && d->n_kv_heads >= 1 && d->n_heads % d->n_kv_heads == 0,
                "n_heads must be a positive multiple of n_kv_heads");
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 160)
        return fail(BLK_EUNSUPPORTED, "attention head_dim must be 64, 128 or 160 (got %lld)",
                    static_cast<long long>(d->head_dim));
    if (d->causal != 1) return fail(BLK_EUNSUPPORTED, "only causal prefill attention is implemented");
    BLK_REQUIRE(d->alibi == 0 || d->alibi == 1, "alibi must be 0 or 1");
    BLK_REQUIRE(std::isfinite(d->softmax_scale), "softmax_scale must be finite");
    const int64_t nq = (d->seq + 127) / 128;
    BLK_REQUIRE(nq * d->batch * d->n_heads <= kI32, "grid too large");
    return BLK_OK;
}

blk_status validate_block(const blk_block_desc* d, const blk_block_weights* w,
                          const blk_q8_weights* q8 = nullptr) {
    BLK_REQUIRE(d && w, "descriptor or weights is NULL");
    blk_status st = validate_qkv_desc(&d->qkv);
    if (st != BLK_OK) return st;
    const auto& q = d->qkv;
    if (q.head_dim != 64 && q.head_dim != 128 && q.head_dim != 160)
        return fail(BLK_EUNSUPPORTED, "head_dim must be 64, 128 or 160");
    BLK_REQUIRE(d->norm_kind == BLK_NORM_LAYERNORM || d->norm_kind == BLK_NORM_RMS, "unknown norm_kind");
    BLK_REQUIRE(d->norm_place == BLK_NORM_PRE || d->norm_place == BLK_NORM_POST, "unknown norm_place");
    BLK_REQUIRE(d->residual == BLK_RESIDUAL_SEQUENTIAL || d->residual == BLK_RESIDUAL_PARALLEL,
                "unknown residual");
    BLK_REQUIRE(d->act == BLK_ACT_SWIGLU || d->act == BLK_ACT_GELU_TANH, "unknown act");
    BLK_REQUIRE(d->alibi == 0 || d->alibi == 1, "alibi must be 0 or 1");
    BLK_REQUIRE(std::isfinite(d->eps) && d->eps >= 0.f, "eps must be >= 0");
    BLK_REQUIRE(d->intermediate >= 8 && d->intermediate % 8 == 0 && d->intermediate <= kI32,
                "intermediate must be a positive multiple of 8");
    BLK_REQUIRE(q.hidden <= 16384, "hidden must be <= 16384");
    if (d->alibi && q.rotary_span != 0)
        return fail(BLK_EUNSUPPORTED,
                    "rotary and ALiBi are exclusive: set rotary_span = 0 for an ALiBi block");
    if (d->alibi && !w->alibi_slopes && !is_pow2(q.n_heads))
        return fail(BLK_EUNSUPPORTED, "standard ALiBi slopes need a power-of-two head count");
    if (d->norm_place == BLK_NORM_POST) {
        if (d->norm_kind != BLK_NORM_RMS || d->residual != BLK_RESIDUAL_SEQUENTIAL)
            return fail(BLK_EUNSUPPORTED, "post-norm blocks are RMSNorm, sequential");
    }
    const bool pre = d->norm_place == BLK_NORM_PRE;
    const bool seq_pre = pre && d->residual == BLK_RESIDUAL_SEQUENTIAL;
    const bool ln = d->norm_kind == BLK_NORM_LAYERNORM;
    const bool swiglu = d->act == BLK_ACT_SWIGLU;
    const bool dense = q8 == nullptr;  // projection weights in the storage dtype
    // Every slot is either used (and then required, except optional biases) or
    // must be NULL: a weight handed to the wrong slot is an error, not ignored.
    struct Slot {
        const void* p;
        const char* name;
        bool used;
        bool required;
    } slots[] = {
        {w->attn_norm_w, "attn_norm_w", pre, pre},
        {w->attn_norm_b, "attn_norm_b", pre && ln, false},
        {w->mlp_norm_w, "mlp_norm_w", seq_pre, seq_pre},
        {w->mlp_norm_b, "mlp_norm_b", seq_pre && ln, false},
        {w->post_attn_norm_w, "post_attn_norm_w", !pre, !pre},
        {w->post_mlp_norm_w, "post_mlp_norm_w", !pre, !pre},
        {w->w_qkv, "w_qkv", dense && true, dense && true},
        {w->b_qkv, "b_qkv", true, false},
        {w->q_norm_w, "q_norm_w", q.qk_norm != BLK_QKNORM_NONE, q.qk_norm != BLK_QKNORM_NONE},
        {w->k_norm_w, "k_norm_w", q.qk_norm != BLK_QKNORM_NONE, q.qk_norm != BLK_QKNORM_NONE},
        {w->w_o, "w_o", dense && true, dense && true},
        {w->b_o, "b_o", true, false},
        {w->w_gate, "w_gate", dense && swiglu, dense && swiglu},
        {w->w_up, "w_up", dense && true, dense && true},
        {w->b_up, "b_up", !swiglu, false},
        {w->w_down, "w_down", dense && true, dense && true},
        {w->b_down, "b_down", true, false},
        {w->alibi_slopes, "alibi_slopes", d->alibi != 0, false},
    };
    for (const Slot& s : slots) {
        if (!s.used && s.p) return fail(BLK_EINVAL, "weight slot %s is not used by this block and must be NULL", s.name);
        if (s.required && !s.p) return fail(BLK_EINVAL, "weight slot %s is required", s.name);
        if (s.p && !aligned16(s.p)) return fail(BLK_EINVAL, "weight slot %s is not 16-byte aligned", s.name);
    }
    if (dense) return BLK_OK;
    // Q8_0 projections: every input width is cut into 32-wide blocks
    BLK_REQUIRE(q.hidden % 32 == 0 && (q.n_heads * q.head_dim) % 32 == 0 &&
                    d->intermediate % 32 == 0,
                "Q8_0 weights need hidden, n_heads * head_dim and intermediate multiples of 32");
    const Slot qslots[] = {
        {q8->q_qkv, "q_qkv", true, true},   {q8->d_qkv, "d_qkv", true, true},
        {q8->q_o, "q_o", true, true},       {q8->d_o, "d_o", true, true},
        {q8->q_gate, "q_gate", swiglu, swiglu}, {q8->d_gate, "d_gate", swiglu, swiglu},
        {q8->q_up, "q_up", true, true},     {q8->d_up, "d_up", true, true},
        {q8->q_down, "q_down", true, true}, {q8->d_down, "d_down", true, true},
    };
    for (const Slot& s : qslots) {
        if (!s.used && s.p) return fail(BLK_EINVAL, "Q8_0 slot %s is not used by this block and must be NULL", s.name);
        if (s.required && !s.p) return fail(BLK_EINVAL, "Q8_0 slot %s is required", s.name);
        if (s.p && !aligned16(s.p)) return fail(BLK_EINVAL, "Q8_0 slot %s is not 16-byte aligned", s.name);
    }
    return BLK_OK;
}

struct FwdLayout {
    size_t n1, q, k, v, o, h, n2, a, h16, tmp, split, total;
};

FwdLayout forward_layout(const blk_block_desc* d) {
    const auto& q = d->qkv;
    const size_t T = static_cast<size_t>(q.batch) * q.seq;
    const size_t D = q.hidden, Hd = q.n_heads * q.head_dim, Kd = q.n_kv_heads * q.head_dim;
    FwdLayout L;
    size_t off = 0;
    auto take = [&](size_t elems) {
        const size_t at = off;
        off += align256(elems * 2);
        return at;
    };
    L.n1 = take(T * D);
    L.q = take(T * Hd);
    L.k = take(T * Kd);
    L.v = take(T * Kd);
    L.o = take(T * Hd);
    L.h = take(2 * T * D);    // fp32 mid-block residual stream
    L.n2 = take(T * D);
    L.a = take(T * static_cast<size_t>(d->intermediate));
    L.h16 = take(T * D);      // storage-dtype copy of h (post-norm MLP input)
    L.tmp = take(2 * T * D);  // fp32 sublayer output (parallel residual, post-norm input)
    L.split = take(kGemmSplitBytes / 2);  // partial tiles + counters of split GEMM rounds
    L.total = off;
    return L;
}

// The dequantize-once Q8_0 path: from this many tokens on, expanding a
// projection's weights once (3 bytes of traffic per weight) costs less than
// the W8A16 kernel's expansion of every weight tile per 128-row tile of x.
constexpr int64_t kQ8DequantMinTokens = 512;

// The projections of a block as (rows, cols) of their weights: QKV, output,
// gate (SwiGLU only), up, down; *n receives how many.
void q8_shapes(const blk_block_desc* d, int64_t (*rc)[2], int* n) {
    const auto& q = d->qkv;
    const int64_t D = q.hidden, Hd = q.n_heads * q.head_dim, Kd = q.n_kv_heads * q.head_dim;
    const int64_t F = d->intermediate;
    int i = 0;
    auto put = [&](int64_t r, int64_t c) {
        rc[i][0] = r;
        rc[i][1] = c;
        ++i;
    };
    put(Hd + 2 * Kd, D);
    put(D, Hd);
    if (d->act == BLK_ACT_SWIGLU) put(F, D);
    put(F, D);
    put(D, F);
    *n = i;
}

// Its scratch after the block's workspace: every projection's weights in the
// storage dtype, each 256-byte aligned, in q8_shapes order.
size_t q8_scratch_bytes(const blk_block_desc* d) {
    int64_t rc[kQ8DequantMaxJobs][2];
    int n = 0;
    q8_shapes(d, rc, &n);
    size_t total = 0;
    for (int i = 0; i < n; ++i) total += align256(static_cast<size_t>(2 * rc[i][0] * rc[i][1]));
    return total;
}

// Records an event after each kernel launch of blk_forward_ex and the kind
// of each launch (see blk_forward_ex in blk.h).
struct StepLog {
    void* const* events;
    int n_events;
    int32_t* kinds;
    int* n_out;
    cudaStream_t s;
    int n = 0;
    bool capturing = false;
    // under stream capture an event record becomes a graph node only when
    // recorded as external
    blk_status record(int i) {
        cudaEvent_t ev = static_cast<cudaEvent_t>(events[i]);
        cudaError_t e = capturing ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                  : cudaEventRecord(ev, s);
        return e == cudaSuccess ? BLK_OK : cuda_fail(e, "cudaEventRecord");
    }
    blk_status begin() {
        if (events && n_events > 0) {
            cudaStreamCaptureStatus cst = cudaStreamCaptureStatusNone;
            cudaError_t e = cudaStreamIsCapturing(s, &cst);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
            capturing = cst == cudaStreamCaptureStatusActive;
            return record(0);
        }
        return BLK_OK;
    }
    blk_status step(int kind) {
        // at most 12 (a block makes at most 9: OLMo-2's eight kernels and
        // the Q8_0 weight expansion)
        if (kinds && n < 12 && (n_events <= 0 || n + 1 < n_events)) kinds[n] = kind;
        ++n;
        if (events && n < n_events) return record(n);
        return BLK_OK;
    }
    blk_status end() {
        if (n_out) *n_out = n;
        return BLK_OK;
    }
};

// Launch the projection (+bias, +rotary when it can be fused) and, when a
// qk-norm or a wider rotary span sits between the projection and attention,
// the in-place qk-norm/rotary kernel.
// split: GEMM scratch (kGemmSplitBytes, counters zero) or nullptr
void set_split(GemmArgs& g, void* split) {
    if (!split) return;
    g.split_ws = static_cast<float*>(split);
    g.split_cnt = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(split) +
                                              static_cast<size_t>(kGemmSplitSlots) * 128 * 256 * 4);
}

// A projection weight in Q8_0 form (codes and scales; q2/d2: SwiGLU's up
// weight beside the gate weight in q/d).
struct Q8W {
    const int8_t* q;
    const void* d;
    const int8_t* q2;
    const void* d2;
};

blk_status run_qkv(const blk_qkv_desc* d, const void* x, const void* w_qkv, const void* b_qkv,
                   const void* q_norm_w, const void* k_norm_w, void* q, void* k, void* v,
                   DType dt, cudaStream_t s, DevState* ds, StepLog* log = nullptr,
                   void* split = nullptr, const Q8W* wq = nullptr) {
    // the GEMM epilogue rotates spans of 16 or 32 dims in registers; other
    // spans, and any qk-norm (which must precede the rotary), run in the
    // qk-norm/rotary kernel after the projection
    const bool fuse_rope = d->qk_norm == BLK_QKNORM_NONE &&
                           (d->rotary_span == 0 || d->rotary_span == 16 || d->rotary_span == 32);
    RopeParams rp = make_rope(fuse_rope ? d->rotary_span : 0, d->rope_base);
    GemmArgs g{};
    g.M = static_cast<int>(d->batch * d->seq);
    g.N = static_cast<int>((d->n_heads + 2 * d->n_kv_heads) * d->head_dim);
    g.K = static_cast<int>(d->hidden);
    g.bias = b_qkv;
    g.q = q;
    g.k = k;
    g.v = v;
    g.S = static_cast<int>(d->seq);
    g.H = static_cast<int>(d->n_heads);
    g.Hk = static_cast<int>(d->n_kv_heads);
    g.d = static_cast<int>(d->head_dim);
    g.interleaved = d->qkv_layout == BLK_QKV_HEAD_INTERLEAVED;
    g.err = ds->err;
    set_split(g, split);
    cudaError_t e = wq ? launch_gemm_q8(dt, EPI_QKV, x, wq->q, wq->d, nullptr, nullptr, g, rp,
                                        ds->sms, s)
                       : launch_gemm(dt, EPI_QKV, x, w_qkv, nullptr, g, rp, ds->sms, s);
    if (e != cudaSuccess) return cuda_fail(e, "qkv projection launch");
    blk_status st;
    if (log && (st = log->step(BLK_STEP_QKV)) != BLK_OK) return st;
    if (!fuse_rope) {
        QkNormRopeArgs a{};
        a.num_sms = ds->sms;
        a.q = q;
        a.k = k;
        a.q_w = q_norm_w;
        a.k_w = k_norm_w;
        a.B = g.M / g.S;
        a.S = g.S;
        a.H = g.H;
        a.Hk = g.Hk;
        a.d = g.d;
        a.mode = d->qk_norm;
        a.eps = d->qk_norm_eps;
        e = launch_qk_norm_rope(dt, a, make_rope(d->rotary_span, d->rope_base), s);
        if (e != cudaSuccess) return cuda_fail(e, "qk-norm/rotary launch");
        if (log && (st = log->step(BLK_STEP_QK_NORM_ROPE)) != BLK_OK) return st;
    }
    return BLK_OK;
}

enum : int { F32_OUT = 1, F32_RES1 = 2, F32_RES2 = 4 };

blk_status run_linear(DType dt, int epi, const void* x, const void* w, const void* w2,
                      const void* bias, const void* r1, const void* r2, void* y, int64_t m,
                      int64_t n, int64_t k, cudaStream_t s, DevState* ds, int f32 = 0,
                      void* split = nullptr, const Q8W* wq = nullptr) {
    // an fp32 output is written through the LINEAR epilogue only
    if ((f32 & F32_OUT) && epi != EPI_LINEAR) return BLK_EUNSUPPORTED;
    GemmArgs g{};
    set_split(g, split);
    g.out_f32 = (f32 & F32_OUT) != 0;
    g.res1_f32 = (f32 & F32_RES1) != 0;
    g.res2_f32 = (f32 & F32_RES2) != 0;
    g.M = static_cast<int>(m);
    g.N = static_cast<int>(n);
    g.K = static_cast<int>(k);
    g.out = y;
    g.bias = bias;
    g.res1 = r1;
    g.res2 = r2;
    g.err = ds->err;
    const RopeParams rp = make_rope(0, 0.f);
    cudaError_t e = wq ? launch_gemm_q8(dt, epi, x, wq->q, wq->d, wq->q2, wq->d2, g, rp, ds->sms, s)
                       : launch_gemm(dt, epi, x, w, w2, g, rp, ds->sms, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    return BLK_OK;
}

blk_status run_attn(const blk_attn_desc* d, const void* q, const void* k, const void* v,
                    const float* slopes, void* o, DType dt, cudaStream_t s, DevState* ds) {
    AttnArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.B = static_cast<int>(d->batch);
    a.S = static_cast<int>(d->seq);
    a.H = static_cast<int>(d->n_heads);
    a.Hk = static_cast<int>(d->n_kv_heads);
    a.d = static_cast<int>(d->head_dim);
    a.scale = d->softmax_scale > 0.f ? d->softmax_scale
                                     : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d->head_dim)));
    a.alibi = d->alibi;
    a.slopes = slopes;
    a.err = ds->err;
    a.num_sms = ds->sms;
    cudaError_t e = launch_attention(dt, a, s);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    return BLK_OK;
}


blk_status forward_impl(const blk_block_desc* d, const blk_block_weights* w,
                        const blk_q8_weights* q8, const void* x, void* y, void* workspace,
                        size_t ws_bytes, blk_dtype dt, blk_stream_t s, void* const* events,
                        int n_events, int32_t* step_kinds, int* n_launches);

}  // namespace

// ------------------------------------------------------------------ ABI --
extern "C" {

const char* blk_status_string(blk_status s) {
    switch (s) {
        case BLK_OK: return "BLK_OK";
        case BLK_EINVAL: return "BLK_EINVAL";
        case BLK_EUNSUPPORTED: return "BLK_EUNSUPPORTED";
        case BLK_ECUDA: return "BLK_ECUDA";
        case BLK_ETIMEOUT: return "BLK_ETIMEOUT";
        case BLK_EWORKSPACE: return "BLK_EWORKSPACE";
    }
    return "BLK_UNKNOWN";
}

const char* blk_last_error(void) { return t_last_error.c_str(); }

int blk_version(void) { return (1 << 16) | 0; }

blk_status blk_check_device_status(blk_stream_t s) {
    DevState* ds = nullptr;
    blk_status st = dev_state(&ds);
    if (st != BLK_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(s));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned word = 0;
    e = cudaMemcpy(&word, ds->err, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (word != DEV_ERR_NONE) {
        const unsigned zero = 0;
        cudaMemcpy(ds->err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        return fail(BLK_ETIMEOUT, "a bounded in-kernel wait gave up (device error code %u)", word);
    }
    return BLK_OK;
}

blk_status blk_selftest_bounded_wait(uint64_t limit_ns, blk_stream_t s) {
    BLK_REQUIRE(limit_ns >= 1000 && limit_ns <= 5000000000ull, "limit_ns must be in [1 us, 5 s]");
    DevState* ds = nullptr;
    blk_status st = dev_state(&ds);
    if (st != BLK_OK) return st;
    bounded_wait_selftest_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(s)>>>(ds->err, limit_ns);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? BLK_OK : cuda_fail(e, "self-test launch");
}

blk_status blk_layernorm_bias(const void* x, const void* residual, const void* gamma,
                              const void* beta, void* y, int64_t rows, int64_t cols, float eps,
                              blk_dtype dt, blk_stream_t s) {
    blk_status st = validate_norm(x, residual, gamma, beta, y, rows, cols, eps, dt);
    if (st != BLK_OK) return st;
    DevState* ds = nullptr;
    if ((st = dev_state(&ds)) != BLK_OK) return st;
    const NormIO io{x, false, residual, false, y, nullptr, ds->err, ds->sms};
    cudaError_t e = launch_norm(to_dt(dt), false, io, gamma, beta, rows, static_cast<int>(cols),
                                eps, reinterpret_cast<cudaStream_t>(s));
    return e == cudaSuccess ? BLK_OK : cuda_fail(e, "layernorm launch");
}

blk_status blk_rmsnorm(const void* x, const void* residual, const void* weight, void* y,
                       int64_t rows, int64_t cols, float eps, blk_dtype dt, blk_stream_t s) {
    blk_status st = validate_norm(x, residual, weight, nullptr, y, rows, cols, eps, dt);
    if (st != BLK_OK) return st;
    DevState* ds = nullptr;
    if ((st = dev_state(&ds)) != BLK_OK) return st;
    const NormIO io{x, false, residual, false, y, nullptr, ds->err, ds->sms};
    cudaError_t e = launch_norm(to_dt(dt), true, io, weight, nullptr, rows, static_cast<int>(cols),
                                eps, reinterpret_cast<cudaStream_t>(s));
    return e == cudaSuccess ? BLK_OK : cuda_fail(e, "rmsnorm launch");
}

blk_status blk_qkv_bias_rope_partial(const blk_qkv_desc* d, const void* x, const void* w_qkv,
                                     const void* b_qkv, const void* q_norm_w,
                                     const void* k_norm_w, void* q, void* k, void* v,
                                     blk_dtype dt, blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    blk_status st = validate_qkv_desc(d);
    if (st != BLK_OK) return st;
    const bool qkn = d->qk_norm != BLK_QKNORM_NONE;
    BLK_CHECK_PTR(x, true);
    BLK_CHECK_PTR(w_qkv, true);
    BLK_CHECK_PTR(b_qkv, false);
    BLK_CHECK_PTR(q_norm_w, qkn);
    BLK_CHECK_PTR(k_norm_w, qkn);
    BLK_REQUIRE(qkn || (!q_norm_w && !k_norm_w), "q_norm_w/k_norm_w must be NULL without qk_norm");
    BLK_CHECK_PTR(q, true);
    BLK_CHECK_PTR(k, true);
    BLK_CHECK_PTR(v, true);
    DevState* ds = nullptr;
    if ((st = dev_state(&ds)) != BLK_OK) return st;
    return run_qkv(d, x, w_qkv, b_qkv, q_norm_w, k_norm_w, q, k, v, to_dt(dt),
                   reinterpret_cast<cudaStream_t>(s), ds);
}

blk_status blk_rope_inplace(void* x, const void* bias, int64_t batch, int64_t n_heads,
                            int64_t seq, int64_t head_dim, int32_t rotary_span, float rope_base,
                            blk_dtype dt, blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    BLK_CHECK_PTR(x, true);
    BLK_CHECK_PTR(bias, false);
    BLK_REQUIRE(batch >= 1 && seq >= 1 && batch * seq <= kI32, "batch*seq out of range");
    BLK_REQUIRE(n_heads >= 1 && head_dim >= 8 && head_dim % 8 == 0 && head_dim <= 256,
                "head_dim must be a multiple of 8 in [8, 256]");
    BLK_REQUIRE(n_heads * head_dim * 4 <= 200 * 1024, "n_heads * head_dim too large");
    BLK_REQUIRE(rotary_span >= 0 && rotary_span % 2 == 0 && rotary_span <= head_dim &&
                    rotary_span / 2 <= kMaxRotaryPairs,
                "rotary_span must be even and in [0, head_dim]");
    BLK_REQUIRE(rotary_span == 0 || (std::isfinite(rope_base) && rope_base > 1.f),
                "rope_base must be > 1 when rotary is on");
    DevState* ds = nullptr;
    blk_status st = dev_state(&ds);
    if (st != BLK_OK) return st;
    QkNormRopeArgs a{};
    a.num_sms = ds->sms;
    a.q = x;
    a.q_bias = bias;
    a.B = static_cast<int>(batch);
    a.S = static_cast<int>(seq);
    a.H = static_cast<int>(n_heads);
    a.Hk = 0;
    a.d = static_cast<int>(head_dim);
    a.mode = QKN_NONE;
    cudaError_t e = launch_qk_norm_rope(to_dt(dt), a, make_rope(rotary_span, rope_base),
                                        reinterpret_cast<cudaStream_t>(s));
    return e == cudaSuccess ? BLK_OK : cuda_fail(e, "rope launch");
}

static blk_status validate_decode_desc(const blk_decode_desc* d) {
    BLK_REQUIRE(d != nullptr, "desc is NULL");
    BLK_REQUIRE(d->batch >= 1 && d->batch <= kI32, "batch out of range");
    BLK_REQUIRE(d->max_seq >= 1 && d->max_seq <= kI32, "max_seq out of range");
    BLK_REQUIRE(d->n_heads >= 1 && d->n_kv_heads >= 1 && d->n_heads % d->n_kv_heads == 0,
                "n_heads must be a positive multiple of n_kv_heads");
    const int64_t g = d->n_heads / d->n_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8)
        return fail(BLK_EUNSUPPORTED, "n_heads / n_kv_heads must be 1, 2, 4 or 8");
    if (d->head_dim != 64 && d->head_dim != 128)
        return fail(BLK_EUNSUPPORTED, "head_dim must be 64 or 128");
    BLK_REQUIRE(d->batch * d->n_heads <= kI32 &&
                    d->batch * d->n_kv_heads * d->max_seq * d->head_dim <= (int64_t(1) << 40),
                "sizes out of range");
    BLK_REQUIRE(d->alibi == 0 || d->alibi == 1, "alibi must be 0 or 1");
    BLK_REQUIRE(std::isfinite(d->softmax_scale), "softmax_scale must be finite");
    return BLK_OK;
}

static size_t decode_ws_bytes(const blk_decode_desc* d) {
    return static_cast<size_t>(d->batch) * d->n_heads * decode_parts_max(d->max_seq) *
           (d->head_dim + 2) * sizeof(float);
}

blk_status blk_attn_decode_workspace_size(const blk_decode_desc* d, size_t* bytes) {
    blk_status st = validate_decode_desc(d);
    if (st != BLK_OK) return st;
    BLK_REQUIRE(bytes != nullptr, "bytes is NULL");
    *bytes = decode_ws_bytes(d);
    return BLK_OK;
}

blk_status blk_attn_decode(const blk_decode_desc* d, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* lens, const float* alibi_slopes,
                           void* o, void* workspace, size_t ws_bytes, blk_dtype dt,
                           blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    blk_status st = validate_decode_desc(d);
    if (st != BLK_OK) return st;
    BLK_CHECK_PTR(q, true);
    BLK_CHECK_PTR(k_cache, true);
    BLK_CHECK_PTR(v_cache, true);
    BLK_CHECK_PTR(o, true);
    BLK_REQUIRE(lens != nullptr && (reinterpret_cast<uintptr_t>(lens) & 3u) == 0,
                "lens must be a 4-byte aligned device pointer");
    BLK_REQUIRE(d->alibi || !alibi_slopes, "alibi_slopes given with alibi = 0");
    if (d->alibi && !alibi_slopes && !is_pow2(d->n_heads))
        return fail(BLK_EUNSUPPORTED, "standard ALiBi slopes need a power-of-two head count");
    BLK_REQUIRE(!alibi_slopes || (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u) == 0,
                "alibi_slopes must be 4-byte aligned");
    const size_t need = decode_ws_bytes(d);
    if (!workspace || ws_bytes < need || !aligned16(workspace))
        return fail(BLK_EWORKSPACE, "workspace needs %zu bytes, 16-byte aligned", need);
    DevState* ds = nullptr;
    if ((st = dev_state(&ds)) != BLK_OK) return st;
    DecodeArgs a{};
    a.q = q;
    a.k = k_cache;
    a.v = v_cache;
    a.o = o;
    a.lens = lens;
    a.slopes = alibi_slopes;
    a.ws = static_cast<float*>(workspace);
    a.B = static_cast<int>(d->batch);
    a.H = static_cast<int>(d->n_heads);
    a.Hk = static_cast<int>(d->n_kv_heads);
    a.d = static_cast<int>(d->head_dim);
    a.S_max = static_cast<int>(d->max_seq);
    a.parts = decode_parts(d->batch, d->n_kv_heads, d->max_seq, d->head_dim, ds->sms);
    a.scale = d->softmax_scale > 0.f ? d->softmax_scale
                                     : 1.0f / std::sqrt(static_cast<float>(d->head_dim));
    a.alibi = d->alibi;
    const cudaError_t e = launch_attention_decode(to_dt(dt), a, reinterpret_cast<cudaStream_t>(s));
    return e == cudaSuccess ? BLK_OK : cuda_fail(e, "decode attention launch");
}

blk_status blk_attn_prefill(const blk_attn_desc* d, const void* q, const void* k, const void* v,
                            const float* alibi_slopes, void* o, blk_dtype dt, blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    blk_status st = validate_attn_desc(d);
    if (st != BLK_OK) return st;
    BLK_CHECK_PTR(q, true);
    BLK_CHECK_PTR(k, true);
    BLK_CHECK_PTR(v, true);
    BLK_CHECK_PTR(o, true);
    BLK_REQUIRE(d->alibi || !alibi_slopes, "alibi_slopes given with alibi = 0");
    if (d->alibi && !alibi_slopes && !is_pow2(d->n_heads))
        return fail(BLK_EUNSUPPORTED, "standard ALiBi slopes need a power-of-two head count");
    BLK_REQUIRE(!alibi_slopes || (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u) == 0,
                "alibi_slopes must be 4-byte aligned");
    DevState* ds = nullptr;
    if ((st = dev_state(&ds)) != BLK_OK) return st;
    return run_attn(d, q, k, v, alibi_slopes, o, to_dt(dt), reinterpret_cast<cudaStream_t>(s), ds);
}

blk_status blk_linear(const void* x, const void* w, const void* bias, const void* res1,
                      const void* res2, void* y, int64_t m, int64_t n, int64_t k, blk_dtype dt,
                      blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    BLK_REQUIRE(m >= 0 && m <= kI32, "m out of range");
    BLK_REQUIRE(n >= 8 && n % 8 == 0 && n <= kI32, "n must be a positive multiple of 8");
    BLK_REQUIRE(k >= 8 && k % 8 == 0 && k <= kI32, "k must be a positive multiple of 8");
    BLK_CHECK_PTR(x, true);
    BLK_CHECK_PTR(w, true);
    BLK_CHECK_PTR(bias, false);
    BLK_CHECK_PTR(res1, false);
    BLK_CHECK_PTR(res2, false);
    BLK_CHECK_PTR(y, true);
    if (m == 0) return BLK_OK;
    DevState* ds = nullptr;
    blk_status st = dev_state(&ds);
    if (st != BLK_OK) return st;
    return run_linear(to_dt(dt), EPI_LINEAR, x, w, nullptr, bias, res1, res2, y, m, n, k,
                      reinterpret_cast<cudaStream_t>(s), ds);
}

blk_status blk_q8_0_quantize(const void* w, int64_t n, int64_t k, int8_t* q, void* d,
                             blk_dtype dt, blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    BLK_REQUIRE(n >= 0 && n <= kI32, "n out of range");
    BLK_REQUIRE(k >= 32 && k % 32 == 0 && k <= kI32, "k must be a positive multiple of 32");
    BLK_REQUIRE(n * (k / 32) <= kI32 * 256LL, "too many blocks");
    BLK_CHECK_PTR(w, true);
    BLK_CHECK_PTR(q, true);
    BLK_CHECK_PTR(d, true);
    if (n == 0) return BLK_OK;
    DevState* ds = nullptr;
    blk_status st = dev_state(&ds);
    if (st != BLK_OK) return st;
    const cudaError_t e = launch_q8_quantize(to_dt(dt), w, n, k, q, d, reinterpret_cast<cudaStream_t>(s));
    return e == cudaSuccess ? BLK_OK : cuda_fail(e, "q8_0 quantize launch");
}

blk_status blk_linear_q8_0(const void* x, const int8_t* q, const void* d, const void* bias,
                           const void* res1, const void* res2, void* y, int64_t m, int64_t n,
                           int64_t k, blk_dtype dt, blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    BLK_REQUIRE(m >= 0 && m <= kI32, "m out of range");
    BLK_REQUIRE(n >= 8 && n % 8 == 0 && n <= kI32, "n must be a positive multiple of 8");
    BLK_REQUIRE(k >= 32 && k % 32 == 0 && k <= kI32, "k must be a positive multiple of 32");
    BLK_CHECK_PTR(x, true);
    BLK_CHECK_PTR(q, true);
    BLK_CHECK_PTR(d, true);
    BLK_CHECK_PTR(bias, false);
    BLK_CHECK_PTR(res1, false);
    BLK_CHECK_PTR(res2, false);
    BLK_CHECK_PTR(y, true);
    if (m == 0) return BLK_OK;
    DevState* ds = nullptr;
    blk_status st = dev_state(&ds);
    if (st != BLK_OK) return st;
    const Q8W wq{q, d, nullptr, nullptr};
    return run_linear(to_dt(dt), EPI_LINEAR, x, nullptr, nullptr, bias, res1, res2, y, m, n, k,
                      reinterpret_cast<cudaStream_t>(s), ds, 0, nullptr, &wq);
}

blk_status blk_mlp_workspace_size(const blk_mlp_desc* d, size_t* bytes) {
    BLK_REQUIRE(d && bytes, "NULL argument");
    BLK_REQUIRE(d->tokens >= 0 && d->intermediate >= 8, "bad sizes");
    *bytes = align256(static_cast<size_t>(d->tokens) * d->intermediate * 2);
    return BLK_OK;
}

blk_status blk_mlp(const blk_mlp_desc* d, const void* x, const void* w_gate, const void* w_up,
                   const void* b_up, const void* w_down, const void* b_down, const void* res1,
                   const void* res2, void* y, void* workspace, size_t ws_bytes, blk_dtype dt,
                   blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    BLK_REQUIRE(d, "descriptor is NULL");
    BLK_REQUIRE(d->act == BLK_ACT_SWIGLU || d->act == BLK_ACT_GELU_TANH, "unknown act");
    BLK_REQUIRE(d->tokens >= 0 && d->tokens <= kI32, "tokens out of range");
    BLK_REQUIRE(d->hidden >= 8 && d->hidden % 8 == 0 && d->hidden <= kI32, "hidden must be a positive multiple of 8");
    BLK_REQUIRE(d->intermediate >= 8 && d->intermediate % 8 == 0 && d->intermediate <= kI32,
                "intermediate must be a positive multiple of 8");
    const bool swiglu = d->act == BLK_ACT_SWIGLU;
    BLK_CHECK_PTR(x, true);
    BLK_CHECK_PTR(w_gate, swiglu);
    BLK_REQUIRE(swiglu || !w_gate, "w_gate must be NULL for GELU_TANH");
    BLK_CHECK_PTR(w_up, true);
    BLK_CHECK_PTR(b_up, false);
    BLK_REQUIRE(!swiglu || !b_up, "b_up is not supported with SWIGLU (must be NULL)");
    BLK_CHECK_PTR(w_down, true);
    BLK_CHECK_PTR(b_down, false);
    BLK_CHECK_PTR(res1, false);
    BLK_CHECK_PTR(res2, false);
    BLK_CHECK_PTR(y, true);
    size_t need = 0;
    blk_mlp_workspace_size(d, &need);
    if (!workspace || ws_bytes < need || !aligned16(workspace))
        return fail(BLK_EWORKSPACE, "workspace needs %zu bytes, 16-byte aligned", need);
    if (d->tokens == 0) return BLK_OK;
    DevState* ds = nullptr;
    blk_status st = dev_state(&ds);
    if (st != BLK_OK) return st;
    const DType t = to_dt(dt);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    st = run_linear(t, swiglu ? EPI_SWIGLU : EPI_GELU, x, swiglu ? w_gate : w_up,
                    swiglu ? w_up : nullptr, b_up, nullptr, nullptr, workspace, d->tokens,
                    d->intermediate, d->hidden, cs, ds);
    if (st != BLK_OK) return st;
    return run_linear(t, EPI_LINEAR, workspace, w_down, nullptr, b_down, res1, res2, y, d->tokens,
                      d->hidden, d->intermediate, cs, ds);
}

blk_status blk_forward_workspace_size(const blk_block_desc* d, size_t* bytes) {
    BLK_REQUIRE(d && bytes, "NULL argument");
    blk_status st = validate_qkv_desc(&d->qkv);
    if (st != BLK_OK) return st;
    BLK_REQUIRE(d->intermediate >= 8 && d->intermediate % 8 == 0, "bad intermediate");
    *bytes = forward_layout(d).total;
    return BLK_OK;
}

blk_status blk_forward_q8_0_workspace_size(const blk_block_desc* d, size_t* bytes) {
    blk_status st = blk_forward_workspace_size(d, bytes);
    if (st != BLK_OK) return st;
    *bytes += q8_scratch_bytes(d);
    return BLK_OK;
}

blk_status blk_forward(const blk_block_desc* d, const blk_block_weights* w, const void* x,
                       void* y, void* workspace, size_t ws_bytes, blk_dtype dt, blk_stream_t s) {
    return blk_forward_ex(d, w, x, y, workspace, ws_bytes, dt, s, nullptr, 0, nullptr, nullptr);
}

blk_status blk_forward_ex(const blk_block_desc* d, const blk_block_weights* w, const void* x,
                          void* y, void* workspace, size_t ws_bytes, blk_dtype dt, blk_stream_t s,
                          void* const* events, int n_events, int32_t* step_kinds, int* n_launches) {
    return forward_impl(d, w, nullptr, x, y, workspace, ws_bytes, dt, s, events, n_events,
                        step_kinds, n_launches);
}

blk_status blk_forward_q8_0(const blk_block_desc* d, const blk_block_weights* w,
                            const blk_q8_weights* q8, const void* x, void* y, void* workspace,
                            size_t ws_bytes, blk_dtype dt, blk_stream_t s) {
    return blk_forward_q8_0_ex(d, w, q8, x, y, workspace, ws_bytes, dt, s, nullptr, 0, nullptr,
                               nullptr);
}

blk_status blk_forward_q8_0_ex(const blk_block_desc* d, const blk_block_weights* w,
                               const blk_q8_weights* q8, const void* x, void* y, void* workspace,
                               size_t ws_bytes, blk_dtype dt, blk_stream_t s,
                               void* const* events, int n_events, int32_t* step_kinds,
                               int* n_launches) {
    BLK_REQUIRE(q8, "Q8_0 weights are NULL");
    return forward_impl(d, w, q8, x, y, workspace, ws_bytes, dt, s, events, n_events, step_kinds,
                        n_launches);
}

}  // extern "C"

namespace {

// The block's composition for dense (q8 == NULL) or Q8_0 projection weights.
blk_status forward_impl(const blk_block_desc* d, const blk_block_weights* w,
                        const blk_q8_weights* q8, const void* x, void* y, void* workspace,
                        size_t ws_bytes, blk_dtype dt, blk_stream_t s, void* const* events,
                        int n_events, int32_t* step_kinds, int* n_launches) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    blk_status st = validate_block(d, w, q8);
    if (st != BLK_OK) return st;
    BLK_CHECK_PTR(x, true);
    BLK_CHECK_PTR(y, true);
    BLK_REQUIRE(x != y, "y must not alias x");
    const FwdLayout L = forward_layout(d);
    if (!workspace || ws_bytes < L.total || !aligned16(workspace))
        return fail(BLK_EWORKSPACE, "workspace needs %zu bytes, 16-byte aligned", L.total);
    BLK_REQUIRE(n_events >= 0 && (events || n_events == 0), "events/n_events mismatch");
    DevState* ds = nullptr;
    if ((st = dev_state(&ds)) != BLK_OK) return st;

    const auto& q = d->qkv;
    const DType t = to_dt(dt);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* n1 = ws + L.n1;
    void* qb = ws + L.q;
    void* kb = ws + L.k;
    void* vb = ws + L.v;
    void* ob = ws + L.o;
    void* hb = ws + L.h;
    void* n2 = ws + L.n2;
    void* ab = ws + L.a;
    void* tmp = ws + L.tmp;
    void* h16 = ws + L.h16;
    void* split = ws + L.split;
    const int64_t T = q.batch * q.seq, D = q.hidden, F = d->intermediate;
    const bool rms = d->norm_kind == BLK_NORM_RMS;
    const bool pre = d->norm_place == BLK_NORM_PRE;
    const bool parallel = d->residual == BLK_RESIDUAL_PARALLEL;
    const bool swiglu = d->act == BLK_ACT_SWIGLU;
    // Q8_0 projection weights (NULL handles: the dense slots of w)
    Q8W wq_qkv{}, wq_o{}, wq_up{}, wq_down{};
    if (q8) {
        wq_qkv = Q8W{q8->q_qkv, q8->d_qkv, nullptr, nullptr};
        wq_o = Q8W{q8->q_o, q8->d_o, nullptr, nullptr};
        wq_up = swiglu ? Q8W{q8->q_gate, q8->d_gate, q8->q_up, q8->d_up}
                       : Q8W{q8->q_up, q8->d_up, nullptr, nullptr};
        wq_down = Q8W{q8->q_down, q8->d_down, nullptr, nullptr};
    }
    const Q8W* pq_qkv = q8 ? &wq_qkv : nullptr;
    const Q8W* pq_o = q8 ? &wq_o : nullptr;
    const Q8W* pq_up = q8 ? &wq_up : nullptr;
    const Q8W* pq_down = q8 ? &wq_down : nullptr;
    // the dense GEMMs' weights: w's, or Q8_0 weights expanded into the
    // scratch after the workspace (dequantize-once path: a workspace of
    // blk_forward_q8_0_workspace_size bytes and at least 512 tokens)
    const void* W_qkv = w->w_qkv;
    const void* W_o = w->w_o;
    const void* W_gate = w->w_gate;
    const void* W_up = w->w_up;
    const void* W_down = w->w_down;
    void* q8_scratch = q8 && T >= kQ8DequantMinTokens && ws_bytes >= L.total + q8_scratch_bytes(d)
                           ? ws + L.total
                           : nullptr;
    cudaError_t e;
    StepLog log{events, n_events, step_kinds, n_launches, cs};
    if ((st = log.begin()) != BLK_OK) return st;
    // the split GEMM rounds' arrival counters start at zero (each launch
    // leaves them zero again)
    e = cudaMemsetAsync(static_cast<uint8_t*>(split) +
                            static_cast<size_t>(kGemmSplitSlots) * 128 * 256 * 4,
                        0, kGemmSplitCounters * sizeof(unsigned), cs);
    if (e != cudaSuccess) return cuda_fail(e, "split counters");
#define BLK_STEP(kind)                                   \
    do {                                                 \
        if ((st = log.step(kind)) != BLK_OK) return st;  \
    } while (0)
    // dequantize-once path: every projection's codes expanded, in one launch,
    // into the scratch; the GEMMs then run dense on them
    if (q8_scratch) {
        int64_t rc[kQ8DequantMaxJobs][2];
        int n_jobs = 0;
        q8_shapes(d, rc, &n_jobs);
        const Q8W* src[kQ8DequantMaxJobs];
        const void** dst[kQ8DequantMaxJobs];
        int k = 0;
        src[k] = pq_qkv, dst[k++] = &W_qkv;
        src[k] = pq_o, dst[k++] = &W_o;
        if (swiglu) src[k] = pq_up, dst[k++] = &W_gate;  // q8_shapes order: gate, then up
        src[k] = pq_up, dst[k++] = &W_up;
        src[k] = pq_down, dst[k++] = &W_down;
        Q8DequantJob jobs[kQ8DequantMaxJobs];
        uint8_t* at = static_cast<uint8_t*>(q8_scratch);
        for (int i = 0; i < n_jobs; ++i) {
            // SwiGLU's up weights are the second pair of wq_up
            const bool second = swiglu && dst[i] == &W_up;
            jobs[i] = Q8DequantJob{second ? src[i]->q2 : src[i]->q, second ? src[i]->d2 : src[i]->d,
                                   at, rc[i][0], rc[i][1]};
            *dst[i] = at;
            at += align256(static_cast<size_t>(2 * rc[i][0] * rc[i][1]));
        }
        e = launch_q8_dequant(t, jobs, n_jobs, cs);
        if (e != cudaSuccess) return cuda_fail(e, "q8_0 dequantize launch");
        BLK_STEP(BLK_STEP_Q8_DEQUANT);
        pq_qkv = pq_o = pq_up = pq_down = nullptr;
    }

    // 1. input norm (absent in the reordered post-norm block)
    const void* attn_in = x;
    if (pre) {
        e = launch_norm(t, rms, NormIO{x, false, nullptr, false, n1, nullptr, ds->err, ds->sms}, w->attn_norm_w,
                        w->attn_norm_b, T, static_cast<int>(D), d->eps, cs);
        if (e != cudaSuccess) return cuda_fail(e, "input norm launch");
        BLK_STEP(BLK_STEP_INPUT_NORM);
        attn_in = n1;
    }
    // 2. projection (+bias), qk-norm, rotary, head split
    st = run_qkv(&q, attn_in, W_qkv, w->b_qkv, w->q_norm_w, w->k_norm_w, qb, kb, vb, t, cs, ds,
                 &log, split, pq_qkv);
    if (st != BLK_OK) return st;
    // 3. causal attention (+ALiBi)
    blk_attn_desc ad{q.batch, q.seq, q.n_heads, q.n_kv_heads, q.head_dim, 0.f, 1, d->alibi};
    st = run_attn(&ad, qb, kb, vb, w->alibi_slopes, ob, t, cs, ds);
    if (st != BLK_OK) return st;
    BLK_STEP(BLK_STEP_ATTENTION);
    const int64_t Hd = q.n_heads * q.head_dim;
    if (parallel) {
        // 4p. attn_out = o W_o^T (+b_o) kept in fp32; mlp on the same normed
        // input; y = x + attn_out + mlp
        st = run_linear(t, EPI_LINEAR, ob, W_o, nullptr, w->b_o, nullptr, nullptr, tmp, T, D, Hd,
                        cs, ds, F32_OUT, split, pq_o);
        if (st != BLK_OK) return st;
        BLK_STEP(BLK_STEP_O_PROJ);
        st = run_linear(t, swiglu ? EPI_SWIGLU : EPI_GELU, attn_in, swiglu ? W_gate : W_up,
                        swiglu ? W_up : nullptr, w->b_up, nullptr, nullptr, ab, T, F, D, cs, ds, 0,
                        split, pq_up);
        if (st != BLK_OK) return st;
        BLK_STEP(BLK_STEP_MLP_UP);
        st = run_linear(t, EPI_LINEAR, ab, W_down, nullptr, w->b_down, x, tmp, y, T, D, F, cs,
                        ds, F32_RES2, split, pq_down);
        if (st != BLK_OK) return st;
        BLK_STEP(BLK_STEP_MLP_DOWN);
        return log.end();
    }
    const void* mlp_in;
    if (pre) {
        // 4. h = x + o W_o^T (+b_o), fp32;  5. n2 = norm(h)
        st = run_linear(t, EPI_LINEAR, ob, W_o, nullptr, w->b_o, x, nullptr, hb, T, D, Hd, cs, ds,
                        F32_OUT, split, pq_o);
        if (st != BLK_OK) return st;
        BLK_STEP(BLK_STEP_O_PROJ);
        e = launch_norm(t, rms, NormIO{hb, true, nullptr, false, n2, nullptr, ds->err, ds->sms}, w->mlp_norm_w,
                        w->mlp_norm_b, T, static_cast<int>(D), d->eps, cs);
        if (e != cudaSuccess) return cuda_fail(e, "mlp norm launch");
        BLK_STEP(BLK_STEP_MLP_NORM);
        mlp_in = n2;
    } else {
        // 4. a = o W_o^T (fp32: the RMS norm rescales it to unit size, so its
        // rounding would be magnified);  5. h = x + RMS(a) * w_post_attn
        // (fp32, and a storage copy for the MLP)
        st = run_linear(t, EPI_LINEAR, ob, W_o, nullptr, w->b_o, nullptr, nullptr, tmp, T, D, Hd,
                        cs, ds, F32_OUT, split, pq_o);
        if (st != BLK_OK) return st;
        BLK_STEP(BLK_STEP_O_PROJ);
        e = launch_norm(t, true, NormIO{tmp, true, x, false, h16, static_cast<float*>(hb), ds->err, ds->sms},
                        w->post_attn_norm_w, nullptr, T, static_cast<int>(D), d->eps, cs);
        if (e != cudaSuccess) return cuda_fail(e, "post-attention norm launch");
        BLK_STEP(BLK_STEP_POST_ATTN_NORM);
        mlp_in = h16;
    }
    // 6. MLP up (+activation)
    st = run_linear(t, swiglu ? EPI_SWIGLU : EPI_GELU, mlp_in, swiglu ? W_gate : W_up,
                    swiglu ? W_up : nullptr, w->b_up, nullptr, nullptr, ab, T, F, D, cs, ds, 0,
                    split, pq_up);
    if (st != BLK_OK) return st;
    BLK_STEP(BLK_STEP_MLP_UP);
    if (pre) {
        // 7. y = h + a W_d^T (+b_d)
        st = run_linear(t, EPI_LINEAR, ab, W_down, nullptr, w->b_down, hb, nullptr, y, T, D, F, cs,
                        ds, F32_RES1, split, pq_down);
        if (st != BLK_OK) return st;
        BLK_STEP(BLK_STEP_MLP_DOWN);
        return log.end();
    }
    // 7. m = a W_d^T;  8. y = h + RMS(m) * w_post_mlp
    st = run_linear(t, EPI_LINEAR, ab, W_down, nullptr, w->b_down, nullptr, nullptr, tmp, T, D, F,
                    cs, ds, F32_OUT, split, pq_down);
    if (st != BLK_OK) return st;
    BLK_STEP(BLK_STEP_MLP_DOWN);
    e = launch_norm(t, true, NormIO{tmp, true, hb, true, y, nullptr, ds->err, ds->sms}, w->post_mlp_norm_w, nullptr,
                    T, static_cast<int>(D), d->eps, cs);
    if (e != cudaSuccess) return cuda_fail(e, "post-mlp norm launch");
    BLK_STEP(BLK_STEP_POST_MLP_NORM);
    return log.end();
#undef BLK_STEP
}

}  // namespace

extern "C" {

blk_status blk_forward_host(const blk_block_desc* d, const blk_block_weights* w,
                            const void* x_host, void* y_host, void* x_dev, void* y_dev,
                            void* workspace, size_t ws_bytes, int32_t n_chunks, blk_dtype dt,
                            blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    blk_status st = validate_block(d, w);
    if (st != BLK_OK) return st;
    BLK_REQUIRE(x_host && y_host, "x_host / y_host is NULL");
    BLK_CHECK_PTR(x_dev, true);
    BLK_CHECK_PTR(y_dev, true);
    BLK_REQUIRE(x_dev != y_dev, "y_dev must not alias x_dev");
    BLK_REQUIRE(n_chunks >= 1 && n_chunks <= kMaxHostChunks, "n_chunks must be in [1, 16]");
    const int64_t B = d->qkv.batch;
    const int chunks = static_cast<int>(n_chunks < B ? n_chunks : B);
    const FwdLayout L = forward_layout(d);
    if (!workspace || ws_bytes < L.total || !aligned16(workspace))
        return fail(BLK_EWORKSPACE, "workspace needs %zu bytes, 16-byte aligned", L.total);
    DevState* ds = nullptr;
    if ((st = dev_state(&ds)) != BLK_OK) return st;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!ds->pipe_init) {
            cudaError_t e = cudaStreamCreateWithFlags(&ds->copy_in, cudaStreamNonBlocking);
            if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ds->copy_out, cudaStreamNonBlocking);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ds->ev_start, cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ds->ev_done, cudaEventDisableTiming);
            for (int i = 0; i < kMaxHostChunks && e == cudaSuccess; ++i) {
                e = cudaEventCreateWithFlags(&ds->ev_in[i], cudaEventDisableTiming);
                if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ds->ev_out[i], cudaEventDisableTiming);
            }
            if (e != cudaSuccess) return cuda_fail(e, "copy stream/event set-up");
            ds->pipe_init = true;
        }
    }
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    const size_t row_bytes = static_cast<size_t>(d->qkv.seq) * d->qkv.hidden * 2;  // one sequence
    // everything earlier on s (a previous call's reads of x_dev / y_dev) comes first
    cudaError_t e = cudaEventRecord(ds->ev_start, cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->copy_in, ds->ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->copy_out, ds->ev_start, 0);
    if (e != cudaSuccess) return cuda_fail(e, "stream ordering");
    int64_t b0[kMaxHostChunks + 1];
    for (int c = 0; c <= chunks; ++c) b0[c] = B * c / chunks;
    for (int c = 0; c < chunks; ++c) {
        const size_t off = static_cast<size_t>(b0[c]) * row_bytes;
        const size_t bytes = static_cast<size_t>(b0[c + 1] - b0[c]) * row_bytes;
        e = cudaMemcpyAsync(static_cast<uint8_t*>(x_dev) + off,
                            static_cast<const uint8_t*>(x_host) + off, bytes,
                            cudaMemcpyHostToDevice, ds->copy_in);
        if (e == cudaSuccess) e = cudaEventRecord(ds->ev_in[c], ds->copy_in);
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    }
    for (int c = 0; c < chunks; ++c) {
        const size_t off = static_cast<size_t>(b0[c]) * row_bytes;
        const size_t bytes = static_cast<size_t>(b0[c + 1] - b0[c]) * row_bytes;
        e = cudaStreamWaitEvent(cs, ds->ev_in[c], 0);
        if (e != cudaSuccess) return cuda_fail(e, "stream ordering");
        blk_block_desc dc = *d;
        dc.qkv.batch = b0[c + 1] - b0[c];
        st = blk_forward(&dc, w, static_cast<const uint8_t*>(x_dev) + off,
                         static_cast<uint8_t*>(y_dev) + off, workspace, ws_bytes, dt, s);
        if (st != BLK_OK) return st;
        e = cudaEventRecord(ds->ev_out[c], cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->copy_out, ds->ev_out[c], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<uint8_t*>(y_host) + off,
                                static_cast<const uint8_t*>(y_dev) + off, bytes,
                                cudaMemcpyDeviceToHost, ds->copy_out);
        if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
    }
    // the call completes on s when the last copy out has landed
    e = cudaEventRecord(ds->ev_done, ds->copy_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ds->ev_done, 0);
    return e == cudaSuccess ? BLK_OK : cuda_fail(e, "stream ordering");
}

namespace {

struct ModelLayout {
    size_t x0, x1, n, blk, total, blk_bytes;
};

ModelLayout model_layout(const blk_model_desc* d) {
    const auto& q = d->block.qkv;
    const size_t act = align256(static_cast<size_t>(q.batch) * q.seq * q.hidden * 2);
    ModelLayout L;
    L.x0 = 0;
    L.x1 = act;
    L.n = 2 * act;
    L.blk = 3 * act;
    L.blk_bytes = forward_layout(&d->block).total;
    L.total = L.blk + L.blk_bytes;
    return L;
}

blk_status validate_model_desc(const blk_model_desc* d) {
    BLK_REQUIRE(d != nullptr, "descriptor is NULL");
    blk_status st = validate_qkv_desc(&d->block.qkv);
    if (st != BLK_OK) return st;
    BLK_REQUIRE(d->block.intermediate >= 8 && d->block.intermediate % 8 == 0,
                "intermediate must be a positive multiple of 8");
    BLK_REQUIRE(d->n_layers >= 0 && d->n_layers <= 4096, "n_layers must be in [0, 4096]");
    BLK_REQUIRE(d->vocab >= 8 && d->vocab % 8 == 0 && d->vocab <= kI32,
                "vocab must be a positive multiple of 8");
    BLK_REQUIRE(d->embed_norm == 0 || d->embed_norm == 1, "embed_norm must be 0 or 1");
    BLK_REQUIRE(d->final_norm == BLK_NORM_LAYERNORM || d->final_norm == BLK_NORM_RMS,
                "unknown final_norm");
    BLK_REQUIRE(std::isfinite(d->final_eps) && d->final_eps >= 0.f, "final_eps must be >= 0");
    BLK_REQUIRE(d->block.qkv.hidden <= 16384, "hidden must be <= 16384");
    return BLK_OK;
}

}  // namespace

blk_status blk_model_workspace_size(const blk_model_desc* d, size_t* bytes) {
    BLK_REQUIRE(bytes != nullptr, "NULL argument");
    blk_status st = validate_model_desc(d);
    if (st != BLK_OK) return st;
    *bytes = model_layout(d).total;
    return BLK_OK;
}

blk_status blk_model_forward(const blk_model_desc* d, const blk_model_weights* w,
                             const int32_t* tokens, void* logits, void* workspace,
                             size_t ws_bytes, blk_dtype dt, blk_stream_t s) {
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    blk_status st = validate_model_desc(d);
    if (st != BLK_OK) return st;
    BLK_REQUIRE(w != nullptr, "weights is NULL");
    BLK_REQUIRE(tokens != nullptr, "tokens is NULL");
    BLK_CHECK_PTR(logits, true);
    BLK_CHECK_PTR(w->embed, true);
    BLK_CHECK_PTR(w->lm_head, true);
    BLK_CHECK_PTR(w->final_norm_w, true);
    BLK_CHECK_PTR(w->final_norm_b, false);
    BLK_REQUIRE(d->final_norm == BLK_NORM_LAYERNORM || !w->final_norm_b,
                "final_norm_b is only read by a LayerNorm final norm");
    if (d->embed_norm) {
        BLK_CHECK_PTR(w->embed_norm_w, true);
        BLK_CHECK_PTR(w->embed_norm_b, false);
    } else {
        BLK_REQUIRE(!w->embed_norm_w && !w->embed_norm_b,
                    "embed_norm weights given but embed_norm is 0");
    }
    BLK_REQUIRE(d->n_layers == 0 || w->layers != nullptr, "layers is NULL");
    for (int32_t l = 0; l < d->n_layers; ++l) {
        st = validate_block(&d->block, &w->layers[l]);
        if (st != BLK_OK) return st;
    }
    const ModelLayout L = model_layout(d);
    if (!workspace || ws_bytes < L.total || !aligned16(workspace))
        return fail(BLK_EWORKSPACE, "workspace needs %zu bytes, 16-byte aligned", L.total);
    DevState* ds = nullptr;
    if ((st = dev_state(&ds)) != BLK_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    const DType t = to_dt(dt);
    const auto& q = d->block.qkv;
    const int64_t T = q.batch * q.seq;
    const int D = static_cast<int>(q.hidden);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* xa = ws + L.x0;
    void* xb = ws + L.x1;
    void* nb = ws + L.n;
    // 1. embedding rows of the tokens
    cudaError_t e = launch_embed_gather(t, tokens, w->embed, xa, T, D, d->vocab, ds->sms, cs);
    if (e != cudaSuccess) return cuda_fail(e, "embedding gather launch");
    // 2. (Bloom) LayerNorm of the embeddings
    if (d->embed_norm) {
        e = launch_norm(t, false, NormIO{xa, false, nullptr, false, xb, nullptr, ds->err, ds->sms},
                        w->embed_norm_w, w->embed_norm_b, T, D, d->block.eps, cs);
        if (e != cudaSuccess) return cuda_fail(e, "embedding norm launch");
        void* tmp = xa;
        xa = xb;
        xb = tmp;
    }
    // 3. the blocks, ping-pong between the two activations
    for (int32_t l = 0; l < d->n_layers; ++l) {
        st = blk_forward(&d->block, &w->layers[l], xa, xb, ws + L.blk, L.blk_bytes, dt, s);
        if (st != BLK_OK) return st;
        void* tmp = xa;
        xa = xb;
        xb = tmp;
    }
    // 4. final norm and the vocabulary projection
    e = launch_norm(t, d->final_norm == BLK_NORM_RMS,
                    NormIO{xa, false, nullptr, false, nb, nullptr, ds->err, ds->sms},
                    w->final_norm_w, w->final_norm_b, T, D, d->final_eps, cs);
    if (e != cudaSuccess) return cuda_fail(e, "final norm launch");
    return run_linear(t, EPI_LINEAR, nb, w->lm_head, nullptr, nullptr, nullptr, nullptr, logits, T,
                      d->vocab, D, cs, ds);
}

constexpr int kMaxPipeDepth = 4;
struct blk_host_pipe {
    blk_block_desc d{};
    blk_dtype dt = BLK_BF16;
    int depth = 0;
    int device = -1;
    size_t io_bytes = 0;  // one batch of x (or y)
    uint8_t* x_dev[kMaxPipeDepth] = {};
    uint8_t* y_dev[kMaxPipeDepth] = {};
    void* ws = nullptr;
    size_t ws_bytes = 0;
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    // ev_fwd[k]: the forward that last read x slot k and wrote y slot k;
    // ev_out[k]: the copy-out that last read y slot k
    cudaEvent_t ev_base = nullptr, ev_flush = nullptr;
    cudaEvent_t ev_in[kMaxPipeDepth] = {}, ev_fwd[kMaxPipeDepth] = {}, ev_out[kMaxPipeDepth] = {};
    int64_t n = 0;            // submits since create or the last flush
    cudaStream_t s = nullptr;  // their stream
    // slot k's forward as a CUDA graph, and the weight pointers it reads
    blk_graph* g[kMaxPipeDepth] = {};
    blk_block_weights gw[kMaxPipeDepth] = {};
};

namespace {

size_t pipe_io_bytes(const blk_block_desc* d) {
    return align256(static_cast<size_t>(d->qkv.batch) * d->qkv.seq * d->qkv.hidden * 2);
}

blk_status pipe_release(blk_host_pipe* p) {
    cudaError_t first = cudaSuccess;
    auto keep = [&](cudaError_t e) {
        if (first == cudaSuccess && e != cudaSuccess) first = e;
    };
    for (int k = 0; k < kMaxPipeDepth; ++k) {
        if (p->g[k] && blk_graph_destroy(p->g[k]) != BLK_OK && first == cudaSuccess)
            first = cudaErrorUnknown;
        if (p->ev_in[k]) keep(cudaEventDestroy(p->ev_in[k]));
        if (p->ev_fwd[k]) keep(cudaEventDestroy(p->ev_fwd[k]));
        if (p->ev_out[k]) keep(cudaEventDestroy(p->ev_out[k]));
    }
    if (p->ev_base) keep(cudaEventDestroy(p->ev_base));
    if (p->ev_flush) keep(cudaEventDestroy(p->ev_flush));
    if (p->copy_in) keep(cudaStreamDestroy(p->copy_in));
    if (p->copy_out) keep(cudaStreamDestroy(p->copy_out));
    delete p;
    return first == cudaSuccess ? BLK_OK : cuda_fail(first, "host pipe release");
}

}  // namespace

blk_status blk_host_pipe_mem_size(const blk_block_desc* d, int32_t depth, size_t* bytes) {
    BLK_REQUIRE(d && bytes, "NULL argument");
    BLK_REQUIRE(depth >= 2 && depth <= kMaxPipeDepth, "depth must be in [2, 4]");
    size_t ws = 0;
    blk_status st = blk_forward_workspace_size(d, &ws);
    if (st != BLK_OK) return st;
    *bytes = 2 * static_cast<size_t>(depth) * pipe_io_bytes(d) + ws;
    return BLK_OK;
}

blk_status blk_host_pipe_create(const blk_block_desc* d, int32_t depth, blk_dtype dt,
                                void* dev_mem, size_t bytes, blk_host_pipe** out) {
    BLK_REQUIRE(out != nullptr, "out is NULL");
    *out = nullptr;
    BLK_REQUIRE(valid_dt(dt), "dtype must be BLK_F16 or BLK_BF16");
    size_t need = 0;
    blk_status st = blk_host_pipe_mem_size(d, depth, &need);
    if (st != BLK_OK) return st;
    BLK_CHECK_PTR(dev_mem, true);
    if (bytes < need) return fail(BLK_EWORKSPACE, "dev_mem needs %zu bytes", need);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    auto* p = new (std::nothrow) blk_host_pipe;
    if (!p) return fail(BLK_ECUDA, "out of host memory");
    p->d = *d;
    p->dt = dt;
    p->depth = depth;
    p->device = dev;
    p->io_bytes = pipe_io_bytes(d);
    uint8_t* m = static_cast<uint8_t*>(dev_mem);
    for (int k = 0; k < depth; ++k) {
        p->x_dev[k] = m + (2 * k) * p->io_bytes;
        p->y_dev[k] = m + (2 * k + 1) * p->io_bytes;
    }
    p->ws = m + 2 * static_cast<size_t>(depth) * p->io_bytes;
    p->ws_bytes = bytes - 2 * static_cast<size_t>(depth) * p->io_bytes;
    e = cudaStreamCreateWithFlags(&p->copy_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->copy_out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_base, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_flush, cudaEventDisableTiming);
    for (int k = 0; k < depth && e == cudaSuccess; ++k) {
        e = cudaEventCreateWithFlags(&p->ev_in[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_fwd[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_out[k], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        pipe_release(p);
        return cuda_fail(e, "host pipe streams/events");
    }
    *out = p;
    return BLK_OK;
}

blk_status blk_host_pipe_submit(blk_host_pipe* p, const blk_block_weights* w, const void* x_host,
                                void* y_host, blk_stream_t s) {
    BLK_REQUIRE(p != nullptr, "pipe is NULL");
    BLK_REQUIRE(x_host && y_host, "x_host / y_host is NULL");
    blk_status st = validate_block(&p->d, w);
    if (st != BLK_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    BLK_REQUIRE(dev == p->device, "the pipe belongs to device %d, current device is %d", p->device,
                dev);
    BLK_REQUIRE(p->n == 0 || cs == p->s,
                "submits between two flushes must use the same stream");
    const int k = static_cast<int>(p->n % p->depth);
    const size_t io = static_cast<size_t>(p->d.qkv.batch) * p->d.qkv.seq * p->d.qkv.hidden * 2;
    if (p->n == 0) {
        p->s = cs;
        e = cudaEventRecord(p->ev_base, cs);
        if (e != cudaSuccess) return cuda_fail(e, "stream ordering");
    }
    // copy in once the forward that last read slot k is done
    e = cudaStreamWaitEvent(p->copy_in, p->n < p->depth ? p->ev_base : p->ev_fwd[k], 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->x_dev[k], x_host, io, cudaMemcpyHostToDevice, p->copy_in);
    if (e == cudaSuccess) e = cudaEventRecord(p->ev_in[k], p->copy_in);
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    // the forward waits for its input and for the copy-out that last read y slot k
    e = cudaStreamWaitEvent(cs, p->ev_in[k], 0);
    if (e == cudaSuccess && p->n >= p->depth) e = cudaStreamWaitEvent(cs, p->ev_out[k], 0);
    if (e != cudaSuccess) return cuda_fail(e, "stream ordering");
    // the forward: slot k's graph, recorded on its first use and again when
    // the weight pointers differ from the recorded ones
    if (!p->g[k] || std::memcmp(&p->gw[k], w, sizeof(*w)) != 0) {
        if (p->g[k]) {
            st = blk_graph_destroy(p->g[k]);
            p->g[k] = nullptr;
            if (st != BLK_OK) return st;
        }
        st = blk_forward_graph_create(&p->d, w, p->x_dev[k], p->y_dev[k], p->ws, p->ws_bytes,
                                      p->dt, nullptr, 0, nullptr, nullptr, &p->g[k]);
        if (st != BLK_OK) return st;
        p->gw[k] = *w;
    }
    st = blk_graph_launch(p->g[k], s);
    if (st != BLK_OK) return st;
    e = cudaEventRecord(p->ev_fwd[k], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->copy_out, p->ev_fwd[k], 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(y_host, p->y_dev[k], io, cudaMemcpyDeviceToHost, p->copy_out);
    if (e == cudaSuccess) e = cudaEventRecord(p->ev_out[k], p->copy_out);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
    ++p->n;
    return BLK_OK;
}

blk_status blk_host_pipe_flush(blk_host_pipe* p, blk_stream_t s) {
    BLK_REQUIRE(p != nullptr, "pipe is NULL");
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    if (p->n == 0) return BLK_OK;
    BLK_REQUIRE(cs == p->s, "flush on the stream of the submits");
    // copy-outs run in submit order on one stream: its tail is the last one
    cudaError_t e = cudaEventRecord(p->ev_flush, p->copy_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, p->ev_flush, 0);
    if (e != cudaSuccess) return cuda_fail(e, "stream ordering");
    p->n = 0;
    return BLK_OK;
}

blk_status blk_host_pipe_destroy(blk_host_pipe* p) {
    if (!p) return BLK_OK;
    return pipe_release(p);
}

constexpr int kMaxForwardEvents = 16;
struct blk_graph {
    cudaGraphExec_t exec = nullptr;
    cudaGraph_t graph = nullptr;  // kept for the event-node handles
    int device = -1;
    int n_events = 0;
    cudaGraphNode_t ev_nodes[kMaxForwardEvents] = {};
};

blk_status blk_forward_graph_create(const blk_block_desc* d, const blk_block_weights* w,
                                    const void* x, void* y, void* workspace, size_t ws_bytes,
                                    blk_dtype dt, void* const* events, int n_events,
                                    int32_t* step_kinds, int* n_launches, blk_graph** out) {
    BLK_REQUIRE(out != nullptr, "out is NULL");
    *out = nullptr;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaStream_t cs = nullptr;
    if ((e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e, "stream for capture");
    if ((e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal)) != cudaSuccess) {
        cudaStreamDestroy(cs);
        return cuda_fail(e, "cudaStreamBeginCapture");
    }
    blk_status st = blk_forward_ex(d, w, x, y, workspace, ws_bytes, dt,
                                   reinterpret_cast<blk_stream_t>(cs), events, n_events,
                                   step_kinds, n_launches);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(cs, &graph);
    cudaStreamDestroy(cs);
    if (st != BLK_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
    blk_graph* g = new (std::nothrow) blk_graph;
    if (!g) {
        cudaGraphDestroy(graph);
        return fail(BLK_EINVAL, "out of host memory");
    }
    g->graph = graph;
    g->device = dev;
    // the capture of one stream is a chain: walk it from its root and keep
    // the event-record nodes in recording order
    size_t n_nodes = 0;
    e = cudaGraphGetRootNodes(graph, nullptr, &n_nodes);
    cudaGraphNode_t node = nullptr;
    if (e == cudaSuccess && n_nodes == 1) e = cudaGraphGetRootNodes(graph, &node, &n_nodes);
    while (e == cudaSuccess && node) {
        cudaGraphNodeType type;
        if ((e = cudaGraphNodeGetType(node, &type)) != cudaSuccess) break;
        if (type == cudaGraphNodeTypeEventRecord && g->n_events < kMaxForwardEvents)
            g->ev_nodes[g->n_events++] = node;
        // edges between kernels launched for programmatic dependent launch
        // carry edge data, which the query must return (it refuses as lossy
        // otherwise); room for two dependents tells a chain link (one) apart
        cudaGraphNode_t next[2] = {};
        cudaGraphEdgeData edge[2] = {};
        size_t n_next = 2;
        if ((e = cudaGraphNodeGetDependentNodes(node, next, edge, &n_next)) != cudaSuccess) break;
        node = n_next == 1 ? next[0] : nullptr;
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&g->exec, graph, 0);
    if (e != cudaSuccess) {
        blk_graph_destroy(g);
        return cuda_fail(e, "graph instantiation");
    }
    *out = g;
    return BLK_OK;
}

blk_status blk_graph_launch(blk_graph* g, blk_stream_t s) {
    BLK_REQUIRE(g != nullptr && g->exec != nullptr, "graph handle is NULL");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    BLK_REQUIRE(dev == g->device, "graph was created on device %d, current device is %d",
                g->device, dev);
    e = cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(s));
    return e == cudaSuccess ? BLK_OK : cuda_fail(e, "cudaGraphLaunch");
}

blk_status blk_graph_set_events(blk_graph* g, void* const* events, int n_events) {
    BLK_REQUIRE(g != nullptr && g->exec != nullptr, "graph handle is NULL");
    BLK_REQUIRE(events != nullptr && n_events >= g->n_events,
                "the graph records %d events, got %d", g->n_events, n_events);
    for (int i = 0; i < g->n_events; ++i) {
        cudaError_t e = cudaGraphExecEventRecordNodeSetEvent(
            g->exec, g->ev_nodes[i], static_cast<cudaEvent_t>(events[i]));
        if (e != cudaSuccess) return cuda_fail(e, "cudaGraphExecEventRecordNodeSetEvent");
    }
    return BLK_OK;
}

blk_status blk_graph_destroy(blk_graph* g) {
    if (!g) return BLK_OK;
    cudaError_t e = g->exec ? cudaGraphExecDestroy(g->exec) : cudaSuccess;
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
    return e == cudaSuccess ? BLK_OK : cuda_fail(e, "cudaGraphExecDestroy");
}

}  // extern "C"
