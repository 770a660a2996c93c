// blk_mlp_noalloc: the MLP of blk_mlp for callers that cannot allocate device
// memory (an engine or plugin host that owns all device memory and forbids
// allocation after start-up; latency-bound code that cannot take
// cudaMalloc's implicit device synchronisation). The [tokens, intermediate]
// activation lives in one file-scope device array instead of a caller
// workspace; everything else is the same two GEMM launches as blk_mlp.
#include <mutex>

#include "internal.h"

namespace blk {

namespace {

constexpr size_t kScratchBytes = BLK_MLP_NOALLOC_SCRATCH_BYTES;

// Held by every device that loads this library until the process exits.
// Shared by all calls: overlapping calls race on it.
static __device__ __align__(256) unsigned char g_mlp_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_mlp_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current, and kept: a device reset in this
// process (cudaDeviceReset) would leave it stale, which the header forbids.
blk_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return report_error_status(BLK_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return report_error_status(BLK_EUNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_mlp_scratch);
        if (e != cudaSuccess || !p)
            return report_error_status(BLK_ECUDA, "cudaGetSymbolAddress(MLP scratch): %s",
                                       cudaGetErrorString(e));
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return BLK_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace blk

using namespace blk;

extern "C" blk_status blk_mlp_noalloc(const blk_mlp_desc* d, const void* x, const void* w_gate,
                                      const void* w_up, const void* b_up, const void* w_down,
                                      const void* b_down, const void* res1, const void* res2,
                                      void* y, blk_dtype dt, blk_stream_t s) {
    if (dt != BLK_F16 && dt != BLK_BF16)
        return report_error_status(BLK_EINVAL, "dtype must be BLK_F16 or BLK_BF16");
    if (!d) return report_error_status(BLK_EINVAL, "descriptor is NULL");
    if (d->act != BLK_ACT_SWIGLU && d->act != BLK_ACT_GELU_TANH)
        return report_error_status(BLK_EINVAL, "unknown act");
    if (d->tokens < 0 || d->tokens > 0x7fffffff)
        return report_error_status(BLK_EINVAL, "tokens out of range");
    if (d->hidden < 8 || d->hidden % 8 || d->hidden > 0x7fffffff)
        return report_error_status(BLK_EINVAL, "hidden must be a positive multiple of 8");
    if (d->intermediate < 8 || d->intermediate % 8 || d->intermediate > 0x7fffffff)
        return report_error_status(BLK_EINVAL, "intermediate must be a positive multiple of 8");
    const bool swiglu = d->act == BLK_ACT_SWIGLU;
    struct P {
        const void* p;
        const char* name;
        bool required;
    } ptrs[] = {{x, "x", true},           {w_gate, "w_gate", swiglu}, {w_up, "w_up", true},
                {b_up, "b_up", false},    {w_down, "w_down", true},   {b_down, "b_down", false},
                {res1, "res1", false},    {res2, "res2", false},      {y, "y", true}};
    for (const P& q : ptrs) {
        if (!q.p && q.required) return report_error_status(BLK_EINVAL, "%s is NULL", q.name);
        if (q.p && !aligned16(q.p))
            return report_error_status(BLK_EINVAL, "%s is not 16-byte aligned", q.name);
    }
    if (!swiglu && w_gate) return report_error_status(BLK_EINVAL, "w_gate must be NULL for GELU_TANH");
    if (swiglu && b_up)
        return report_error_status(BLK_EINVAL, "b_up is not supported with SWIGLU (must be NULL)");
    const size_t need = static_cast<size_t>(d->tokens) * static_cast<size_t>(d->intermediate) * 2;
    if (need > kScratchBytes)
        return report_error_status(BLK_EWORKSPACE,
                                   "tokens * intermediate * 2 = %zu bytes exceeds the %zu-byte "
                                   "scratch of blk_mlp_noalloc; use blk_mlp with a workspace",
                                   need, kScratchBytes);
    if (d->tokens == 0) return BLK_OK;

    int sms = 0;
    unsigned* err = nullptr;
    blk_status st = current_device_info(&sms, &err);
    if (st != BLK_OK) return st;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != BLK_OK) return st;

    const DType t = dt == BLK_F16 ? DType::F16 : DType::BF16;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    RopeParams rp;
    memset(&rp, 0, sizeof(rp));
    GemmArgs g{};
    g.M = static_cast<int>(d->tokens);
    g.N = static_cast<int>(d->intermediate);
    g.K = static_cast<int>(d->hidden);
    g.out = scratch;
    g.bias = b_up;
    g.err = err;
    cudaError_t e = launch_gemm(t, swiglu ? EPI_SWIGLU : EPI_GELU, x, swiglu ? w_gate : w_up,
                                swiglu ? w_up : nullptr, g, rp, sms, cs);
    if (e != cudaSuccess)
        return report_error_status(BLK_ECUDA, "mlp up launch: %s", cudaGetErrorString(e));
    GemmArgs g2{};
    g2.M = static_cast<int>(d->tokens);
    g2.N = static_cast<int>(d->hidden);
    g2.K = static_cast<int>(d->intermediate);
    g2.out = y;
    g2.bias = b_down;
    g2.res1 = res1;
    g2.res2 = res2;
    g2.err = err;
    e = launch_gemm(t, EPI_LINEAR, scratch, w_down, nullptr, g2, rp, sms, cs);
    if (e != cudaSuccess)
        return report_error_status(BLK_ECUDA, "mlp down launch: %s", cudaGetErrorString(e));
    return BLK_OK;
}
