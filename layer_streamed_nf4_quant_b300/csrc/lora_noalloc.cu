// lora_nf4_fwd_static_scratch: the single NF4 linear + LoRA forward without any device
// allocation, for callers that cannot call cudaMalloc.
//
// Who needs it: code that may not allocate device memory -- a plug-in hosted by a framework
// that owns every byte of device memory and forbids its plug-ins to call cudaMalloc, or a
// latency-critical serving path that must never enter the driver's allocator.  Such a caller
// still owns its inputs and outputs but cannot provide the split-K workspace that
// lora_nf4_fwd asks for, nor let the library allocate its per-device error word lazily.
//
// Instead, the scratch this variant needs lives in file-scope __device__ arrays: a
// kStaticScratchBytes (16 MiB) buffer for the fp32 split-K partial sums and one 32-bit error
// word.  Every GPU that loads the library holds them until the process exits.  Host code
// cannot use these names as device addresses, so on its first call on each device (with
// that device current) the entry point looks their addresses up with cudaGetSymbolAddress,
// clears the error word, and caches both; that first call must therefore not happen inside
// a stream capture.  All calls on a device share the same scratch: calls whose kernels
// overlap on the GPU (for example on two streams without ordering) race and must not be
// made.  The partial sums are fully written before they are read, so only the error word
// has to start at zero.  A device-wait timeout of a call made without device_status stays in
// the word until lsn_check() or the next call with device_status reads and clears it.
#include <mutex>

#include "lsn_internal.h"
#include "tc_gemm.h"

namespace lsn {

constexpr size_t kStaticScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
static __device__ __align__(256) uint32_t g_static_err[64];

namespace {

struct StaticAddrs {
    void* scratch = nullptr;
    uint32_t* err = nullptr;
};

std::mutex g_static_mu;
StaticAddrs g_static_addr[64];

// Looks up (once per device, with that device current) the device addresses of the static
// scratch and error word, and clears the error word.
int static_addresses(StaticAddrs* out) {
    int dev = 0;
    LSN_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(LSN_EINVAL, "static scratch: device index out of range");
    std::lock_guard<std::mutex> lk(g_static_mu);
    StaticAddrs& a = g_static_addr[dev];
    if (!a.scratch) {
        void* s = nullptr;
        void* e = nullptr;
        LSN_CUDA_TRY(cudaGetSymbolAddress(&s, g_static_scratch));
        LSN_CUDA_TRY(cudaGetSymbolAddress(&e, g_static_err));
        LSN_CUDA_TRY(cudaMemset(e, 0, sizeof(g_static_err)));
        LSN_CUDA_TRY(cudaDeviceSynchronize());
        a.err = static_cast<uint32_t*>(e);
        a.scratch = s;
    }
    *out = a;
    return LSN_OK;
}

}  // namespace

int static_error_take(uint32_t* v) {
    *v = 0;
    int dev = 0;
    LSN_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return LSN_OK;
    uint32_t* w = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_static_mu);
        w = g_static_addr[dev].err;
    }
    if (!w) return LSN_OK;   // the entry point has not run on this device
    LSN_CUDA_TRY(cudaMemcpy(v, w, sizeof(uint32_t), cudaMemcpyDeviceToHost));
    if (*v) LSN_CUDA_TRY(cudaMemset(w, 0, sizeof(uint32_t)));
    return LSN_OK;
}

}  // namespace lsn

using namespace lsn;

extern "C" int lora_nf4_fwd_static_scratch(const nf4_view* W, const uint16_t* X, int64_t M, const uint16_t* A,
                                           const uint16_t* B, int r, float scale, const uint16_t* residual,
                                           uint16_t* Y, uint16_t* T_out, uint32_t* device_status,
                                           void* stream) {
    // the same checks (shapes, NULLs, 16-byte alignment of every pointer) as lora_nf4_fwd
    int rc = check_linear_fwd("lora_nf4_fwd_static_scratch", W, X, M, A, B, r, residual, Y, T_out, true);
    if (rc) return rc;
    // the same plans (and so the same split decisions) as lora_nf4_fwd, so both give the same bits
    GemmPlan gt, gy;
    rc = plan_linear_fwd(&gt, &gy, W, X, M, A, B, r, scale, residual, Y, T_out);
    if (rc) return rc;
    const size_t need_t = gt.partial_bytes(), need_y = gy.partial_bytes();
    const size_t need = need_t > need_y ? need_t : need_y;
    if (need > kStaticScratchBytes)
        return fail(LSN_ENOMEM,
                    "lora_nf4_fwd_static_scratch: this shape needs %zu bytes of split-K scratch; the static "
                    "scratch holds %zu bytes (use lora_nf4_fwd with a caller workspace)",
                    need, kStaticScratchBytes);
    StaticAddrs sa;
    rc = static_addresses(&sa);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* scratch = static_cast<float*>(sa.scratch);
    gt.set_error_word(sa.err);   // T = bf16(X A^T)
    rc = gt.launch(s, scratch, kStaticScratchBytes);
    if (rc) return rc;
    gy.set_error_word(sa.err);   // Y = bf16(X W^T + s T B^T [+ residual])
    rc = gy.launch(s, scratch, kStaticScratchBytes);
    if (rc) return rc;
    if (device_status) {
        // synchronous status read: wait for this call's kernels, read and clear the word
        LSN_CUDA_TRY(cudaStreamSynchronize(s));
        uint32_t v = 0;
        LSN_CUDA_TRY(cudaMemcpy(&v, sa.err, sizeof(v), cudaMemcpyDeviceToHost));
        *device_status = v;
        if (v) {
            LSN_CUDA_TRY(cudaMemset(sa.err, 0, sizeof(uint32_t)));
            return fail(LSN_ETIMEOUT, "lora_nf4_fwd_static_scratch: a device wait ran out (site %u)", v & 0xFFFFFFu);
        }
    }
    return LSN_OK;
}
