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

inline size_t partial_bytes(int splits, int64_t m, int64_t n) {
    return splits > 1 ? (size_t)splits * (size_t)m * (size_t)n * sizeof(float) : 0;
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
    const int K = (int)W->k_in, N = (int)W->n_out, m = (int)M;
    // the same split decisions as lora_nf4_fwd, so both give the same bits
    const int bn = N <= 64 ? 64 : (N <= 128 ? 128 : 256);
    const LinearFwdSplits sp = linear_fwd_splits(M, N, K, r);
    const int st = sp.t, sy = sp.y;
    const size_t need_t = partial_bytes(st, M, r), need_y = partial_bytes(sy, M, N);
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
    {   // T = bf16(X A^T)
        GemmPlan g;
        g.set_error_word(sa.err);
        int mx = g.map(X, M, K, K, kBM);
        int ma = g.map(A, r, K, K, 64);
        g.problem(m, r, 64, A_KMAJOR, EPI_BF16, T_out, r, 1.0f, r, st);
        g.seg(mx, 0, B_TMA_K, ma, 0, 0, K);
        rc = g.launch(s, scratch, kStaticScratchBytes);
        if (rc) return rc;
    }
    {   // Y = bf16(X W^T + s T B^T [+ residual])
        GemmPlan g;
        g.set_error_word(sa.err);
        int mx = g.map(X, M, K, K, kBM);
        int mt = g.map(T_out, M, r, r, kBM);
        int wv = g.nf4(W->base, N, K);
        g.problem(m, N, bn, A_KMAJOR, EPI_BF16, Y, N, 1.0f, N, sy, residual, N);
        g.seg(mx, 0, B_NF4_K, wv, 0, 0, K);
        g.seg_scaled(mt, 0, B, r, N, r, scale);
        rc = g.launch(s, scratch, kStaticScratchBytes);
        if (rc) return rc;
    }
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
