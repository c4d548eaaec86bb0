// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "lsn.h"

namespace lsn {

// Records a thread-local error message and returns `code`.
int fail(int code, const char* fmt, ...);
// Records a CUDA error (with the failing call's text) and returns LSN_ECUDA.
int cuda_fail(cudaError_t e, const char* what);

#define LSN_CUDA_TRY(call)                                            \
    do {                                                              \
        cudaError_t lsn_e_ = (call);                                  \
        if (lsn_e_ != cudaSuccess) return ::lsn::cuda_fail(lsn_e_, #call); \
    } while (0)

// Device error word of the current device (lazily allocated, zeroed).  Kernels write
// (kind << 24 | detail) into it; kinds below.  Returns nullptr and sets the error on failure.
uint32_t* device_error_word();
enum DeviceErrorKind : uint32_t {
    kDevErrTimeout = 1u,   // a bounded spin-wait ran out (detail: site id)
    kDevErrTag = 2u,       // layer image tag mismatch (detail: expected layer)
};

class GemmPlan;
// The two launches of the single-linear forward (T, then Y) as plans, exactly as
// lora_nf4_fwd builds them: lora_nf4_fwd_static_scratch uses them, so the two give the same
// bits.  Returns the plans' status.
int plan_linear_fwd(GemmPlan* gt, GemmPlan* gy, const nf4_view* W, const uint16_t* X, int64_t M, const uint16_t* A,
                    const uint16_t* B, int r, float scale, const uint16_t* residual, uint16_t* Y, uint16_t* T_out);
// Argument checks of the single-linear forward entry points (shapes, NULLs, 16-byte
// alignment of every operand and output).  adapter == false: A, B and T_out are not used.
int check_linear_fwd(const char* who, const nf4_view* W, const uint16_t* X, int64_t M, const uint16_t* A,
                     const uint16_t* B, int r, const uint16_t* residual, const uint16_t* Y,
                     const uint16_t* T_out, bool adapter);
// Reads and clears the static-scratch entry point's error word of the current device
// (0 if that entry point has not been called on it).
int static_error_take(uint32_t* v);

// Launch accounting: every kernel launch site calls note_launch().
void note_launch();
// GEMM profiling hooks (no-ops unless lsn_profile_enable(1) was called).
bool profiling();
void* profile_begin(cudaStream_t s);                       // returns a token or nullptr
void profile_end(void* token, cudaStream_t s, double flops);

// NF4 codebook as computed by the library (host, fp32, ascending).
const float* nf4_levels();

// Layer image header (first 64 bytes of every layer image).
struct LayerHeader {
    uint32_t magic;        // kImageMagic
    uint32_t layer;
    uint64_t image_bytes;
    uint32_t d_model, d_kv, d_ff, n_mats;
    uint32_t rank_unused;
    uint8_t pad[28];
};
static_assert(sizeof(LayerHeader) == 64, "layer header is 64 bytes");
constexpr uint32_t kImageMagic = 0x314E534Cu;   // "LSN1"

// Projection indices in canonical order.
enum Proj { kQ = 0, kK, kV, kGate, kUp, kO, kDown, kNumProj };

// (n_out, k_in) of a projection.
void proj_shape(const lsn_stack_desc* d, int p, int64_t* n, int64_t* k);

// Packed-matrix section offsets (bytes, relative to the matrix start).
struct Nf4Layout {
    size_t codes, absmax, scale, offset, total;
    int64_t blocks, groups;
};
bool nf4_layout(int64_t n_out, int64_t k_in, Nf4Layout* out);

}  // namespace lsn
