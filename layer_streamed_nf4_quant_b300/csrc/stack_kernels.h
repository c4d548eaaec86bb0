// Launchers of the memory-bound layer kernels (internal interface).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lsn.h"

namespace lsn {

constexpr int kLossBlocks = 296;   // fixed grid of the loss reductions (fixes their order): 2 per SM

// h = bf16(x * rstd), rstd = (mean(x^2) + eps)^-1/2.  If header is non-null, block 0 also
// checks the layer image tag against `layer` and records a mismatch in the error word.
int launch_rmsnorm_fwd(const uint16_t* x, uint16_t* h, float* rstd, int M, int D, float eps,
                       const void* header, uint32_t layer, cudaStream_t s);
// Checks a layer image's tag (magic and layer index) and records a mismatch.
int launch_tag_check(const void* header, uint32_t layer, cudaStream_t s);
// dx += rstd*dh - rstd^3 * x * mean(dh*x)  (in place), dx_bf = bf16(dx).
int launch_rmsnorm_bwd(const uint16_t* x, const float* rstd, const float* dh, float* dx, uint16_t* dx_bf,
                       int M, int D, cudaStream_t s);
// a = bf16(silu(y[:, og:og+F]) * y[:, ou:ou+F]).
int launch_silu_mul(const uint16_t* y, int64_t ldy, int og, int ou, uint16_t* a, int M, int F, cudaStream_t s);
// part[2b], part[2b+1] = block sums of k^2 and v^2 (kLossBlocks blocks).
int launch_kv_sumsq(const uint16_t* y, int64_t ldy, int ok, int ov, int dkv, int M, float* part, cudaStream_t s);
// dx = x/(T*D) (fp32 and bf16) and the scalar loss from x's and the layers' k/v sums, with
// T = norm_tokens the token count the means are taken over (M, or a data-parallel batch's).
int launch_loss(const uint16_t* x, int M, double norm_tokens, int D, int dkv, int n_layers, float kv_coef, float* dx,
                uint16_t* dx_bf, float* xpart, const float* kvpart, float* loss, cudaStream_t s);
// out = in[0] + in[1] + ... (rank order, fp32), in = [n_ranks][n].
int launch_sum_ranks(const float* in, int n_ranks, int64_t n, float* out, cudaStream_t s);
// The k, v, gate and up columns of dY_cat (bf16): 2c k/(M dkv), 2c v/(M dkv), dgate, dup,
// from da (fp32 [M x F]) and the forward outputs; the dq columns are written by the GEMM.
int launch_dy_build(const float* da, const uint16_t* y, uint16_t* dy, int M, int D, int dkv, int F,
                    float kv_coef, cudaStream_t s);

// One AdamW step over n fp32 parameters (bf16 copy into pb when non-null).
int launch_adamw(const lsn_adamw_hparams& hp, float* p, uint16_t* pb, const float* g, float* m, float* v, int64_t n,
                 cudaStream_t s);

}  // namespace lsn
