// Memory-bound kernels of the synthetic decoder layer: RMSNorm forward/backward, SiLU-mul,
// the loss and its seed gradients, and the assembly of the fused QKVGU output gradient.
// Every reduction runs in a fixed order (fixed grid, fixed shuffle tree), so results are
// bit-reproducible.
//
// Layer definition (the workload description of the Llama-3.1-8B-shaped layer): unit-weight
// RMSNorm with eps, q/k/v/gate/up projections, a = silu(gate) * up, x' = x + o(q) + down(a);
// loss = 0.5 mean(x_L^2) + sum_l c (mean(k_l^2) + mean(v_l^2)).
#include <cuda_bf16.h>

#include "lsn_internal.h"
#include "stack_kernels.h"

namespace lsn {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Fixed-order warp sum to lane 0, broadcast back to every lane.
__device__ __forceinline__ float warp_sum_bcast(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
    return __shfl_sync(0xffffffffu, v, 0);
}

// Fixed-order block sum (blockDim.x == 256) of one value per thread; result valid in thread 0.
__device__ __forceinline__ float block_sum256(float v, float* sh) {
    sh[threadIdx.x] = v;
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
        if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
        __syncthreads();
    }
    return sh[0];
}

// ------------------------------------------------------------------------ layer tag

__global__ void tag_check_kernel(const LayerHeader* hdr, uint32_t expect_layer, uint32_t* err) {
    if (threadIdx.x == 0 && (hdr->magic != kImageMagic || hdr->layer != expect_layer))
        atomicCAS(err, 0u, (kDevErrTag << 24) | (expect_layer & 0xFFFFFFu));
}

// ------------------------------------------------------------------------- RMSNorm

__global__ void rmsnorm_fwd_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ h,
                                   float* __restrict__ rstd, int M, int D, float eps,
                                   const LayerHeader* hdr, uint32_t expect_layer, uint32_t* err) {
    if (hdr && blockIdx.x == 0 && threadIdx.x == 0) {
        if (hdr->magic != kImageMagic || hdr->layer != expect_layer)
            atomicCAS(err, 0u, (kDevErrTag << 24) | (expect_layer & 0xFFFFFFu));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + warp;
    if (row >= M) return;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)row * D);
    float ss = 0.f;
    for (int c = lane; c < D / 8; c += 32) {
        const uint4 v = xr[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = bf_lo(w[j]), b = bf_hi(w[j]);
            ss = __fadd_rn(ss, __fmul_rn(a, a));
            ss = __fadd_rn(ss, __fmul_rn(b, b));
        }
    }
    ss = warp_sum_bcast(ss);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)D), eps)));
    if (lane == 0) rstd[row] = r;
    uint4* hr = reinterpret_cast<uint4*>(h + (int64_t)row * D);
    for (int c = lane; c < D / 8; c += 32) {
        const uint4 v = xr[c];
        uint4 o;
        o.x = bf2(__fmul_rn(bf_lo(v.x), r), __fmul_rn(bf_hi(v.x), r));
        o.y = bf2(__fmul_rn(bf_lo(v.y), r), __fmul_rn(bf_hi(v.y), r));
        o.z = bf2(__fmul_rn(bf_lo(v.z), r), __fmul_rn(bf_hi(v.z), r));
        o.w = bf2(__fmul_rn(bf_lo(v.w), r), __fmul_rn(bf_hi(v.w), r));
        hr[c] = o;
    }
}

// dx = dx_next + rstd*dh - rstd^3 * x * mean(dh * x); also writes a bf16 copy of dx.
__global__ void rmsnorm_bwd_kernel(const uint16_t* __restrict__ x, const float* __restrict__ rstd,
                                   const float* __restrict__ dh, float* __restrict__ dx,
                                   uint16_t* __restrict__ dx_bf, int M, int D) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + warp;
    if (row >= M) return;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)row * D);
    const float4* dr = reinterpret_cast<const float4*>(dh + (int64_t)row * D);
    float dot = 0.f;
    for (int c = lane; c < D / 8; c += 32) {
        const uint4 v = xr[c];
        const float4 d0 = dr[2 * c], d1 = dr[2 * c + 1];
        dot = __fadd_rn(dot, __fmul_rn(d0.x, bf_lo(v.x)));
        dot = __fadd_rn(dot, __fmul_rn(d0.y, bf_hi(v.x)));
        dot = __fadd_rn(dot, __fmul_rn(d0.z, bf_lo(v.y)));
        dot = __fadd_rn(dot, __fmul_rn(d0.w, bf_hi(v.y)));
        dot = __fadd_rn(dot, __fmul_rn(d1.x, bf_lo(v.z)));
        dot = __fadd_rn(dot, __fmul_rn(d1.y, bf_hi(v.z)));
        dot = __fadd_rn(dot, __fmul_rn(d1.z, bf_lo(v.w)));
        dot = __fadd_rn(dot, __fmul_rn(d1.w, bf_hi(v.w)));
    }
    dot = warp_sum_bcast(dot);
    const float r = rstd[row];
    const float c3 = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), __fdiv_rn(dot, (float)D));
    float4* xo = reinterpret_cast<float4*>(dx + (int64_t)row * D);
    uint4* bo = reinterpret_cast<uint4*>(dx_bf + (int64_t)row * D);
    for (int c = lane; c < D / 8; c += 32) {
        const uint4 v = xr[c];
        const float4 d0 = dr[2 * c], d1 = dr[2 * c + 1];
        float4 g0 = xo[2 * c], g1 = xo[2 * c + 1];
        const float xs[8] = {bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y),
                             bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w)};
        const float ds[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
        float gs[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j)
            gs[j] = __fsub_rn(__fadd_rn(gs[j], __fmul_rn(r, ds[j])), __fmul_rn(c3, xs[j]));
        xo[2 * c] = make_float4(gs[0], gs[1], gs[2], gs[3]);
        xo[2 * c + 1] = make_float4(gs[4], gs[5], gs[6], gs[7]);
        bo[c] = make_uint4(bf2(gs[0], gs[1]), bf2(gs[2], gs[3]), bf2(gs[4], gs[5]), bf2(gs[6], gs[7]));
    }
}

// The same backward with one 128-thread block per row, for D <= 4096: each thread keeps its
// (at most four) 16-byte pieces of x and dh in registers between the dot product and the
// update, so the row is read once.  The dot product adds each thread's pieces in order, then
// the warps' sums in warp order: a fixed order.
constexpr int kNormBwdThreads = 128;
constexpr int kNormBwdPieces = 4;   // 16-byte pieces of x per thread: D <= 8 * 128 * 4
__global__ void __launch_bounds__(kNormBwdThreads) rmsnorm_bwd_row_kernel(const uint16_t* __restrict__ x,
                                                                         const float* __restrict__ rstd,
                                                                         const float* __restrict__ dh,
                                                                         float* __restrict__ dx,
                                                                         uint16_t* __restrict__ dx_bf, int D) {
    __shared__ float wsum[kNormBwdThreads / 32];
    const int row = blockIdx.x;
    const int np = D / 8;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)row * D);
    const float4* dr = reinterpret_cast<const float4*>(dh + (int64_t)row * D);
    uint4 xv[kNormBwdPieces];
    float4 d0[kNormBwdPieces], d1[kNormBwdPieces];
#pragma unroll
    for (int i = 0; i < kNormBwdPieces; ++i) {
        const int c = threadIdx.x + i * kNormBwdThreads;
        if (c < np) {
            xv[i] = xr[c];
            d0[i] = dr[2 * c];
            d1[i] = dr[2 * c + 1];
        }
    }
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < kNormBwdPieces; ++i) {
        const int c = threadIdx.x + i * kNormBwdThreads;
        if (c < np) {
            const uint4 v = xv[i];
            dot = __fadd_rn(dot, __fmul_rn(d0[i].x, bf_lo(v.x)));
            dot = __fadd_rn(dot, __fmul_rn(d0[i].y, bf_hi(v.x)));
            dot = __fadd_rn(dot, __fmul_rn(d0[i].z, bf_lo(v.y)));
            dot = __fadd_rn(dot, __fmul_rn(d0[i].w, bf_hi(v.y)));
            dot = __fadd_rn(dot, __fmul_rn(d1[i].x, bf_lo(v.z)));
            dot = __fadd_rn(dot, __fmul_rn(d1[i].y, bf_hi(v.z)));
            dot = __fadd_rn(dot, __fmul_rn(d1[i].z, bf_lo(v.w)));
            dot = __fadd_rn(dot, __fmul_rn(d1[i].w, bf_hi(v.w)));
        }
    }
    dot = warp_sum_bcast(dot);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = dot;
    __syncthreads();
    float tot = wsum[0];
#pragma unroll
    for (int w = 1; w < kNormBwdThreads / 32; ++w) tot = __fadd_rn(tot, wsum[w]);
    const float r = rstd[row];
    const float c3 = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), __fdiv_rn(tot, (float)D));
    float4* xo = reinterpret_cast<float4*>(dx + (int64_t)row * D);
    uint4* bo = reinterpret_cast<uint4*>(dx_bf + (int64_t)row * D);
#pragma unroll
    for (int i = 0; i < kNormBwdPieces; ++i) {
        const int c = threadIdx.x + i * kNormBwdThreads;
        if (c < np) {
            const uint4 v = xv[i];
            const float4 g0 = xo[2 * c], g1 = xo[2 * c + 1];
            const float xs[8] = {bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y),
                                 bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w)};
            const float ds[8] = {d0[i].x, d0[i].y, d0[i].z, d0[i].w, d1[i].x, d1[i].y, d1[i].z, d1[i].w};
            float gs[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j)
                gs[j] = __fsub_rn(__fadd_rn(gs[j], __fmul_rn(r, ds[j])), __fmul_rn(c3, xs[j]));
            xo[2 * c] = make_float4(gs[0], gs[1], gs[2], gs[3]);
            xo[2 * c + 1] = make_float4(gs[4], gs[5], gs[6], gs[7]);
            bo[c] = make_uint4(bf2(gs[0], gs[1]), bf2(gs[2], gs[3]), bf2(gs[4], gs[5]), bf2(gs[6], gs[7]));
        }
    }
}

// --------------------------------------------------------------------------- SiLU-mul

__device__ __forceinline__ float silu_f(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g))); }

// a = bf16(silu(g) * u); g, u are column blocks of the fused projection output.
__global__ void silu_mul_kernel(const uint16_t* __restrict__ y, int64_t ldy, int og, int ou,
                                uint16_t* __restrict__ a, int M, int F) {
    const int64_t chunks = (int64_t)M * (F / 8);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < chunks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / (F / 8);
        const int c = (int)(i - row * (F / 8)) * 8;
        const uint4 g = *reinterpret_cast<const uint4*>(y + row * ldy + og + c);
        const uint4 u = *reinterpret_cast<const uint4*>(y + row * ldy + ou + c);
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[j] = bf2(__fmul_rn(silu_f(bf_lo(gw[j])), bf_lo(uw[j])),
                       __fmul_rn(silu_f(bf_hi(gw[j])), bf_hi(uw[j])));
        *reinterpret_cast<uint4*>(a + row * F + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ------------------------------------------------------------------ loss and seeds

// Per-block sums of k^2 and v^2 over rows blockIdx.x, blockIdx.x + kLossBlocks, ...  The
// block's rows are cut into 16-byte pieces (dkv / 8 per row, for k and for v) and thread t
// takes pieces t, t + 256, ... in order, four at a time so that their loads are in flight
// together; every thread's order and the block tree are fixed, so the sums do not depend on
// timing.
__global__ void kv_sumsq_kernel(const uint16_t* __restrict__ y, int64_t ldy, int ok, int ov, int dkv,
                                int M, float* __restrict__ part) {
    __shared__ float sh[256];
    float sk = 0.f, sv = 0.f;
    const int ppr = dkv / 8;   // pieces per row
    const int rows = blockIdx.x < M ? (M - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int64_t total = (int64_t)rows * ppr;
    auto piece = [&](int64_t p, uint4& k, uint4& v) {
        const int64_t row = blockIdx.x + (p / ppr) * (int64_t)gridDim.x;
        const int c = (int)(p % ppr) * 8;
        k = *reinterpret_cast<const uint4*>(y + row * ldy + ok + c);
        v = *reinterpret_cast<const uint4*>(y + row * ldy + ov + c);
    };
    auto add = [&](const uint4& k, const uint4& v) {
        const uint32_t kw[4] = {k.x, k.y, k.z, k.w}, vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sk = __fadd_rn(sk, __fmul_rn(bf_lo(kw[j]), bf_lo(kw[j])));
            sk = __fadd_rn(sk, __fmul_rn(bf_hi(kw[j]), bf_hi(kw[j])));
            sv = __fadd_rn(sv, __fmul_rn(bf_lo(vw[j]), bf_lo(vw[j])));
            sv = __fadd_rn(sv, __fmul_rn(bf_hi(vw[j]), bf_hi(vw[j])));
        }
    };
    int64_t p = threadIdx.x;
    for (; p + 3 * 256 < total; p += 4 * 256) {
        uint4 k[4], v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) piece(p + u * 256, k[u], v[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u) add(k[u], v[u]);
    }
    for (; p < total; p += 256) {
        uint4 k, v;
        piece(p, k, v);
        add(k, v);
    }
    const float tk = block_sum256(sk, sh);
    __syncthreads();
    const float tv = block_sum256(sv, sh);
    if (threadIdx.x == 0) {
        part[2 * blockIdx.x] = tk;
        part[2 * blockIdx.x + 1] = tv;
    }
}

// Seed gradient dx = x / (M*D) (fp32 and bf16) and per-block sums of x^2.
__global__ void loss_seed_kernel(const uint16_t* __restrict__ x, int M, int D, float inv_md,
                                 float* __restrict__ dx, uint16_t* __restrict__ dx_bf,
                                 float* __restrict__ part) {
    __shared__ float sh[256];
    float s = 0.f;
    for (int row = blockIdx.x; row < M; row += gridDim.x) {
        for (int c = threadIdx.x * 8; c < D; c += 256 * 8) {
            const uint4 v = *reinterpret_cast<const uint4*>(x + (int64_t)row * D + c);
            const float xs[8] = {bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y),
                                 bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w)};
            float g[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                s = __fadd_rn(s, __fmul_rn(xs[j], xs[j]));
                g[j] = __fmul_rn(xs[j], inv_md);
            }
            float4* o = reinterpret_cast<float4*>(dx + (int64_t)row * D + c);
            o[0] = make_float4(g[0], g[1], g[2], g[3]);
            o[1] = make_float4(g[4], g[5], g[6], g[7]);
            *reinterpret_cast<uint4*>(dx_bf + (int64_t)row * D + c) =
                make_uint4(bf2(g[0], g[1]), bf2(g[2], g[3]), bf2(g[4], g[5]), bf2(g[6], g[7]));
        }
    }
    const float t = block_sum256(s, sh);
    if (threadIdx.x == 0) part[blockIdx.x] = t;
}

// loss = 0.5 * Sx / (M D) + sum_l coef (Sk_l + Sv_l) / (M dkv), summed in a fixed order in fp64.
// Sum over the kLossFinalThreads threads of one block, in a fixed tree order (fp64).
constexpr int kLossFinalThreads = 128;
__device__ __forceinline__ double block_sum_f64(double v, double* sh) {
    sh[threadIdx.x] = v;
    __syncthreads();
    for (int s = kLossFinalThreads / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
        __syncthreads();
    }
    const double t = sh[0];
    __syncthreads();   // sh is reused by the next sum
    return t;
}

// loss = 0.5 * sum(x^2) / (M D) + coef / (M dkv) * sum over layers of sum(k^2 + v^2), from the
// per-block partial sums.  One block; thread t takes the blocks b = t, t + 128, ... in order and
// the threads' sums meet in a fixed tree, so the result does not depend on timing.
__global__ void loss_final_kernel(const float* __restrict__ xpart, const float* __restrict__ kvpart,
                                  int n_layers, int nb, double inv_md, double coef_inv_mkv,
                                  float* __restrict__ loss) {
    __shared__ double sh[kLossFinalThreads];
    double sx = 0.0;
    for (int b = threadIdx.x; b < nb; b += kLossFinalThreads) sx += (double)xpart[b];
    double l = 0.5 * block_sum_f64(sx, sh) * inv_md;
    for (int layer = 0; layer < n_layers; ++layer) {
        const float* kv = kvpart + (size_t)layer * nb * 2;
        double skv = 0.0;
        for (int b = threadIdx.x; b < nb; b += kLossFinalThreads) skv += (double)kv[2 * b] + (double)kv[2 * b + 1];
        l += coef_inv_mkv * block_sum_f64(skv, sh);
    }
    if (threadIdx.x == 0) *loss = (float)l;
}

// ------------------------------------------------------------- backward dY assembly

// dY_cat's [dk | dv | dgate | dup] columns (bf16) from da (fp32 [M x F]), the forward outputs
// (k, v, gate, up) and the k/v loss coefficient; the dq columns come from the GEMM.
__global__ void dy_build_kernel(const float* __restrict__ da_in, const uint16_t* __restrict__ y,
                                uint16_t* __restrict__ dy, int M, int D, int dkv, int F, float kv_coef) {
    const int ldy = D + 2 * dkv + 2 * F;
    const int ok = D, og = D + 2 * dkv, ou = og + F;   // v follows k directly
    const int per_row = (2 * dkv) / 8 + F / 8;
    const int64_t total = (int64_t)M * per_row;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / per_row;
        int c = (int)(i - row * per_row) * 8;
        const uint16_t* yr = y + row * ldy;
        uint16_t* orow = dy + row * ldy;
        if (c < 2 * dkv) {
            const int col = ok + c;   // k block then v block are adjacent
            const uint4 v = *reinterpret_cast<const uint4*>(yr + col);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = bf2(__fmul_rn(kv_coef, bf_lo(w[j])), __fmul_rn(kv_coef, bf_hi(w[j])));
            *reinterpret_cast<uint4*>(orow + col) = make_uint4(o[0], o[1], o[2], o[3]);
            continue;
        }
        c -= 2 * dkv;
        const float* dr = da_in + row * F;
        const float4 a0 = *reinterpret_cast<const float4*>(dr + c);
        const float4 a1 = *reinterpret_cast<const float4*>(dr + c + 4);
        const float da[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint4 g4 = *reinterpret_cast<const uint4*>(yr + og + c);
        const uint4 u4 = *reinterpret_cast<const uint4*>(yr + ou + c);
        const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, uw[4] = {u4.x, u4.y, u4.z, u4.w};
        float dg[8], du[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float gg[2] = {bf_lo(gw[j]), bf_hi(gw[j])};
            const float uu[2] = {bf_lo(uw[j]), bf_hi(uw[j])};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float g = gg[e];
                const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g)));
                const float d = da[2 * j + e];
                // dg = da * u * sig(g) * (1 + g (1 - sig(g))),  du = da * g * sig(g)
                const float t = __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sg)));
                dg[2 * j + e] = __fmul_rn(__fmul_rn(__fmul_rn(d, uu[e]), sg), t);
                du[2 * j + e] = __fmul_rn(__fmul_rn(d, g), sg);
            }
        }
        *reinterpret_cast<uint4*>(orow + og + c) =
            make_uint4(bf2(dg[0], dg[1]), bf2(dg[2], dg[3]), bf2(dg[4], dg[5]), bf2(dg[6], dg[7]));
        *reinterpret_cast<uint4*>(orow + ou + c) =
            make_uint4(bf2(du[0], du[1]), bf2(du[2], du[3]), bf2(du[4], du[5]), bf2(du[6], du[7]));
    }
}

// -------------------------------------------------------------------------- AdamW

__global__ void adamw_kernel(float* __restrict__ p, uint16_t* __restrict__ pb, const float* __restrict__ g,
                             float* __restrict__ m, float* __restrict__ v, int64_t n, float lr, float b1, float b2,
                             float eps, float wd, float bc1, float bc2) {
    const float omb1 = 1.0f - b1, omb2 = 1.0f - b2;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float gi = g[i];
        const float mi = __fadd_rn(__fmul_rn(b1, m[i]), __fmul_rn(omb1, gi));
        const float vi = __fadd_rn(__fmul_rn(b2, v[i]), __fmul_rn(omb2, __fmul_rn(gi, gi)));
        const float mh = __fdiv_rn(mi, bc1);
        const float vh = __fdiv_rn(vi, bc2);
        const float pi = p[i];
        const float upd = __fadd_rn(__fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), eps)), __fmul_rn(wd, pi));
        const float pn = __fsub_rn(pi, __fmul_rn(lr, upd));
        m[i] = mi;
        v[i] = vi;
        p[i] = pn;
        if (pb) {
            __nv_bfloat16 h = __float2bfloat16_rn(pn);
            pb[i] = *reinterpret_cast<uint16_t*>(&h);
        }
    }
}

// ---------------------------------------------------------------------- launchers

static inline unsigned grid_for(int64_t work, int per_block) {
    int64_t b = (work + per_block - 1) / per_block;
    if (b < 1) b = 1;
    if (b > 148 * 16) b = 148 * 16;
    return (unsigned)b;
}

int launch_rmsnorm_fwd(const uint16_t* x, uint16_t* h, float* rstd, int M, int D, float eps,
                       const void* header, uint32_t layer, cudaStream_t s) {
    uint32_t* err = header ? device_error_word() : nullptr;
    if (header && !err) return LSN_ECUDA;
    rmsnorm_fwd_kernel<<<(M + 7) / 8, 256, 0, s>>>(x, h, rstd, M, D, eps,
                                                   static_cast<const LayerHeader*>(header), layer, err);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

int launch_tag_check(const void* header, uint32_t layer, cudaStream_t s) {
    uint32_t* err = device_error_word();
    if (!err) return LSN_ECUDA;
    tag_check_kernel<<<1, 32, 0, s>>>(static_cast<const LayerHeader*>(header), layer, err);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

int launch_rmsnorm_bwd(const uint16_t* x, const float* rstd, const float* dh, float* dx, uint16_t* dx_bf,
                       int M, int D, cudaStream_t s) {
    if (D <= 8 * kNormBwdThreads * kNormBwdPieces)
        rmsnorm_bwd_row_kernel<<<M, kNormBwdThreads, 0, s>>>(x, rstd, dh, dx, dx_bf, D);
    else
        rmsnorm_bwd_kernel<<<(M + 7) / 8, 256, 0, s>>>(x, rstd, dh, dx, dx_bf, M, D);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

int launch_silu_mul(const uint16_t* y, int64_t ldy, int og, int ou, uint16_t* a, int M, int F, cudaStream_t s) {
    silu_mul_kernel<<<grid_for((int64_t)M * F / 8, 256), 256, 0, s>>>(y, ldy, og, ou, a, M, F);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

int launch_kv_sumsq(const uint16_t* y, int64_t ldy, int ok, int ov, int dkv, int M, float* part, cudaStream_t s) {
    kv_sumsq_kernel<<<kLossBlocks, 256, 0, s>>>(y, ldy, ok, ov, dkv, M, part);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

int launch_loss(const uint16_t* x, int M, double norm_tokens, int D, int dkv, int n_layers, float kv_coef, float* dx,
                uint16_t* dx_bf, float* xpart, const float* kvpart, float* loss, cudaStream_t s) {
    const double md = norm_tokens * (double)D;
    loss_seed_kernel<<<kLossBlocks, 256, 0, s>>>(x, M, D, (float)(1.0 / md), dx, dx_bf, xpart);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    loss_final_kernel<<<1, kLossFinalThreads, 0, s>>>(xpart, kvpart, n_layers, kLossBlocks, 1.0 / md,
                                       (double)kv_coef / (norm_tokens * (double)dkv), loss);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

int launch_dy_build(const float* da, const uint16_t* y, uint16_t* dy, int M, int D, int dkv, int F,
                    float kv_coef, cudaStream_t s) {
    const int64_t work = (int64_t)M * (2 * dkv / 8 + F / 8);
    dy_build_kernel<<<grid_for(work, 256), 256, 0, s>>>(da, y, dy, M, D, dkv, F, kv_coef);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

// out[i] = sum over ranks in rank order (fp32, left to right).
// (no __restrict__: out may alias in[0]; each thread reads its elements before writing them)
// kVec: four elements per thread through 16-byte accesses.  Rank r's row starts at in + r*n,
// which is 16-byte aligned for every r only when n is a multiple of 4 (in and out are), so
// the launcher takes the vector form only then.
template <bool kVec>
__global__ void sum_ranks_kernel(const float* in, int n_ranks, int64_t n, float* out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t first = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (kVec) {
        const int64_t n4 = n / 4;
        for (int64_t i = first; i < n4; i += stride) {
            float4 acc = reinterpret_cast<const float4*>(in)[i];
            for (int r = 1; r < n_ranks; ++r) {
                const float4 v = reinterpret_cast<const float4*>(in + (int64_t)r * n)[i];
                acc.x = __fadd_rn(acc.x, v.x);
                acc.y = __fadd_rn(acc.y, v.y);
                acc.z = __fadd_rn(acc.z, v.z);
                acc.w = __fadd_rn(acc.w, v.w);
            }
            reinterpret_cast<float4*>(out)[i] = acc;
        }
    } else {
        for (int64_t i = first; i < n; i += stride) {
            float acc = in[i];
            for (int r = 1; r < n_ranks; ++r) acc = __fadd_rn(acc, in[(int64_t)r * n + i]);
            out[i] = acc;
        }
    }
}

int launch_sum_ranks(const float* in, int n_ranks, int64_t n, float* out, cudaStream_t s) {
    if (n == 0) return LSN_OK;
    if (n % 4 == 0)
        sum_ranks_kernel<true><<<grid_for(n / 4, 256), 256, 0, s>>>(in, n_ranks, n, out);
    else
        sum_ranks_kernel<false><<<grid_for(n, 256), 256, 0, s>>>(in, n_ranks, n, out);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

int launch_adamw(const lsn_adamw_hparams& hp, float* p, uint16_t* pb, const float* g, float* m, float* v, int64_t n,
                 cudaStream_t s) {
    const double bc1 = 1.0 - pow((double)hp.beta1, (double)hp.step);
    const double bc2 = 1.0 - pow((double)hp.beta2, (double)hp.step);
    adamw_kernel<<<grid_for(n, 256), 256, 0, s>>>(p, pb, g, m, v, n, hp.lr, hp.beta1, hp.beta2, hp.eps,
                                                  hp.weight_decay, (float)bc1, (float)bc2);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

}  // namespace lsn

extern "C" int lsn_adamw_step(const lsn_adamw_hparams* hp, float* p, uint16_t* p_bf16, const float* g, float* m,
                              float* v, size_t n, void* stream) {
    using namespace lsn;
    if (!hp || !p || !g || !m || !v || n == 0) return fail(LSN_EINVAL, "lsn_adamw_step: bad arguments");
    if (hp->step < 1 || !(hp->beta1 >= 0.f && hp->beta1 < 1.f) || !(hp->beta2 >= 0.f && hp->beta2 < 1.f))
        return fail(LSN_EINVAL, "lsn_adamw_step: need step >= 1 and betas in [0, 1)");
    return launch_adamw(*hp, p, p_bf16, g, m, v, (int64_t)n, static_cast<cudaStream_t>(stream));
}
