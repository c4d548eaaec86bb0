// C entry points of the single frozen-NF4 linear with its LoRA branch (forward and
// backward) and the test-only dequantiser, assembled from grouped tcgen05 GEMM launches.
//
// "Can You Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's Layer Streaming Explained", section
// "How Soup's layer streaming actually works", step 1: the base W is frozen (no dW), only the
// LoRA factors A, B train.
#include <string.h>

#include "lsn_internal.h"
#include "tc_gemm.h"

namespace lsn {

static inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }
static inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
static inline int bn_for(int64_t n) { return n <= 64 ? 64 : (n <= 128 ? 128 : 256); }

struct LinearShape {
    int64_t M, N, K;
    int r;
};

// The launches of the single linear, as plans.  Given null pointers and a dry plan they size
// the workspace with exactly the split decisions of the real launch (the split planner sees
// the same problems).  The LoRA k-steps of the Y launch are a tail: the adapter-disabled
// launch splits the base contraction the same way.
static void plan_fwd_T(GemmPlan& g, const LinearShape& s, const uint16_t* X, const uint16_t* A, uint16_t* T) {
    const int K = (int)s.K;
    int mx = g.map(X, s.M, K, K, kBM);
    int ma = g.map(A, s.r, K, K, 64);
    g.problem((int)s.M, s.r, 64, A_KMAJOR, EPI_BF16, T, s.r, 1.0f, s.r, kAutoSplits);
    g.seg(mx, 0, B_TMA_K, ma, 0, 0, K);
}

static void plan_fwd_Y(GemmPlan& g, const LinearShape& s, const void* W, const uint16_t* X, const uint16_t* T,
                       const uint16_t* B, float scale, const uint16_t* residual, uint16_t* Y, bool adapter) {
    const int K = (int)s.K, N = (int)s.N;
    int mx = g.map(X, s.M, K, K, kBM);
    int wv = g.nf4(W, N, K);
    g.problem((int)s.M, N, bn_for(N), A_KMAJOR, EPI_BF16, Y, N, 1.0f, N, kAutoSplits, residual, N);
    g.seg(mx, 0, B_NF4_K, wv, 0, 0, K);
    if (adapter) g.seg_scaled(g.map(T, s.M, s.r, s.r, kBM), 0, B, s.r, N, s.r, scale);
}

static void plan_bwd_dT(GemmPlan& g, const LinearShape& s, const uint16_t* dY, const uint16_t* B, float scale,
                        uint16_t* dT) {
    const int N = (int)s.N;
    int my = g.map(dY, s.M, N, N, kBM);
    int mb = g.map(B, N, s.r, s.r, 64);
    g.problem((int)s.M, s.r, 64, A_KMAJOR, EPI_BF16, dT, s.r, scale, s.r, kAutoSplits);
    g.seg(my, 0, B_TMA_MN, mb, 0, 0, N);
}

// dB = s dY^T T ; dA^T = X^T dT ; dX (+)= dY W + dT A   (one grouped launch; dX optional)
static void plan_bwd_main(GemmPlan& g, const LinearShape& s, const void* W, const uint16_t* X, const uint16_t* T,
                          const uint16_t* dY, const uint16_t* A, const uint16_t* dT, float scale, float* dX,
                          bool want_dX, bool accumulate_dX, float* dA, float* dB) {
    const int K = (int)s.K, N = (int)s.N, m = (int)s.M, r = s.r;
    int my_mn = g.map(dY, s.M, N, N, 64);
    int mt_mn = g.map(T, s.M, r, r, 64);
    int mx_mn = g.map(X, s.M, K, K, 64);
    int mdt_mn = g.map(dT, s.M, r, r, 64);
    g.problem(N, r, 64, A_MNMAJOR, EPI_F32, dB, r, scale, r, kAutoSplits);
    g.seg(my_mn, 0, B_TMA_MN, mt_mn, 0, 0, m);
    g.problem(K, r, 64, A_MNMAJOR, EPI_F32_T, dA, K, 1.0f, r, kAutoSplits);
    g.seg(mx_mn, 0, B_TMA_MN, mdt_mn, 0, 0, m);
    if (want_dX) {
        int my = g.map(dY, s.M, N, N, kBM);
        int mdt = g.map(dT, s.M, r, r, kBM);
        int ma_mn = g.map(A, r, K, K, 64);
        int wv = g.nf4(W, N, K);
        g.problem(m, K, bn_for(K), A_KMAJOR, accumulate_dX ? EPI_F32_ACC : EPI_F32, dX, K, 1.0f, K, kAutoSplits);
        g.seg(my, 0, B_NF4_MN, wv, 0, 0, N);
        g.seg(mdt, 0, B_TMA_MN, ma_mn, 0, 0, r, true);
    }
}

// Workspace of the forward: the T launch's partial slabs, then the Y launch's.
struct FwdWs { size_t t, y; };
static FwdWs fwd_ws(const LinearShape& s) {
    GemmPlan gt(true), gy(true);
    plan_fwd_T(gt, s, nullptr, nullptr, nullptr);
    plan_fwd_Y(gy, s, nullptr, nullptr, nullptr, nullptr, 1.0f, nullptr, nullptr, true);
    return FwdWs{align256(gt.partial_bytes()), align256(gy.partial_bytes())};
}

// Workspace of the backward: dT (bf16 [M x r]), the dT launch's partials, the main launch's
// partials (with or without dX, whichever needs more).
struct BwdWs { size_t dt_out, dt, main; };
static BwdWs bwd_ws(const LinearShape& s) {
    GemmPlan g1(true), g2(true), g3(true);
    plan_bwd_dT(g1, s, nullptr, nullptr, 1.0f, nullptr);
    plan_bwd_main(g2, s, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 1.0f, nullptr, true, false, nullptr,
                  nullptr);
    plan_bwd_main(g3, s, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 1.0f, nullptr, false, false, nullptr,
                  nullptr);
    const size_t a = g2.partial_bytes(), b = g3.partial_bytes();
    return BwdWs{align256((size_t)s.M * s.r * 2), align256(g1.partial_bytes()), align256(a > b ? a : b)};
}

static int check_linear(const nf4_view* W, int64_t M, int r, const void* X) {
    if (!W || !W->base || !X) return fail(LSN_EINVAL, "lora: NULL argument");
    if (W->k_in < 64 || W->k_in % 64 || W->n_out < 8 || W->n_out % 8)
        return fail(LSN_EINVAL, "lora: need k_in %% 64 == 0 and n_out %% 8 == 0");
    if (r < 8 || r > 64 || r % 8) return fail(LSN_EINVAL, "lora: r must be 8..64, a multiple of 8");
    if (M < 1 || M > (1 << 30)) return fail(LSN_EINVAL, "lora: bad M");
    if (!al16(W->base) || !al16(X)) return fail(LSN_EINVAL, "lora: pointers must be 16-byte aligned");
    return LSN_OK;
}

int plan_linear_fwd(GemmPlan* gt, GemmPlan* gy, const nf4_view* W, const uint16_t* X, int64_t M, const uint16_t* A,
                    const uint16_t* B, int r, float scale, const uint16_t* residual, uint16_t* Y, uint16_t* T_out) {
    const LinearShape s{M, W->n_out, W->k_in, r};
    plan_fwd_T(*gt, s, X, A, T_out);
    plan_fwd_Y(*gy, s, W->base, X, T_out, B, scale, residual, Y, true);
    return gt->status() ? gt->status() : gy->status();
}

int check_linear_fwd(const char* who, const nf4_view* W, const uint16_t* X, int64_t M, const uint16_t* A,
                     const uint16_t* B, int r, const uint16_t* residual, const uint16_t* Y,
                     const uint16_t* T_out, bool adapter) {
    if (!W || !W->base || !X || !Y || (adapter && (!A || !B || !T_out)))
        return fail(LSN_EINVAL, "%s: NULL argument", who);
    if (W->k_in < 64 || W->k_in % 64 || W->n_out < 8 || W->n_out % 8)
        return fail(LSN_EINVAL, "%s: need k_in %% 64 == 0 and n_out %% 8 == 0", who);
    if (r < 8 || r > 64 || r % 8) return fail(LSN_EINVAL, "%s: r must be 8..64, a multiple of 8", who);
    if (M < 1 || M > (1 << 30)) return fail(LSN_EINVAL, "%s: bad M", who);
    if (!al16(W->base) || !al16(X) || !al16(Y) || (residual && !al16(residual)) ||
        (adapter && (!al16(A) || !al16(B) || !al16(T_out))))
        return fail(LSN_EINVAL, "%s: pointers must be 16-byte aligned", who);
    return LSN_OK;
}

}  // namespace lsn

using namespace lsn;

extern "C" {

size_t lora_nf4_workspace_bytes(int64_t M, int64_t n_out, int64_t k_in, int r) {
    if (M < 1 || M > (1 << 30) || n_out < 8 || n_out % 8 || k_in < 64 || k_in % 64 || r < 8 || r > 64 || r % 8)
        return 0;
    const LinearShape s{M, n_out, k_in, r};
    const FwdWs f = fwd_ws(s);
    const BwdWs b = bwd_ws(s);
    const size_t a = f.t + f.y, c = b.dt_out + b.dt + b.main;
    return (a > c ? a : c) + 256;
}

int lora_nf4_fwd_plan(int64_t M, int64_t n_out, int64_t k_in, int r, int* t_splits, int* y_splits,
                      size_t* t_partial_bytes, size_t* y_partial_bytes) {
    if (M < 1 || M > (1 << 30) || n_out < 8 || n_out % 8 || k_in < 64 || k_in % 64 || r < 8 || r > 64 || r % 8)
        return fail(LSN_EINVAL, "lora_nf4_fwd_plan: shape refused by lora_nf4_fwd");
    const LinearShape s{M, n_out, k_in, r};
    GemmPlan gt(true), gy(true);
    plan_fwd_T(gt, s, nullptr, nullptr, nullptr);
    plan_fwd_Y(gy, s, nullptr, nullptr, nullptr, nullptr, 1.0f, nullptr, nullptr, true);
    if (gt.status() || gy.status()) return gt.status() ? gt.status() : gy.status();
    if (t_splits) *t_splits = gt.splits_of(0);
    if (y_splits) *y_splits = gy.splits_of(0);
    if (t_partial_bytes) *t_partial_bytes = gt.partial_bytes();
    if (y_partial_bytes) *y_partial_bytes = gy.partial_bytes();
    return LSN_OK;
}

int nf4_dequant(const nf4_view* W, uint16_t* out, void* stream) {
    if (!W || !W->base || !out) return fail(LSN_EINVAL, "nf4_dequant: NULL argument");
    Nf4Layout L;
    if (!nf4_layout(W->n_out, W->k_in, &L) || !al16(W->base) || !al16(out))
        return fail(LSN_EINVAL, "nf4_dequant: bad view or alignment");
    Nf4Dev d;
    const int rc = nf4_view_dev(W->base, W->n_out, W->k_in, &d);
    if (rc) return rc;
    return nf4_dequant_many(&d, &out, 1, static_cast<cudaStream_t>(stream));
}

int lora_nf4_fwd(const nf4_view* W, const uint16_t* X, int64_t M, const uint16_t* A, const uint16_t* B,
                 int r, float scale, const uint16_t* residual, uint16_t* Y, uint16_t* T_out, void* ws,
                 size_t ws_bytes, void* stream) {
    // A == B == NULL: the adapter is disabled; Y is the frozen linear alone
    const bool adapter = A || B;
    int rc = check_linear_fwd("lora_nf4_fwd", W, X, M, A, B, r, residual, Y, T_out, adapter);
    if (rc) return rc;
    const LinearShape s{M, W->n_out, W->k_in, r};
    const FwdWs f = fwd_ws(s);
    if (ws_bytes < f.t + f.y || (f.t + f.y && !ws))
        return fail(LSN_ENOMEM, "lora_nf4_fwd: workspace %zu < %zu", ws_bytes, f.t + f.y);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    if (adapter) {   // T = bf16(X A^T)
        GemmPlan g;
        plan_fwd_T(g, s, X, A, T_out);
        rc = g.launch(st, reinterpret_cast<float*>(wsb), f.t);
        if (rc) return rc;
    }
    {   // Y = bf16(X W^T + s T B^T [+ residual])
        GemmPlan g;
        plan_fwd_Y(g, s, W->base, X, T_out, B, scale, residual, Y, adapter);
        rc = g.launch(st, reinterpret_cast<float*>(wsb ? wsb + f.t : nullptr), ws_bytes - f.t);
        if (rc) return rc;
    }
    return LSN_OK;
}

int lora_nf4_bwd(const nf4_view* W, const uint16_t* X, const uint16_t* T, const uint16_t* dY, int64_t M,
                 const uint16_t* A, const uint16_t* B, int r, float scale, float* dX, int accumulate_dX,
                 float* dA, float* dB, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_linear(W, M, r, X);
    if (rc) return rc;
    if (!T || !dY || !A || !B || !dA || !dB) return fail(LSN_EINVAL, "lora_nf4_bwd: NULL argument");
    if (!al16(T) || !al16(dY) || !al16(A) || !al16(B) || !al16(dA) || !al16(dB) || (dX && !al16(dX)))
        return fail(LSN_EINVAL, "lora_nf4_bwd: pointers must be 16-byte aligned");
    const LinearShape s{M, W->n_out, W->k_in, r};
    const BwdWs b = bwd_ws(s);
    const size_t need = b.dt_out + b.dt + b.main;
    if (ws_bytes < need || !ws) return fail(LSN_ENOMEM, "lora_nf4_bwd: workspace %zu < %zu", ws_bytes, need);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    uint16_t* dT = reinterpret_cast<uint16_t*>(wsb);
    {   // dT = bf16(s dY B)
        GemmPlan g;
        plan_bwd_dT(g, s, dY, B, scale, dT);
        rc = g.launch(st, reinterpret_cast<float*>(wsb + b.dt_out), b.dt);
        if (rc) return rc;
    }
    {   // dB, dA and dX in one grouped launch
        GemmPlan g;
        plan_bwd_main(g, s, W->base, X, T, dY, A, dT, scale, dX, dX != nullptr, accumulate_dX != 0, dA, dB);
        rc = g.launch(st, reinterpret_cast<float*>(wsb + b.dt_out + b.dt), b.main);
        if (rc) return rc;
    }
    return LSN_OK;
}

}  // extern "C"
