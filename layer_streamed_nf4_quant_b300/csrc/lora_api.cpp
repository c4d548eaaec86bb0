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
static inline int tiles_of(int64_t m, int64_t n, int bn) { return pair_tiles(m, n, bn); }
static inline int bn_for(int64_t n) { return n <= 64 ? 64 : (n <= 128 ? 128 : 256); }
static inline int ksteps_of(int64_t k) { return (int)((k + kBK - 1) / kBK); }

struct LinearShape {
    int64_t M, N, K;
    int r;
};

// Split counts used by the forward / backward launches (shared with the workspace query).
struct FwdSplits { int t, y; };
struct BwdSplits { int dt, db, da, dx; };

// The LoRA k-steps of the Y launch are a tail (they go to the last split), so the splits
// divide the base contraction only: the adapter-disabled launch splits it the same way.
static FwdSplits fwd_splits(const LinearShape& s) {
    FwdSplits f;
    f.t = choose_splits(tiles_of(s.M, s.r, 64), ksteps_of(s.K));
    f.y = choose_splits(tiles_of(s.M, s.N, bn_for(s.N)), ksteps_of(s.K));
    return f;
}

LinearFwdSplits linear_fwd_splits(int64_t M, int64_t n_out, int64_t k_in, int r) {
    const FwdSplits f = fwd_splits(LinearShape{M, n_out, k_in, r});
    return LinearFwdSplits{f.t, f.y};
}

static BwdSplits bwd_splits(const LinearShape& s) {
    BwdSplits b;
    b.dt = choose_splits(tiles_of(s.M, s.r, 64), ksteps_of(s.N));
    const int tiles2 = tiles_of(s.N, s.r, 64) + tiles_of(s.K, s.r, 64) + tiles_of(s.M, s.K, bn_for(s.K));
    b.db = choose_splits(tiles2, ksteps_of(s.M));
    b.da = b.db;
    b.dx = choose_splits(tiles2, ksteps_of(s.N));
    return b;
}

static size_t partial_bytes(int splits, int64_t m, int64_t n) {
    return splits > 1 ? align256((size_t)splits * m * n * sizeof(float)) : 0;
}

static size_t fwd_ws(const LinearShape& s) {
    FwdSplits f = fwd_splits(s);
    return partial_bytes(f.t, s.M, s.r) + partial_bytes(f.y, s.M, s.N);
}

static size_t bwd_ws(const LinearShape& s) {
    BwdSplits b = bwd_splits(s);
    return align256((size_t)s.M * s.r * 2) + partial_bytes(b.dt, s.M, s.r) + partial_bytes(b.db, s.N, s.r) +
           partial_bytes(b.da, s.K, s.r) + partial_bytes(b.dx, s.M, s.K);
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
    if (M < 1 || n_out < 1 || k_in < 64 || r < 8 || r > 64) return 0;
    LinearShape s{M, n_out, k_in, r};
    size_t a = fwd_ws(s), b = bwd_ws(s);
    return (a > b ? a : b) + 256;
}

int nf4_dequant(const nf4_view* W, uint16_t* out, void* stream) {
    if (!W || !W->base || !out) return fail(LSN_EINVAL, "nf4_dequant: NULL argument");
    Nf4Layout L;
    if (!nf4_layout(W->n_out, W->k_in, &L) || !al16(W->base) || !al16(out))
        return fail(LSN_EINVAL, "nf4_dequant: bad view or alignment");
    const uint8_t* b = static_cast<const uint8_t*>(W->base);
    Nf4Dev d;
    d.codes = b + L.codes;
    d.absmax = b + L.absmax;
    d.scale = reinterpret_cast<const float*>(b + L.scale);
    d.offset = reinterpret_cast<const float*>(b + L.offset);
    d.n_out = W->n_out;
    d.k_in = W->k_in;
    return nf4_dequant_launch(d, out, static_cast<cudaStream_t>(stream));
}

int lora_nf4_fwd(const nf4_view* W, const uint16_t* X, int64_t M, const uint16_t* A, const uint16_t* B,
                 int r, float scale, const uint16_t* residual, uint16_t* Y, uint16_t* T_out, void* ws,
                 size_t ws_bytes, void* stream) {
    // A == B == NULL: the adapter is disabled; Y is the frozen linear alone
    const bool adapter = A || B;
    int rc = check_linear_fwd("lora_nf4_fwd", W, X, M, A, B, r, residual, Y, T_out, adapter);
    if (rc) return rc;
    const LinearShape s{M, W->n_out, W->k_in, r};
    if (ws_bytes < fwd_ws(s) || (fwd_ws(s) && !ws))
        return fail(LSN_ENOMEM, "lora_nf4_fwd: workspace %zu < %zu", ws_bytes, fwd_ws(s));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const FwdSplits f = fwd_splits(s);
    const int K = (int)s.K, N = (int)s.N, m = (int)M;

    // T = bf16(X A^T)
    if (adapter) {
        GemmPlan g;
        int mx = g.map(X, M, K, K, kBM);
        int ma = g.map(A, r, K, K, 64);
        g.problem(m, r, 64, A_KMAJOR, EPI_BF16, T_out, r, 1.0f, r, f.t);
        g.seg(mx, 0, B_TMA_K, ma, 0, 0, K);
        rc = g.launch(st, static_cast<float*>(ws), ws_bytes);
        if (rc) return rc;
    }
    // Y = bf16(X W^T + s T B^T [+ residual])
    {
        uint8_t* wsb = static_cast<uint8_t*>(ws) + partial_bytes(f.t, s.M, s.r);
        GemmPlan g;
        int mx = g.map(X, M, K, K, kBM);
        int wv = g.nf4(W->base, N, K);
        g.problem(m, N, bn_for(N), A_KMAJOR, EPI_BF16, Y, N, 1.0f, N, f.y, residual, N);
        g.seg(mx, 0, B_NF4_K, wv, 0, 0, K);
        if (adapter) g.seg_scaled(g.map(T_out, M, r, r, kBM), 0, B, r, N, r, scale);
        rc = g.launch(st, reinterpret_cast<float*>(wsb), ws_bytes - (wsb - static_cast<uint8_t*>(ws)));
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
    if (ws_bytes < bwd_ws(s) || !ws)
        return fail(LSN_ENOMEM, "lora_nf4_bwd: workspace %zu < %zu", ws_bytes, bwd_ws(s));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const BwdSplits b = bwd_splits(s);
    const int K = (int)s.K, N = (int)s.N, m = (int)M;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    uint16_t* dT = reinterpret_cast<uint16_t*>(wsb);
    size_t off = align256((size_t)M * r * 2);

    // dT = bf16(s dY B)
    {
        GemmPlan g;
        int my = g.map(dY, M, N, N, kBM);
        int mb = g.map(B, N, r, r, 64);
        g.problem(m, r, 64, A_KMAJOR, EPI_BF16, dT, r, scale, r, b.dt);
        g.seg(my, 0, B_TMA_MN, mb, 0, 0, N);
        rc = g.launch(st, reinterpret_cast<float*>(wsb + off), ws_bytes - off);
        if (rc) return rc;
        off += partial_bytes(b.dt, s.M, s.r);
    }
    // dB = s dY^T T ; dA^T = X^T dT ; dX (+)= dY W + dT A   (one grouped launch)
    {
        GemmPlan g;
        int my_mn = g.map(dY, M, N, N, 64);
        int mt_mn = g.map(T, M, r, r, 64);
        int mx_mn = g.map(X, M, K, K, 64);
        int mdt_mn = g.map(dT, M, r, r, 64);
        g.problem(N, r, 64, A_MNMAJOR, EPI_F32, dB, r, scale, r, b.db);
        g.seg(my_mn, 0, B_TMA_MN, mt_mn, 0, 0, m);
        g.problem(K, r, 64, A_MNMAJOR, EPI_F32_T, dA, K, 1.0f, r, b.da);
        g.seg(mx_mn, 0, B_TMA_MN, mdt_mn, 0, 0, m);
        if (dX) {
            int my = g.map(dY, M, N, N, kBM);
            int mdt = g.map(dT, M, r, r, kBM);
            int ma_mn = g.map(A, r, K, K, 64);
            int wv = g.nf4(W->base, N, K);
            g.problem(m, K, bn_for(K), A_KMAJOR, accumulate_dX ? EPI_F32_ACC : EPI_F32, dX, K, 1.0f, K, b.dx);
            g.seg(my, 0, B_NF4_MN, wv, 0, 0, N);
            g.seg(mdt, 0, B_TMA_MN, ma_mn, 0, 0, r, true);
        }
        rc = g.launch(st, reinterpret_cast<float*>(wsb + off), ws_bytes - off);
        if (rc) return rc;
    }
    return LSN_OK;
}

}  // extern "C"
