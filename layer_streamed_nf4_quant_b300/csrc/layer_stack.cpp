// layer_stack_step: the forward sweep, the loss and the reverse backward sweep over the
// synthetic decoder-layer stack, with every layer's packed weights coming through the
// two-slot stream pool (or from a resident device store).
//
// "Can You Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's Layer Streaming Explained":
//   section "How Soup's layer streaming actually works" -- one layer at a time in reusable
//   VRAM buffers, the next prefetched while the current computes, every layer read again in
//   the backward pass;
//   section "The gradient bug also reveals something important about AI benchmarks" -- the
//   streamed run must give the resident run's forward output and LoRA gradients.
// Both modes below enqueue the same kernels with the same arguments except the weight
// addresses, and no kernel's arithmetic depends on an address, so they agree bit for bit.
//
// Per layer (s = alpha / r, canonical projection order q, k, v, gate, up, o, down):
//   forward : h = rmsnorm(x); T_cat = h A_cat^T; [q|k|v|g|u] = h W_p^T + s T_p B_p^T;
//             a = silu(g) u; T_od = [q A_o^T | a A_d^T]; x' = x + [q|a][W_o|W_d]^T + s T_od [B_o|B_d]^T
//   backward: dT_od = s dx' [B_o|B_d]; dB_o,d; dA_o,d; [dq|da] = dx' [W_o|W_d] + dT_od [A_o;A_d];
//             dY_cat = [dq | dk | dv | dg | du]; dT_cat = s dY_p B_p; dB_p; dA_p;
//             dh = sum_p dY_p W_p + dT_cat A_cat;  dx = dx' + rmsnorm'(dh)
#include <string.h>

#include <algorithm>
#include <vector>

#include "lsn_internal.h"
#include "stack_kernels.h"
#include "tc_gemm.h"

using namespace lsn;

namespace {

inline size_t a256(size_t x) { return (x + 255) / 256 * 256; }

struct Dims {
    int L, D, dkv, F, r, M, Ncat;
    double norm_M;   // tokens the loss means are taken over (M, or a data-parallel batch's count)
    float s, eps, coef;
    int np[kNumProj];   // n_out per projection
    int kp[kNumProj];   // k_in per projection
    int coff[5];        // column offset of q, k, v, gate, up in the fused output
};

struct Buffers {
    std::vector<uint16_t*> x;    // L+1 (x[0] = caller's x0)
    std::vector<uint16_t*> h, y, a, tcat, tod;
    std::vector<float*> rstd;
    float* dx = nullptr;
    uint16_t* dx_bf = nullptr;
    uint16_t* dtod = nullptr;
    float* da = nullptr;   // dloss/da (fp32 [M x F]); dq goes straight into dY_cat as bf16
    uint16_t* dy = nullptr;
    uint16_t* dtcat = nullptr;
    float* dh = nullptr;
    float* kvpart = nullptr;
    float* xpart = nullptr;
    float* partial = nullptr;
    size_t partial_bytes = 0;
    // backward with decoded weights: one layer's W_o, W_down, then W_q..W_up, as bf16
    uint16_t* wdec = nullptr;
    // reference (adapter disabled) pass: residual stream ping-pong and per-layer scratch
    uint16_t* xr[2] = {nullptr, nullptr};
    uint16_t* hr = nullptr;
    float* rstdr = nullptr;
    uint16_t* yr = nullptr;
    uint16_t* ar = nullptr;
};

bool make_dims(const lsn_stack_desc* d, int64_t M, Dims* o) {
    if (!d || d->n_layers < 1 || d->d_model < 256 || d->d_model % 256 || d->d_kv < 256 || d->d_kv % 256 ||
        d->d_ff < 256 || d->d_ff % 256 || d->rank < 8 || d->rank > 64 || d->rank % 8 || M < 1 ||
        M > (1 << 24))
        return false;
    o->L = d->n_layers;
    o->D = d->d_model;
    o->dkv = d->d_kv;
    o->F = d->d_ff;
    o->r = d->rank;
    o->M = (int)M;
    o->norm_M = (double)M;
    o->Ncat = o->D + 2 * o->dkv + 2 * o->F;
    o->s = d->lora_alpha / (float)d->rank;
    o->eps = d->rms_eps;
    o->coef = d->kv_loss_coef;
    for (int p = 0; p < kNumProj; ++p) {
        int64_t n, k;
        proj_shape(d, p, &n, &k);
        o->np[p] = (int)n;
        o->kp[p] = (int)k;
    }
    o->coff[0] = 0;
    o->coff[1] = o->D;
    o->coff[2] = o->D + o->dkv;
    o->coff[3] = o->D + 2 * o->dkv;
    o->coff[4] = o->D + 2 * o->dkv + o->F;
    return true;
}

// The backward reads packed NF4 inside its GEMMs unless the caller asks for each layer's W to
// be decoded to bf16 scratch first (bwd_weights = 2).
bool dense_bwd(const Dims&, const lsn_step_opts& o) { return o.bwd_weights == 2; }

// bf16 elements of the decoded-weight scratch: the larger of [W_o, W_down] and [W_q .. W_up].
size_t wdec_elems(const Dims& d) {
    size_t od = (size_t)d.np[kO] * d.kp[kO] + (size_t)d.np[kDown] * d.kp[kDown], qu = 0;
    for (int p = 0; p < 5; ++p) qu += (size_t)d.np[p] * d.kp[p];
    return od > qu ? od : qu;
}

// Lays the activations and scratch out in ws (base == nullptr: only sizes).  Returns bytes.
// With recompute, only x_l is kept per layer; h, rstd, the projections, a and the T's live in
// one set of buffers that the reverse sweep refills by recomputing the layer.
size_t layout(const Dims& d, uint8_t* base, const uint16_t* x0, Buffers* b, size_t partial_bytes,
              const lsn_step_opts& o) {
    size_t off = 0;
    auto take = [&](size_t bytes) -> uint8_t* {
        uint8_t* p = base ? base + off : nullptr;
        off += a256(bytes);
        return p;
    };
    const size_t M = (size_t)d.M;
    b->x.assign(d.L + 1, nullptr);
    b->h.assign(d.L, nullptr);
    b->y.assign(d.L, nullptr);
    b->a.assign(d.L, nullptr);
    b->tcat.assign(d.L, nullptr);
    b->tod.assign(d.L, nullptr);
    b->rstd.assign(d.L, nullptr);
    b->x[0] = const_cast<uint16_t*>(x0);
    for (int l = 0; l < d.L; ++l) {
        b->x[l + 1] = reinterpret_cast<uint16_t*>(take(M * d.D * 2));
        if (o.recompute && l > 0) {
            b->h[l] = b->h[0];
            b->rstd[l] = b->rstd[0];
            b->y[l] = b->y[0];
            b->a[l] = b->a[0];
            b->tcat[l] = b->tcat[0];
            b->tod[l] = b->tod[0];
            continue;
        }
        b->h[l] = reinterpret_cast<uint16_t*>(take(M * d.D * 2));
        b->rstd[l] = reinterpret_cast<float*>(take(M * 4));
        b->y[l] = reinterpret_cast<uint16_t*>(take(M * d.Ncat * 2));
        b->a[l] = reinterpret_cast<uint16_t*>(take(M * d.F * 2));
        b->tcat[l] = reinterpret_cast<uint16_t*>(take(M * 5 * d.r * 2));
        b->tod[l] = reinterpret_cast<uint16_t*>(take(M * 2 * d.r * 2));
    }
    b->dx = reinterpret_cast<float*>(take(M * d.D * 4));
    b->dx_bf = reinterpret_cast<uint16_t*>(take(M * d.D * 2));
    b->dtod = reinterpret_cast<uint16_t*>(take(M * 2 * d.r * 2));
    b->da = reinterpret_cast<float*>(take(M * d.F * 4));
    b->dy = reinterpret_cast<uint16_t*>(take(M * d.Ncat * 2));
    b->dtcat = reinterpret_cast<uint16_t*>(take(M * 5 * d.r * 2));
    b->dh = reinterpret_cast<float*>(take(M * d.D * 4));
    b->kvpart = reinterpret_cast<float*>(take((size_t)d.L * kLossBlocks * 2 * 4));
    b->xpart = reinterpret_cast<float*>(take((size_t)kLossBlocks * 4));
    if (o.reference_pass) {
        b->xr[0] = reinterpret_cast<uint16_t*>(take(M * d.D * 2));
        b->xr[1] = reinterpret_cast<uint16_t*>(take(M * d.D * 2));
        b->hr = reinterpret_cast<uint16_t*>(take(M * d.D * 2));
        b->rstdr = reinterpret_cast<float*>(take(M * 4));
        b->yr = reinterpret_cast<uint16_t*>(take(M * d.Ncat * 2));
        b->ar = reinterpret_cast<uint16_t*>(take(M * d.F * 2));
    }
    if (dense_bwd(d, o)) b->wdec = reinterpret_cast<uint16_t*>(take(wdec_elems(d) * 2));
    b->partial = reinterpret_cast<float*>(take(partial_bytes));
    b->partial_bytes = partial_bytes;
    return off;
}

struct Ctx {
    Dims d;
    Buffers b;
    lsn_step_opts o{};
    cudaStream_t s = nullptr;
    bool dry = false;
    size_t partial_need = 0;
    size_t img_off[kNumProj];
    size_t img_bytes = 0;
    size_t la[kNumProj], lb[kNumProj];   // LoRA element offsets (A_p, B_p)
    // streamed mode: the layer being computed; need() makes the compute stream wait for a byte
    // range of its image (a no-op for a resident store, or when nothing is being computed)
    lsn_pool* pool = nullptr;
    int layer = -1;

    int need(size_t begin, size_t end) {
        if (dry || !pool || layer < 0) return LSN_OK;
        const void* p = nullptr;
        return stream_pool_wait_range(pool, layer, begin, end, s, &p, 0);
    }
    // the header and q, k, v, gate, up / o and down
    int need_qkvgu() { return need(0, img_off[kO]); }
    int need_od() { return need(img_off[kO], img_bytes); }

    int run(GemmPlan& g) {
        if (g.status()) return g.status();
        if (dry) {
            partial_need = std::max(partial_need, g.partial_bytes());
            return LSN_OK;
        }
        return g.launch(s, b.partial, b.partial_bytes);
    }
    const void* mat(const uint8_t* img, int p) const { return img ? img + img_off[p] : nullptr; }
    // decoded-weight scratch: bf16 matrix p of a group laid out from `first` on
    uint16_t* wd(int first, int p) const {
        if (!b.wdec) return nullptr;
        size_t off = 0;
        for (int q = first; q < p; ++q) off += (size_t)d.np[q] * d.kp[q];
        return b.wdec + off;
    }
    // decodes projections first .. last of the layer image into the scratch
    int decode(const uint8_t* img, int first, int last) {
        if (dry) return LSN_OK;
        Nf4Dev w[kNumProj];
        uint16_t* out[kNumProj];
        for (int p = first; p <= last; ++p) {
            const int rc = nf4_view_dev(mat(img, p), d.np[p], d.kp[p], &w[p - first]);
            if (rc) return rc;
            out[p - first] = wd(first, p);
        }
        return nf4_dequant_many(w, out, last - first + 1, s);
    }
    const uint16_t* A(const uint16_t* lo, int p) const { return lo ? lo + la[p] : nullptr; }
    const uint16_t* B(const uint16_t* lo, int p) const { return lo ? lo + lb[p] : nullptr; }
    float* dA(float* g, int p) const { return g ? g + la[p] : nullptr; }
    float* dB(float* g, int p) const { return g ? g + lb[p] : nullptr; }
};

#define RC(x)                    \
    do {                         \
        int rc_ = (x);           \
        if (rc_) return rc_;     \
    } while (0)

// --------------------------------------------------------------------------- forward

// recompute: the reverse sweep's refill of this layer's stored activations (the output x'
// and the loss terms are already known, so the O+down GEMM and the k/v sums are skipped).
int fwd_layer(Ctx& c, int l, const uint8_t* img, const uint16_t* lora, bool recompute = false) {
    const Dims& d = c.d;
    const Buffers& b = c.b;
    const int M = d.M, D = d.D, r = d.r;
    if (!c.dry) RC(launch_rmsnorm_fwd(b.x[l], b.h[l], b.rstd[l], M, D, d.eps, img, (uint32_t)l, c.s));
    {   // T_cat = bf16(h A_cat^T)
        GemmPlan g(c.dry);
        int mh = g.map(b.h[l], M, D, D, kBM);
        int ma = g.map(c.A(lora, kQ), 5 * r, D, D, 64);
        g.problem(M, 5 * r, 64, A_KMAJOR, EPI_BF16, b.tcat[l], 5 * r, 1.0f, 5 * r, kAutoSplits);
        g.seg(mh, 0, B_TMA_K, ma, 0, 0, D);
        RC(c.run(g));
    }
    {   // q, k, v, gate, up = bf16(h W_p^T + s T_p B_p^T)
        GemmPlan g(c.dry);
        int mh = g.map(b.h[l], M, D, D, kBM);
        int mt = g.map(b.tcat[l], M, 5 * r, 5 * r, kBM);
        for (int p = 0; p < 5; ++p) {
            int v = g.nf4(c.mat(img, p), d.np[p], D);
            g.problem(M, d.np[p], 256, A_KMAJOR, EPI_BF16, b.y[l] ? b.y[l] + d.coff[p] : nullptr, d.Ncat, 1.0f,
                      d.np[p], kAutoSplits);
            g.seg(mh, 0, B_NF4_K, v, 0, 0, D);
            g.seg_scaled(mt, p * r, c.B(lora, p), r, d.np[p], r, d.s);
        }
        RC(c.run(g));
    }
    if (!c.dry) RC(launch_silu_mul(b.y[l], d.Ncat, d.coff[3], d.coff[4], b.a[l], M, d.F, c.s));
    {   // T_o = bf16(q A_o^T), T_d = bf16(a A_d^T)
        GemmPlan g(c.dry);
        int mq = g.map(b.y[l], M, D, d.Ncat, kBM);
        int ma = g.map(b.a[l], M, d.F, d.F, kBM);
        int mao = g.map(c.A(lora, kO), r, D, D, 64);
        int mad = g.map(c.A(lora, kDown), r, d.F, d.F, 64);
        g.problem(M, r, 64, A_KMAJOR, EPI_BF16, b.tod[l], 2 * r, 1.0f, r, kAutoSplits);
        g.seg(mq, 0, B_TMA_K, mao, 0, 0, D);
        g.problem(M, r, 64, A_KMAJOR, EPI_BF16, b.tod[l] ? b.tod[l] + r : nullptr, 2 * r, 1.0f, r, kAutoSplits);
        g.seg(ma, 0, B_TMA_K, mad, 0, 0, d.F);
        RC(c.run(g));
    }
    if (recompute) return LSN_OK;
    RC(c.need_od());
    {   // x' = bf16(x + q W_o^T + a W_d^T + s T_o B_o^T + s T_d B_d^T)
        GemmPlan g(c.dry);
        int mq = g.map(b.y[l], M, D, d.Ncat, kBM);
        int ma = g.map(b.a[l], M, d.F, d.F, kBM);
        int mt = g.map(b.tod[l], M, 2 * r, 2 * r, kBM);
        int vo = g.nf4(c.mat(img, kO), D, D);
        int vd = g.nf4(c.mat(img, kDown), D, d.F);
        g.problem(M, D, 256, A_KMAJOR, EPI_BF16, b.x[l + 1], D, 1.0f, D, kAutoSplits, b.x[l], D);
        g.seg(mq, 0, B_NF4_K, vo, 0, 0, D);
        g.seg(ma, 0, B_NF4_K, vd, 0, 0, d.F);
        g.seg_scaled(mt, 0, c.B(lora, kO), r, D, r, d.s);
        g.seg_scaled(mt, r, c.B(lora, kDown), r, D, r, d.s);
        RC(c.run(g));
    }
    if (!c.dry)
        RC(launch_kv_sumsq(b.y[l], d.Ncat, d.coff[1], d.coff[2], d.dkv, M, b.kvpart + (size_t)l * kLossBlocks * 2, c.s));
    return LSN_OK;
}

// ------------------------------------------------------- reference (adapter disabled)

// The frozen base alone on the same streamed weights: the LoRA contraction steps are left
// out of the GEMMs (not multiplied by zero).  xin -> xout, scratch shared by all layers.
int ref_layer(Ctx& c, const uint8_t* img, const uint16_t* xin, uint16_t* xout) {
    const Dims& d = c.d;
    const Buffers& b = c.b;
    const int M = d.M, D = d.D;
    if (!c.dry) RC(launch_rmsnorm_fwd(xin, b.hr, b.rstdr, M, D, d.eps, nullptr, 0, c.s));
    {
        GemmPlan g(c.dry);
        int mh = g.map(b.hr, M, D, D, kBM);
        for (int p = 0; p < 5; ++p) {
            int v = g.nf4(c.mat(img, p), d.np[p], D);
            g.problem(M, d.np[p], 256, A_KMAJOR, EPI_BF16, b.yr ? b.yr + d.coff[p] : nullptr, d.Ncat, 1.0f, d.np[p],
                      kAutoSplits);
            g.seg(mh, 0, B_NF4_K, v, 0, 0, D);
        }
        RC(c.run(g));
    }
    if (!c.dry) RC(launch_silu_mul(b.yr, d.Ncat, d.coff[3], d.coff[4], b.ar, M, d.F, c.s));
    {
        GemmPlan g(c.dry);
        int mq = g.map(b.yr, M, D, d.Ncat, kBM);
        int ma = g.map(b.ar, M, d.F, d.F, kBM);
        int vo = g.nf4(c.mat(img, kO), D, D);
        int vd = g.nf4(c.mat(img, kDown), D, d.F);
        g.problem(M, D, 256, A_KMAJOR, EPI_BF16, xout, D, 1.0f, D, kAutoSplits, xin, D);
        g.seg(mq, 0, B_NF4_K, vo, 0, 0, D);
        g.seg(ma, 0, B_NF4_K, vd, 0, 0, d.F);
        RC(c.run(g));
    }
    return LSN_OK;
}

// -------------------------------------------------------------------------- backward

int bwd_layer(Ctx& c, int l, const uint8_t* img, const uint16_t* lora, float* grad) {
    const Dims& d = c.d;
    const Buffers& b = c.b;
    const int M = d.M, D = d.D, F = d.F, r = d.r;
    RC(c.need_od());
    {   // dT_o = bf16(s dx' B_o), dT_d = bf16(s dx' B_d)
        GemmPlan g(c.dry);
        int mdx = g.map(b.dx_bf, M, D, D, kBM);
        int mbo = g.map(c.B(lora, kO), D, r, r, 64);
        int mbd = g.map(c.B(lora, kDown), D, r, r, 64);
        const int sp = kAutoSplits;
        g.problem(M, r, 64, A_KMAJOR, EPI_BF16, b.dtod, 2 * r, d.s, r, sp);
        g.seg(mdx, 0, B_TMA_MN, mbo, 0, 0, D);
        g.problem(M, r, 64, A_KMAJOR, EPI_BF16, b.dtod ? b.dtod + r : nullptr, 2 * r, d.s, r, sp);
        g.seg(mdx, 0, B_TMA_MN, mbd, 0, 0, D);
        RC(c.run(g));
    }
    const bool dense = dense_bwd(c.d, c.o);
    if (dense) RC(c.decode(img, kO, kDown));
    {   // dB_o, dB_d, dA_o, dA_d and [dq | da] = dx' [W_o | W_d] + dT_od [A_o ; A_d]
        GemmPlan g(c.dry);
        int mdx_mn = g.map(b.dx_bf, M, D, D, 64);
        int mtod_mn = g.map(b.tod[l], M, 2 * r, 2 * r, 64);
        int mq_mn = g.map(b.y[l], M, D, d.Ncat, 64);
        int ma_mn = g.map(b.a[l], M, F, F, 64);
        int mdtod_mn = g.map(b.dtod, M, 2 * r, 2 * r, 64);
        int mdx = g.map(b.dx_bf, M, D, D, kBM);
        int mdtod = g.map(b.dtod, M, 2 * r, 2 * r, kBM);
        int mao = g.map(c.A(lora, kO), r, D, D, 64);
        int mad = g.map(c.A(lora, kDown), r, F, F, 64);
        // W_o, W_down: packed NF4 decoded by the GEMM, or the bf16 copies decoded above
        const int bsrc = dense ? B_TMA_MN : B_NF4_MN;
        const int vo = dense ? g.map(c.wd(kO, kO), D, D, D, 64) : g.nf4(c.mat(img, kO), D, D);
        const int vd = dense ? g.map(c.wd(kO, kDown), D, F, F, 64) : g.nf4(c.mat(img, kDown), D, F);
        const int ws = kAutoSplits, xs = kAutoSplits;
        g.problem(D, r, 64, A_MNMAJOR, EPI_F32, c.dB(grad, kO), r, d.s, r, ws);
        g.seg(mdx_mn, 0, B_TMA_MN, mtod_mn, 0, 0, M);
        g.problem(D, r, 64, A_MNMAJOR, EPI_F32, c.dB(grad, kDown), r, d.s, r, ws);
        g.seg(mdx_mn, 0, B_TMA_MN, mtod_mn, 0, r, M);
        g.problem(D, r, 64, A_MNMAJOR, EPI_F32_T, c.dA(grad, kO), D, 1.0f, r, ws);
        g.seg(mq_mn, 0, B_TMA_MN, mdtod_mn, 0, 0, M);
        g.problem(F, r, 64, A_MNMAJOR, EPI_F32_T, c.dA(grad, kDown), F, 1.0f, r, ws);
        g.seg(ma_mn, 0, B_TMA_MN, mdtod_mn, 0, r, M);
        // dq: only its bf16 rounding is used (as dY_q), so it is written into dY_cat directly
        g.problem(M, D, 256, A_KMAJOR, EPI_BF16, b.dy, d.Ncat, 1.0f, D, xs);
        g.seg(mdx, 0, bsrc, vo, 0, 0, D);
        g.seg(mdtod, 0, B_TMA_MN, mao, 0, 0, r, true);
        g.problem(M, F, 256, A_KMAJOR, EPI_F32, b.da, F, 1.0f, F, xs);
        g.seg(mdx, 0, bsrc, vd, 0, 0, D);
        g.seg(mdtod, r, B_TMA_MN, mad, 0, 0, r, true);
        RC(c.run(g));
    }
    if (!c.dry)
        RC(launch_dy_build(b.da, b.y[l], b.dy, M, D, d.dkv, F, (float)(2.0 * d.coef / (d.norm_M * d.dkv)), c.s));
    RC(c.need_qkvgu());
    if (!c.dry) RC(launch_tag_check(img, (uint32_t)l, c.s));
    if (dense) RC(c.decode(img, kQ, kUp));
    {   // dT_p = bf16(s dY_p B_p)
        GemmPlan g(c.dry);
        int mdy = g.map(b.dy, M, d.Ncat, d.Ncat, kBM);
        for (int p = 0; p < 5; ++p) {
            int mb = g.map(c.B(lora, p), d.np[p], r, r, 64);
            g.problem(M, r, 64, A_KMAJOR, EPI_BF16, b.dtcat ? b.dtcat + p * r : nullptr, 5 * r, d.s, r, kAutoSplits);
            g.seg(mdy, d.coff[p], B_TMA_MN, mb, 0, 0, d.np[p]);
        }
        RC(c.run(g));
    }
    {   // dB_p, dA_p and dh = sum_p dY_p W_p + dT_cat A_cat
        GemmPlan g(c.dry);
        int mdyp[5];
        for (int p = 0; p < 5; ++p) mdyp[p] = g.map(b.dy ? b.dy + d.coff[p] : nullptr, M, d.np[p], d.Ncat, 64);
        int mtcat_mn = g.map(b.tcat[l], M, 5 * r, 5 * r, 64);
        int mh_mn = g.map(b.h[l], M, D, D, 64);
        int mdtcat_mn = g.map(b.dtcat, M, 5 * r, 5 * r, 64);
        int mdy = g.map(b.dy, M, d.Ncat, d.Ncat, kBM);
        int mdtcat = g.map(b.dtcat, M, 5 * r, 5 * r, kBM);
        int macat = g.map(c.A(lora, kQ), 5 * r, D, D, 64);
        const int ws = kAutoSplits;
        for (int p = 0; p < 5; ++p) {
            g.problem(d.np[p], r, 64, A_MNMAJOR, EPI_F32, c.dB(grad, p), r, d.s, r, ws);
            g.seg(mdyp[p], 0, B_TMA_MN, mtcat_mn, 0, p * r, M);
        }
        for (int p = 0; p < 5; ++p) {
            g.problem(D, r, 64, A_MNMAJOR, EPI_F32_T, c.dA(grad, p), D, 1.0f, r, ws);
            g.seg(mh_mn, 0, B_TMA_MN, mdtcat_mn, 0, p * r, M);
        }
        g.problem(M, D, 256, A_KMAJOR, EPI_F32, b.dh, D, 1.0f, D, kAutoSplits);
        for (int p = 0; p < 5; ++p) {
            const int v = dense ? g.map(c.wd(kQ, p), d.np[p], D, D, 64) : g.nf4(c.mat(img, p), d.np[p], D);
            g.seg(mdy, d.coff[p], dense ? B_TMA_MN : B_NF4_MN, v, 0, 0, d.np[p]);
        }
        g.seg(mdtcat, 0, B_TMA_MN, macat, 0, 0, 5 * r, true);
        RC(c.run(g));
    }
    if (!c.dry) RC(launch_rmsnorm_bwd(b.x[l], b.rstd[l], b.dh, b.dx, b.dx_bf, M, D, c.s));
    return LSN_OK;
}

int init_ctx(Ctx& c, const lsn_stack_desc* desc, int64_t M) {
    if (!make_dims(desc, M, &c.d)) return fail(LSN_EINVAL, "layer stack: bad descriptor or M");
    RC(lsn_layer_image_offsets(desc, c.img_off));
    c.img_bytes = lsn_layer_image_bytes(desc);
    size_t lo[2 * kNumProj];
    RC(lsn_lora_offsets(desc, lo));
    for (int p = 0; p < kNumProj; ++p) {
        c.la[p] = lo[p];
        c.lb[p] = lo[kNumProj + p];
    }
    return LSN_OK;
}

size_t partial_need(const lsn_stack_desc* desc, int64_t M, const lsn_step_opts& o) {
    Ctx c;
    if (init_ctx(c, desc, M)) return 0;
    c.dry = true;
    c.o = o;
    layout(c.d, nullptr, nullptr, &c.b, 0, o);
    if (fwd_layer(c, 0, nullptr, nullptr) || bwd_layer(c, 0, nullptr, nullptr, nullptr)) return 0;
    if (o.reference_pass && ref_layer(c, nullptr, nullptr, nullptr)) return 0;
    return c.partial_need;
}

lsn_step_opts opts_or_default(const lsn_step_opts* o) {
    lsn_step_opts d{};
    return o ? *o : d;
}

}  // namespace

extern "C" {

size_t lsn_stack_workspace_bytes_ex(const lsn_stack_desc* desc, int64_t M, const lsn_step_opts* opts) {
    Ctx c;
    if (init_ctx(c, desc, M)) return 0;
    const lsn_step_opts o = opts_or_default(opts);
    Buffers b;
    return layout(c.d, nullptr, nullptr, &b, partial_need(desc, M, o), o) + 256;
}

int lsn_sum_ranks(const float* in, int n_ranks, size_t n, float* out, void* stream) {
    if (!in || !out || n_ranks < 1 || (reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return fail(LSN_EINVAL, "lsn_sum_ranks: NULL or misaligned buffer, or no rank");
    if (out != in && out < in + (size_t)n_ranks * n && in < out + n)
        return fail(LSN_EINVAL, "lsn_sum_ranks: out overlaps in other than as in[0]");
    return launch_sum_ranks(in, n_ranks, (int64_t)n, out, static_cast<cudaStream_t>(stream));
}

size_t lsn_stack_workspace_bytes(const lsn_stack_desc* desc, int64_t M) {
    return lsn_stack_workspace_bytes_ex(desc, M, nullptr);
}

int layer_stack_step_ex(lsn_pool* pool, const void* resident_store, const lsn_stack_desc* desc,
                        const lsn_step_opts* opts, const uint16_t* x0, int64_t M, const uint16_t* const* lora,
                        float* const* grads, float* loss_out, uint16_t* x_out, uint16_t* x_ref_out, float* dx0,
                        void* ws, size_t ws_bytes, void* stream) {
    Ctx c;
    RC(init_ctx(c, desc, M));
    c.o = opts_or_default(opts);
    if (!x0 || !lora || !grads || !loss_out || !ws || (!pool && !resident_store))
        return fail(LSN_EINVAL, "layer_stack_step: NULL argument");
    if (c.o.token_count < 0 || (c.o.token_count > 0 && c.o.token_count < M))
        return fail(LSN_EINVAL, "layer_stack_step: token_count must be 0 or at least M");
    if (c.o.token_count > 0) c.d.norm_M = (double)c.o.token_count;
    if (c.o.bwd_weights < 0 || c.o.bwd_weights > 2)
        return fail(LSN_EINVAL, "layer_stack_step: bwd_weights must be 0, 1 or 2");
    if (c.o.adamw && c.o.grads_ready)
        return fail(LSN_EINVAL, "layer_stack_step: AdamW inside the step cannot follow a gradient hook "
                                "(the hook's exchange must finish first; run lsn_adamw_step after it)");
    if ((reinterpret_cast<uintptr_t>(ws) & 255) || (reinterpret_cast<uintptr_t>(x0) & 15))
        return fail(LSN_EINVAL, "layer_stack_step: ws must be 256-byte and x0 16-byte aligned");
    for (int l = 0; l < c.d.L; ++l)
        if (!lora[l] || !grads[l] || (reinterpret_cast<uintptr_t>(lora[l]) & 15) ||
            (reinterpret_cast<uintptr_t>(grads[l]) & 15))
            return fail(LSN_EINVAL, "layer_stack_step: LoRA / grad blob %d missing or misaligned", l);
    if (c.o.adamw) {
        const lsn_adamw_state* st = c.o.adamw;
        if (!st->master || !st->m || !st->v || !st->lora_out || st->hp.step < 1)
            return fail(LSN_EINVAL, "layer_stack_step: incomplete AdamW state");
        for (int l = 0; l < c.d.L; ++l)
            if (!st->master[l] || !st->m[l] || !st->v[l] || !st->lora_out[l])
                return fail(LSN_EINVAL, "layer_stack_step: AdamW state of layer %d missing", l);
    }
    const size_t pneed = partial_need(desc, M, c.o);
    const size_t need = layout(c.d, nullptr, nullptr, &c.b, pneed, c.o);
    if (ws_bytes < need) return fail(LSN_ENOMEM, "layer_stack_step: workspace %zu < %zu", ws_bytes, need);
    layout(c.d, static_cast<uint8_t*>(ws), x0, &c.b, pneed, c.o);
    c.s = static_cast<cudaStream_t>(stream);
    const size_t img_bytes = c.img_bytes;
    const uint8_t* res = static_cast<const uint8_t*>(resident_store);
    const int L = c.d.L;
    c.pool = pool;
    // the layer's image address; streamed, the compute stream first waits for the part of it
    // the layer's first GEMMs read (the rest is waited for by Ctx::need before its GEMMs)
    auto image = [&](int l, bool od_first, const uint8_t** img) -> int {
        c.layer = l;
        if (!pool) {
            *img = res + (size_t)l * img_bytes;
            return LSN_OK;
        }
        const void* p = nullptr;
        int rc = od_first ? stream_pool_wait_range(pool, l, c.img_off[kO], img_bytes, stream, &p, 0)
                          : stream_pool_wait_range(pool, l, 0, c.img_off[kO], stream, &p, 0);
        *img = static_cast<const uint8_t*>(p);
        return rc;
    };

    // forward sweep, prefetching one layer ahead; the reference pass (if any) runs on the
    // same slot before it is released, so it costs no extra copy
    if (pool) RC(stream_pool_prefetch_ex(pool, 0, 0));
    const uint16_t* xr_in = x0;
    for (int l = 0; l < L; ++l) {
        if (pool && l + 1 < L) RC(stream_pool_prefetch_ex(pool, l + 1, 0));
        const uint8_t* img;
        RC(image(l, false, &img));
        RC(fwd_layer(c, l, img, lora[l]));
        if (c.o.reference_pass) {
            uint16_t* xr_out = c.b.xr[l & 1];
            RC(ref_layer(c, img, xr_in, xr_out));
            xr_in = xr_out;
        }
        if (pool) RC(stream_pool_release(pool, l, stream));
    }
    const size_t act = (size_t)c.d.M * c.d.D;
    if (c.o.x_layers_out)
        for (int l = 0; l < L; ++l)
            LSN_CUDA_TRY(cudaMemcpyAsync(c.o.x_layers_out + (size_t)l * act, c.b.x[l + 1], act * 2,
                                         cudaMemcpyDeviceToDevice, c.s));
    RC(launch_loss(c.b.x[L], c.d.M, c.d.norm_M, c.d.D, c.d.dkv, L, c.d.coef, c.b.dx, c.b.dx_bf, c.b.xpart, c.b.kvpart,
                   loss_out, c.s));
    // reverse sweep, re-streaming every layer (and recomputing its activations if asked); the
    // backward of a layer starts with o and down, so those are copied first -- unless the
    // layer is recomputed, which starts with q..up
    c.layer = -1;
    const int rev = c.o.recompute ? 0 : 1;
    if (pool) RC(stream_pool_prefetch_ex(pool, L - 1, rev));
    for (int l = L - 1; l >= 0; --l) {
        if (pool && l - 1 >= 0) RC(stream_pool_prefetch_ex(pool, l - 1, rev));
        const uint8_t* img;
        RC(image(l, rev != 0, &img));
        if (c.o.recompute) RC(fwd_layer(c, l, img, lora[l], true));
        RC(bwd_layer(c, l, img, lora[l], grads[l]));
        if (c.o.grads_ready) c.o.grads_ready(c.o.hook_user, l, grads[l], lsn_lora_elems(desc), stream);
        if (c.o.dx_layers_out)
            LSN_CUDA_TRY(cudaMemcpyAsync(c.o.dx_layers_out + (size_t)l * act, c.b.dx, act * 4,
                                         cudaMemcpyDeviceToDevice, c.s));
        if (c.o.adamw) {
            const lsn_adamw_state* st = c.o.adamw;
            RC(launch_adamw(st->hp, st->master[l], st->lora_out[l], grads[l], st->m[l], st->v[l],
                            (int64_t)lsn_lora_elems(desc), c.s));
        }
        if (pool) RC(stream_pool_release(pool, l, stream));
    }
    c.layer = -1;
    if (x_out)
        LSN_CUDA_TRY(cudaMemcpyAsync(x_out, c.b.x[L], (size_t)c.d.M * c.d.D * 2, cudaMemcpyDeviceToDevice, c.s));
    if (x_ref_out && c.o.reference_pass)
        LSN_CUDA_TRY(cudaMemcpyAsync(x_ref_out, xr_in, (size_t)c.d.M * c.d.D * 2, cudaMemcpyDeviceToDevice, c.s));
    if (dx0) LSN_CUDA_TRY(cudaMemcpyAsync(dx0, c.b.dx, (size_t)c.d.M * c.d.D * 4, cudaMemcpyDeviceToDevice, c.s));
    return LSN_OK;
}

int layer_stack_step(lsn_pool* pool, const void* resident_store, const lsn_stack_desc* desc, const uint16_t* x0,
                     int64_t M, const uint16_t* const* lora, float* const* grads, float* loss_out, uint16_t* x_out,
                     float* dx0, void* ws, size_t ws_bytes, void* stream) {
    return layer_stack_step_ex(pool, resident_store, desc, nullptr, x0, M, lora, grads, loss_out, x_out, nullptr, dx0,
                               ws, ws_bytes, stream);
}

}  // extern "C"
