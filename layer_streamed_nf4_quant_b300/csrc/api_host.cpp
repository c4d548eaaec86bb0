// Host side of the library: error reporting, the NF4 codebook, the host quantiser
// (nf4_pack), layer images and LoRA blob layouts.
//
// NF4: "Can You Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's Layer Streaming Explained",
// section "Why NF4 matters so much" (QLoRA's 4-bit format for the frozen base); packing as
// the workload description fixes it (64-weight blocks, uint8 absmax codes, fp32 scale and
// offset per 256 blocks).  Every decision below is an IEEE fp64 or fp32 operation in a
// stated order, so the bytes do not depend on the thread count or the machine.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <thread>
#include <vector>

#include "lsn_internal.h"

namespace lsn {

static thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(LSN_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

static std::mutex g_dev_mu;
static uint32_t* g_dev_err[64] = {nullptr};

uint32_t* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        fail(LSN_ECUDA, "cudaGetDevice failed");
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_err[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaMalloc(&p, 64);
        if (e != cudaSuccess) {
            cuda_fail(e, "cudaMalloc(device error word)");
            return nullptr;
        }
        e = cudaMemset(p, 0, 64);
        if (e != cudaSuccess) {
            cuda_fail(e, "cudaMemset(device error word)");
            return nullptr;
        }
        g_dev_err[dev] = static_cast<uint32_t*>(p);
    }
    return g_dev_err[dev];
}

// ------------------------------------------------------------------- launch accounting

static std::atomic<uint64_t> g_launches(0);
static std::atomic<bool> g_profiling(false);

struct ProfEvent {
    cudaEvent_t start, end;
    double flops;
};
static std::mutex g_prof_mu;
static std::vector<ProfEvent> g_prof_pending, g_prof_spare;
static uint64_t g_prof_launches = 0;
static double g_prof_ms = 0.0, g_prof_flops = 0.0;

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
bool profiling() { return g_profiling.load(std::memory_order_relaxed); }

void* profile_begin(cudaStream_t s) {
    if (!profiling()) return nullptr;
    ProfEvent* e = new (std::nothrow) ProfEvent();
    if (!e) return nullptr;
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        if (!g_prof_spare.empty()) {
            *e = g_prof_spare.back();
            g_prof_spare.pop_back();
        } else if (cudaEventCreate(&e->start) != cudaSuccess || cudaEventCreate(&e->end) != cudaSuccess) {
            delete e;
            return nullptr;
        }
    }
    if (cudaEventRecord(e->start, s) != cudaSuccess) {
        delete e;
        return nullptr;
    }
    return e;
}

void profile_end(void* token, cudaStream_t s, double flops) {
    if (!token) return;
    ProfEvent* e = static_cast<ProfEvent*>(token);
    e->flops = flops;
    cudaEventRecord(e->end, s);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_pending.push_back(*e);
    delete e;
}

// ------------------------------------------------------------------------- codebook
// Standard-normal upper quantile by Newton's method on the complementary error function:
// solve 0.5*erfc(x/sqrt(2)) = 1 - p for x, starting from the Abramowitz-Stegun 26.2.23
// rational approximation.  p in (0.5, 1).
static double normal_quantile_upper(double p) {
    const double q = 1.0 - p;                 // exact for p in [0.5, 1]
    const double t = sqrt(-2.0 * log(q));
    double x = t - (2.515517 + 0.802853 * t + 0.010328 * t * t) /
                       (1.0 + 1.432788 * t + 0.189269 * t * t + 0.001308 * t * t * t);
    const double inv_sqrt2 = 0.70710678118654752440;
    const double inv_sqrt2pi = 0.39894228040143267794;
    for (int it = 0; it < 100; ++it) {
        double tail = 0.5 * erfc(x * inv_sqrt2);
        double pdf = inv_sqrt2pi * exp(-0.5 * x * x);
        double dx = (tail - q) / pdf;
        x += dx;
        if (fabs(dx) <= 1e-17 * fabs(x)) break;
    }
    return x;
}

static float g_levels[16];
static std::once_flag g_levels_once;

static void build_levels() {
    // QLoRA's asymmetric NormalFloat: 8 positive levels at probabilities delta + i*step,
    // step = (1/2 - delta)/8, i = 0..7; 7 negative levels at delta + j*step', step' =
    // (1/2 - delta)/7, j = 0..6; an exact zero; all divided by the quantile of delta.
    const double delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0);
    const double zmax = normal_quantile_upper(delta);
    double lv[16];
    int n = 0;
    const double sn = (0.5 - delta) / 7.0;
    for (int j = 0; j < 7; ++j) {
        double p = (double)j * sn + delta;
        lv[n++] = -normal_quantile_upper(p) / zmax;
    }
    lv[n++] = 0.0;
    const double sp = (0.5 - delta) / 8.0;
    for (int i = 7; i >= 0; --i) {
        double p = (double)i * sp + delta;
        lv[n++] = normal_quantile_upper(p) / zmax;
    }
    for (int i = 0; i < 16; ++i) g_levels[i] = (float)lv[i];
}

const float* nf4_levels() {
    std::call_once(g_levels_once, build_levels);
    return g_levels;
}

// --------------------------------------------------------------------------- layout

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool nf4_layout(int64_t n_out, int64_t k_in, Nf4Layout* o) {
    if (n_out < 1 || k_in < 64 || k_in % 64 != 0) return false;
    const int64_t nw = n_out * k_in;
    o->blocks = nw / 64;
    o->groups = (o->blocks + 255) / 256;
    o->codes = 0;
    o->absmax = align_up((size_t)(nw / 2), 16);
    o->scale = o->absmax + align_up((size_t)o->blocks, 16);
    o->offset = o->scale + align_up((size_t)(4 * o->groups), 16);
    o->total = o->offset + align_up((size_t)(4 * o->groups), 16);
    return true;
}

void proj_shape(const lsn_stack_desc* d, int p, int64_t* n, int64_t* k) {
    switch (p) {
        case kQ: *n = d->d_model; *k = d->d_model; break;
        case kK: case kV: *n = d->d_kv; *k = d->d_model; break;
        case kGate: case kUp: *n = d->d_ff; *k = d->d_model; break;
        case kO: *n = d->d_model; *k = d->d_model; break;
        default: *n = d->d_model; *k = d->d_ff; break;   // down
    }
}

// ------------------------------------------------------------------------ quantiser

static inline float round_up_f32(double x) {
    float f = (float)x;
    if ((double)f < x) f = nextafterf(f, INFINITY);
    return f;
}

// a' = fp32(fp32(q*scale) + lo).  q*scale is exact in fp64; each rounding to fp32 is the
// correctly rounded fp32 operation.
static inline float deq_absmax(int q, float scale, float lo) {
    float t = (float)((double)q * (double)scale);
    return (float)((double)t + (double)lo);
}

template <class F>
static void parallel_for(int64_t n, int n_threads, F&& f) {
    if (n <= 0) return;
    int t = n_threads > 0 ? n_threads : (int)std::max(1u, std::thread::hardware_concurrency());
    t = (int)std::min<int64_t>(t, n);
    if (t <= 1) {
        f(0, n);
        return;
    }
    std::vector<std::thread> th;
    int64_t chunk = (n + t - 1) / t;
    for (int i = 0; i < t; ++i) {
        int64_t b = i * chunk, e = std::min(n, b + chunk);
        if (b >= e) break;
        th.emplace_back([&f, b, e] { f(b, e); });
    }
    for (auto& x : th) x.join();
}

static int pack_matrix(const float* W, int64_t n_out, int64_t k_in, uint8_t* dst, int n_threads) {
    Nf4Layout L;
    nf4_layout(n_out, k_in, &L);
    const int64_t nb = L.blocks, G = L.groups;
    std::vector<float> absmax(nb), aq(nb);
    std::vector<uint8_t> qcode(nb);
    std::atomic<bool> nonfinite(false);

    parallel_for(nb, n_threads, [&](int64_t b0, int64_t b1) {
        for (int64_t b = b0; b < b1; ++b) {
            const float* w = W + b * 64;
            float m = 0.f;
            bool bad = false;
            for (int i = 0; i < 64; ++i) {
                float a = fabsf(w[i]);
                if (!(a <= 3.4028234663852886e38f)) bad = true;   // NaN or Inf
                m = a > m ? a : m;
            }
            if (bad) nonfinite.store(true, std::memory_order_relaxed);
            absmax[b] = m;
        }
    });
    if (nonfinite.load()) return fail(LSN_EINVAL, "nf4_pack: W holds NaN or Inf");

    std::vector<float> scale(G), offset(G);
    parallel_for(G, n_threads, [&](int64_t g0, int64_t g1) {
        for (int64_t g = g0; g < g1; ++g) {
            const int64_t b0 = g * 256, b1 = std::min(nb, b0 + 256);
            float lo = absmax[b0], hi = absmax[b0];
            for (int64_t b = b0; b < b1; ++b) {
                lo = std::min(lo, absmax[b]);
                hi = std::max(hi, absmax[b]);
            }
            float s = round_up_f32(((double)hi - (double)lo) / 255.0);
            for (;;) {
                bool short_any = false;
                for (int64_t b = b0; b < b1; ++b) {
                    int q = 0;
                    if (s > 0.f) {
                        double v = ceil(((double)absmax[b] - (double)lo) / (double)s);
                        q = v < 0.0 ? 0 : (v > 255.0 ? 255 : (int)v);
                    }
                    float ap = deq_absmax(q, s, lo);
                    while (ap < absmax[b] && q < 255) {
                        ++q;
                        ap = deq_absmax(q, s, lo);
                    }
                    if (ap < absmax[b]) short_any = true;
                    qcode[b] = (uint8_t)q;
                    aq[b] = ap;
                }
                if (!short_any) break;
                s = nextafterf(s, INFINITY);
            }
            scale[g] = s;
            offset[g] = lo;
        }
    });

    // Nearest level of n = w / a' by counting the fp64 midpoints strictly below n.
    const float* c = nf4_levels();
    double mid[15];
    for (int i = 0; i < 15; ++i) mid[i] = ((double)c[i] + (double)c[i + 1]) / 2.0;
    parallel_for(nb, n_threads, [&](int64_t b0, int64_t b1) {
        for (int64_t b = b0; b < b1; ++b) {
            const float* w = W + b * 64;
            const double a = (double)aq[b];
            uint8_t* out = dst + L.codes + b * 32;
            for (int i = 0; i < 64; i += 2) {
                uint8_t code[2];
                for (int j = 0; j < 2; ++j) {
                    double n = a == 0.0 ? 0.0 : (double)w[i + j] / a;
                    int k = 0;
                    for (int m = 0; m < 15; ++m) k += (mid[m] < n) ? 1 : 0;
                    code[j] = (uint8_t)k;
                }
                out[i / 2] = (uint8_t)((code[0] << 4) | code[1]);
            }
        }
    });
    memcpy(dst + L.absmax, qcode.data(), (size_t)nb);
    memset(dst + L.absmax + nb, 0, L.scale - L.absmax - (size_t)nb);
    memcpy(dst + L.scale, scale.data(), 4 * (size_t)G);
    memset(dst + L.scale + 4 * G, 0, L.offset - L.scale - 4 * (size_t)G);
    memcpy(dst + L.offset, offset.data(), 4 * (size_t)G);
    memset(dst + L.offset + 4 * G, 0, L.total - L.offset - 4 * (size_t)G);
    return LSN_OK;
}

static bool desc_ok(const lsn_stack_desc* d) {
    return d && d->n_layers >= 1 && d->d_model >= 64 && d->d_model % 256 == 0 && d->d_kv >= 64 &&
           d->d_kv % 256 == 0 && d->d_ff >= 64 && d->d_ff % 256 == 0 && d->rank >= 8 &&
           d->rank <= 64 && d->rank % 8 == 0;
}

static void image_offsets(const lsn_stack_desc* d, size_t off[kNumProj], size_t* total) {
    size_t cur = 256;
    for (int p = 0; p < kNumProj; ++p) {
        int64_t n, k;
        proj_shape(d, p, &n, &k);
        Nf4Layout L;
        nf4_layout(n, k, &L);
        off[p] = cur;
        cur = align_up(cur + L.total, 256);
    }
    *total = cur;
}

}  // namespace lsn

using namespace lsn;

extern "C" {

const char* lsn_last_error(void) { return g_err; }

int lsn_abi_version(void) { return 4; }

uint64_t lsn_launch_count(void) { return g_launches.load(); }

int lsn_profile_enable(int on) {
    g_profiling.store(on != 0);
    return LSN_OK;
}

int lsn_profile_read(lsn_profile* out, int reset) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto& e : g_prof_pending) {
        cudaError_t r = cudaEventSynchronize(e.end);
        if (r != cudaSuccess) return cuda_fail(r, "lsn_profile_read: cudaEventSynchronize");
        float ms = 0.f;
        r = cudaEventElapsedTime(&ms, e.start, e.end);
        if (r != cudaSuccess) return cuda_fail(r, "lsn_profile_read: cudaEventElapsedTime");
        g_prof_ms += ms;
        g_prof_flops += e.flops;
        g_prof_launches += 1;
        g_prof_spare.push_back(e);
    }
    g_prof_pending.clear();
    if (out) {
        out->gemm_launches = g_prof_launches;
        out->gemm_ms = g_prof_ms;
        out->gemm_flops = g_prof_flops;
    }
    if (reset) {
        g_prof_launches = 0;
        g_prof_ms = 0.0;
        g_prof_flops = 0.0;
    }
    return LSN_OK;
}

int lsn_check(void* stream, uint32_t* detail) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t* w = device_error_word();
    if (!w) return LSN_ECUDA;
    uint32_t v = 0;
    LSN_CUDA_TRY(cudaMemcpy(&v, w, 4, cudaMemcpyDeviceToHost));
    if (v) LSN_CUDA_TRY(cudaMemset(w, 0, 4));
    // the static-scratch entry point keeps its own word: collect it here as well
    uint32_t vs = 0;
    int rc = static_error_take(&vs);
    if (rc) return rc;
    if (!v) v = vs;
    if (detail) *detail = v;
    if (v == 0) return LSN_OK;
    uint32_t kind = v >> 24;
    if (kind == kDevErrTag)
        return fail(LSN_ECORRUPT, "layer image tag mismatch (expected layer %u)", v & 0xFFFFFFu);
    return fail(LSN_ETIMEOUT, "device bounded wait ran out (site %u)", v & 0xFFFFFFu);
}

int lsn_nf4_codebook(float* out) {
    if (!out) return fail(LSN_EINVAL, "lsn_nf4_codebook: out is NULL");
    memcpy(out, nf4_levels(), 16 * sizeof(float));
    return LSN_OK;
}

size_t nf4_packed_bytes(int64_t n_out, int64_t k_in) {
    Nf4Layout L;
    return nf4_layout(n_out, k_in, &L) ? L.total : 0;
}

int nf4_pack(const float* W, int64_t n_out, int64_t k_in, void* dst, size_t dst_bytes,
             int n_threads) {
    Nf4Layout L;
    if (!W || !dst) return fail(LSN_EINVAL, "nf4_pack: NULL pointer");
    if (!nf4_layout(n_out, k_in, &L))
        return fail(LSN_EINVAL, "nf4_pack: need n_out >= 1 and k_in a positive multiple of 64");
    if (dst_bytes < L.total)
        return fail(LSN_EINVAL, "nf4_pack: dst_bytes %zu < %zu", dst_bytes, L.total);
    return pack_matrix(W, n_out, k_in, static_cast<uint8_t*>(dst), n_threads);
}

size_t lsn_layer_image_bytes(const lsn_stack_desc* d) {
    if (!desc_ok(d)) return 0;
    size_t off[kNumProj], total;
    image_offsets(d, off, &total);
    return total;
}

int lsn_layer_image_offsets(const lsn_stack_desc* d, size_t* offsets) {
    if (!desc_ok(d) || !offsets) return fail(LSN_EINVAL, "lsn_layer_image_offsets: bad desc");
    size_t total;
    image_offsets(d, offsets, &total);
    return LSN_OK;
}

int lsn_layer_image_pack(const lsn_stack_desc* d, int layer, const float* const* W, void* dst,
                         size_t dst_bytes, int n_threads) {
    if (!desc_ok(d) || !W || !dst) return fail(LSN_EINVAL, "lsn_layer_image_pack: bad arguments");
    size_t off[kNumProj], total;
    image_offsets(d, off, &total);
    if (dst_bytes < total) return fail(LSN_EINVAL, "lsn_layer_image_pack: dst too small");
    uint8_t* base = static_cast<uint8_t*>(dst);
    LayerHeader h;
    memset(&h, 0, sizeof(h));
    h.magic = kImageMagic;
    h.layer = (uint32_t)layer;
    h.image_bytes = total;
    h.d_model = (uint32_t)d->d_model;
    h.d_kv = (uint32_t)d->d_kv;
    h.d_ff = (uint32_t)d->d_ff;
    h.n_mats = kNumProj;
    memset(base, 0, 256);
    memcpy(base, &h, sizeof(h));
    size_t prev_end = 256;
    for (int p = 0; p < kNumProj; ++p) {
        if (!W[p]) return fail(LSN_EINVAL, "lsn_layer_image_pack: W[%d] is NULL", p);
        int64_t n, k;
        proj_shape(d, p, &n, &k);
        if (off[p] > prev_end) memset(base + prev_end, 0, off[p] - prev_end);
        int rc = pack_matrix(W[p], n, k, base + off[p], n_threads);
        if (rc != LSN_OK) return rc;
        prev_end = off[p] + nf4_packed_bytes(n, k);
    }
    if (total > prev_end) memset(base + prev_end, 0, total - prev_end);
    return LSN_OK;
}

size_t lsn_lora_elems(const lsn_stack_desc* d) {
    if (!desc_ok(d)) return 0;
    size_t e = 0;
    for (int p = 0; p < kNumProj; ++p) {
        int64_t n, k;
        proj_shape(d, p, &n, &k);
        e += (size_t)d->rank * (size_t)(n + k);
    }
    return e;
}

int lsn_lora_offsets(const lsn_stack_desc* d, size_t* offsets) {
    if (!desc_ok(d) || !offsets) return fail(LSN_EINVAL, "lsn_lora_offsets: bad desc");
    size_t cur = 0;
    for (int p = 0; p < kNumProj; ++p) {
        int64_t n, k;
        proj_shape(d, p, &n, &k);
        offsets[p] = cur;
        cur += (size_t)d->rank * (size_t)k;
    }
    for (int p = 0; p < kNumProj; ++p) {
        int64_t n, k;
        proj_shape(d, p, &n, &k);
        offsets[kNumProj + p] = cur;
        cur += (size_t)n * (size_t)d->rank;
    }
    return LSN_OK;
}

}  // extern "C"
