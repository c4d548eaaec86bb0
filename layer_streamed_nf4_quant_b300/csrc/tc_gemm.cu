// Grouped tcgen05 GEMM for sm_103a with the NF4 block-dequant stage fused into its operand
// producer, plus the fixed-order split reduction and the test-only dequant kernel.
//
// The hot path of layer-streamed LoRA ("Can You Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's
// Layer Streaming Explained", "How Soup's layer streaming actually works" and "Why NF4
// matters so much"): the frozen NF4 base W is applied forward (y = x W^T) and transposed
// backward (dX = dY W) once per layer while the layer sits in a streamed VRAM slot.  Here W
// is decoded 64 weights (one absmax block) at a time by producer warps directly into the
// 128-byte-swizzled shared-memory operand tiles that tcgen05.mma reads, so bf16 W need not
// exist in HBM (nf4_dequant_many writes it there when a caller prefers a dense operand: the
// backward at large token counts).  The LoRA branch enters as extra contraction steps of the same accumulator
// (s*T*B^T forward, dT*A backward), so one fp32 TMEM accumulator holds the full result.
//
// Clusters of two CTAs (one per SM) share each tile through cta_group::2 MMAs; persistent
// over a static tile order.  CTA roles (512 threads; warp w runs on sub-partition w % 4):
//   warp 0       TMA producer of A (and of dense B) tiles
//   warp 1       TMEM allocator (both CTAs) and, in the even CTA, the single-thread UMMA issuer
//   warp 9       in the odd CTA: relays "stage full" to the even CTA
//   warps 4-7    epilogue: TMEM -> registers -> swizzled shared staging -> coalesced stores
//   warps 2, 3, 8, 10, 11, 12, 14, 15
//                B producer: NF4 decode / scaled LoRA-B rows into shared memory
// The issuer's sub-partition (1) carries no producer warp: the decode's ALU stream would take
// the issue slots the MMA instructions need (measured: two decode-like warps beside the
// issuer cut the pair-MMA rate to 69 %, the same warps on the other sub-partitions cost
// nothing).
// Every tile has a fixed K order and a fixed owner; split-K partials are reduced in split
// order by gemm_reduce; the accumulate mode adds the old output value once per element per
// launch.  So every launch is bit-reproducible and independent of where
// the weights live.
#include <cuda_bf16.h>
#include <string.h>

#include <map>
#include <mutex>
#include <vector>

#include "lsn_internal.h"
#include "tc_gemm.h"
#include "tc_ptx.cuh"

namespace lsn {

static_assert(sizeof(GemmParams) <= 32764, "kernel parameters must fit the 32 KB limit");

constexpr int kRasterGroup = 8;   // at most this many M-pairs per raster group
constexpr int kDequantWarpsPerStep = 4;   // one of the two producer groups
constexpr int kRelayWarp = 9;

// Producer warps: group * 4 + slot of warp w, or -1.  Each group of four spans sub-partitions
// 0, 2 and 3; none is on sub-partition 1, the MMA issuer's.
__device__ __forceinline__ int producer_index(int w) {
    switch (w) {
        case 8: return 0;
        case 2: return 1;
        case 10: return 2;
        case 3: return 3;
        case 12: return 4;
        case 14: return 5;
        case 11: return 6;
        case 15: return 7;
        default: return -1;
    }
}
constexpr int kEpiWarp0 = 4;
constexpr int kEpiStageBytes = 32 * 128;   // one staging tile: 32 rows of 128 bytes
constexpr size_t kGemmSmemBytes = 1024 + (size_t)kStages * (kStageABytes + kStageBBytes) +
                                  4 * 2 * kEpiStageBytes + 8 * (3 * kStages + 3) + 128;
static_assert(kGemmSmemBytes <= 227 * 1024, "shared memory per CTA");

// Wait-site ids recorded in the device error word when a bounded wait runs out.
enum : uint32_t { kSiteEmptyTma = 1, kSiteFull = 2, kSiteAccEmpty = 3, kSiteAccFull = 4,
                  kSiteEmptyDeq = 5, kSitePeerFull = 6, kSiteRelay = 7, kSiteDrain = 8 };

// No "memory" clobber: the store stays ordered with the other volatile asm statements (the
// proxy fence, the barrier arrives), and the compiler may keep values it loaded from the
// kernel parameters in registers across it instead of reloading them after every store.
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo_elem, float hi_elem) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo_elem, hi_elem);   // .x (low half) = first
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The raw bytes of one 64-weight NF4 block: its 32 code bytes, its absmax code and its
// group's scale and offset.  Loaded one step ahead of the decode to hide memory latency.
struct Nf4Block {
    uint4 c0, c1;
    uint32_t q;
    float sc, off;
};

__device__ __forceinline__ void nf4_load_block(const Nf4Dev& w, int64_t row, int64_t col0, Nf4Block& b) {
    const int64_t e0 = row * w.k_in + col0;
    const int64_t blk = e0 >> 6;
    const uint4* src = reinterpret_cast<const uint4*>(w.codes + (e0 >> 1));
    b.c0 = __ldg(src);
    b.c1 = __ldg(src + 1);
    b.q = __ldg(w.absmax + blk);
    const int64_t g = blk >> 8;
    b.sc = __ldg(w.scale + g);
    b.off = __ldg(w.offset + g);
}

// Decodes one block into 32 words of packed bf16 pairs (element order preserved).  Every
// weight is bf16_rn(fp32(level[code] * a')), a' = fp32(fp32(q * scale) + offset): the 16
// possible values of the block are computed first, with exactly that rounding, and split
// into a low-byte and a high-byte table (four registers each).  Each code then indexes the
// tables with byte permutes: prmt picks entries 0-7 and 8-15 by the code's low three bits,
// a sign-replicating prmt turns the code's top bit into a byte mask that selects between
// them, and a final prmt interleaves low and high bytes into bf16 pairs.
__device__ __forceinline__ void nf4_decode_regs(const Nf4Block& bk, const float (&lv)[16], uint32_t (&o)[32]) {
    const float a = __fadd_rn(__fmul_rn((float)bk.q, bk.sc), bk.off);
    uint32_t P[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) P[j] = pack_bf16x2(__fmul_rn(lv[2 * j], a), __fmul_rn(lv[2 * j + 1], a));
    // byte k of L0..L3 / H0..H3: low / high byte of the value of code 4*i + k
    const uint32_t L0 = prmt(P[0], P[1], 0x6420u), L1 = prmt(P[2], P[3], 0x6420u);
    const uint32_t L2 = prmt(P[4], P[5], 0x6420u), L3 = prmt(P[6], P[7], 0x6420u);
    const uint32_t H0 = prmt(P[0], P[1], 0x7531u), H1 = prmt(P[2], P[3], 0x7531u);
    const uint32_t H2 = prmt(P[4], P[5], 0x7531u), H3 = prmt(P[6], P[7], 0x7531u);
    const uint32_t wd[8] = {bk.c0.x, bk.c0.y, bk.c0.z, bk.c0.w, bk.c1.x, bk.c1.y, bk.c1.z, bk.c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // selector nibbles: codes of weights 1, 0, 3, 2 of this group of four
            // (weight 2k sits in the high nibble of byte k)
            const uint32_t S = h ? (wd[i] >> 16) : wd[i];
            const uint32_t S7 = S & 0x7777u;
            const uint32_t M = prmt(S << 4, S, 0xD9C8u);   // 0xFF where the code is >= 8
            const uint32_t lo = (prmt(L0, L1, S7) & ~M) | (prmt(L2, L3, S7) & M);
            const uint32_t hi = (prmt(H0, H1, S7) & ~M) | (prmt(H2, H3, S7) & M);
            o[4 * i + 2 * h] = prmt(lo, hi, 0x4051u);       // weights 0, 1
            o[4 * i + 2 * h + 1] = prmt(lo, hi, 0x6273u);   // weights 2, 3
        }
    }
}

// One row of a dense bf16 matrix (k <= 64 elements, k % 8 == 0) times `scale`, zero padded,
// as 32 words of bf16 pairs.
__device__ __forceinline__ void scaled_row(const uint16_t* src, int k, float scale, uint32_t (&o)[32]) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (ch * 8 < k) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
            const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = __uint_as_float(in[j] << 16);
                const float hi = __uint_as_float(in[j] & 0xFFFF0000u);
                w[j] = pack_bf16x2(__fmul_rn(lo, scale), __fmul_rn(hi, scale));
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) o[4 * ch + j] = w[j];
    }
}

struct TileInfo {
    int prob, m0, n0, split, ks_begin, ks_end;
    bool half0, half1;   // whether each 128-row half of this CTA's M tile holds any row
};

__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int t, uint32_t rank) {
    int pi = 0;
    while (pi + 1 < p.n_probs && t >= p.probs[pi + 1].tile_begin) ++pi;
    const Problem& pr = p.probs[pi];
    const int l = t - pr.tile_begin;
    const int per_split = pr.tiles_m * pr.tiles_n;   // tiles_m counts M-pairs
    const int s = l / per_split;
    const int r = l - s * per_split;
    // grouped raster: pr.raster M-pairs sweep all N tiles together, so the A rows of the
    // group stay in L2 while B streams past them once per group
    const int rg = pr.raster;
    const int g = r / (rg * pr.tiles_n);
    const int first_m = g * rg;
    const int gm = min(rg, pr.tiles_m - first_m);
    const int rr = r - g * rg * pr.tiles_n;
    const int nt = rr / gm;
    const int mt = first_m + (rr - nt * gm);
    TileInfo ti;
    ti.prob = pi;
    ti.m0 = (2 * mt + (int)rank) * kBM;
    ti.n0 = nt * pr.bn;
    ti.split = s;
    const int64_t kb = pr.ksteps_split;
    ti.ks_begin = (int)(kb * s / pr.splits);
    ti.ks_end = s + 1 == pr.splits ? pr.ksteps : (int)(kb * (s + 1) / pr.splits);
    ti.half0 = ti.m0 < pr.m;
    ti.half1 = ti.m0 + 128 < pr.m;
    return ti;
}

// Maps a problem-level k-step to (segment index, k-step within the segment).
__device__ __forceinline__ void locate(const GemmParams& p, const Problem& pr, int ks, int& seg,
                                       int& kk) {
    int s = pr.seg_begin;
    int k = ks;
    while (s + 1 < pr.seg_begin + pr.seg_count && k >= p.segs[s].ksteps) {
        k -= p.segs[s].ksteps;
        ++s;
    }
    seg = s;
    kk = k;
}

__device__ __forceinline__ bool seg_b_mn(int b_src) { return b_src == B_NF4_MN || b_src == B_TMA_MN; }

// Position in the cluster's flattened sequence of (tile, k-step); every role walks it.
struct SeqPos {
    int t;        // schedule tile (>= total_tiles: finished)
    TileInfo ti;
    int ks;       // problem-level k-step
    int si, kk;   // segment and k-step within it
};

__device__ __forceinline__ void seq_tile(const GemmParams& p, SeqPos& s, uint32_t rank) {
    if (s.t < p.total_tiles) {
        s.ti = decode_tile(p, s.t, rank);
        s.ks = s.ti.ks_begin;
        locate(p, p.probs[s.ti.prob], s.ks, s.si, s.kk);
    }
}

__device__ __forceinline__ void seq_begin(const GemmParams& p, SeqPos& s, uint32_t rank) {
    s.t = (int)ptx::cluster_id_x();
    seq_tile(p, s, rank);
}

__device__ __forceinline__ void seq_next(const GemmParams& p, SeqPos& s, uint32_t rank) {
    if (s.t >= p.total_tiles) return;
    if (++s.ks >= s.ti.ks_end) {
        s.t += (int)ptx::n_clusters_x();
        seq_tile(p, s, rank);
        return;
    }
    if (++s.kk >= p.segs[s.si].ksteps) {
        ++s.si;
        s.kk = 0;
    }
}

// What one B-producer thread writes for one k-step: one 128-byte row of this CTA's half of
// the B tile.  A pair MMA takes N/2 of B's rows (K-major) or N/2 of its columns (MN-major,
// in whole 64-column atoms) from each CTA's shared memory at the same offset.
enum : int { kJobNone = 0, kJobNf4 = 1, kJobZero = 2, kJobScaled = 3 };
struct DeqJob {
    int kind;
    int w;              // NF4 matrix index
    int64_t row, col0;  // the block W[row][col0 .. col0+63]
    uint32_t dst_off;   // byte offset of the 128-byte row within the stage's B half-tile
    uint32_t swz;       // swizzle phase of that row
    const uint16_t* sp; // kJobScaled: source row, its length and the factor
    int sk;
    float ss;
};

// j: row job within this CTA's half of the B tile, 0 .. bn/2 - 1.
__device__ __forceinline__ DeqJob make_deq_job(const GemmParams& p, const SeqPos& s, int j, uint32_t rank) {
    DeqJob d{};
    d.kind = kJobNone;
    const Problem& pr = p.probs[s.ti.prob];
    const int half = pr.bn >> 1;
    if (j >= half) return d;
    const KSeg& sg = p.segs[s.si];
    const int kk = s.kk;
    const int nb = s.ti.n0 + (int)rank * half;   // first output column of this CTA's half
    if (sg.b_src == B_NF4_K) {
        const Nf4Dev& w = p.nf4[sg.b_idx];
        d.w = sg.b_idx;
        d.row = (int64_t)sg.b_n0 + nb + j;
        d.col0 = (int64_t)sg.b_k0 + (int64_t)kk * kBK;
        d.dst_off = j * 128;
        d.swz = j & 7;
        d.kind = (d.row < w.n_out && d.col0 < w.k_in) ? kJobNf4 : kJobZero;
    } else if (sg.b_src == B_NF4_MN) {
        const int r = j & 63;      // contraction row within the k-step
        const int a = j >> 6;      // local 64-column atom
        const Nf4Dev& w = p.nf4[sg.b_idx];
        const int kin = kk * kBK + r;
        d.w = sg.b_idx;
        d.row = (int64_t)sg.b_k0 + kin;
        d.col0 = (int64_t)sg.b_n0 + nb + 64 * a;
        d.dst_off = a * 8192 + r * 128;
        d.swz = r & 7;
        d.kind = (kin < sg.k_len && d.row < w.n_out && d.col0 < w.k_in) ? kJobNf4 : kJobZero;
    } else if (sg.b_src == B_SCALED_K) {
        const int64_t n = (int64_t)nb + j;
        d.dst_off = j * 128;
        d.swz = j & 7;
        if (n < sg.b_rows) {
            d.kind = kJobScaled;
            d.sp = sg.b_ptr + n * sg.b_ld;
            d.sk = sg.k_len;
            d.ss = sg.b_scale;
        } else {
            d.kind = kJobZero;
        }
    }
    return d;
}

// ----------------------------------------------------------------------------- epilogue

// Epilogue of one warp: its 32 accumulator rows (lane = row row0 + lane), 128 bytes of each
// row per step (64 bf16 or 32 fp32 columns).  Each step writes the values row by row into one
// of the warp's two 4 KB staging tiles in shared memory (16-byte pieces XOR-swizzled by row,
// so neither the row-wise writes nor the column-wise reads conflict), then reads the tile
// back so that every 8 lanes hold one 128-byte row segment and store it with st.global.v4:
// coalesced, with no bulk-copy unit, proxy fence or completion wait on the path (the bulk
// tensor stores this replaces shared the copy unit with the A loads and waited for it).  The
// two tiles alternate, so one __syncwarp per step orders a tile's writes before its reads and
// its reads before its next writes.  The arithmetic per element: alpha * acc, then the
// residual (bf16 outputs) or, for EPI_F32_ACC, the old value of the output (one fp32
// addition per element), then the rounding.
struct EpiStage {
    uint32_t base;   // this warp's two staging tiles
    uint32_t buf;    // the tile written next
};

// The per-problem values the epilogue needs, copied into registers once per tile.
struct EpiArgs {
    int epi, m, n_valid, split;
    float alpha;
    void* out;
    int64_t ldo;
    int64_t part_stride;
    const uint16_t* residual;
    int64_t ldr;
};

// Register copies of kernel parameters.  The empty asm hides where the value came from, so the
// compiler keeps it in a register (or spills it to the stack) instead of re-reading the
// parameter inside the epilogue loop, where a constant-cache miss costs hundreds of cycles.
__device__ __forceinline__ int reg_copy(int v) { asm volatile("mov.b32 %0, %0;" : "+r"(v)); return v; }
__device__ __forceinline__ float reg_copy(float v) { asm volatile("mov.b32 %0, %0;" : "+f"(v)); return v; }
__device__ __forceinline__ int64_t reg_copy(int64_t v) { asm volatile("mov.b64 %0, %0;" : "+l"(v)); return v; }
template <class T>
__device__ __forceinline__ T* reg_copy(T* v) {
    uint64_t u = reinterpret_cast<uint64_t>(v);
    asm volatile("mov.b64 %0, %0;" : "+l"(u));
    return reinterpret_cast<T*>(u);
}

__device__ __forceinline__ EpiArgs epi_args(const Problem& pr, int split) {
    EpiArgs a;
    a.epi = reg_copy(pr.epi);
    a.m = reg_copy(pr.m);
    a.n_valid = reg_copy(pr.n_valid);
    a.split = reg_copy(split);
    a.alpha = reg_copy(pr.alpha);
    a.out = reg_copy(pr.out);
    a.ldo = reg_copy(pr.ldo);
    a.part_stride = reg_copy(pr.part_stride);
    a.residual = reg_copy(pr.residual);
    a.ldr = reg_copy(pr.ldr);
    return a;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Output stores are not read again by this kernel: evict-first keeps L2 for the A rows.
__device__ __forceinline__ void st_global_v4_ef(void* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// One step: w = this lane's 128 bytes of row row0 + lane (kElemBytes per element), written
// to the output columns col0 .. col0 + 128 / kElemBytes.
template <int kElemBytes>
__device__ __forceinline__ void epi_flush(const EpiArgs& a, int row0, int col0, const uint32_t (&w)[32], EpiStage& st,
                                          int lane, uint64_t pol) {
    const uint32_t tile = st.base + st.buf * kEpiStageBytes;
    const uint32_t swz = (uint32_t)(lane & 7);
#pragma unroll
    for (int g = 0; g < 8; ++g)
        st_shared_v4(tile + (uint32_t)lane * 128u + ((((uint32_t)g) ^ swz) << 4), w[4 * g], w[4 * g + 1],
                     w[4 * g + 2], w[4 * g + 3]);
    __syncwarp();
    constexpr int kPer16 = 16 / kElemBytes;   // elements per 16-byte piece
    const int c = lane & 7;                   // this lane's piece of each row segment
    const int col = col0 + c * kPer16;
    const bool col_ok = col < a.n_valid;      // n_valid is a multiple of 8: pieces are whole
    char* base = static_cast<char*>(a.out);
    if (a.epi == EPI_PARTIAL) base += (int64_t)a.split * a.part_stride * 4;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int r = 4 * j + (lane >> 3);
        const int row = row0 + r;
        uint4 v = ld_shared_v4(tile + (uint32_t)r * 128u + ((((uint32_t)c) ^ (uint32_t)(r & 7)) << 4));
        if (row < a.m && col_ok) {
            void* o = base + ((int64_t)row * a.ldo + col) * kElemBytes;
            if (kElemBytes == 4 && a.epi == EPI_F32_ACC) {
                const float4 old = *reinterpret_cast<const float4*>(o);
                v.x = __float_as_uint(old.x + __uint_as_float(v.x));
                v.y = __float_as_uint(old.y + __uint_as_float(v.y));
                v.z = __float_as_uint(old.z + __uint_as_float(v.z));
                v.w = __float_as_uint(old.w + __uint_as_float(v.w));
            }
            st_global_v4_ef(o, v, pol);
        }
    }
    st.buf ^= 1u;
}

// fp32 outputs, 32 columns per step (EPI_F32, EPI_F32_ACC, EPI_PARTIAL; EPI_F32_T is written
// directly, transposed).
__device__ __forceinline__ void epi_chunk(const EpiArgs& a, int row0, int col0, const uint32_t (&r)[32], EpiStage& st,
                                          int lane, uint64_t pol) {
    const float al = a.alpha;
    if (a.epi == EPI_F32_T) {
        // transposed output: for a fixed column the lanes write consecutive rows
        const int row = row0 + lane;
        if (row < a.m && col0 < a.n_valid) {
            float* o = static_cast<float*>(a.out);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < a.n_valid) o[(int64_t)(col0 + j) * a.ldo + row] = __uint_as_float(r[j]) * al;
        }
        __syncwarp();
        return;
    }
    if (col0 >= a.n_valid) return;   // warp-uniform
    const float a2 = a.epi == EPI_PARTIAL ? 1.0f : al;
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(__uint_as_float(r[j]) * a2);
    epi_flush<4>(a, row0, col0, w, st, lane, pol);
}

// bf16 output, 64 columns (two 32-column accumulator chunks) per step.
__device__ __forceinline__ void epi_pair_bf16(const EpiArgs& a, int row0, int col0, const uint32_t (&ra)[32],
                                              const uint32_t (&rb)[32], EpiStage& st, int lane, uint64_t pol) {
    if (col0 >= a.n_valid) return;   // warp-uniform
    const float al = a.alpha;
    const bool unit = al == 1.0f;   // x * 1.0f == x exactly, so the multiply is skipped
    const int row = row0 + lane;
    const bool res_row = a.residual != nullptr && row < a.m;
    const uint16_t* rp = res_row ? a.residual + (int64_t)row * a.ldr + col0 : nullptr;
    uint32_t w[32];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const uint32_t(&r)[32] = g < 4 ? ra : rb;
        const int gg = g & 3;
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = unit ? __uint_as_float(r[8 * gg + j]) : __uint_as_float(r[8 * gg + j]) * al;
        if (res_row && col0 + 8 * g < a.n_valid) {
            const uint4 r4 = *reinterpret_cast<const uint4*>(rp + 8 * g);
            const uint32_t rw[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] += __uint_as_float(rw[j] << 16);
                f[2 * j + 1] += __uint_as_float(rw[j] & 0xFFFF0000u);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) w[4 * g + j] = pack_bf16x2(f[2 * j], f[2 * j + 1]);
    }
    epi_flush<2>(a, row0, col0, w, st, lane, pol);
}

// ------------------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(kGemmThreads, 1) tc_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + kStages * kStageABytes;
    const uint32_t sStg = sB + kStages * kStageBBytes;   // epilogue staging, two tiles per warp
    const uint32_t sBar = sStg + 4 * 2 * kEpiStageBytes;
    auto full_bar = [&](int s) { return sBar + 8u * s; };
    auto pfull_bar = [&](int s) { return sBar + 8u * (kStages + s); };
    auto empty_bar = [&](int s) { return sBar + 8u * (2 * kStages + s); };
    const uint32_t acc_full = sBar + 8u * (3 * kStages);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t drain_bar = acc_empty + 8u;   // the issuer's own MMAs have all finished
    uint8_t* const gmisc = gbase + (sBar - base) + 8 * (3 * kStages + 3);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(gmisc);
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gmisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();   // 0 (issues the pair MMAs) or 1
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1 + kDequantWarpsPerStep);   // own TMA + own producer group
            ptx::mbar_init(pfull_bar(s), 1);                         // the peer's stage is full
            ptx::mbar_init(empty_bar(s), 1);                         // the pair MMAs read the stage
        }
        ptx::mbar_init(acc_full, 1);
        ptx::mbar_init(acc_empty, 256);   // both CTAs' epilogue threads (used in the even CTA)
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 512);
        ptx::tmem_relinquish_pair();
    }
    __syncthreads();
    ptx::cluster_sync();   // both CTAs' barriers are initialised before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // A rows are read again by the later N tiles of their raster group: keep them in
            // L2 ahead of the streamed weights and outputs
            const uint64_t pol_keep = ptx::policy_evict_last();
            SeqPos s;
            seq_begin(p, s, rank);
            uint32_t n_steps = 0;
            for (uint32_t i = 0; s.t < p.total_tiles; ++i, seq_next(p, s, rank)) {
                const uint32_t stage = i % kStages, phase = (i / kStages) & 1u;
                // everything the copies need is read before the stage is free
                const Problem& pr = p.probs[s.ti.prob];
                const KSeg& sg = p.segs[s.si];
                const int half = pr.bn >> 1;
                const uint32_t bar = full_bar(stage);
                const uint32_t a_dst = sA + stage * kStageABytes;
                const uint32_t b_dst = sB + stage * kStageBBytes;
                const int bsrc = sg.b_src;
                const uint32_t bytes = kStageABytes + ((bsrc == B_TMA_K || bsrc == B_TMA_MN) ? half * kBK * 2 : 0);
                const int ak = sg.a_k0 + s.kk * kBK;
                const bool a_k = pr.a_major == A_KMAJOR;
                const CUtensorMap* amap = &p.maps[sg.a_map];
                const CUtensorMap* bmap = &p.maps[sg.b_idx];
                const int bk = sg.b_k0 + s.kk * kBK;
                const int nb = sg.b_n0 + s.ti.n0 + (int)rank * half;
                const int m0 = s.ti.m0;
                if (!ptx::mbar_wait_bounded_cta(empty_bar(stage), phase ^ 1u, abort_flag, p.err, kSiteEmptyTma))
                    break;
                ptx::mbar_arrive_expect_tx(bar, bytes);
                if (a_k) {
                    ptx::tma_load_2d_hint(a_dst, amap, ak, m0, bar, pol_keep);
                } else {
#pragma unroll
                    for (int q = 0; q < kBM / 64; ++q)
                        ptx::tma_load_2d_hint(a_dst + q * 8192, amap, m0 + 64 * q, ak, bar, pol_keep);
                }
                if (bsrc == B_TMA_K) {
                    ptx::tma_load_2d(b_dst, bmap, bk, nb, bar);
                } else if (bsrc == B_TMA_MN) {
                    for (int q = 0; q < half / 64; ++q)
                        ptx::tma_load_2d(b_dst + q * 8192, bmap, nb + 64 * q, bk, bar);
                }
                n_steps = i + 1;
            }
            // Wait for the last release of every stage: the pair MMAs' commits arrive on this
            // CTA's empty barriers asynchronously, and they must land before the CTA exits.
            if (!*abort_flag) {
                for (uint32_t st = 0; st < (uint32_t)kStages && st < n_steps; ++st) {
                    const uint32_t last = st + ((n_steps - 1 - st) / kStages) * kStages;
                    if (!ptx::mbar_wait_bounded_cta(empty_bar(st), (last / kStages) & 1u, abort_flag, p.err,
                                                kSiteEmptyTma))
                        break;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ pair UMMA issuer (rank 0)
        // One thread issues every pair MMA, so its own instructions per k-step bound the
        // tensor rate when the stages are ready (they nearly always are): the tile's k-steps
        // are walked segment by segment with no parameter loads inside, and the stage
        // barriers are polled with test_wait.
        if (lane == 0 && leader) {
            uint32_t acc_phase = 0;
            uint32_t i = 0;
            // Operand descriptors at stage 0; the start-address field (address / 16, bits 0-13)
            // takes the stage, block and k16 offsets by plain addition (shared memory < 256 KB).
            const uint64_t dA_k = ptx::smem_desc_sw128(sA, 16, 1024), dA_mn = ptx::smem_desc_sw128(sA, 8192, 1024);
            const uint64_t dB_k = ptx::smem_desc_sw128(sB, 16, 1024), dB_mn = ptx::smem_desc_sw128(sB, 8192, 1024);
            constexpr uint32_t kHalfA16 = (kStageABytes / 2) >> 4;   // the second 128-row block
            bool ok = true;
            for (int t = (int)ptx::cluster_id_x(); ok && t < p.total_tiles; t += (int)ptx::n_clusters_x()) {
                const TileInfo ti = decode_tile(p, t, rank);
                const Problem& pr = p.probs[ti.prob];
                if (!ptx::mbar_wait_bounded(acc_empty, acc_phase ^ 1u, abort_flag, p.err, kSiteAccEmpty)) break;
                ptx::tc_fence_after();
                const bool a_mn = pr.a_major == A_MNMAJOR;
                const uint64_t dA = a_mn ? dA_mn : dA_k;
                const uint32_t a_k16 = a_mn ? (2048u >> 4) : (32u >> 4);
                const uint32_t idesc_bk = ptx::idesc_bf16_f32(pr.bn, a_mn ? 1 : 0, 0, 256);
                const uint32_t idesc_bmn = ptx::idesc_bf16_f32(pr.bn, a_mn ? 1 : 0, 1, 256);
                const uint32_t tmem_h1 = tmem + (uint32_t)pr.bn;
                const bool h0 = ti.half0, h1 = ti.half1;
                int si, kk;
                locate(p, pr, ti.ks_begin, si, kk);
                uint32_t acc = 0u;   // the tile's first MMA overwrites the accumulator
                for (int ks = ti.ks_begin; ok && ks < ti.ks_end; ++si, kk = 0) {
                    const bool b_mn = seg_b_mn(p.segs[si].b_src);
                    const int seg_end = ks + (p.segs[si].ksteps - kk) < ti.ks_end ? ks + (p.segs[si].ksteps - kk)
                                                                                   : ti.ks_end;
                    const uint32_t idesc = b_mn ? idesc_bmn : idesc_bk;
                    const uint64_t dB = b_mn ? dB_mn : dB_k;
                    const uint32_t b_k16 = b_mn ? (2048u >> 4) : (32u >> 4);
                    for (; ks < seg_end; ++ks, ++i) {
                        const uint32_t stage = i % kStages, phase = (i / kStages) & 1u;
                        if (!ptx::mbar_poll_bounded<false>(full_bar(stage), phase, abort_flag, p.err, kSiteFull) ||
                            !ptx::mbar_poll_bounded<true>(pfull_bar(stage), phase, abort_flag, p.err, kSitePeerFull)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint64_t a0 = dA + ((stage * (uint32_t)kStageABytes) >> 4);
                        const uint64_t b0 = dB + ((stage * (uint32_t)kStageBBytes) >> 4);
#pragma unroll
                        for (int k4 = 0; k4 < kBK / 16; ++k4) {
                            // rows of block h: 128 of this CTA's tile and 128 of the peer's
                            const uint64_t bd = b0 + (uint64_t)(k4 * b_k16);
                            const uint64_t ad = a0 + (uint64_t)(k4 * a_k16);
                            if (h0) ptx::umma_f16_pair(tmem, ad, bd, idesc, acc);
                            if (h1) ptx::umma_f16_pair(tmem_h1, ad + kHalfA16, bd, idesc, acc);
                            acc = 1u;
                        }
                        ptx::umma_commit_pair_mc(empty_bar(stage), 0x3);
                    }
                }
                if (!ok) break;
                ptx::umma_commit_pair_mc(acc_full, 0x3);
                acc_phase ^= 1u;
            }
            // Every pair MMA this thread issued has finished before the CTAs may release
            // TMEM and shared memory, on the normal path and after an abort alike.
            ptx::umma_commit_pair_mc(drain_bar, 0x1);
            volatile int no_abort = 0;   // this wait does not end early on an abort
            if (!ptx::mbar_wait_bounded(drain_bar, 0, &no_abort, p.err, kSiteDrain)) *abort_flag = 1;
        }
    } else if (warp == kRelayWarp) {
        // ------------------------------------------- relay of stage readiness (rank 1)
        if (lane == 0 && !leader) {
            const uint32_t remote_pfull0 = ptx::mapa(pfull_bar(0), 0);
            SeqPos s;
            seq_begin(p, s, rank);
            for (uint32_t i = 0; s.t < p.total_tiles; ++i, seq_next(p, s, rank)) {
                const uint32_t stage = i % kStages, phase = (i / kStages) & 1u;
                if (!ptx::mbar_wait_bounded_cta(full_bar(stage), phase, abort_flag, p.err, kSiteRelay)) break;
                ptx::mbar_arrive_remote(remote_pfull0 + 8u * stage);
            }
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // ------------------------------------------------------------------- epilogue
        const int q = warp - kEpiWarp0;
        uint32_t acc_phase = 0;
        const uint32_t acc_empty_dst = leader ? acc_empty : ptx::mapa(acc_empty, 0);
        EpiStage est{sStg + (uint32_t)q * 2u * kEpiStageBytes, 0u};
        const uint64_t pol_out = ptx::policy_evict_first();
        for (int t = (int)ptx::cluster_id_x(); t < p.total_tiles; t += (int)ptx::n_clusters_x()) {
            const TileInfo ti = decode_tile(p, t, rank);
            const TileInfo t0 = decode_tile(p, t, 0);   // which blocks the pair MMAs wrote
            const Problem& pr = p.probs[ti.prob];
            const EpiArgs ea = epi_args(pr, ti.split);
            int ok = 0;
            if (lane == 0) ok = ptx::mbar_wait_bounded(acc_full, acc_phase, abort_flag, p.err, kSiteAccFull);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ptx::tc_fence_after();
            // chunks of 32 columns over both 128-row blocks; the TMEM load of the next chunk
            // is in flight while the current one is staged (tcgen05.ld and its wait are
            // warp-collective: every path through epi_chunk ends reconverged)
            const int h_first = t0.half0 ? 0 : 1, h_last = t0.half1 ? 1 : 0;
            const int per_h_log = pr.bn == 256 ? 3 : 2;   // 32-column chunks per block: bn / 32
            const int n_chunks = (h_last - h_first + 1) << per_h_log;
            const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
            auto chunk_h = [&](int i) { return h_first + (i >> per_h_log); };
            auto chunk_c = [&](int i) { return (i & ((1 << per_h_log) - 1)) * 32; };
            uint32_t ra[32], rb[32];
            __syncwarp();
            const int bn = reg_copy(pr.bn), m0 = reg_copy(ti.m0), n0 = reg_copy(ti.n0);
            if (ea.epi == EPI_BF16) {
                // chunk pairs (the N tile is 128 or 256 wide, so pairs never straddle a block)
                for (int i = 0; i < n_chunks; i += 2) {
                    ptx::tmem_ld32_issue(tq + (uint32_t)(chunk_h(i) * bn + chunk_c(i)), ra);
                    ptx::tmem_ld32_issue(tq + (uint32_t)(chunk_h(i + 1) * bn + chunk_c(i + 1)), rb);
                    ptx::tmem_ld_wait(ra);
                    ptx::tmem_ld_wait(rb);
                    epi_pair_bf16(ea, m0 + chunk_h(i) * 128 + q * 32, n0 + chunk_c(i), ra, rb, est, lane, pol_out);
                }
            } else {
            ptx::tmem_ld32_issue(tq + (uint32_t)(chunk_h(0) * bn + chunk_c(0)), ra);
            ptx::tmem_ld_wait(ra);
            for (int i = 0; i < n_chunks; i += 2) {
                if (i + 1 < n_chunks) ptx::tmem_ld32_issue(tq + (uint32_t)(chunk_h(i + 1) * bn + chunk_c(i + 1)), rb);
                epi_chunk(ea, m0 + chunk_h(i) * 128 + q * 32, n0 + chunk_c(i), ra, est, lane, pol_out);
                if (i + 1 >= n_chunks) break;
                ptx::tmem_ld_wait(rb);
                if (i + 2 < n_chunks) ptx::tmem_ld32_issue(tq + (uint32_t)(chunk_h(i + 2) * bn + chunk_c(i + 2)), ra);
                epi_chunk(ea, m0 + chunk_h(i + 1) * 128 + q * 32, n0 + chunk_c(i + 1), rb, est, lane, pol_out);
                if (i + 2 < n_chunks) ptx::tmem_ld_wait(ra);
            }
            }
            ptx::tc_fence_before();
            if (leader) ptx::mbar_arrive(acc_empty_dst);
            else ptx::mbar_arrive_remote(acc_empty_dst);
            acc_phase ^= 1u;
        }
    } else if (producer_index(warp) >= 0) {
        // --------------------------------------------------------------- B producer
        // Two groups of four warps take alternate k-steps of the sequence, so two k-steps
        // are being decoded at once; each thread owns one 128-byte row of this CTA's half of
        // the B tile.
        const int dt = producer_index(warp) * 32 + lane;   // 0 .. 255
        const int grp = dt >> 7;
        const int gt = dt & 127;
        SeqPos s;
        seq_begin(p, s, rank);
        uint32_t i = 0;
        if (grp == 1) {
            seq_next(p, s, rank);
            i = 1;
        }
        DeqJob cur{};
        Nf4Block cb{};
        if (s.t < p.total_tiles) {
            cur = make_deq_job(p, s, gt, rank);
            if (cur.kind == kJobNf4) nf4_load_block(p.nf4[cur.w], cur.row, cur.col0, cb);
        }
        while (s.t < p.total_tiles) {
            SeqPos sn = s;
            seq_next(p, sn, rank);
            seq_next(p, sn, rank);
            DeqJob nxt{};
            Nf4Block nb{};
            if (sn.t < p.total_tiles) {
                nxt = make_deq_job(p, sn, gt, rank);
                if (nxt.kind == kJobNf4) nf4_load_block(p.nf4[nxt.w], nxt.row, nxt.col0, nb);
            }
            const uint32_t stage = i % kStages, phase = (i / kStages) & 1u;
            // the row is decoded into registers before the stage is free; only the stores wait
            uint32_t o[32];
            if (cur.kind == kJobNf4) {
                nf4_decode_regs(cb, p.levels, o);
            } else if (cur.kind == kJobScaled) {
                scaled_row(cur.sp, cur.sk, cur.ss, o);
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) o[k] = 0u;
            }
            int ok = 0;
            if (lane == 0)
                ok = ptx::mbar_wait_bounded_cta(empty_bar(stage), phase ^ 1u, abort_flag, p.err, kSiteEmptyDeq);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (cur.kind != kJobNone) {
                const uint32_t dst = sB + stage * kStageBBytes + cur.dst_off;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    st_shared_v4(dst + (uint32_t)((ch ^ (int)cur.swz) << 4), o[4 * ch], o[4 * ch + 1],
                                 o[4 * ch + 2], o[4 * ch + 3]);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(full_bar(stage));
            cur = nxt;
            cb = nb;
            s = sn;
            i += 2;
        }
    }

    __syncthreads();
    // An abort in either CTA is an abort of the pair: tell the peer, then both settle.
    if (threadIdx.x == 0 && *abort_flag)
        ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u), 1u);
    ptx::cluster_sync();   // no CTA leaves while the pair may still use its memory
    if (*abort_flag) {
        // let copies already in flight land before the CTAs release their resources
        if (threadIdx.x == 0) ptx::settle_ns(50000);
        __syncthreads();
        ptx::cluster_sync();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem, 512);
    }
}

// ----------------------------------------------------------------------- split reduce

struct ReduceJob {
    const float* partial;
    void* out;
    const uint16_t* residual;
    int64_t part_stride, ldo, ldr;
    int splits, m, n, epi, n_valid;
    float alpha;
    int64_t begin;   // first work item of this job in the launch
};
constexpr int kMaxReduceJobs = kMaxProbs;
struct ReduceJobs {
    ReduceJob j[kMaxReduceJobs];
    int count;
    int64_t total;
};

// Sums the split partials of every split problem of one GEMM launch in split order and
// applies each problem's final epilogue (four columns per work item).
__global__ void gemm_reduce_kernel(const __grid_constant__ ReduceJobs jobs) {
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < jobs.total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        int k = 0;
        while (k + 1 < jobs.count && idx >= jobs.j[k + 1].begin) ++k;
        const ReduceJob& jb = jobs.j[k];
        const int64_t local = idx - jb.begin;
        const int n4 = jb.n_valid / 4;
        int row, c4;
        if (jb.epi == EPI_F32_T) {   // consecutive threads on consecutive rows: coalesced stores
            c4 = (int)(local / jb.m);
            row = (int)(local - (int64_t)c4 * jb.m);
        } else {
            row = (int)(local / n4);
            c4 = (int)(local - (int64_t)row * n4);
        }
        const int col = c4 * 4;
        const float* src = jb.partial + (int64_t)row * jb.n + col;
        float4 acc = *reinterpret_cast<const float4*>(src);
        for (int s = 1; s < jb.splits; ++s) {
            const float4 y = *reinterpret_cast<const float4*>(src + (int64_t)s * jb.part_stride);
            acc.x += y.x; acc.y += y.y; acc.z += y.z; acc.w += y.w;
        }
        float f[4] = {acc.x * jb.alpha, acc.y * jb.alpha, acc.z * jb.alpha, acc.w * jb.alpha};
        if (jb.epi == EPI_BF16) {
            if (jb.residual) {
                const uint2 r2 = *reinterpret_cast<const uint2*>(jb.residual + (int64_t)row * jb.ldr + col);
                f[0] += __uint_as_float(r2.x << 16);
                f[1] += __uint_as_float(r2.x & 0xFFFF0000u);
                f[2] += __uint_as_float(r2.y << 16);
                f[3] += __uint_as_float(r2.y & 0xFFFF0000u);
            }
            uint2 w;
            w.x = pack_bf16x2(f[0], f[1]);
            w.y = pack_bf16x2(f[2], f[3]);
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(jb.out) + (int64_t)row * jb.ldo + col) = w;
        } else if (jb.epi == EPI_F32_T) {
            float* o = static_cast<float*>(jb.out);
            for (int j = 0; j < 4; ++j) o[(int64_t)(col + j) * jb.ldo + row] = f[j];
        } else {
            float* o = static_cast<float*>(jb.out) + (int64_t)row * jb.ldo + col;
            float4 x = make_float4(f[0], f[1], f[2], f[3]);
            if (jb.epi == EPI_F32_ACC) {
                const float4 y = *reinterpret_cast<const float4*>(o);
                x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
            }
            *reinterpret_cast<float4*>(o) = x;
        }
    }
}

// --------------------------------------------------------------------------- dequant

// Many matrices at once, 32 blocks per warp; the decoded rows are transposed through shared
// memory so that every store instruction writes 512 contiguous bytes.
struct DequantParams {
    Nf4Dev w[kMaxNf4];
    uint16_t* out[kMaxNf4];
    int64_t group_begin[kMaxNf4 + 1];   // first 32-block group of each matrix; [n] = total
    int n;
    Nf4Levels lvl;
};
constexpr int kDequantWarps = 8;

__global__ void __launch_bounds__(kDequantWarps * 32) nf4_dequant_many_kernel(const __grid_constant__ DequantParams p) {
    __shared__ __align__(128) uint8_t stage[kDequantWarps][32 * 128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = ptx::smem_u32(&stage[warp][0]);
    const int64_t total = p.group_begin[p.n];
    for (int64_t g = (int64_t)blockIdx.x * kDequantWarps + warp; g < total;
         g += (int64_t)gridDim.x * kDequantWarps) {
        int m = 0;
        while (m + 1 < p.n && g >= p.group_begin[m + 1]) ++m;
        const Nf4Dev& w = p.w[m];
        const int64_t nb = w.n_out * (w.k_in >> 6);
        const int64_t b0 = (g - p.group_begin[m]) * 32;
        const int64_t b = b0 + lane;
        if (b < nb) {
            const int64_t kb = w.k_in >> 6;
            const int64_t row = b / kb;
            Nf4Block bk;
            nf4_load_block(w, row, (b - row * kb) * 64, bk);
            uint32_t o[32];
            nf4_decode_regs(bk, p.lvl.v, o);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared_v4(base + (uint32_t)lane * 128u + (((uint32_t)c ^ (uint32_t)(lane & 7)) << 4), o[4 * c],
                             o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        }
        __syncwarp();
        uint4* dst = reinterpret_cast<uint4*>(p.out[m] + b0 * 64);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int idx = j * 32 + lane;   // 16-byte piece of the group's 4 KB
            const int r = idx >> 3, c = idx & 7;
            if (b0 + r < nb) dst[idx] = ld_shared_v4(base + (uint32_t)r * 128u + (((uint32_t)c ^ (uint32_t)(r & 7)) << 4));
        }
        __syncwarp();
    }
}

// =========================================================================== host side

static int launch_reduce(const ReduceJobs& jobs, cudaStream_t s);

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

int num_sms() {
    static int sms[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!sms[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        sms[dev] = v;
    }
    return sms[dev];
}

// Largest number of CTA pairs of the GEMM kernel that can be resident at once (per device).
static int max_pair_clusters() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev]) return cached[dev];
    if (cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmemBytes) !=
        cudaSuccess) {
        fail(LSN_ECUDA, "cudaFuncSetAttribute(max dynamic shared memory) failed");
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * 74, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = kGemmSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel, &cfg);
    if (e != cudaSuccess || n < 1) {
        fail(LSN_ECUDA, "cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
        return 0;
    }
    cached[dev] = n;
    return n;
}

// The epilogue stores 16-byte pieces of output rows: the output (or partial slab) and its
// row stride must keep every piece 16-byte aligned.
static int check_out(const Problem& pr) {
    if (pr.epi == EPI_F32_T) return LSN_OK;   // written element by element
    const int64_t es = pr.epi == EPI_BF16 ? 2 : 4;
    if ((pr.ldo * es) % 16 || pr.ldo < pr.n_valid || (reinterpret_cast<uintptr_t>(pr.out) & 15))
        return fail(LSN_EINVAL, "gemm: output rows must be 16-byte aligned multiples of 16 bytes");
    return LSN_OK;
}

// ------------------------------------------------------------------ split-K planner

namespace {

constexpr int kPlanPairs = 74;                  // CTA pairs of a 148-SM part
constexpr double kPlanEpiSteps = 7.0;           // epilogue of one tile, in k-step times
constexpr double kPlanReduceBytesPerStep = 3.75e6;   // partial bytes reduced per k-step time
constexpr double kPlanReduceLaunchSteps = 8.0;  // the reduction launch itself

struct PlanProblem {
    int64_t units;      // tiles of one split (M-pairs x N tiles)
    int kb;             // k-steps the splits divide (a LoRA tail is left out of the estimate, so
                        // that a problem gets the same splits with and without its tail)
    double part_bytes;  // fp32 partial bytes of one split slab
    double out_bytes;   // bytes of the final output
};

// Estimated launch time (in k-step times) of the static schedule with split counts s[].
double plan_estimate(const PlanProblem* pp, int n, const int* s) {
    int64_t total = 0;
    for (int i = 0; i < n; ++i) total += pp[i].units * s[i];
    const int P = total < kPlanPairs ? (int)total : kPlanPairs;
    if (P < 1) return 0.0;
    double load[kPlanPairs] = {0.0};
    int64_t t = 0;
    double reduce = 0.0;
    bool any_split = false;
    for (int i = 0; i < n; ++i) {
        const int si = s[i];
        for (int j = 0; j < si; ++j) {
            // the tiles of split j: units consecutive schedule slots of equal length
            const double len = (double)((int64_t)pp[i].kb * (j + 1) / si - (int64_t)pp[i].kb * j / si) +
                               kPlanEpiSteps;
            const int64_t c = pp[i].units;
            const int64_t full = c / P, rem = c % P;
            const int start = (int)(t % P);
            for (int q = 0; q < P; ++q) {
                const int64_t pos = (q - start + P) % P;   // order of pair q from the block start
                load[q] += len * (double)(full + (pos < rem ? 1 : 0));
            }
            t += c;
        }
        if (si > 1) {
            any_split = true;
            reduce += (si * pp[i].part_bytes + pp[i].out_bytes) / kPlanReduceBytesPerStep;
        }
    }
    double mk = 0.0;
    for (int q = 0; q < P; ++q) mk = load[q] > mk ? load[q] : mk;
    return mk + (any_split ? reduce + kPlanReduceLaunchSteps : 0.0);
}

std::mutex g_plan_mu;
std::map<std::vector<int64_t>, std::vector<int>> g_plan_cache;

}  // namespace

void GemmPlan::resolve_splits() {
    if (resolved_) return;
    resolved_ = true;
    const int n = p_.n_probs;
    PlanProblem pp[kMaxProbs];
    int s[kMaxProbs], maxs[kMaxProbs];
    bool any_auto = false;
    std::vector<int64_t> key;
    key.reserve(8 * n);
    for (int i = 0; i < n; ++i) {
        const Problem& pr = p_.probs[i];
        const int64_t tm = ((pr.m + kBM - 1) / kBM + 1) / 2, tn = (pr.n + pr.bn - 1) / pr.bn;
        pp[i].units = tm * tn;
        pp[i].kb = pr.ksteps_split;
        pp[i].part_bytes = 4.0 * pr.m * pr.n;
        pp[i].out_bytes = (double)pr.m * pr.n_valid * (pr.epi == EPI_BF16 ? 2 : 4);
        maxs[i] = pr.ksteps_split / 2 < 32 ? pr.ksteps_split / 2 : 32;
        if (maxs[i] < 1) maxs[i] = 1;
        if (pr.splits == kAutoSplits) {
            any_auto = true;
            s[i] = 1;
        } else {
            s[i] = pr.splits < pr.ksteps_split ? pr.splits : (pr.ksteps_split > 0 ? pr.ksteps_split : 1);
            maxs[i] = s[i];
        }
        key.insert(key.end(), {(int64_t)pr.m, (int64_t)pr.n, (int64_t)pr.bn, (int64_t)pr.ksteps_split,
                               (int64_t)pr.epi, (int64_t)pr.n_valid, (int64_t)pr.splits});
    }
    if (any_auto) {
        bool hit = false;
        {
            std::lock_guard<std::mutex> lk(g_plan_mu);
            auto it = g_plan_cache.find(key);
            if (it != g_plan_cache.end()) {
                for (int i = 0; i < n; ++i) s[i] = it->second[i];
                hit = true;
            }
        }
        if (!hit) {
            // coordinate descent over the auto problems, two rounds, smallest split on ties
            double best = plan_estimate(pp, n, s);
            for (int round = 0; round < 2; ++round) {
                for (int i = 0; i < n; ++i) {
                    if (p_.probs[i].splits != kAutoSplits || pp[i].units >= 2 * kPlanPairs) continue;
                    const int keep = s[i];
                    int arg = keep;
                    for (int c = 1; c <= maxs[i]; ++c) {
                        s[i] = c;
                        const double e = plan_estimate(pp, n, s);
                        if (e < best - 1e-9 || (e <= best + 1e-9 && c < arg)) {
                            best = e < best ? e : best;
                            arg = c;
                        }
                    }
                    s[i] = arg;
                    best = plan_estimate(pp, n, s);
                }
            }
            std::lock_guard<std::mutex> lk(g_plan_mu);
            g_plan_cache[key] = std::vector<int>(s, s + n);
        }
    }
    for (int i = 0; i < n; ++i) p_.probs[i].splits = s[i];
}

int GemmPlan::splits_of(int i) {
    if (i < 0 || i >= p_.n_probs) return 0;
    resolve_splits();
    return p_.probs[i].splits;
}

GemmPlan::GemmPlan(bool dry) : dry_(dry) { memset(&p_, 0, sizeof(p_)); }

int GemmPlan::map(const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    if (status_) return -1;
    if (n_maps_ >= kMaxMaps) return status_ = fail(LSN_EINVAL, "gemm: too many tensor maps");
    map_box_[n_maps_] = box_rows;
    if (dry_) return n_maps_++;
    if (!ptr || rows < 1 || cols < 1 || ld < cols || (reinterpret_cast<uintptr_t>(ptr) & 15) ||
        (ld * 2) % 16 || box_rows < 1 || box_rows > 256)
        return status_ = fail(LSN_EINVAL, "gemm: operand must be 16-byte aligned with 16-byte rows");
    EncodeTiledFn enc = encode_fn();
    if (!enc) return status_ = fail(LSN_ECUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = enc(&p_.maps[n_maps_], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return status_ = fail(LSN_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return n_maps_++;
}

int GemmPlan::nf4(const void* base, int64_t n_out, int64_t k_in) {
    if (status_) return -1;
    Nf4Layout L;
    if (n_nf4_ >= kMaxNf4) return status_ = fail(LSN_EINVAL, "gemm: too many NF4 matrices");
    if (dry_) {
        p_.nf4[n_nf4_].n_out = n_out;
        p_.nf4[n_nf4_].k_in = k_in;
        return n_nf4_++;
    }
    if (!base || (reinterpret_cast<uintptr_t>(base) & 15) || !nf4_layout(n_out, k_in, &L))
        return status_ = fail(LSN_EINVAL, "gemm: bad NF4 view");
    const uint8_t* b = static_cast<const uint8_t*>(base);
    Nf4Dev& d = p_.nf4[n_nf4_];
    d.codes = b + L.codes;
    d.absmax = b + L.absmax;
    d.scale = reinterpret_cast<const float*>(b + L.scale);
    d.offset = reinterpret_cast<const float*>(b + L.offset);
    d.n_out = n_out;
    d.k_in = k_in;
    return n_nf4_++;
}

int GemmPlan::problem(int m, int n, int bn, int a_major, int epi, void* out, int64_t ldo, float alpha,
                      int n_valid, int splits, const uint16_t* residual, int64_t ldr) {
    if (status_) return -1;
    if (p_.n_probs >= kMaxProbs) return status_ = fail(LSN_EINVAL, "gemm: too many problems");
    if (bn < kMinBN) bn = kMinBN;   // a pair MMA needs at least one 64-wide atom per CTA
    if (m < 1 || n < 1 || !(bn == 128 || bn == 256) || (!out && !dry_) || n_valid < 1 ||
        n_valid > n || n_valid % 8 || splits < 0 || (reinterpret_cast<uintptr_t>(out) & 15))
        return status_ = fail(LSN_EINVAL, "gemm: bad problem");
    Problem& pr = p_.probs[p_.n_probs];
    memset(&pr, 0, sizeof(pr));
    pr.m = m;
    pr.n = n;
    pr.bn = bn;
    pr.a_major = a_major;
    pr.seg_begin = n_segs_;
    pr.seg_count = 0;
    pr.splits = splits;
    pr.epi = epi;
    pr.out = out;
    pr.ldo = ldo;
    pr.alpha = alpha;
    pr.n_valid = n_valid;
    pr.residual = residual;
    pr.ldr = ldr;
    return p_.n_probs++;
}

int GemmPlan::seg(int a_map, int a_k0, int b_src, int b_idx, int b_k0, int b_n0, int k_len, bool tail) {
    if (status_) return -1;
    if (p_.n_probs == 0 || n_segs_ >= kMaxSegs || k_len < 1 || (a_k0 % 8) || a_map < 0 || a_map >= n_maps_)
        return status_ = fail(LSN_EINVAL, "gemm: bad segment");
    if (!tail && p_.probs[p_.n_probs - 1].ksteps != p_.probs[p_.n_probs - 1].ksteps_split)
        return status_ = fail(LSN_EINVAL, "gemm: a base segment after a tail segment");
    if ((b_src == B_TMA_K || b_src == B_TMA_MN) && (b_idx < 0 || b_idx >= n_maps_))
        return status_ = fail(LSN_EINVAL, "gemm: bad B map");
    {
        // every TMA box must deliver exactly the bytes the kernel expects for its stage
        const Problem& pr = p_.probs[p_.n_probs - 1];
        const int want_a = pr.a_major == A_KMAJOR ? kBM : 64;
        if (map_box_[a_map] != want_a) return status_ = fail(LSN_EINVAL, "gemm: A map box rows mismatch");
        if (b_src == B_TMA_K && map_box_[b_idx] != pr.bn / 2)
            return status_ = fail(LSN_EINVAL, "gemm: K-major B map box rows must be half the N tile");
        if (b_src == B_TMA_MN && map_box_[b_idx] != 64)
            return status_ = fail(LSN_EINVAL, "gemm: MN-major B map box rows must be 64");
    }
    if ((b_src == B_NF4_K || b_src == B_NF4_MN) && (b_idx < 0 || b_idx >= n_nf4_ || b_k0 % 64 || b_n0 % 64))
        return status_ = fail(LSN_EINVAL, "gemm: bad NF4 segment");
    KSeg& s = p_.segs[n_segs_];
    memset(&s, 0, sizeof(s));
    s.a_map = a_map;
    s.a_k0 = a_k0;
    s.b_src = b_src;
    s.b_idx = b_idx;
    s.b_k0 = b_k0;
    s.b_n0 = b_n0;
    s.k_len = k_len;
    s.ksteps = (k_len + kBK - 1) / kBK;
    Problem& pr = p_.probs[p_.n_probs - 1];
    pr.seg_count++;
    pr.ksteps += s.ksteps;
    if (!tail) pr.ksteps_split += s.ksteps;
    return n_segs_++;
}

int GemmPlan::seg_scaled(int a_map, int a_k0, const uint16_t* b_ptr, int b_ld, int b_rows, int k_len,
                         float b_scale) {
    if (status_) return -1;
    if ((!b_ptr && !dry_) || k_len < 8 || k_len > 64 || k_len % 8 || b_ld % 8 ||
        (reinterpret_cast<uintptr_t>(b_ptr) & 15))
        return status_ = fail(LSN_EINVAL, "gemm: bad scaled segment");
    int s = seg(a_map, a_k0, B_SCALED_K, 0, 0, 0, k_len, true);
    if (s < 0) return s;
    p_.segs[s].b_ptr = b_ptr;
    p_.segs[s].b_ld = b_ld;
    p_.segs[s].b_rows = b_rows;
    p_.segs[s].b_scale = b_scale;
    return s;
}

size_t GemmPlan::partial_bytes() {
    if (status_) return 0;
    resolve_splits();
    size_t b = 0;
    for (int i = 0; i < p_.n_probs; ++i) {
        const Problem& pr = p_.probs[i];
        if (pr.splits > 1) b += (size_t)pr.splits * pr.m * pr.n * sizeof(float);
    }
    return b;
}

int GemmPlan::launch(cudaStream_t s, float* partial_ws, size_t ws_bytes) {
    if (status_) return status_;
    if (p_.n_probs == 0) return LSN_OK;
    if (dry_) return LSN_OK;
    resolve_splits();
    // partial-sum slabs for split problems
    struct Final { int epi; void* out; int64_t ldo; float alpha; const uint16_t* res; int64_t ldr; };
    Final fin[kMaxProbs];
    size_t off = 0;
    int tiles = 0;
    for (int i = 0; i < p_.n_probs; ++i) {
        Problem& pr = p_.probs[i];
        if (pr.seg_count == 0) return status_ = fail(LSN_EINVAL, "gemm: problem without segments");
        pr.tiles_m = ((pr.m + kBM - 1) / kBM + 1) / 2;   // M-pairs: one per CTA pair
        pr.tiles_n = (pr.n + pr.bn - 1) / pr.bn;
        // raster group: as many M-pairs as keep their A rows (512 x K bf16 each) within
        // about 48 MB of L2, between 1 and kRasterGroup
        {
            int64_t k_total = 0;
            for (int j = 0; j < pr.seg_count; ++j) k_total += p_.segs[pr.seg_begin + j].k_len;
            const int64_t a_pair = 2 * (int64_t)kBM * k_total * 2;
            int rg = (int)((48ll << 20) / (a_pair > 0 ? a_pair : 1));
            pr.raster = rg < 1 ? 1 : (rg > kRasterGroup ? kRasterGroup : rg);
        }
        pr.tile_begin = tiles;
        tiles += pr.tiles_m * pr.tiles_n * pr.splits;
        fin[i] = {pr.epi, pr.out, pr.ldo, pr.alpha, pr.residual, pr.ldr};
        if (pr.splits > 1) {
            const size_t need = (size_t)pr.splits * pr.m * pr.n * sizeof(float);
            if (!partial_ws || off + need > ws_bytes)
                return status_ = fail(LSN_ENOMEM, "gemm: split-K workspace too small");
            pr.out = reinterpret_cast<uint8_t*>(partial_ws) + off;
            pr.ldo = pr.n;
            pr.part_stride = (int64_t)pr.m * pr.n;
            pr.epi = EPI_PARTIAL;
            pr.residual = nullptr;
            off += need;
        }
    }
    p_.total_tiles = tiles;
    for (int i = 0; i < p_.n_probs; ++i) {
        int rc = check_out(p_.probs[i]);
        if (rc) return status_ = rc;
    }
    memcpy(p_.levels, nf4_levels(), sizeof(p_.levels));
    p_.err = ext_err_ ? ext_err_ : device_error_word();
    if (!p_.err) return LSN_ECUDA;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = kGemmSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = max_pair_clusters();
    if (clusters < 1) return status_ = LSN_ECUDA;
    if (tiles < clusters) clusters = tiles;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    void* prof = profile_begin(s);
    LSN_CUDA_TRY(cudaLaunchKernelEx(&cfg, tc_gemm_kernel, p_));
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    if (prof) {
        double flops = 0.0;
        for (int i = 0; i < p_.n_probs; ++i) {
            const Problem& pr = p_.probs[i];
            double k = 0.0;
            for (int j = 0; j < pr.seg_count; ++j) k += (double)p_.segs[pr.seg_begin + j].k_len;
            flops += 2.0 * (double)pr.m * (double)pr.n_valid * k;
        }
        profile_end(prof, s, flops);
    }
    ReduceJobs jobs;
    memset(&jobs, 0, sizeof(jobs));
    for (int i = 0; i < p_.n_probs; ++i) {
        const Problem& pr = p_.probs[i];
        if (pr.epi != EPI_PARTIAL) continue;
        ReduceJob& j = jobs.j[jobs.count++];
        j.partial = static_cast<const float*>(pr.out);
        j.out = fin[i].out;
        j.residual = fin[i].res;
        j.part_stride = pr.part_stride;
        j.ldo = fin[i].ldo;
        j.ldr = fin[i].ldr;
        j.splits = pr.splits;
        j.m = pr.m;
        j.n = pr.n;
        j.epi = fin[i].epi;
        j.n_valid = pr.n_valid;
        j.alpha = fin[i].alpha;
        j.begin = jobs.total;
        jobs.total += (int64_t)pr.m * (pr.n_valid / 4);
    }
    return launch_reduce(jobs, s);
}

static int launch_reduce(const ReduceJobs& jobs, cudaStream_t s) {
    if (jobs.count == 0) return LSN_OK;
    int64_t blocks = (jobs.total + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    gemm_reduce_kernel<<<(unsigned)blocks, 256, 0, s>>>(jobs);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

int nf4_view_dev(const void* base, int64_t n_out, int64_t k_in, Nf4Dev* out) {
    Nf4Layout L;
    if (!base || !out || (reinterpret_cast<uintptr_t>(base) & 15) || !nf4_layout(n_out, k_in, &L))
        return fail(LSN_EINVAL, "nf4: bad NF4 view");
    const uint8_t* b = static_cast<const uint8_t*>(base);
    out->codes = b + L.codes;
    out->absmax = b + L.absmax;
    out->scale = reinterpret_cast<const float*>(b + L.scale);
    out->offset = reinterpret_cast<const float*>(b + L.offset);
    out->n_out = n_out;
    out->k_in = k_in;
    return LSN_OK;
}

int nf4_dequant_many(const Nf4Dev* w, uint16_t* const* out, int n, cudaStream_t s) {
    if (n < 1 || n > kMaxNf4 || !w || !out) return fail(LSN_EINVAL, "nf4_dequant_many: bad matrix count");
    DequantParams p;
    memset(&p, 0, sizeof(p));
    p.n = n;
    memcpy(p.lvl.v, nf4_levels(), sizeof(p.lvl.v));
    int64_t g = 0;
    for (int i = 0; i < n; ++i) {
        if (!out[i] || (reinterpret_cast<uintptr_t>(out[i]) & 15) || w[i].n_out < 1 || w[i].k_in < 64 || w[i].k_in % 64)
            return fail(LSN_EINVAL, "nf4_dequant_many: bad output or shape");
        p.w[i] = w[i];
        p.out[i] = out[i];
        p.group_begin[i] = g;
        g += (w[i].n_out * (w[i].k_in / 64) + 31) / 32;
    }
    p.group_begin[n] = g;
    int64_t blocks = (g + kDequantWarps - 1) / kDequantWarps;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    nf4_dequant_many_kernel<<<(unsigned)blocks, kDequantWarps * 32, 0, s>>>(p);
    note_launch();
    LSN_CUDA_TRY(cudaGetLastError());
    return LSN_OK;
}

}  // namespace lsn
