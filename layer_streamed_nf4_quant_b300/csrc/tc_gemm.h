// Grouped tcgen05 GEMM with an NF4-dequantising operand producer (internal interface).
//
// One launch runs up to kMaxProbs independent GEMM "problems"
//     D[m x n] = sum over K-segments of  A_seg[m x k] * B_seg[n x k]^T
// on a persistent grid.  A always arrives by TMA (K-major or MN-major tiles).  B arrives by
// TMA (dense bf16), is decoded from packed NF4 by producer warps straight into the
// swizzled shared-memory operand layout (K-major for y = x W^T, MN-major for dX = dY W), or
// is loaded and scaled by the producer warps (the LoRA B factor times s).  Accumulation is
// fp32 in TMEM; the epilogue writes bf16, fp32, fp32 added into the output, fp32 transposed,
// or fp32 split-K partials that one reduction launch per GEMM launch sums in a fixed order.
// Split-K counts are chosen per launch by a planner that replays the kernel's static schedule
// on a fixed 148-SM machine (GemmPlan::resolve_splits).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lsn {

constexpr int kBM = 256;        // rows per CTA tile: two 128-row blocks, each half of a pair MMA
constexpr int kBK = 64;         // contraction per stage: one NF4 block, one 128-byte row
constexpr int kStages = 4;
constexpr int kMaxBN = 256;
constexpr int kMinBN = 128;     // a pair MMA splits B's N over the two CTAs in 64-wide atoms
constexpr int kStageABytes = kBM * kBK * 2;
constexpr int kStageBBytes = (kMaxBN / 2) * kBK * 2;   // this CTA's half of the B tile
constexpr int kGemmThreads = 512;
constexpr int kMaxMaps = 16;
constexpr int kMaxNf4 = 8;
constexpr int kMaxSegs = 20;
constexpr int kMaxProbs = 16;
// splits argument of GemmPlan::problem: let the launch planner choose the split-K count
constexpr int kAutoSplits = 0;

enum ASrc : int { A_KMAJOR = 0, A_MNMAJOR = 1 };
enum BSrc : int {
    B_NF4_K = 0,     // packed NF4 W [n_out x k_in]; tile rows = W rows (output n)
    B_NF4_MN = 1,    // packed NF4 W; contraction over W rows, output over W columns
    B_TMA_K = 2,     // dense bf16 [n x k] via TMA, K-major
    B_TMA_MN = 3,    // dense bf16 [k x n] via TMA, MN-major
    B_SCALED_K = 4,  // dense bf16 [n x k<=64] loaded and multiplied by b_scale
};
enum Epi : int {
    EPI_BF16 = 0,     // out bf16 = alpha*acc (+ residual)
    EPI_F32 = 1,      // out fp32 = alpha*acc
    EPI_F32_ACC = 2,  // out fp32 += alpha*acc
    EPI_F32_T = 3,    // out fp32 [n x m] (transposed) = alpha*acc
    EPI_PARTIAL = 4,  // partial fp32 [split][m][n] = acc (reduced by gemm_reduce)
};

struct KSeg {
    int a_map;         // tensor map of A
    int a_k0;          // contraction offset into A (elements)
    int b_src;
    int b_idx;         // NF4 view index (B_NF4_*) or tensor map (B_TMA_*)
    int b_k0;          // contraction offset into B
    int b_n0;          // output offset into B
    int k_len;         // contraction length of the segment
    int ksteps;        // ceil(k_len / 64)
    const uint16_t* b_ptr;  // B_SCALED_K: rows of length b_ld
    int b_ld;
    int b_rows;        // B_SCALED_K: valid rows
    float b_scale;
};

struct Problem {
    int m, n;          // output rows / columns
    int bn;            // N tile: 64, 128 or 256
    int a_major;
    int seg_begin, seg_count;
    int ksteps;        // total over the segments
    int ksteps_split;  // k-steps of the leading (non-tail) segments, which the splits divide;
                       // the tail segments' k-steps all go to the last split
    int splits;
    int tiles_m, tiles_n;
    int raster;        // M-pairs per raster group (set at launch)
    int tile_begin;
    int epi;
    void* out;
    int64_t ldo;       // output leading dimension (elements); for EPI_F32_T: row stride of out
    const uint16_t* residual;
    int64_t ldr;
    float alpha;
    int n_valid;       // columns to write
    int64_t part_stride;  // EPI_PARTIAL: elements per split slab (m * n)
};

struct Nf4Dev {
    const uint8_t* codes;
    const uint8_t* absmax;
    const float* scale;
    const float* offset;
    int64_t n_out, k_in;
};

struct GemmParams {   // 128-byte aligned through CUtensorMap
    CUtensorMap maps[kMaxMaps];
    Nf4Dev nf4[kMaxNf4];
    KSeg segs[kMaxSegs];
    Problem probs[kMaxProbs];
    float levels[16];
    uint32_t* err;
    int n_probs;
    int total_tiles;
};

// Host-side assembly of one grouped launch.
class GemmPlan {
   public:
    // dry: shapes only (no pointers are checked, no tensor maps encoded, nothing launched);
    // used to size workspaces with exactly the split decisions of the real launch.
    explicit GemmPlan(bool dry = false);
    // Dense bf16 matrix [rows x cols] (row stride ld elements) as an A or B operand.
    // kmajor: box 64 (cols) x box_rows; otherwise box 64 x 64.  Returns the map index or < 0.
    int map(const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows);
    int nf4(const void* base, int64_t n_out, int64_t k_in);
    // Starts a problem; segments added next belong to it.  splits = kAutoSplits leaves the
    // split-K count to the launch planner (see resolve_splits).
    int problem(int m, int n, int bn, int a_major, int epi, void* out, int64_t ldo, float alpha,
                int n_valid, int splits = kAutoSplits, const uint16_t* residual = nullptr,
                int64_t ldr = 0);
    // tail: a LoRA contraction appended to the base one.  Tail segments follow every
    // non-tail segment of their problem, and all their k-steps belong to the last split, so
    // the base k-steps are split exactly as in the same problem without the tail.
    int seg(int a_map, int a_k0, int b_src, int b_idx, int b_k0, int b_n0, int k_len, bool tail = false);
    // Always a tail segment.
    int seg_scaled(int a_map, int a_k0, const uint16_t* b_ptr, int b_ld, int b_rows, int k_len,
                   float b_scale);
    // Bytes of split-K partial workspace the launch needs (after the planner's choice).
    size_t partial_bytes();
    // Split-K count of problem i (after the planner's choice).
    int splits_of(int i);
    // Launches the GEMM and the split reductions (a dry plan only validates).
    int launch(cudaStream_t s, float* partial_ws, size_t ws_bytes);
    int status() const { return status_; }
    // Device error word the kernel reports bounded-wait timeouts into (default: the
    // library's lazily allocated per-device word).
    void set_error_word(uint32_t* w) { ext_err_ = w; }

   private:
    // Chooses the split count of every kAutoSplits problem (once per plan).  The estimate
    // replays the kernel's static schedule -- tile t on CTA pair t mod P, every split of a
    // problem in order -- on a fixed P = 74 pairs (a 148-SM part, whatever the device), so
    // the choice, and with it the summation order, never depends on the device; it adds the
    // time the fixed-order reduction needs for the fp32 partial slabs.  Among equal
    // estimates the smaller split count wins.  Choices are cached by problem shapes.
    void resolve_splits();
    bool resolved_ = false;
    GemmParams p_;
    int n_maps_ = 0, n_nf4_ = 0, n_segs_ = 0;
    int map_box_[kMaxMaps] = {0};   // box rows of each map (the kernel's byte counts rely on it)
    int status_ = 0;
    bool dry_ = false;
    uint32_t* ext_err_ = nullptr;
};

int num_sms();

// Work units of a problem: one per CTA pair = two 256-row M tiles x one N tile (>= 128 wide).
inline int pair_tiles(int64_t m, int64_t n, int bn) {
    const int64_t bnn = bn < kMinBN ? kMinBN : bn;
    const int64_t mt = (m + kBM - 1) / kBM;
    return (int)(((mt + 1) / 2) * ((n + bnn - 1) / bnn));
}


struct Nf4Levels {
    float v[16];
};
// Device view of a packed NF4 matrix at base (16-byte aligned).
int nf4_view_dev(const void* base, int64_t n_out, int64_t k_in, Nf4Dev* out);
// Decodes n (<= kMaxNf4) packed NF4 matrices into dense row-major bf16 [n_out x k_in] at
// out[i] (16-byte aligned), in one launch: the same values, bit for bit, that the GEMM's
// producer warps write into its operand tiles.  Each warp decodes 32 consecutive blocks
// (4 KB of output) and stores them through shared memory in whole 512-byte rows.
int nf4_dequant_many(const Nf4Dev* w, uint16_t* const* out, int n, cudaStream_t s);

}  // namespace lsn
