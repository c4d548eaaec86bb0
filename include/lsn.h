/*
 * lsn.h -- C ABI of the layer-streamed NF4-LoRA library (liblsn.so), B300 / sm_103a.
 *
 * What the library computes comes from the pages on Soup's layer streaming:
 *   [P1] "Can You Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's Layer Streaming Explained"
 *   [P2] "Fine tune an 8B model on a 4GB laptop GPU (Soup setup)"
 *   [P4] the rug.gal radar item "soup-fine-tune-8b-4gb-laptop-gpu-layer-streaming"
 * and from the workload description they are measured on (NF4 blocksize 64, uint8 absmax
 * per block, fp32 scale + offset per 256 absmax; Llama-3.1-8B-shaped synthetic layers).
 *
 * Conventions (all entry points):
 *   - Every function returns an int status: LSN_OK (0) or a negative LSN_E* code.  Nothing
 *     aborts, throws across the ABI or traps on the device.  lsn_last_error() returns a
 *     thread-local message for the last failure on the calling thread.
 *   - bf16 tensors are passed as uint16_t pointers to bf16 bit patterns; every matrix is
 *     row-major with the stated shape and a row stride equal to its width.
 *   - "device" pointers are CUDA device memory of the current device, owned by the caller.
 *     "host" pointers are host memory owned by the caller.  The library owns only the
 *     opaque pool handle, its CUDA events and a per-device error word.
 *   - `stream` arguments are cudaStream_t values passed as void*.  Device work is enqueued
 *     asynchronously on that stream; inputs must stay valid until it completes.
 *   - Kernels never spin without a bound.  A device-side failure (a bounded wait that ran out,
 *     a layer image whose tag does not match the expected layer) is recorded in the device
 *     error word and reported by the next lsn_check() or stream_pool_wait() as LSN_ECORRUPT
 *     or LSN_ETIMEOUT.
 */
#ifndef LSN_H
#define LSN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LSN_OK        0
#define LSN_EINVAL   -1   /* bad argument: null pointer, shape, alignment, unpinned store   */
#define LSN_ENOMEM   -2   /* a host allocation or the caller's workspace is too small        */
#define LSN_ECUDA    -3   /* a CUDA runtime/driver call failed                               */
#define LSN_ETIMEOUT -4   /* a bounded wait (host poll or device spin) ran out                */
#define LSN_ESTATE   -5   /* call out of order: e.g. prefetch into a slot still in use        */
#define LSN_ECORRUPT -6   /* a layer image tag did not match the layer the kernels expected   */

/* Thread-local text of the last error on the calling thread ("" if none).  Never NULL. */
const char* lsn_last_error(void);

/* ABI version of this header (incremented on any incompatible change). */
int lsn_abi_version(void);

/* Reads and clears the device error word of the current device after synchronising
 * `stream` (NULL: the legacy default stream).  Returns LSN_OK, LSN_ETIMEOUT (a kernel's
 * bounded wait ran out) or LSN_ECORRUPT (layer tag mismatch); LSN_ECUDA if the
 * synchronisation itself failed.  `detail` (nullable, host) receives the raw word.  The
 * error word of lora_nf4_fwd_static_scratch (if that entry point has run on this device) is
 * read and cleared as well, so a timeout of any call is reported here. */
int lsn_check(void* stream, uint32_t* detail);

/* Launch accounting and opt-in kernel timing (process-wide).
 * lsn_launch_count: number of kernels this library has launched so far (all devices).
 * lsn_profile_enable(1): from then on every GEMM launch is bracketed by two CUDA events on
 * its own stream and its algorithmic FLOPs (2 * m * n * k summed over its problems, no
 * padding) are recorded; lsn_profile_read synchronises on those events, adds their device
 * times up and (reset != 0) clears the totals. */
typedef struct {
    uint64_t gemm_launches;   /* timed GEMM launches since the last reset */
    double   gemm_ms;         /* summed device time of those launches     */
    double   gemm_flops;      /* summed algorithmic FLOPs of those launches */
} lsn_profile;
uint64_t lsn_launch_count(void);
int lsn_profile_enable(int on);
int lsn_profile_read(lsn_profile* out, int reset);

/* ------------------------------------------------------------------------------ NF4 ---
 * NF4 storage of the frozen base ([P1] "Why NF4 matters so much": QLoRA's 4-bit NormalFloat,
 * about a quarter of bf16).  Codebook: the 16 QLoRA levels -- standard-normal quantiles at
 * 8 evenly spaced probabilities from delta = 1 - (1/30 + 1/32)/2 towards 1/2 on the positive
 * side, 7 on the negative side, plus an exact zero -- divided by the largest, rounded once
 * to fp32.  Quantisation of W [n_out x k_in] (row-major, fp32):
 *   blocks of 64 consecutive weights along k_in; absmax a_b = max |w| (fp32);
 *   groups of 256 consecutive blocks: lo = min a_b, hi = max a_b,
 *   scale = smallest fp32 >= (hi - lo)/255, q_b = ceil((a_b - lo)/scale) clamped to 0..255,
 *   a'_b = fp32(fp32(q_b*scale) + lo); q_b is raised while a'_b < a_b, and the group's scale
 *   raised one fp32 ulp (group redone) if q_b would pass 255;
 *   code = nearest level of w / a'_b (fp64), ties to the lower level; the zero level
 *   when a'_b = 0;
 *   dequantised weight = bf16_rne(fp32(level[code] * a'_b)).
 * Packed matrix (all offsets from the start of the matrix, every section 16-byte aligned):
 *   codes  : n_out*k_in/2 bytes, weight 2j in the high nibble of byte j
 *   absmax : n_out*k_in/64 uint8 codes q_b
 *   scale  : G fp32 values,  G = ceil(n_out*k_in/64/256)
 *   offset : G fp32 values (lo)
 */

/* Writes the 16 fp32 levels (ascending) into out[16] (host). */
int lsn_nf4_codebook(float* out);

/* Bytes of one packed matrix (0 if k_in is not a positive multiple of 64 or n_out < 1). */
size_t nf4_packed_bytes(int64_t n_out, int64_t k_in);

/* Host quantiser.  W: host fp32 [n_out x k_in], finite (NaN/Inf -> LSN_EINVAL);
 * k_in % 64 == 0.  dst: host buffer of dst_bytes >= nf4_packed_bytes() (may be pinned; it
 * is written with plain stores).  n_threads <= 0 uses the hardware concurrency. */
int nf4_pack(const float* W, int64_t n_out, int64_t k_in, void* dst, size_t dst_bytes,
             int n_threads);

/* A packed matrix in device memory: base points at its codes section (16-byte aligned). */
typedef struct {
    const void* base;
    int64_t n_out;
    int64_t k_in;
} nf4_view;

/* Test entry: dequantises W into out (device bf16 [n_out x k_in]) with the same decode the
 * GEMMs use.  The GEMMs themselves never write dequantised weights to HBM. */
int nf4_dequant(const nf4_view* W, uint16_t* out, void* stream);

/* ---------------------------------------------------------------- LoRA linear (one W) ---
 * [P1] "How Soup's layer streaming actually works", step 1 "The base model is frozen":
 * W is frozen, only the LoRA factors train.  With s = scale (alpha / r):
 *   forward : T = bf16(X A^T);  Y = bf16(X W^T + s T B^T [+ residual])
 *             (A == B == NULL in lora_nf4_fwd: the adapter is disabled, Y = bf16(X W^T
 *             [+ residual]) and T_out is not written and may be NULL.  The LoRA k-steps
 *             are appended to the last split-K slice, so the base contraction is summed in
 *             the same order with or without the adapter: B = 0 gives the adapter-disabled
 *             Y bit for bit.)
 *   backward: dT = bf16(s dY B); dB = s dY^T T; dA = dT^T X; dX = dY W + dT A   (no dW)
 * fp32 accumulation on the tensor cores; every reduction has a fixed order (split-K
 * partials are summed in split order; accumulate_dX adds each element exactly once, so the
 * order of those additions never matters), so repeated calls give identical bits.  s is
 * applied exactly when it is a power of two.
 * Shapes: X [M x k_in], A [r x k_in], B [n_out x r], dY/Y/residual [M x n_out], T [M x r];
 * dX [M x k_in] fp32, dA [r x k_in] fp32, dB [n_out x r] fp32 (overwritten).
 * Limits: k_in % 64 == 0, n_out % 8 == 0, r in {8, 16, 24, ..., 64}, M >= 1.
 * All pointers are device pointers and 16-byte aligned; ws is a device workspace of at
 * least lora_nf4_workspace_bytes() bytes (LSN_ENOMEM if smaller). */
size_t lora_nf4_workspace_bytes(int64_t M, int64_t n_out, int64_t k_in, int r);

int lora_nf4_fwd(const nf4_view* W, const uint16_t* X, int64_t M,
                 const uint16_t* A, const uint16_t* B, int r, float scale,
                 const uint16_t* residual /* nullable */, uint16_t* Y, uint16_t* T_out,
                 void* ws, size_t ws_bytes, void* stream);

/* Diagnostics (host only, no device work): the split-K counts lora_nf4_fwd uses for this shape
 * in its two launches -- T = X A^T and Y = X W^T + s T B^T -- and the fp32 partial-sum bytes
 * each launch needs (0 when it is not split).  The counts come from the library's launch
 * planner, which replays the GEMM's static tile schedule on a fixed 148-SM machine, so they
 * (and the summation order they fix) do not depend on the device.  Every output pointer is
 * nullable.  LSN_EINVAL for a shape lora_nf4_fwd refuses. */
int lora_nf4_fwd_plan(int64_t M, int64_t n_out, int64_t k_in, int r, int* t_splits, int* y_splits,
                      size_t* t_partial_bytes, size_t* y_partial_bytes);

/* lora_nf4_fwd for callers that cannot allocate device memory (a plug-in inside a framework
 * that owns all device memory, or a serving path that must not enter the allocator).  The
 * pages have no counterpart of it.  Same arguments and results as lora_nf4_fwd, bit for bit,
 * but no workspace: the split-K partial sums go to a 16 MiB file-scope __device__ buffer and
 * device-side wait timeouts to a file-scope __device__ word, both held by every GPU that
 * loads the library until the process exits.  It calls no cudaMalloc/cudaFree (with the
 * opt-in profiler off).  Its first call on each device looks the buffers' addresses up with
 * cudaGetSymbolAddress and clears the word (synchronously), so make that first call before
 * any stream capture.  All calls on a device share the buffer: calls whose kernels overlap on
 * the GPU race.  A shape whose split-K partials exceed 16 MiB is rejected with LSN_ENOMEM.
 * A, B and T_out are required here (no adapter-disabled mode); every pointer is checked for
 * NULL and 16-byte alignment exactly as in lora_nf4_fwd (LSN_EINVAL).
 * device_status (host, nullable): if given, the call synchronises `stream`, stores the word
 * there, clears it and returns LSN_ETIMEOUT if a device wait ran out.  A timeout of an earlier
 * call made without device_status that lsn_check() has not collected yet is reported by that
 * read too. */
int lora_nf4_fwd_static_scratch(const nf4_view* W, const uint16_t* X, int64_t M,
                                const uint16_t* A, const uint16_t* B, int r, float scale,
                                const uint16_t* residual /* nullable */, uint16_t* Y,
                                uint16_t* T_out, uint32_t* device_status, void* stream);

/* accumulate_dX != 0 adds into dX instead of overwriting it.  dX may be NULL (skipped). */
int lora_nf4_bwd(const nf4_view* W, const uint16_t* X, const uint16_t* T, const uint16_t* dY,
                 int64_t M, const uint16_t* A, const uint16_t* B, int r, float scale,
                 float* dX, int accumulate_dX, float* dA, float* dB,
                 void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------- two-slot stream pool ---
 * [P1] "How Soup's layer streaming actually works", steps 2-4, and [P2] "Step 2, train":
 * the packed base lives in pinned host RAM; each decoder layer is copied into one of two
 * reusable VRAM buffers while the previous layer computes, prefetched one ahead, and every
 * layer is read again in the backward sweep.
 * Slots are used round-robin in prefetch order, starting at `first_slot`.  A prefetch
 * enqueues, on copy_stream: a wait on the slot's slot-free event (recorded by the release
 * of its previous layer), one cudaMemcpyAsync of the layer image, and the copy-done event.
 * stream_pool_wait makes the compute stream wait on copy-done and returns the slot's device
 * address; stream_pool_release records slot-free on the compute stream. */
typedef struct lsn_pool lsn_pool;

typedef struct {
    uint64_t bytes_copied;    /* host->device bytes of completed prefetches            */
    uint64_t copies;          /* completed prefetches                                  */
    uint64_t skipped;         /* prefetches satisfied by a layer already in its slot    */
    double   copy_ms;         /* summed device time of the copies (copy-stream events) */
    double   wait_ms;         /* summed host time spent polling in stream_pool_wait    */
} lsn_pool_stats;

/* pinned_store: host memory from cudaHostAlloc/cudaMallocHost or cudaHostRegister, of
 * store_bytes (LSN_EINVAL if it is not page-locked); layer l occupies
 * [layer_offset[l], layer_offset[l] + layer_bytes) of it.  layer_offset (host array of
 * n_layers) is copied.  slot0/slot1: device buffers of at least layer_bytes, 256-byte
 * aligned, owned by the caller.  reuse_resident != 0 lets a prefetch of the layer that a
 * slot already holds skip the copy.  first_slot is 0 or 1. */
int stream_pool_create(const void* pinned_store, size_t store_bytes, const size_t* layer_offset,
                       size_t layer_bytes, int n_layers, void* slot0, void* slot1,
                       void* copy_stream, int first_slot, int reuse_resident, lsn_pool** out);
/* LSN_ESTATE if the slot this prefetch would use still holds a layer that was prefetched
 * or waited on and not released. */
int stream_pool_prefetch(lsn_pool* pool, int layer);
/* Makes compute_stream wait for the layer's copy and returns its device address in
 * *dev_image.  timeout_ms > 0 also polls the copy on the host and returns LSN_ETIMEOUT if it
 * has not finished in time (the stream wait is enqueued either way).  LSN_ESTATE if the
 * layer was not prefetched. */
int stream_pool_wait(lsn_pool* pool, int layer, void* compute_stream, const void** dev_image,
                     int timeout_ms);
/* Records slot-free for the layer's slot on compute_stream (after its last kernel). */
int stream_pool_release(lsn_pool* pool, int layer, void* compute_stream);
/* Synchronises the copy stream and fills *out. */
int stream_pool_stats(lsn_pool* pool, lsn_pool_stats* out);
int stream_pool_reset_stats(lsn_pool* pool);
/* Sub-layer streaming.  Splits every layer image into n_chunks byte ranges [chunk_offset[c],
 * chunk_offset[c + 1]) with chunk_offset[0] = 0, ascending, 256-byte aligned, the last chunk
 * ending at layer_bytes (chunk_offset: host array of n_chunks, 1 <= n_chunks <= 8; ignored for
 * n_chunks = 1).  A prefetch then issues one cudaMemcpyAsync per chunk, each followed by that
 * chunk's copy-done event, so the compute stream can start on the chunks it needs first
 * (stream_pool_wait_range) while the others are still copying.  Bytes and results are the
 * same as with whole-layer copies.  LSN_ESTATE while a slot holds a prefetched or waited
 * layer (call it before the first prefetch or after every layer is released); it forgets the
 * slots' contents.  [P1] "Did a correctness bug invalidate the Llama 3.1 8B result?": the
 * pages' wrong-gradient bug lived in how large layers were transferred; the tests check the
 * chunked stream bit for bit against the resident run on a layer above 172 MiB. */
int stream_pool_set_chunks(lsn_pool* pool, int n_chunks, const size_t* chunk_offset);
/* stream_pool_prefetch with the chunk order: ascending (reverse == 0) or descending.  The
 * reverse sweep of layer_stack_step copies o and down (the end of the image) first because
 * its backward needs them first.  stream_pool_prefetch(pool, l) is
 * stream_pool_prefetch_ex(pool, l, 0). */
int stream_pool_prefetch_ex(lsn_pool* pool, int layer, int reverse);
/* stream_pool_wait for the bytes [begin, end) of the layer image only: the compute stream
 * waits for the copy-done event of the last chunk, in this prefetch's copy order, that covers
 * the range (chunks land in copy order on the one copy stream).  LSN_EINVAL if the range is
 * empty or outside the image.  stream_pool_wait is the range [0, layer_bytes). */
int stream_pool_wait_range(lsn_pool* pool, int layer, size_t begin, size_t end, void* compute_stream,
                           const void** dev_image, int timeout_ms);
/* Statistics of one chunk index over all layers (synchronises the copy stream): bytes_copied,
 * copies and copy_ms of that chunk's transfers; the other fields are zero. */
int stream_pool_chunk_stats(lsn_pool* pool, int chunk, lsn_pool_stats* out);
/* Fault injection for tests: every later prefetch first runs a host callback on the copy
 * stream that sleeps `usec` microseconds (0 turns it off, at most 10 s).  Results must not
 * change; only the copies come later. */
int stream_pool_set_copy_delay_us(lsn_pool* pool, int usec);
/* Synchronises the copy stream and frees the handle and its events (not the slots). */
int stream_pool_destroy(lsn_pool* pool);

/* ---------------------------------------------------------------- synthetic layer stack ---
 * One decoder layer (Llama-3.1-8B-shaped, no attention; o acts on q directly):
 *   h = bf16(x * (mean(x^2) + eps)^-1/2)                 (unit RMSNorm weight)
 *   p = bf16(h W_p^T + s T_p B_p^T),  T_p = bf16(h A_p^T)    for p in q, k, v, gate, up
 *   a = bf16(silu(gate) * up)
 *   x' = bf16(x + q W_o^T + s T_o B_o^T + a W_d^T + s T_d B_d^T),
 *        T_o = bf16(q A_o^T), T_d = bf16(a A_d^T)
 * loss = 0.5 mean(x_L^2) + sum_l c (mean(k_l^2) + mean(v_l^2))
 * layer_stack_step runs the forward sweep, the loss and the reverse backward sweep and writes
 * every layer's dA_p, dB_p.  With a pool, every layer of both sweeps comes through the pool
 * (prefetched one ahead); with pool == NULL the layers are read from a resident device store.
 * The same kernels run in the same order either way, so the results are bit-identical.
 *
 * Layer image (host store, slot, resident store): a 64-byte header {uint32 magic 0x314E534C
 * ("LSN1"), uint32 layer index, uint64 image bytes, uint32 d_model, d_kv, d_ff, ...} and then
 * the seven packed matrices q, k, v, gate, up, o, down, each starting at a 256-byte aligned
 * offset (lsn_layer_image_offsets).
 * LoRA blob of one layer (bf16 device; grads use the same layout in fp32):
 *   A_q, A_k, A_v, A_gate, A_up, A_o, A_down  (each [r x K_p])  then
 *   B_q, B_k, B_v, B_gate, B_up, B_o, B_down  (each [N_p x r])
 * Projections always come in the order q, k, v, gate, up, o, down ("canonical order"). */
typedef struct {
    int32_t n_layers;
    int32_t d_model;      /* 4096  */
    int32_t d_kv;         /* 1024  */
    int32_t d_ff;         /* 14336 */
    int32_t rank;         /* r: 8..64, multiple of 8 */
    float   lora_alpha;   /* s = lora_alpha / rank */
    float   rms_eps;      /* 1e-5 */
    float   kv_loss_coef; /* c = 1e-3 */
} lsn_stack_desc;

/* Bytes of one layer image, and the byte offsets of the seven matrices within it
 * (offsets[7] in canonical order). */
size_t lsn_layer_image_bytes(const lsn_stack_desc* desc);
int lsn_layer_image_offsets(const lsn_stack_desc* desc, size_t* offsets);
/* Host packer of one layer image: W[p] are host fp32 matrices [N_p x K_p] in canonical
 * order.  Writes the header and the seven packed matrices. */
int lsn_layer_image_pack(const lsn_stack_desc* desc, int layer, const float* const* W,
                         void* dst, size_t dst_bytes, int n_threads);
/* Elements of one layer's LoRA blob (A's then B's), and the element offsets of A_p / B_p
 * (offsets[14]: the seven A_p then the seven B_p, canonical order). */
size_t lsn_lora_elems(const lsn_stack_desc* desc);
int lsn_lora_offsets(const lsn_stack_desc* desc, size_t* offsets);
/* Device workspace bytes layer_stack_step needs for M tokens (stored activations of every
 * layer plus backward scratch). */
size_t lsn_stack_workspace_bytes(const lsn_stack_desc* desc, int64_t M);

/* pool: a pool over the desc->n_layers images, or NULL to read resident_store (device,
 * layer l at byte offset l * lsn_layer_image_bytes()).
 * x0: device bf16 [M x d_model].  lora: host array of n_layers device pointers to LoRA blobs.
 * grads: host array of n_layers device pointers to fp32 gradient blobs (overwritten).
 * loss_out: device fp32 [1].  x_out (nullable): device bf16 [M x d_model] receives x_L.
 * dx0 (nullable): device fp32 [M x d_model] receives dloss/dx0.
 * ws: device workspace of ws_bytes >= lsn_stack_workspace_bytes(desc, M). */
int layer_stack_step(lsn_pool* pool, const void* resident_store, const lsn_stack_desc* desc,
                     const uint16_t* x0, int64_t M, const uint16_t* const* lora,
                     float* const* grads, float* loss_out, uint16_t* x_out, float* dx0,
                     void* ws, size_t ws_bytes, void* stream);

/* Options of layer_stack_step_ex (zero-initialise; NULL means all zero).
 *
 * recompute: checkpointed backward ([P1] "How Soup's layer streaming actually works", step 4:
 *   under gradient checkpointing the backward recomputes the forward and so reads every
 *   layer again).  Only x_l is kept per layer; the reverse sweep refills h, rstd, the
 *   projections, a and the T's of each layer from its re-streamed weights before its
 *   backward.  The workspace shrinks from about 115.6 KB to 8 KB per token per layer (plus
 *   one layer's set); results are bit-identical to the stored-activation run.
 * reference_pass: preference-pair reuse ([P4] "In detail": the DPO reference model is the
 *   same base stream with the adapter disabled).  In the forward sweep each layer also runs
 *   the frozen base alone (the LoRA contraction steps are left out, not multiplied by zero)
 *   on its own residual stream from x0, against the same streamed slot before it is
 *   released, so no layer is copied more often than without it.  The backward and the loss
 *   concern the policy (adapter) branch only; x_ref_out receives the reference output. */
/* AdamW hyper-parameters (decoupled weight decay); step = t >= 1 sets the bias corrections. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int32_t step;
} lsn_adamw_hparams;

/* Optimizer state for the fused update of layer_stack_step_ex: per layer, device fp32
 * arrays of lsn_lora_elems() (master copy, first and second moment) and the bf16 LoRA blob
 * that receives bf16(master) after the update (normally the blob the step reads). */
typedef struct {
    lsn_adamw_hparams hp;
    float* const* master;
    float* const* m;
    float* const* v;
    uint16_t* const* lora_out;
} lsn_adamw_state;

/* Host callback of layer_stack_step_ex: called on the calling thread right after the
 * backward of `layer` (its dA and dB in grad, `elems` fp32 values) has been enqueued on
 * `stream`, and before that layer's fused AdamW update (if any) is enqueued.  It may enqueue
 * work on `stream` or record an event there and work on another stream; it must not wait
 * for the device.  Data-parallel training uses it to start each layer's gradient exchange
 * while the next layer's backward runs. */
typedef void (*lsn_layer_hook)(void* user, int32_t layer, float* grad, size_t elems, void* stream);

typedef struct {
    int32_t recompute;
    int32_t reference_pass;
    /* How the backward's two transposed GEMMs ([dq | da] and dh) read W:
     *   0 or 1: packed NF4, decoded by the GEMM's producer warps into its operand tiles (bf16
     *      W never exists in HBM);
     *   2: each layer's W decoded once into bf16 scratch in the workspace (the same values,
     *      bit for bit, so the results are identical), then read by TMA as a dense operand.
     * Other values: LSN_EINVAL.  The workspace size depends on it (lsn_stack_workspace_bytes_ex). */
    int32_t bwd_weights;
    int32_t reserved[5];
    /* nullable: when set, each layer's AdamW update runs in the reverse sweep right after
     * that layer's dA/dB are written (they are still written to grads). */
    const lsn_adamw_state* adamw;
    /* nullable, device bf16 [n_layers][M][d_model]: slice l receives x_{l+1}, the output of
     * layer l, at the end of the forward sweep (for per-layer checks). */
    uint16_t* x_layers_out;
    /* nullable, device fp32 [n_layers][M][d_model]: slice l receives dloss/dx_l, the gradient
     * with respect to layer l's input, right after layer l's backward. */
    float* dx_layers_out;
    /* Tokens the loss means are taken over (0: M).  A data-parallel rank that holds M of a
     * global batch of token_count tokens passes the global count: its loss, dx and dA/dB are
     * then its exact share, and the ranks' sums are the global ones. */
    int64_t token_count;
    /* nullable: called after every layer's backward (see lsn_layer_hook).  Not together with
     * adamw (LSN_EINVAL): the update has to see the exchanged gradients, so a step with a hook
     * leaves the update to lsn_adamw_step once the hook's work is done. */
    lsn_layer_hook grads_ready;
    void* hook_user;
} lsn_step_opts;

size_t lsn_stack_workspace_bytes_ex(const lsn_stack_desc* desc, int64_t M, const lsn_step_opts* opts);

/* One AdamW step over n parameters (the pages set lr 2e-5 in "Fine tune an 8B model on a
 * 4GB laptop GPU (Soup setup)", "Step 1, the config"; they name no optimizer):
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   p = p - lr ((m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps) + wd p)
 * p, m, v: device fp32 [n] (updated in place); g: device fp32 [n]; p_bf16 (nullable): device
 * bf16 [n] receives bf16(p).  All pointers 16-byte aligned.  Elementwise, in fp32. */
int lsn_adamw_step(const lsn_adamw_hparams* hp, float* p, uint16_t* p_bf16, const float* g, float* m,
                   float* v, size_t n, void* stream);

/* Fixed-order sum over ranks (the reduction of data-parallel gradients): out[i] =
 * ((in[0][i] + in[1][i]) + in[2][i]) + ... in fp32, rank order, for i < n, where in is the
 * device array [n_ranks][n] the ranks' gradients were gathered into.  Every rank that sums the
 * same gathered array gets the same bits, whatever order a collective would have added them
 * in.  out may alias in[0].  Pointers 16-byte aligned; n_ranks >= 1. */
int lsn_sum_ranks(const float* in, int n_ranks, size_t n, float* out, void* stream);

/* layer_stack_step with options.  x_ref_out (nullable, device bf16 [M x d_model]) receives
 * the reference-pass output when opts->reference_pass is set. */
int layer_stack_step_ex(lsn_pool* pool, const void* resident_store, const lsn_stack_desc* desc,
                        const lsn_step_opts* opts, const uint16_t* x0, int64_t M,
                        const uint16_t* const* lora, float* const* grads, float* loss_out,
                        uint16_t* x_out, uint16_t* x_ref_out, float* dx0, void* ws, size_t ws_bytes,
                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LSN_H */
