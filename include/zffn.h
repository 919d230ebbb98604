/*
 * zffn.h -- C ABI of the fused Q4_K SwiGLU feed-forward library (GB300, sm_103a).
 *
 * The block computed is
 *     y = W_down . ( silu(W_gate . x)  (*)  (W_up . x) ),   silu(g) = g / (1 + e^-g)
 * with the hidden state of width H projected up twice to the intermediate
 * width I and back down ("Fused SwiGLU MLP: ZINC RDNA4 Down-Projection
 * Bandwidth", section "The MLP is two trips up to a wider width").  Weights
 * stay in Q4_K super-blocks and are unpacked on chip on their way into the
 * multiply (same page, FAQ "Why is fusing the SwiGLU intermediate harder than
 * fusing the weight dequant?"); the SwiGLU intermediate is produced and
 * consumed on chip and never written to device memory (same page, section
 * "Why this fusion is harder than the last one").
 *
 * Q4_K layout used throughout (144 bytes per 256 weights, little endian):
 *   bytes 0..1 d (binary16), 2..3 dmin (binary16), 4..15 twelve bytes holding
 *   eight 6-bit (scale, min) pairs, 16..143 the 4-bit codes; code byte 32g+l
 *   holds weight 64g+l (low nibble) and weight 64g+32+l (high nibble);
 *   w = d*scale*q - dmin*min.
 * A matrix of R rows and C columns is R consecutive rows of ceil(C/256)
 * consecutive blocks (zffn_q4k_row_bytes(C) bytes per row).  Weights past
 * column C in a row's last block are ignored.
 *
 * Conventions for every entry point:
 *   - Pointers named x, y, h, gamma, logits, W*, blocks, out, expert_* are
 *     DEVICE pointers owned by the caller; the library never frees or retains
 *     them.  Pointers named *_host are host memory (the host pipeline only).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call is asynchronous and stream-ordered; none synchronises the host
 *     except zffn_get_device_error and the host pipeline's sync and destroy,
 *     and none reads device data on the host.
 *   - Argument checks run on the host before anything is launched; a failed
 *     check returns ZFFN_ERR_INVALID_ARG (or ZFFN_ERR_UNSUPPORTED) and launches
 *     nothing.  A failed launch returns ZFFN_ERR_CUDA.
 *   - Every device-side wait is bounded.  A wait that runs out records
 *     ZFFN_ERR_TIMEOUT in the device error word (read with
 *     zffn_get_device_error) and the kernel returns; it never traps or hangs.
 *   - The current CUDA device at the time of the call is the device used.
 */
#ifndef ZFFN_H
#define ZFFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZFFN_OK = 0,
    ZFFN_ERR_INVALID_ARG = 1,  /* a host-side argument check failed; nothing launched */
    ZFFN_ERR_UNSUPPORTED = 2,  /* valid call, shape/device this build does not handle */
    ZFFN_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed                 */
    ZFFN_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out                   */
    ZFFN_ERR_NO_WORKSPACE = 5  /* library workspace could not be allocated             */
} zffn_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *zffn_status_string(zffn_status s);

/* Bytes of one Q4_K row of `cols` weights: ceil(cols/256) * 144.  0 if cols <= 0. */
size_t zffn_q4k_row_bytes(int64_t cols);

/* Unpack Q4_K to fp32.
 *   blocks: rows * zffn_q4k_row_bytes(cols) bytes (any alignment).
 *   out:    fp32 [rows][cols] row-major.
 * Each output is the correctly rounded fp32 value of d*scale*q - dmin*min (the
 * two products are exact in fp32), so the result is bit-exact.
 * Errors: INVALID_ARG if a pointer is NULL or rows/cols <= 0. */
zffn_status zffn_q4k_dequant(const void *blocks, float *out, int64_t rows, int64_t cols,
                             void *stream);

/* Quantise fp32 weights to Q4_K with the min/max quantiser (the pages name no
 * quantiser; the source workloads quantise fp32 weights "min/max"):
 *   per 32-weight sub-block: lo = min(0, min w), hi = max w,
 *                            scale = (hi-lo)/15, min = -lo;
 *   per block: d = fp16(max scale / 63), dmin = fp16(max min / 63),
 *              sc = clamp(rint(scale/d), 0, 63), m = clamp(rint(min/dmin), 0, 63);
 *   per weight: q = clamp(rint((w + dmin*m) / (d*sc)), 0, 15);
 * every step in IEEE fp32 round-to-nearest-even (0 where a divisor is 0).
 * Columns past `cols` in a row's last block are quantised as zeros.
 *   w:      fp32 [rows][cols] row-major.
 *   blocks: output, rows * zffn_q4k_row_bytes(cols) bytes.
 * Errors: INVALID_ARG if a pointer is NULL or rows/cols <= 0. */
zffn_status zffn_q4k_quantize(const float *w, void *blocks, int64_t rows, int64_t cols,
                              void *stream);

/* Dense SwiGLU block over T tokens.
 *   x:  bf16 [T][H] row-major, 16-byte aligned.
 *   Wg, Wu: Q4_K, I rows of H/256 blocks (W_gate, W_up: [I x H]), 16-byte aligned.
 *   Wd: Q4_K, H rows of ceil(I/256) blocks (W_down: [H x I]), 16-byte aligned.
 *   y:  fp32 [T][H] row-major, overwritten, 16-byte aligned.
 * Requirements: T >= 1, H % 256 == 0, I % 64 == 0, 256 <= H <= 16384,
 * 64 <= I <= 65536.  T = 1 runs the memory-bound single-token kernel; larger T
 * run the tensor-core prefill kernel (the switch-over can be changed with
 * zffn_set_option).  Accumulation is fp32.  Operands of the tensor-core path:
 * the gate/up product takes x and the unpacked W_gate, W_up in fp16 (x
 * converted once per call; each sub-block's scale d*sc and offset dmin*m
 * rounded to fp16, then one fused multiply-add per weight); the down product
 * takes 16 times the unpacked W_down (formed the same way) and the SwiGLU
 * intermediate as fp16(h / 16), so that its result needs no rescaling.  fp16
 * values saturate at +-65504: |x| above that, a W_gate or W_up sub-block with
 * d*sc > 128 or dmin*m > 65504, a W_down sub-block with d*sc > 8 or
 * dmin*m > 4094, or |h| above 1.05e6, is clamped on that path (far outside
 * quantised weights and normalised activations).
 * Uses library workspace (see zffn_reserve): the single-token path's
 * intermediate strip, and the prefill path's fp16 copy of x (T*H*2 bytes).
 * Errors: INVALID_ARG (NULL, misaligned, bad sizes), CUDA, NO_WORKSPACE. */
zffn_status zffn_swiglu_q4k(const void *x, const void *Wg, const void *Wu, const void *Wd,
                            float *y, int T, int H, int I, void *stream);

/* As zffn_swiglu_q4k, but adds the block's output to y instead of overwriting
 * it: y += W_down . (silu(W_gate . x) (*) (W_up . x)) -- the residual
 * connection around the block.  y must hold valid fp32 values on entry. */
zffn_status zffn_swiglu_q4k_residual(const void *x, const void *Wg, const void *Wu,
                                     const void *Wd, float *y, int T, int H, int I,
                                     void *stream);

/* RMSNorm of the residual stream into the block's input:
 *     x[t][c] = bf16( h[t][c] / sqrt(mean_c' h[t][c']^2 + eps) * gamma[c] )
 * ("Four bottlenecks, one CUDA backend...", section "Bottleneck 3 -- Gemma
 * decode is launch-latency bound": the rms_norm and the residual accumulate
 * around a block; the pages do not write RMSNorm out, this is the usual form).
 * Sum of squares and scaling in fp32, one rounding to bf16 (round to nearest
 * even).
 *   h: fp32 [T][H] (device), read only.  gamma: fp32 [H] (device).
 *   x: output, bf16 [T][H] (device).
 * Requirements: T >= 1, 256 <= H <= 16384, H % 256 == 0, 0 <= eps <= 1,
 * 16-byte aligned pointers.  Errors: INVALID_ARG (nothing launched), CUDA. */
zffn_status zffn_rmsnorm_bf16(const float *h, const float *gamma, float eps, void *x, int T,
                              int H, void *stream);

/* The block with its normalisation and residual connection, as a pre-norm
 * transformer layer applies it to the residual stream h:
 *     h[t] += W_down . (silu(W_gate . x[t]) (*) (W_up . x[t])),
 *     x = zffn_rmsnorm_bf16(h, gamma, eps)
 * T = 1 (when the single-token kernels take the sizes): the normalisation
 * runs inside the gate/up kernel, which reads the fp32 row and gamma and
 * builds x itself; then the down kernel adds into h (two launches, no
 * workspace copy of x; x may differ from zffn_rmsnorm_bf16's in the last bf16
 * place of rare elements, the sum of squares being reduced in another order).
 * Otherwise two launch groups in stream order: the normalisation into library
 * workspace (bf16 [T][H], see zffn_reserve), then the block accumulating
 * into h.
 *   h: fp32 [T][H] (device), read and updated in place.
 *   gamma: fp32 [H]; Wg, Wu, Wd as for zffn_swiglu_q4k.
 * Requirements as zffn_swiglu_q4k and zffn_rmsnorm_bf16.
 * Errors: INVALID_ARG, CUDA, NO_WORKSPACE. */
zffn_status zffn_swiglu_q4k_prenorm_residual(float *h, const float *gamma, float eps,
                                             const void *Wg, const void *Wu, const void *Wd,
                                             int T, int H, int I, void *stream);

/* Host pipeline: the dense block over inputs and outputs in host memory, with
 * the host-to-device copy of each submission's x and the device-to-host copy
 * of its y overlapped with the blocks of the neighbouring submissions (an
 * upload stream, a compute stream and a download stream of the library's own,
 * ordered by events per slot; `depth` slots of device x and y, allocated once
 * at creation).  The source pages have no counterpart; it is how a caller
 * that keeps activations on the host feeds the block without idling it.
 *   zffn_pipeline_create: *out = a pipeline for blocks of T tokens of width H
 *     and intermediate width I; 2 <= depth <= ZFFN_PIPELINE_MAX_DEPTH.  Uses
 *     the current device.  Errors: INVALID_ARG, CUDA, NO_WORKSPACE (device
 *     memory: depth * T * H * 6 bytes).
 *   zffn_pipeline_submit: queues upload(x_host) -> block -> download(y_host)
 *     and returns without waiting.  x_host: bf16 [T][H], y_host: fp32 [T][H],
 *     host memory (page-locked for the copies to overlap; pageable memory
 *     works, with the copies serialised by the driver); both must stay valid
 *     and x_host unchanged until zffn_pipeline_sync returns.  Wg, Wu, Wd:
 *     device Q4_K weights as for zffn_swiglu_q4k; the pipeline's streams do
 *     not wait for other streams, so the weights must be complete before the
 *     call (synchronise the stream that wrote them).  Must be called on the
 *     pipeline's device.  Errors: INVALID_ARG, CUDA, NO_WORKSPACE.
 *   zffn_pipeline_sync: waits for every submission so far (their y_host
 *     hold the results).  Device-side errors are reported by
 *     zffn_get_device_error as for the other calls.
 *   zffn_pipeline_destroy: waits, then frees everything (NULL is ignored). */
#define ZFFN_PIPELINE_MAX_DEPTH 4
typedef struct zffn_pipeline zffn_pipeline;
zffn_status zffn_pipeline_create(zffn_pipeline **out, int T, int H, int I, int depth);
zffn_status zffn_pipeline_submit(zffn_pipeline *p, const void *x_host, const void *Wg,
                                 const void *Wu, const void *Wd, float *y_host);
/* As zffn_pipeline_submit for the routed block (zffn_moe_swiglu_q4k): x_host and
 * y_host in host memory as above; expert_ids, expert_weights (device, [T][top_k],
 * e.g. from zffn_moe_router_topk) and the stacked expert weights as for
 * zffn_moe_swiglu_q4k, complete before the call and unchanged until
 * zffn_pipeline_sync returns. */
zffn_status zffn_pipeline_submit_moe(zffn_pipeline *p, const void *x_host,
                                     const int32_t *expert_ids, const float *expert_weights,
                                     const void *Wg, const void *Wu, const void *Wd, int E,
                                     int top_k, float *y_host);
zffn_status zffn_pipeline_sync(zffn_pipeline *p);
void zffn_pipeline_destroy(zffn_pipeline *p);

/* Block formats of W_down.  The pages name Q5_K, Q6_K and Q5_1 expert and down
 * matrices next to Q4_K ("Four bottlenecks, one CUDA backend...", section
 * "Bottleneck 2": the routed layers' down projection in Q5_K or Q5_1; section
 * "Bottleneck 4": Q5_K and Q6_K) without laying them out; the arrangement used
 * is GGUF's:
 *   ZFFN_FMT_Q5_K  176 bytes / 256 weights: fp16 d, fp16 dmin, 12 scale bytes
 *     packed as Q4_K, qh[32], qs[128]; code = nibble (as Q4_K) + 16 * bit
 *     (k/32) of qh[k%32]; w = d*sc*q - dmin*m.
 *   ZFFN_FMT_Q6_K  210 bytes / 256 weights: ql[128], qh[64], int8 scales[16],
 *     fp16 d; w = d * scales[k/16] * (q - 32), q of 6 bits (4 from ql, 2 from
 *     qh).
 *   ZFFN_FMT_Q5_1  24 bytes / 32 weights: fp16 d, fp16 m, 32-bit qh, qs[16];
 *     w = d*q + m, q of 5 bits. */
typedef enum {
    ZFFN_FMT_Q4_K = 0,
    ZFFN_FMT_Q5_K = 1,
    ZFFN_FMT_Q6_K = 2,
    ZFFN_FMT_Q5_1 = 3
} zffn_format;

/* Bytes of one row of `cols` weights in format fmt (0 for cols <= 0 or an
 * unknown format). */
size_t zffn_row_bytes_fmt(int fmt, int64_t cols);

/* fp32 [rows][cols] from rows of blocks of format fmt, bit-exact (every product
 * in the formats is exact in fp32; at most the final addition rounds).
 * Errors: INVALID_ARG, CUDA. */
zffn_status zffn_dequant_fmt(int fmt, const void *blocks, float *out, int64_t rows,
                             int64_t cols, void *stream);

/* The block with W_gate and W_up in Q4_K and W_down in format wd_fmt (rows of
 * zffn_row_bytes_fmt(wd_fmt, I) bytes) ("Four bottlenecks, one CUDA
 * backend...", section "Bottleneck 4": Q4_K, Q5_K and Q6_K GEMMs of prefill).
 * ZFFN_FMT_Q4_K is zffn_swiglu_q4k.
 *   T = 1: the single-token kernels, every format.  Wd must be 4-byte aligned
 *     (its rows need not be: Q6_K rows are 210-byte multiples; a 16-byte
 *     aligned Wd is copied faster).  h is held in shared memory as int16
 *     with one fp32 scale per 32 and one fp32 sum per 16 values (2.375 bytes
 *     a value); UNSUPPORTED when top_k * I such values plus the row buffers
 *     (66 KB for Q5_K, 72 KB for Q5_1, 90 KB for Q6_K) exceed a block's
 *     shared memory (227 KB: at top_k = 1 every I for Q5_K and Q5_1, I <=
 *     58688 for Q6_K; at top_k = 8, I <= 8576, 8256 and 7296).
 *   T > 1: every format on the grouped tensor-core kernel (the routed
 *     kernel's groups of 32 token rows; a dense block runs as one expert), Wd
 *     and y 16-byte aligned.  Its weights are unpacked once per group of 32
 *     tokens, so it suits routed layers and short prompts rather than long
 *     prefills.  Q6_K rows (210-byte blocks, row pitches not a multiple of 16
 *     bytes) are copied row by row instead of by TMA boxes: slower (about
 *     1.3x the Q5_K call at the routed T = 256 layer).
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA, NO_WORKSPACE. */
zffn_status zffn_swiglu_q4k_wd(const void *x, const void *Wg, const void *Wu, const void *Wd,
                               int wd_fmt, float *y, int T, int H, int I, void *stream);

/* The routed block (as zffn_moe_swiglu_q4k) with every expert's W_down in
 * format wd_fmt; the same formats and restrictions as zffn_swiglu_q4k_wd (at
 * T > 1 the grouped tensor-core kernel). */
zffn_status zffn_moe_swiglu_q4k_wd(const void *x, const int32_t *expert_ids,
                                   const float *expert_weights, const void *Wg, const void *Wu,
                                   const void *Wd, int wd_fmt, float *y, int T, int H, int I,
                                   int E, int top_k, void *stream);

/* Mixture-of-experts SwiGLU block:
 *     y[t] = sum_{j < top_k} expert_weights[t][j] * FFN_{expert_ids[t][j]}(x[t])
 * ("Four bottlenecks, one CUDA backend...", section "Bottleneck 2 -- MoE decode
 * was paying for its routing twice": the chosen expert ids are read from a
 * device buffer by the kernels; nothing is read back to the host).
 *   x:  bf16 [T][H].
 *   expert_ids: int32 [T][top_k] (device).  An id outside [0, E) contributes 0.
 *   expert_weights: fp32 [T][top_k] (device).
 *   Wg, Wu: E stacked experts, each I rows of H/256 blocks.
 *   Wd: E stacked experts, each H rows of ceil(I/256) blocks.
 *   y:  fp32 [T][H], overwritten.
 * Requirements as zffn_swiglu_q4k, plus 1 <= E <= 4096, 1 <= top_k <= 64,
 * T * top_k <= 2^24, expert_ids and expert_weights 4-byte aligned.
 * T = 1: one cooperative launch when every block's share of the token's
 * expert weights fits in its shared memory (see ZFFN_OPT_TOKEN_KERNEL and
 * zffn_single_token_launches), else the two single-token kernels; T > 1:
 * routing, gathering and a tensor-core kernel.
 * Uses library workspace (see zffn_reserve).
 * Errors: INVALID_ARG, CUDA, NO_WORKSPACE. */
zffn_status zffn_moe_swiglu_q4k(const void *x, const int32_t *expert_ids,
                                const float *expert_weights, const void *Wg, const void *Wu,
                                const void *Wd, float *y, int T, int H, int I, int E,
                                int top_k, void *stream);

/* Router of a routed block: for every token, the top_k experts by router
 * logit and softmax weights over the chosen logits, written to device buffers
 * that zffn_moe_swiglu_q4k reads as they are ("Four bottlenecks, one CUDA
 * backend...", section "Bottleneck 2 -- MoE decode was paying for its routing
 * twice": the layer computes router logits and picks the top-k experts; section
 * "What's next, and what it's worth": a GPU-side step drops the last router
 * round-trip).  The pages do not state the weighting; the softmax over the
 * chosen k logits is the reading used here.
 *   logits: fp32 [T][E] row-major (device).
 *   expert_ids: output, int32 [T][top_k] (device): the chosen experts from the
 *     highest logit down; equal logits go to the lower index; -0 equals +0; a
 *     NaN logit ranks below every number (-inf included), NaNs by index.
 *   expert_weights: output, fp32 [T][top_k] (device):
 *     exp(l_j - l_0) / sum_i exp(l_i - l_0) over the chosen logits, l_0 the
 *     largest, in fp32 (IEEE arithmetic for infinities and NaNs).
 * Requirements: T >= 1, 1 <= E <= 4096, 1 <= top_k <= min(E, 64), T*E <= 2^31,
 * 4-byte aligned pointers.  All buffers are the caller's; nothing is read back
 * to the host.
 * Errors: INVALID_ARG (checked on the host, nothing launched), CUDA. */
zffn_status zffn_moe_router_topk(const float *logits, int32_t *expert_ids,
                                 float *expert_weights, int T, int E, int top_k,
                                 void *stream);

/* The routed block with a scale on each expert's down projection
 * ("Four bottlenecks, one CUDA backend...", section "Bottleneck 2 -- MoE decode
 * was paying for its routing twice": a routed layer's per-expert
 * down-projection scale is applied inside the batched path, not folded away):
 *     y[t] (+)= sum_{j < top_k} expert_weights[t][j] * down_scale[e] * FFN_e(x[t]),
 *     e = expert_ids[t][j]
 *   down_scale: fp32 [E] (device, 4-byte aligned), or NULL for every scale 1.
 *     It multiplies the routing weight of each (token, slot) in fp32 before the
 *     down projection's output is added.
 *   wd_fmt: block format of every expert's W_down (zffn_format), with the
 *     same rules as zffn_moe_swiglu_q4k_wd.
 *   accumulate: 0 overwrites y, non-zero adds the block's output to y.
 *   The other arguments as for zffn_moe_swiglu_q4k (expert_ids and
 *   expert_weights must not be NULL).
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA, NO_WORKSPACE. */
zffn_status zffn_moe_swiglu_q4k_scaled(const void *x, const int32_t *expert_ids,
                                       const float *expert_weights, const float *down_scale,
                                       const void *Wg, const void *Wu, const void *Wd, int wd_fmt,
                                       float *y, int T, int H, int I, int E, int top_k,
                                       int accumulate, void *stream);

/* As zffn_moe_swiglu_q4k, but y += the routed block's output. */
zffn_status zffn_moe_swiglu_q4k_residual(const void *x, const int32_t *expert_ids,
                                         const float *expert_weights, const void *Wg,
                                         const void *Wu, const void *Wd, float *y, int T, int H,
                                         int I, int E, int top_k, void *stream);

/* Single-token dense block (T = 1) that allocates no device memory.  The
 * source pages have no counterpart of this entry point.  It is for callers
 * that cannot let the library call cudaMalloc/cudaFree during a call -- for
 * example a server whose own allocator already owns all device memory, or a
 * loop that forbids allocation after start-up.  It computes the same block as
 * zffn_swiglu_q4k with T = 1 (same kernels), but its scratch (the fp32
 * intermediate strip) lives in one fixed array compiled into the library:
 * 64 KB that every GPU loading the library keeps until exit.
 *   x: bf16 [H]; Wg, Wu, Wd and y as for zffn_swiglu_q4k with T = 1.
 * Limits: I <= 16384 (the array's size); larger I returns ZFFN_ERR_INVALID_ARG
 * and zffn_last_error() says why.  The first call on a device looks up the
 * array's device address with cudaGetSymbolAddress, so make that first call
 * before capturing any stream.  All calls share the array and it keeps the
 * last call's contents; calls whose launches overlap on the GPU race on it.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
zffn_status zffn_swiglu_q4k_token_static(const void *x, const void *Wg, const void *Wu,
                                         const void *Wd, float *y, int H, int I, void *stream);

/* Allocate (or grow) the current device's workspace for calls up to the given
 * sizes, so that later calls allocate nothing (call it before capturing calls
 * into a CUDA graph).  Calls that share a device share its workspace: issue
 * them on one stream, or order them, since concurrent calls race on it.
 * Errors: INVALID_ARG (a size < 1), NO_WORKSPACE. */
zffn_status zffn_reserve(int T_max, int H_max, int I_max, int E_max, int top_k_max);

/* Release every workspace the library holds (all devices).  Not stream-ordered:
 * the caller makes sure no call is still running. */
void zffn_release(void);

/* Bytes of workspace the library currently holds on the current device (0 if
 * none has been allocated, or after zffn_release).  Host-side query; launches
 * nothing and allocates nothing. */
size_t zffn_workspace_bytes(void);

/* Kernel launches one routed single-token call (zffn_moe_swiglu_q4k with
 * T = 1 and Q4_K W_down) of these sizes makes on the current device under the
 * current options (ZFFN_OPT_TOKEN_KERNEL): 1 for the one cooperative launch,
 * 2 for the gate/up and down pair; -1 without a device or for sizes outside
 * [1, 65536] (top_k in [1, 64]).  Host-side query; launches nothing. */
int zffn_single_token_launches(int H, int I, int E, int top_k);

/* Description of the last failure a call on this host thread reported: the
 * CUDA error behind a ZFFN_ERR_CUDA, or the failed check behind a
 * ZFFN_ERR_INVALID_ARG.  A successful call leaves it unchanged.  Static
 * string, never NULL; "no error" before the first failure. */
const char *zffn_last_error(void);

/* Synchronise `stream`, then return and clear the current device's error word:
 * ZFFN_OK, or ZFFN_ERR_TIMEOUT if a bounded device wait ran out since the last
 * read.  ZFFN_ERR_CUDA if the synchronisation itself failed.  On
 * ZFFN_ERR_TIMEOUT it also resets the grid-barrier count of the one-launch
 * routed path in the device's workspace (a barrier that ran out leaves it
 * mid-count), so the caller must have no call of the library still running
 * on the device (the calls share the workspace anyway). */
zffn_status zffn_get_device_error(void *stream);

/* Tunables (process-wide).  ZFFN_OPT_MATVEC_MAX_T: 1 (default) sends single-token
 * calls (T = 1, dense or routed) to the memory-bound single-token kernel; 0
 * sends every call to the tensor-core kernels (any value > 1 acts as 1).
 * ZFFN_OPT_MOE_KERNEL chooses the tensor-core kernel of routed calls: 0
 * (default) the grouped kernel (groups of 32 gathered rows of one expert, the
 * weights on the MMA's M side) when T * top_k <= 48 * E and the prefill
 * kernel on 128-row expert tiles otherwise; 1 always the grouped kernel; 2
 * always the 128-row tiles.
 * ZFFN_OPT_TOKEN_KERNEL chooses the single-token routed path (Q4_K W_down):
 * 0 (default) one cooperative launch (every block asks for all of its gate/up
 * and down rows at once, computes its h rows, meets the other blocks at a
 * grid barrier, then its output rows) whenever each block's share of the
 * token's expert weights fits in its shared memory, else the two-kernel
 * pair; 1 always the two-kernel pair (gate/up, then down as its
 * programmatic dependent).
 * Returns the previous value, or -1 for an unknown key. */
enum { ZFFN_OPT_MATVEC_MAX_T = 1, ZFFN_OPT_MOE_KERNEL = 2, ZFFN_OPT_TOKEN_KERNEL = 3 };
int zffn_set_option(int key, int value);

/* Self-test of the bounded-wait machinery: launches one block that waits on an
 * mbarrier nothing will ever complete, with a budget of `budget_cycles` SM
 * clocks; the wait gives up, records ZFFN_ERR_TIMEOUT in the device error word
 * and the kernel returns normally.  Errors: INVALID_ARG (budget < 1), CUDA. */
zffn_status zffn_selftest_wait_timeout(int64_t budget_cycles, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ZFFN_H */
