/*
 * moe_decode.h -- C ABI of libmoe_decode.so, an output-centric ("warp decode")
 * small-batch mixture-of-experts decode layer for NVIDIA GB300 (sm_103a).
 *
 * The layer (the warp-decode post, cursor.com/blog/warp-decode, sections
 * "The classic MoE path" and "How the two kernels work"):
 *
 *   for every token t and routed slot j (e = topk_ids[t,j]) and neuron i:
 *     g = sum_K dq(W_gateup[e, i,   K]) * x[t,K]
 *     u = sum_K dq(W_gateup[e, I+i, K]) * x[t,K]
 *     h[t,j,i] = bf16( SiLU(g) * u )                     (moe_gate_up)
 *   for every token t and output dimension r:
 *     y[t,r] = bf16( sum_j topk_w[t,j] * sum_i dq(W_down[e_j, r, i]) * h[t,j,i] )
 *                                                        (moe_down)
 *
 * dq() is MXFP8 dequantisation: one E4M3 code per element and one UE8M0
 * exponent per 32 consecutive elements along the reduction axis (the block
 * format named in the GC-MoE summary, onedev.kr/papers/1690, "How it is
 * used"): dq = E4M3(code) * 2^(scale - 127). With MOE_FLAG_MXFP4 it is MXFP4
 * dequantisation instead, the routed-weight format of the same page and
 * section: one E2M1 code per element (1 sign, 2 exponent bits with bias 1,
 * 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two codes to a
 * byte, with the same UE8M0 scales. Dot products accumulate in FP32; h and y
 * are rounded to BF16 (round to nearest even).
 *
 * Conventions shared by every call:
 *   - Tensors are row-major and contiguous. bf16 tensors are passed as
 *     uint16_t bit patterns. Device pointers are marked "device".
 *   - Weights are borrowed: the handle keeps the pointers, never copies, and
 *     the caller keeps them alive and unchanged until moe_decode_destroy.
 *   - Compute calls only enqueue work on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and return at once. Argument errors are detected
 *     on the host, return a non-zero status and enqueue nothing.
 *   - T = 0 is a successful no-op. T may exceed 32: the library then works
 *     through the tokens 32 at a time (expert dedup applies within a group).
 *   - An expert id outside [0, E) contributes nothing (its h slice is zero)
 *     and sets MOE_DEVICE_BAD_ID in the handle's device error word, read with
 *     moe_decode_get_error. Nothing traps and nothing spins.
 *   - Duplicate ids in a token's row are legal; their contributions add.
 *   - Results are bitwise reproducible run to run (no atomics on data).
 *   - Calls on one handle may run concurrently on different streams, with two
 *     exceptions: moe_decode_layer with T = 1 (its one-launch form shares the
 *     handle's grid-barrier counter, so such calls must be ordered on one
 *     stream) and moe_decode_forward_host (which shares staging buffers).
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,       /* null pointer, negative size, T > max_T ... */
  MOE_ERR_UNSUPPORTED_SHAPE = 2, /* H or I not a multiple of 32, k > 32, E > 1024 ... */
  MOE_ERR_MISALIGNED = 3,        /* a pointer breaks the alignment stated below */
  MOE_ERR_CUDA = 4,              /* a CUDA runtime call failed */
  MOE_ERR_DEVICE_FAULT = 5       /* moe_decode_get_error found a latched device flag */
} moe_status_t;

/* Bits of the device error word. */
#define MOE_DEVICE_BAD_ID 0x1u     /* some topk_id was outside [0, E) */
#define MOE_DEVICE_TIMEOUT 0x2u    /* a bounded device wait gave up (results undefined) */

/* Flags of moe_decode_config_t. */
#define MOE_FLAG_NO_PDL 0x1u       /* launch without programmatic dependent launch */
#define MOE_FLAG_HOST_COPY 0x2u    /* moe_decode_forward_host always copies through
                                      the device staging buffers */
#define MOE_FLAG_MXFP4 0x4u        /* the weights are MXFP4, not MXFP8 (see
                                      moe_decode_create) */
#define MOE_FLAG_WARP_MMA 0x8u     /* warp-decode calls of 16 to 32 tokens form
                                      their products on the warp-level MMA
                                      (kernels moe_gate_up_tma, moe_down_mma):
                                      faster when a few experts serve many of
                                      the tokens, slower when each expert
                                      serves one or two (the default then) */

typedef struct {
  int32_t E;      /* experts, 1..1024 */
  int32_t k;      /* routed experts per token, 1..min(E, 32) */
  int32_t H;      /* hidden size, multiple of 32 */
  int32_t I;      /* intermediate size per expert, multiple of 32 */
  int32_t max_T;  /* largest T any call will pass (sizes host-side checks and
                     the staging buffers of moe_decode_forward_host) */
  uint32_t flags; /* MOE_FLAG_* */
} moe_decode_config_t;

typedef struct moe_decode* moe_decode_t;

/*
 * Create a handle for one layer on the current CUDA device.
 *   w_gateup  device uint8 [E, 2I, H]   E4M3 codes; rows [0,I) gate, [I,2I) up
 *   s_gateup  device uint8 [E, 2I, H/32] UE8M0 scale codes
 *   w_down    device uint8 [E, H, I]    E4M3 codes
 *   s_down    device uint8 [E, H, I/32] UE8M0 scale codes
 * With MOE_FLAG_MXFP4 in cfg->flags, w_gateup is uint8 [E, 2I, H/2] and
 * w_down uint8 [E, H, I/2]: E2M1 codes, element 2c of a row in the low
 * nibble of byte c and element 2c+1 in its high nibble; the scales are as
 * above. w_gateup and w_down must be 32-byte aligned; the scale arrays need
 * no alignment (16-byte aligned scale arrays enable the one-launch
 * single-token layer, which with MXFP4 also needs H a multiple of 1024). Allocates 32 bytes of device
 * state (the error word and the one-launch kernel's launch and grid-barrier
 * counters), one CUDA event and one non-blocking stream (for
 * moe_decode_get_error) and, when max_T > 0, the staging buffers of
 * moe_decode_forward_host. *out receives the handle; on error *out is NULL.
 */
moe_status_t moe_decode_create(const moe_decode_config_t* cfg,
                               const uint8_t* w_gateup, const uint8_t* s_gateup,
                               const uint8_t* w_down, const uint8_t* s_down,
                               moe_decode_t* out);

/* Release the handle and its device allocations (not the weights). NULL is a no-op. */
moe_status_t moe_decode_destroy(moe_decode_t handle);

/*
 * Router: softmax over the E logits of each token, keep the k largest
 * (ties to the lower expert id, ids in decreasing weight order), renormalise
 * the kept weights to sum to one. The warp-decode post ("The classic MoE
 * path") routes each token to k of E experts; the renormalisation follows the
 * usual top-k router.
 *   logits    device float [T, E]  (4-byte aligned)
 *   topk_ids  device int32 [T, k]  out
 *   topk_w    device float [T, k]  out
 * Weights are computed in FP32 as exp(l_j - l_max) / sum over the kept j.
 */
moe_status_t moe_route(moe_decode_t handle, int32_t T, const float* logits,
                       int32_t* topk_ids, float* topk_w, void* stream);

/*
 * Per-step expert dedup schedule, exactly as the kernels build it (exported
 * for inspection; the kernels rebuild it on chip and never read this).
 * For T <= 32 tokens:
 *   uniq     device int32 [min(E, T*k)]    ascending unique valid expert ids
 *   offsets  device int32 [min(E, T*k)+1]  pairs of uniq[u] are pairs[offsets[u]:offsets[u+1]]
 *   pairs    device int32 [T*k]            flattened slots p = t*k + j, ascending within an expert
 *   n_uniq   device int32 [1]              number of unique experts
 * Entries past n_uniq / offsets[n_uniq] are left unchanged.
 */
moe_status_t moe_dedup_schedule(moe_decode_t handle, int32_t T, const int32_t* topk_ids,
                                int32_t* uniq, int32_t* offsets, int32_t* pairs,
                                int32_t* n_uniq, void* stream);

/*
 * Gate/up projection (the warp-decode post, "How the two kernels work", first
 * two paragraphs). Each unique expert's gate and up rows are streamed once
 * per group of tokens and serve every token routed to it. The kernel depends
 * on T and the shape (moe_decode_kernel_name reports it):
 * moe_gate_up_3d_batched (x read through L1), moe_gate_up_3d_batched_xs (x
 * staged in shared memory as power-of-two-scaled f16 blocks), or, from 16
 * tokens, moe_gate_up_tma (16-neuron weight tiles streamed by TMA into a
 * shared-memory ring, products on mma.sync with FP32 accumulation). Groups
 * are at most 32 tokens, fewer when that lets x fit in shared memory.
 *   x         device bf16 [T, H]     32-byte aligned
 *   topk_ids  device int32 [T, k]
 *   h         device bf16 [T, k, I]  out, 32-byte aligned
 */
moe_status_t moe_gate_up(moe_decode_t handle, int32_t T, const uint16_t* x,
                         const int32_t* topk_ids, uint16_t* h, void* stream);

/*
 * Down projection with the routing-weighted sum over the top-k experts (the
 * warp-decode post, "How the two kernels work", third paragraph onward).
 * Kernel by T and shape: moe_down_3d_batched (one warp per output y[t, r]),
 * from 2 tokens moe_down_tma (a 16-row tile of y[t] per item, each distinct
 * routed expert's rows streamed by TMA, one warp per row), from 16 tokens
 * moe_down_mma (one CTA per 16-row tile of y for every token, each unique
 * expert's rows streamed once, products on mma.sync); no atomics in any.
 *   h         device bf16 [T, k, I]  32-byte aligned
 *   topk_ids  device int32 [T, k]
 *   topk_w    device float [T, k]
 *   y         device bf16 [T, H]     out
 */
moe_status_t moe_down(moe_decode_t handle, int32_t T, const uint16_t* h,
                      const int32_t* topk_ids, const float* topk_w, uint16_t* y,
                      void* stream);

/*
 * The whole layer: moe_gate_up then moe_down on one stream. The down kernel
 * is launched as a programmatic dependent of the gate/up kernel and fetches
 * its weight rows (which depend only on topk_ids) while the gate/up kernel
 * drains; topk_ids and topk_w must therefore be complete before this call's
 * work starts on `stream`, which stream order guarantees. h is the caller's
 * [T, k, I] bf16 buffer (32-byte aligned).
 * With T = 1, when moe_decode_fused_layer(handle) is 1, both projections run
 * as one cooperative launch of one CTA per SM (kernel moe_layer_fused_t1): a
 * producer warp streams the CTA's gate/up rows and then its down rows with
 * TMA tensor copies, fifteen consumer warps compute, and the CTAs meet at a
 * grid barrier (a bounded wait; on timeout it sets MOE_DEVICE_TIMEOUT) once h
 * is written. h is still written to the caller's buffer. Such calls on one
 * handle must not run concurrently (they share the handle's counters).
 * With T >= 64 tokens (or any T after moe_decode_set_path(handle,
 * MOE_PATH_TENSOR)), when moe_decode_tensor_path(handle) is 1, the layer runs
 * expert-centric on the tensor cores instead, in groups of up to 256 tokens
 * (the warp-decode post, "Warp decode and Composer training": large batches
 * favour packing tokens per expert; the operand-swapped MMA is the GC-MoE
 * summary's, onedev.kr/papers/1690, "How it is used"). Per group, four
 * launches: moe_tc_prep (the unique experts, each one's (token, slot) pairs,
 * x gathered into expert order), moe_tc_gate_up and moe_tc_down (weights
 * decoded exactly to bf16 into tensor memory as the A operand of
 * tcgen05.mma kind::f16, 128 weight rows by up to 64 pairs a tile, FP32
 * accumulators in tensor memory), moe_tc_combine (the routing-weighted sum
 * in slot order). Every unique expert is streamed once per group. h is
 * written to the caller's buffer as on the other path. The path keeps a
 * workspace sized at create and is not thread-safe across concurrent calls
 * on one handle (they share it); calls on one stream are ordered.
 */
moe_status_t moe_decode_layer(moe_decode_t handle, int32_t T, const uint16_t* x,
                              const int32_t* topk_ids, const float* topk_w,
                              uint16_t* h, uint16_t* y, void* stream);

/*
 * The whole layer from and to HOST memory, waiting for the stream before it
 * returns. The kernels read x, topk_ids and topk_w and write y in place when
 * the device can address the host buffers: always on a device that accesses
 * pageable host memory coherently (cudaDevAttrPageableMemoryAccess, e.g. a
 * Grace-Blackwell part over its chip-to-chip link), else when all four are
 * page-locked (cudaHostAlloc or torch pin_memory). Otherwise, or with
 * MOE_FLAG_HOST_COPY, x, topk_ids and topk_w are copied to the handle's device
 * staging buffers, moe_decode_layer runs, and y is copied back. h goes to the
 * handle's staging buffer either way. T <= max_T. Calls on one handle must not
 * overlap (they share the staging buffers).
 *   x_host [T,H] bf16, ids_host [T,k] int32, w_host [T,k] float, y_host [T,H] bf16 out
 */
moe_status_t moe_decode_forward_host(moe_decode_t handle, int32_t T, const uint16_t* x_host,
                                     const int32_t* ids_host, const float* w_host,
                                     uint16_t* y_host, void* stream);

/*
 * Read and clear the handle's device error word. *device_flags receives the
 * MOE_DEVICE_* bits latched since the last read; the return value is
 * MOE_ERR_DEVICE_FAULT when any bit was set, MOE_OK otherwise.
 * moe_decode_get_error first waits for the work of this handle's most recent
 * call that was not being captured into a CUDA graph (an event the handle
 * records after each call's launches), and for nothing else: kernels of other
 * streams and other libraries keep running. The read and the clear run on a
 * private non-blocking stream of the handle. Errors of earlier calls made on
 * another stream may still be in flight then; after replaying a graph, or to
 * cover every call made on one stream, use moe_decode_get_error_stream, which
 * waits for `stream` (a cudaStream_t) instead.
 */
moe_status_t moe_decode_get_error(moe_decode_t handle, uint32_t* device_flags);
moe_status_t moe_decode_get_error_stream(moe_decode_t handle, void* stream,
                                         uint32_t* device_flags);

/* Static, human-readable name of a status. */
const char* moe_status_string(moe_status_t status);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t moe_decode_version(void);

/*
 * Diagnostic: 1 when moe_decode_layer with T = 1 runs as one persistent
 * launch (both projections in one cooperative kernel, TMA-streamed weights,
 * a grid barrier between them) for this handle, 0 when it falls back to the
 * two kernels (shape or alignment outside that kernel's limits: H a multiple
 * of 512 (of 1024 with MOE_FLAG_MXFP4), I a multiple of 128, scale arrays
 * 16-byte aligned, enough shared memory), -1 for a NULL handle.
 */
int32_t moe_decode_fused_layer(moe_decode_t handle);

/*
 * Which form moe_decode_layer and moe_decode_forward_host take:
 *   MOE_PATH_AUTO    (the default) the tensor-core path when the handle
 *                    supports it, T >= 16 and 2 T k >= 3 E (1.5 or more
 *                    routed slots per expert on average), output-centric
 *                    warp decode otherwise
 *   MOE_PATH_WARP    always warp decode (the one-launch kernel at T = 1)
 *   MOE_PATH_TENSOR  always the tensor-core path; MOE_ERR_UNSUPPORTED_SHAPE
 *                    when moe_decode_tensor_path(handle) is 0
 * moe_gate_up and moe_down always run warp decode. Not synchronised with
 * calls in flight on other threads.
 */
#define MOE_PATH_AUTO 0
#define MOE_PATH_WARP 1
#define MOE_PATH_TENSOR 2
moe_status_t moe_decode_set_path(moe_decode_t handle, int32_t path);

/* The path (MOE_PATH_WARP or MOE_PATH_TENSOR) a layer call with T tokens
 * takes on this handle; -1 for a NULL handle or T < 1. */
int32_t moe_decode_path(moe_decode_t handle, int32_t T);

/*
 * Diagnostic: 1 when the handle can run the tensor-core path, 0 when not, -1
 * for a NULL handle. It needs max_T >= 1, H a multiple of 512, I a multiple
 * of 128, 16-byte aligned scale arrays, and weights that all decode to normal
 * bf16 values, so that the decode is exact: every scale code in 10..142
 * (MXFP8) or 2..142 (MXFP4), and no E4M3 NaN code (checked once, at create,
 * by a pass over both projections; the weights must not change afterwards).
 * Its workspace, allocated at create, holds min(max_T, 256) * k pairs: x and
 * h in expert order (bf16) and FP32 partial rows of y, (2H + 2I + 4H) bytes
 * a pair, plus the schedule.
 */
int32_t moe_decode_tensor_path(moe_decode_t handle);

/*
 * Diagnostic: the name of the kernel that moe_gate_up (which = 0) or moe_down
 * (which = 1) launches for T tokens on this handle (for T > 32, for each
 * group of 32): "moe_gate_up_tma", "moe_gate_up_3d_batched_xs" or
 * "moe_gate_up_3d_batched"; "moe_down_mma", "moe_down_tma" or
 * "moe_down_3d_batched"; "moe_tc_gate_up" and "moe_tc_down" when a layer
 * call with T tokens takes the tensor-core path. A static string; "" for a
 * NULL handle, T <= 0 or another `which`. (moe_decode_layer with T = 1 uses
 * moe_layer_fused_t1 when moe_decode_fused_layer says so.)
 */
const char* moe_decode_kernel_name(moe_decode_t handle, int32_t T, int32_t which);

/*
 * Test support: the launch plan the library would make, computed on the host
 * alone (no device, no allocation) for a configuration, a device with
 * num_sms SMs and smem_per_block bytes of opt-in shared memory per CTA, and
 * calls of T tokens. The weight pointers are taken as suitably aligned.
 *   fused*        the one-launch single-token layer: whether it fits, its
 *                 K-chunk (weights per row per stage), ring slots and slot
 *                 bytes, down rows per chunk and chunks per slot, and its
 *                 dynamic shared memory
 *   gate_up_*     tokens per gate/up launch, its kernel (0 reads x through
 *                 L1, 1 stages x, 2 TMA ring with mma.sync), ring slots (0
 *                 without a ring) and dynamic shared memory
 *   down_*        down kernel for min(T, 32) tokens (0 one warp per output,
 *                 1 TMA ring token by token, 2 TMA ring with mma.sync), ring
 *                 slots and dynamic shared memory
 * Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED_SHAPE as
 * moe_decode_create would for the configuration.
 */
typedef struct {
  int32_t fused, fused_kc, fused_slots, fused_slot_bytes, fused_down_rows, fused_down_per_slot,
      fused_smem;
  int32_t gate_up_group, gate_up_kernel, gate_up_slots, gate_up_smem;
  int32_t down_kernel, down_slots, down_smem;
} moe_decode_plan_t;
moe_status_t moe_decode_plan(const moe_decode_config_t* cfg, int32_t num_sms,
                             int32_t smem_per_block, int32_t T, moe_decode_plan_t* out);

/*
 * Test support for failure detection (the pages have no counterpart): moves
 * this handle's launch counter far ahead of its grid-barrier counter, so that
 * the next one-launch call's grid barrier can never be met. Every CTA's
 * bounded wait then gives up (after a few seconds), sets MOE_DEVICE_TIMEOUT
 * and the launch completes with unspecified y; moe_decode_get_error reports
 * it and, on a timeout, sets both counters back to zero, so later calls run
 * normally. Nothing faults or hangs. Enqueued on the default stream and
 * synchronised; returns MOE_ERR_INVALID_ARG for NULL, MOE_ERR_UNSUPPORTED_SHAPE
 * when the handle does not use the one-launch form.
 */
moe_status_t moe_decode_arm_barrier_timeout(moe_decode_t handle);

/*
 * The whole layer without any device allocation. The pages have no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc, such as code that runs inside another framework's memory
 * pool, plugin enqueue functions that must not allocate, or real-time loops
 * where an allocation may block. It takes no handle (creating one allocates)
 * and keeps the intermediate h, plus an internal error word, in one
 * fixed-size array in the library's static device memory, which every GPU
 * that loads the library holds until the process exits.
 *
 *   cfg, w_gateup, s_gateup, w_down, s_down   as for moe_decode_create
 *                                              (cfg->max_T is ignored)
 *   x, topk_ids, topk_w, y                     as for moe_decode_layer
 *
 * T * k * I * 2 bytes of h must fit in MOE_NOALLOC_SCRATCH_BYTES (1 MiB,
 * e.g. T = 32 tokens at k = 8, I = 2048); a larger call returns
 * MOE_ERR_UNSUPPORTED_SHAPE and enqueues nothing. The first call on a device
 * looks up the array's device address and sets the kernels' attributes for
 * that device; make that first call before any stream capture. All calls on
 * a device share the one array and it keeps the previous call's contents
 * (nothing in it needs to start at zero: every h value the down kernel reads
 * is written earlier in the same call), so calls whose work overlaps on the
 * GPU, for example on two streams, race and corrupt each other's h.
 * Out-of-range expert ids still contribute nothing, but this call has no way
 * to report them. Nor can it report a bounded device wait that gave up
 * (MOE_DEVICE_TIMEOUT on a handle): with T = 1 the one-launch kernel's CTAs
 * wait for one another on counters kept in the same array, and if such a
 * wait runs out (for example because an overlapping call on another stream
 * holds the SMs), that call's y is unspecified and nothing says so. Every
 * call advances those counters by the same fixed amount whatever happens in
 * it, so a later call that does not overlap another one is unaffected. The
 * call plans its launches (kernel choice and TMA tensor maps) on the host and
 * keeps the plan of the latest configuration and weight pointers per device,
 * so repeated calls with the same layer skip that work.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status_t moe_decode_layer_noalloc(const moe_decode_config_t* cfg,
                                      const uint8_t* w_gateup, const uint8_t* s_gateup,
                                      const uint8_t* w_down, const uint8_t* s_down, int32_t T,
                                      const uint16_t* x, const int32_t* topk_ids,
                                      const float* topk_w, uint16_t* y, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_H */
