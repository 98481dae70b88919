/*
 * fp8rl.h -- C ABI of the GB300 (sm_103a) FP8 W8A8 rollout linear path.
 *
 * The path, as the FP8-RL pages describe it ("FP8-RL: A Practical and Stable
 * Low-Precision Stack for LLM Reinforcement Learning"):
 *   1. weight sync: bf16 weights are quantised to E4M3 with one scale per
 *      128x128 block, once per RL step ("Method steps", steps 1 and 2;
 *      format and block formula in "Prerequisites / FP8 quantisation format");
 *   2. activations are quantised dynamically in every forward pass (step 1),
 *      here in 1x128 groups along K;
 *   3. the linears run as W8A8 FP8 GEMMs with fp32 accumulation and bf16
 *      output ("Core method": compute-level W8A8; "Results": FP8 GEMM
 *      kernels), including the MoE expert linears fc1/fc2 (step 1), whose
 *      token-to-expert assignment is a fixed, replayed integer routing
 *      ("MoE RL routing replay (R3)", section 4).
 *   The scale is fp32 (the main variant) or UE8M0, a power of two stored as a
 *   biased 8-bit exponent ("Results", scale-format ablation).
 *
 * Numerics (readings of the pages, fixed here so that results are bit-exact):
 *   scale      = amax / 448 in IEEE fp32 (a block of zeros gets scale 1.0);
 *   UE8M0      = 2^e, e the smallest integer with 448 * 2^e >= amax, clamped
 *                to [-127, 127], stored as the byte e + 127 (zeros: 127);
 *   code       = E4M3 round-to-nearest-even, saturating at +-448, of the fp32
 *                quotient x / scale (UE8M0: the exact x * 2^-e); the sign bit
 *                of x is kept, so -0 gives 0x80;
 *   GEMM       = Y[m][n] = bf16_rne( sum_kb sx[kb][m] * sw[n/128][kb] * P_kb[m][n] )
 *                with P_kb the fp32-accumulated E4M3 products over the 128-wide
 *                K chunk kb, scales applied in fp32 and one rounding at the end
 *                ("Where Rounding Happens Matters": round once, at the end of
 *                the fused region).
 *
 * Conventions for every call:
 *   - Pointers named d_* or documented as device pointers are device memory;
 *     the caller allocates and owns all of it.  The library allocates no
 *     memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream).  Results are ready once the stream
 *     is synchronised.
 *   - Overlapped launches: fp8rl_quant_act_group and the GEMMs at decode
 *     sizes (dense, m <= 64, and up to 128 for the narrow shapes that debug
 *     key 10 lists; fp8rl_gemm_act_quant at m <= 16) are launched
 *     with programmatic stream serialisation, and let the next kernel of the
 *     stream start before they complete.  Such a kernel may begin while the kernel before it on the
 *     stream is still running; it waits for that kernel's completion before
 *     it reads any activation or scale of X and before it writes anything,
 *     but the decode GEMM reads its first weight tiles (wq) before that wait.
 *     No kernel of this library that lets a dependent start early writes
 *     weights; a caller whose own kernel writes wq and triggers its
 *     dependents early (griddepcontrol.launch_dependents) must not enqueue a
 *     decode-size GEMM on that weight right behind it.
 *   - Arguments are validated on the host before any launch; a call that
 *     returns a validation error (INVALID_ARG, SHAPE, ALIGNMENT) launched
 *     nothing.
 *   - Matrices are row-major with an explicit leading dimension in elements.
 *   - No call throws; every call returns an fp8rl_status.
 *   - Non-finite inputs give unspecified codes.
 */
#ifndef FP8RL_H
#define FP8RL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP8RL_API __attribute__((visibility("default")))
#else
#define FP8RL_API
#endif

typedef enum {
    FP8RL_OK = 0,
    FP8RL_ERR_INVALID_ARG = 1, /* null pointer, negative size, unknown enum  */
    FP8RL_ERR_SHAPE = 2,       /* a size the operation does not support      */
    FP8RL_ERR_ALIGNMENT = 3,   /* pointer or leading dimension misaligned    */
    FP8RL_ERR_UNSUPPORTED = 4, /* device is not sm_103 / feature unavailable */
    FP8RL_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed       */
    FP8RL_ERR_TIMEOUT = 6,     /* a device-side bounded wait ran out         */
    FP8RL_ERR_DEVICE_CHECK = 7 /* a device-side bounds check failed (builds
                                  with FP8RL_DEBUG only; the store was skipped) */
} fp8rl_status;

typedef enum {
    FP8RL_SCALE_FP32 = 0,  /* one fp32 scale per block or group          */
    FP8RL_SCALE_UE8M0 = 1  /* one byte per block or group: exponent + 127 */
} fp8rl_scale_fmt;

/*
 * Weight-sync quantisation of one bf16 matrix W [n][k] to E4M3 with one scale
 * per 128x128 block ("Prerequisites / FP8 quantisation format": per-block
 * scale, W_hat = round(W / scale); "Method steps", step 2: done at every
 * weight sync).
 *   w_bf16   device, bf16 [n][k], row stride ldw elements (ldw >= k)
 *   q_e4m3   device, E4M3 bytes [n][k], row stride ldq bytes (ldq >= k)
 *   w_scale  device, [ceil(n/128)][ceil(k/128)] row-major; fp32 or uint8 (fmt)
 * Partial edge blocks take amax over their valid elements only.
 * n == 0 or k == 0 is a no-op.
 * Errors: INVALID_ARG (null pointer, n/k < 0, ld < k, bad fmt),
 *         ALIGNMENT (w_bf16, q_e4m3 not 16-byte aligned, or w_scale not
 *         4-byte aligned for fp32), CUDA (launch failure).
 * Rows whose byte stride is not a multiple of 16 take a slower scalar path.
 */
FP8RL_API fp8rl_status fp8rl_quant_weight_blockwise(const void* w_bf16, int64_t n, int64_t k,
                                                    int64_t ldw, void* q_e4m3, int64_t ldq,
                                                    void* w_scale, fp8rl_scale_fmt fmt,
                                                    void* stream);

/* One matrix of a batched weight sync. */
typedef struct {
    const void* w_bf16; /* device, bf16 [n][k], row stride ldw       */
    void* q_e4m3;       /* device, E4M3 [n][k], row stride ldq       */
    void* w_scale;      /* device, [ceil(n/128)][ceil(k/128)]         */
    int64_t n, k, ldw, ldq;
} fp8rl_weight_desc;

/*
 * Weight sync of many matrices in one pass (a whole model: every linear of
 * every layer).  Same numerics and layout per matrix as
 * fp8rl_quant_weight_blockwise.  `descs` is HOST memory, read during the
 * call only; the descriptors travel to the device inside the launch
 * parameters, so no device-side table is needed.  Matrices are processed as
 * one grid of 128x128 blocks; large counts are split into a few launches.
 * Errors: as fp8rl_quant_weight_blockwise, for any descriptor; count < 0 or a
 * null descs with count > 0 is INVALID_ARG.  count == 0 is a no-op.
 */
FP8RL_API fp8rl_status fp8rl_quant_weight_blockwise_batched(const fp8rl_weight_desc* descs,
                                                            int32_t count, fp8rl_scale_fmt fmt,
                                                            void* stream);

/*
 * Weight sync from HOST memory to HOST memory ("Method steps", step 2: the
 * trainer's bf16 weights are quantised to FP8 at every weight sync).  Same
 * numerics and output layout per matrix as fp8rl_quant_weight_blockwise.
 *   descs      HOST array of `count` descriptors, read during the call only;
 *              their w_bf16, q_e4m3 and w_scale are HOST pointers (any
 *              alignment; row strides ldw, ldq in elements / bytes).  Pinned
 *              memory (cudaHostAlloc, cudaHostRegister) lets the copies run
 *              asynchronously and overlap; pageable memory gives the same
 *              bytes, but then each copy makes the calling thread wait.
 *   d_staging  DEVICE buffer of staging_bytes, owned by the caller, 256-byte
 *              aligned, cut into `slots` (2..8) equal slots; its contents are
 *              overwritten.  fp8rl_host_sync_staging_bytes(rows, k, slots, fmt)
 *              is the size that holds chunks of `rows` rows of a width-k matrix.
 * Each matrix is cut into chunks of whole 128-row block rows, as many as fit a
 * slot (a chunk's codes and scale rows are exactly the whole matrix's); per
 * chunk, a host-to-device copy into a slot, the quantiser, and the copies of
 * the codes and scale rows back to the host run on three streams of the
 * library's own (made once per device and context), chained by events per
 * slot, so both directions of the host link and the kernels overlap.  The
 * work starts after everything enqueued on `stream` before the call (and after
 * the previous call's copies have left the staging slots); work enqueued on
 * `stream` after the call starts after the last copy back, so the host codes
 * and scales are valid once `stream` has been synchronised.  The host buffers
 * must stay alive and untouched until then.  Calls on one device are
 * serialised by the library.
 * Errors: INVALID_ARG (count < 0, null pointers, slots outside 2..8, ldw or
 *         ldq < k, negative sizes), ALIGNMENT (d_staging not 256-byte
 *         aligned), SHAPE (a slot cannot hold one 128-row block row of some
 *         matrix), CUDA.  count == 0 is a no-op.
 */
FP8RL_API size_t fp8rl_host_sync_staging_bytes(int64_t rows, int64_t k, int32_t slots, fp8rl_scale_fmt fmt);
FP8RL_API fp8rl_status fp8rl_quant_weight_host_batched(const fp8rl_weight_desc* descs, int32_t count,
                                                       fp8rl_scale_fmt fmt, void* d_staging,
                                                       size_t staging_bytes, int32_t slots, void* stream);

/*
 * Dynamic activation quantisation in 1x128 groups along K (one scale per token
 * and per 128 columns; "Method steps", step 1: activations quantised in every
 * forward pass).
 *   x_bf16   device, bf16 [m][k], row stride ldx elements
 *   q_e4m3   device, E4M3 [m][k], row stride ldq bytes
 *   x_scale  device, [ceil(k/128)][m] (group-major, so that a GEMM reads one
 *            contiguous run of m scales per K chunk); fp32 or uint8 (fmt)
 * A partial last group takes amax over its valid columns.
 * Errors: as fp8rl_quant_weight_blockwise.
 */
FP8RL_API fp8rl_status fp8rl_quant_act_group(const void* x_bf16, int64_t m, int64_t k, int64_t ldx,
                                             void* q_e4m3, int64_t ldq, void* x_scale,
                                             fp8rl_scale_fmt fmt, void* stream);

/*
 * FP8 KV cache, per-step scale calibration ("Method steps", step 3: the
 * K/V quantisation scales are recomputed from the first forward of every RL
 * step, before its rollout, so that they follow the freshly synced weights).
 * One fp32 scale per tensor (the pages leave the granularity open; per tensor
 * is the plain reading): scale = amax / 448 over the calibration pass, 1.0 for
 * an all-zero tensor.
 *   k_bf16, v_bf16  device, bf16 [tokens][kv_dim], row strides ldk, ldv
 *   q_bf16          device, bf16 [tokens][q_dim] (row stride ldq), or null
 *   d_scales        device, float [3] (q given) or [2]: K, V (, Q) scales;
 *                   written on the stream, never read back on the host
 * Three kernels (zero the words, reduce, convert): the first starts once
 * everything before it on the stream has completed, each later one starts
 * while the one before it runs (overlapped launches, debug key 13) and
 * waits for it before it writes d_scales; work enqueued after the call sees
 * the finished scales.
 * Errors: INVALID_ARG (negative sizes, short strides, null pointers),
 *         ALIGNMENT (element alignment), CUDA.
 */
FP8RL_API fp8rl_status fp8rl_kv_calibrate(const void* k_bf16, const void* v_bf16, const void* q_bf16,
                                          int64_t tokens, int64_t kv_dim, int64_t ldk, int64_t ldv,
                                          int64_t q_dim, int64_t ldq, float* d_scales, void* stream);

/*
 * Quantised append to the FP8 KV cache: row t of K and V, divided by the
 * calibrated scale (IEEE fp32 quotient), rounded to nearest-even E4M3 and
 * saturated at +-448, is written to cache row d_slot_mapping[t] (the flat
 * slot index of a paged cache: block * block_size + offset).  Slots outside
 * [0, num_slots), e.g. -1 for padding, are skipped; slot values are device
 * data and are not read on the host.
 *   k_bf16, v_bf16  device, bf16 [tokens][kv_dim], row strides ldk, ldv
 *   d_slot_mapping  device, int32 [tokens]
 *   k_cache, v_cache device, E4M3 [num_slots][ld_cache]
 *   d_scales        device, float [2]: the K and V scales of fp8rl_kv_calibrate
 * Rows that are 16-byte aligned go through the vector path; any layout is
 * accepted.  Errors: INVALID_ARG, ALIGNMENT (element alignment), CUDA.
 */
FP8RL_API fp8rl_status fp8rl_kv_append(const void* k_bf16, const void* v_bf16, int64_t tokens, int64_t kv_dim,
                                       int64_t ldk, int64_t ldv, const int32_t* d_slot_mapping, void* k_cache,
                                       void* v_cache, int64_t ld_cache, int64_t num_slots, const float* d_scales,
                                       void* stream);

/*
 * Block-scaled W8A8 GEMM: Y = X W^T with E4M3 operands, fp32 accumulation per
 * 128-wide K chunk on the tensor cores, the two chunk scales applied in fp32,
 * and one bf16 round-to-nearest-even at the end ("Core method": W8A8
 * linears; "Where Rounding Happens Matters": round once).
 *   xq       device, E4M3 [m][k] row-major (row stride k)
 *   x_scale  device, [k/128][m] (layout of fp8rl_quant_act_group)
 *   wq       device, E4M3 [n][k] row-major (row stride k)
 *   w_scale  device, [n/128][k/128] (layout of fp8rl_quant_weight_blockwise)
 *   y_bf16   device, bf16 [m][n] row-major (row stride n)
 * n and k must be multiples of 128 (SHAPE otherwise); m >= 0 is free.
 * xq, wq and y_bf16 must be 16-byte aligned, the scales 4-byte (fp32).
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, UNSUPPORTED (not an sm_103 device),
 *         CUDA; a device-side wait that runs out is reported as TIMEOUT by
 *         the next fp8rl_sync_status.
 */
FP8RL_API fp8rl_status fp8rl_gemm_blockscaled(const void* xq, const void* x_scale, const void* wq,
                                              const void* w_scale, void* y_bf16, int64_t m,
                                              int64_t n, int64_t k, fp8rl_scale_fmt fmt,
                                              void* stream);

/*
 * The activation quantisation and the block-scaled GEMM in one call: X (bf16)
 * is quantised in 1x128 groups exactly as fp8rl_quant_act_group quantises it
 * (its codes and scales are written to xq and x_scale), and Y = X W^T is
 * computed from them exactly as fp8rl_gemm_blockscaled computes it, so the
 * results are bit for bit those of the two calls ("Method steps", step 1:
 * activations quantised dynamically in every forward pass, then the W8A8
 * linear).  At decode sizes (m <= 16, ldx a multiple of 8, X 16-byte
 * aligned) one kernel does both: it quantises each 128-wide chunk of X as it
 * streams the weights (one launch instead of two; measured on GB300 as fast
 * as the two overlapped launches over a Qwen3-8B decode layer, faster for
 * the smaller projections, slower for the wide gate-up); otherwise the call
 * runs the two kernels.
 *   x_bf16   device, bf16 [m][k], row stride ldx elements (ldx >= k)
 *   wq, w_scale, y_bf16, m, n, k, fmt   as fp8rl_gemm_blockscaled
 *   xq       device, E4M3 [m][k] row-major (row stride k), 16-byte aligned:
 *            receives the activation codes
 *   x_scale  device, [k/128][m], fp32 or uint8 (fmt): receives the scales
 * Errors: as fp8rl_gemm_blockscaled (xq and x_scale are checked as its X
 * operands), INVALID_ARG for a null x_bf16 or ldx < k.  n == 0 quantises X
 * only; m == 0 is a no-op.
 */
FP8RL_API fp8rl_status fp8rl_gemm_act_quant(const void* x_bf16, int64_t ldx, const void* wq,
                                            const void* w_scale, void* y_bf16, int64_t m, int64_t n,
                                            int64_t k, fp8rl_scale_fmt fmt, void* xq, void* x_scale,
                                            void* stream);

/*
 * Fused gate-up projection of a gated MLP: the block-scaled GEMM against the
 * fused gate/up weight, SiLU(gate) * up computed from the fp32 accumulators
 * (never rounded to bf16), and that result quantised to E4M3 in 1x128 groups
 * along its columns, ready to be the down projection's activation ("Method
 * steps", step 1: activations quantised dynamically; "Where Rounding Happens
 * Matters", "the overall scheme": keep the fused region's intermediate in fp32
 * and round once).  Replaces the bf16 gate-up output, the SwiGLU and the
 * activation quantisation pass of the unfused path.
 *   xq, x_scale      as fp8rl_gemm_blockscaled, [m][k] and [k/128][m]
 *   wq_gate_up       device, E4M3 [2 * inter][k]: the gate and up weights with
 *                    their 128-row blocks interleaved: gate rows 0..127, up
 *                    rows 0..127, gate rows 128..255, up rows 128..255, ...
 *                    (a row order, not arithmetic: the 128x128 block
 *                    quantisation of either layout is the same)
 *   w_scale_gate_up  device, [2 * inter / 128][k/128], in the same block order
 *   hq               device, E4M3 [m][inter] (row stride inter)
 *   h_scale          device, [inter/128][m] (layout of fp8rl_quant_act_group)
 * inter and k must be multiples of 128 (SHAPE otherwise).  fmt applies to the
 * input scales and to h_scale alike.  Alignment and errors as
 * fp8rl_gemm_blockscaled (hq takes the place of y_bf16).
 */
FP8RL_API fp8rl_status fp8rl_gemm_swiglu_quant(const void* xq, const void* x_scale, const void* wq_gate_up,
                                               const void* w_scale_gate_up, int64_t m, int64_t inter,
                                               int64_t k, void* hq, void* h_scale, fp8rl_scale_fmt fmt,
                                               void* stream);

/*
 * The same fused gate-up path over MoE expert row segments (the expert
 * layout of fp8rl_grouped_gemm_blockscaled): expert e's rows
 * offsets[e] .. offsets[e+1]-1 use wq_gate_up[e], each expert's weight with
 * the interleaved block order above.
 *   wq_gate_up       device, E4M3 [num_experts][2 * inter][k]
 *   w_scale_gate_up  device, [num_experts][2 * inter / 128][k/128]
 *   hq               device, E4M3 [rows][inter];  h_scale [inter/128][rows]
 * Errors: as fp8rl_grouped_gemm_blockscaled.
 */
FP8RL_API fp8rl_status fp8rl_grouped_gemm_swiglu_quant(const void* xq, const void* x_scale,
                                                       const void* wq_gate_up, const void* w_scale_gate_up,
                                                       const int32_t* d_offsets, int64_t num_experts,
                                                       int64_t rows, int64_t inter, int64_t k, void* hq,
                                                       void* h_scale, fp8rl_scale_fmt fmt, void* stream);

/*
 * Bytes of workspace that fp8rl_gemm_blockscaled_ws needs on the current
 * device (a 256-byte header, one flag word and one 128 x 256 fp32 tile per SM;
 * about 20 MB on a 152-SM part).  The size does not depend on the shape.
 * Errors: INVALID_ARG (null bytes), UNSUPPORTED (not an sm_103 device).
 */
FP8RL_API fp8rl_status fp8rl_gemm_workspace_size(size_t* bytes);

/*
 * fp8rl_gemm_blockscaled with a caller-provided workspace, which lets shapes
 * whose 128-row tiles would fill the SMs unevenly (e.g. m = 1024) use a
 * stream-K schedule: the K iterations of all tiles are divided evenly over one
 * cooperative wave of CTAs; a CTA that computes the later K chunks of a tile
 * publishes its fp32 partial tile in the workspace, and the CTA holding the
 * tile's first chunks adds the published parts in CTA order and rounds to
 * bf16 once.  The arithmetic per output element is that of
 * fp8rl_gemm_blockscaled (same per-chunk products and scales) with the fp32
 * chunk partial sums added in a different, fixed order; results are
 * deterministic for a given shape and device.  Other shapes run exactly as in
 * fp8rl_gemm_blockscaled and leave the workspace untouched.
 *   workspace        device, 256-byte aligned, at least
 *                    fp8rl_gemm_workspace_size bytes, owned by the caller.
 *                    Zero-fill it once before its first use; the library
 *                    keeps it consistent from then on (also after a TIMEOUT).
 *                    Calls that may run at the same time (other streams or
 *                    threads) need workspaces of their own.
 *   workspace_bytes  its size
 * Other arguments as fp8rl_gemm_blockscaled.
 * Errors: as fp8rl_gemm_blockscaled; a null or short workspace is
 *         INVALID_ARG, a misaligned one ALIGNMENT.
 */
FP8RL_API fp8rl_status fp8rl_gemm_blockscaled_ws(const void* xq, const void* x_scale, const void* wq,
                                                 const void* w_scale, void* y_bf16, int64_t m,
                                                 int64_t n, int64_t k, fp8rl_scale_fmt fmt,
                                                 void* workspace, size_t workspace_bytes,
                                                 void* stream);

/*
 * fp8rl_gemm_blockscaled_ws without a caller workspace: the stream-K scratch
 * is a fixed 24 MiB device array inside the library, so the call allocates
 * nothing.  (No counterpart in the method's description: a convenience of
 * this library.)  Meant for callers that cannot allocate device memory on
 * their path: C code with no device allocator of its own, or loops where an
 * allocation could synchronise the device or fail under memory pressure.
 *   Set-up: the first call on each device, with that device current, looks
 *   the array up and zeroes its header and flags (a synchronous memset and
 *   device synchronisation); make that first call before any stream capture
 *   begins.  Later calls only launch.
 *   Capacity: the scratch the stream-K schedule needs (a 1 KB header and
 *   flags, one 128 x 256 fp32 tile per SM: 19.9 MB on 152 SMs) must fit in
 *   24 MiB; a device that needs more gets UNSUPPORTED and nothing runs.
 *   Races: every call on a device shares the one array.  Calls that may run
 *   at the same time (on different streams, or from different threads
 *   without ordering) corrupt each other's partial tiles; issue them on one
 *   stream, or give each concurrent caller its own workspace through
 *   fp8rl_gemm_blockscaled_ws.
 * Results are bit-identical to fp8rl_gemm_blockscaled_ws for the same
 * arguments.  Arguments and errors as fp8rl_gemm_blockscaled; CUDA if the
 * first-call set-up fails.
 */
FP8RL_API fp8rl_status fp8rl_gemm_blockscaled_static(const void* xq, const void* x_scale,
                                                     const void* wq, const void* w_scale,
                                                     void* y_bf16, int64_t m, int64_t n, int64_t k,
                                                     fp8rl_scale_fmt fmt, void* stream);

/*
 * Grouped (MoE expert) block-scaled GEMM over row segments: for every expert e,
 * rows offsets[e] .. offsets[e+1]-1 of X are multiplied by expert e's weights
 * ("Method steps", step 1: MoE fc1 / fc2 are quantised; "MoE RL routing
 * replay (R3)": the routing is a fixed integer assignment, so the segments
 * are known before the call).
 *   xq        device, E4M3 [rows][k] (rows grouped by expert)
 *   x_scale   device, [k/128][rows]
 *   wq        device, E4M3 [num_experts][n][k]
 *   w_scale   device, [num_experts][n/128][k/128]
 *   d_offsets device, int32 [num_experts + 1], offsets[0] == 0, non-decreasing,
 *             offsets[num_experts] == rows.  Not read on the host; values
 *             outside that contract give unspecified output (rows outside every
 *             segment are left unwritten), never an out-of-bounds access.
 *   y_bf16    device, bf16 [rows][n]
 * Errors: as fp8rl_gemm_blockscaled; num_experts < 1 is INVALID_ARG.
 */
FP8RL_API fp8rl_status fp8rl_grouped_gemm_blockscaled(const void* xq, const void* x_scale,
                                                      const void* wq, const void* w_scale,
                                                      const int32_t* d_offsets, int64_t num_experts,
                                                      int64_t rows, int64_t n, int64_t k,
                                                      void* y_bf16, fp8rl_scale_fmt fmt,
                                                      void* stream);

/*
 * The device E4M3 codec alone: out[i] = E4M3 code of the fp32 in[i],
 * round-to-nearest-even, saturating at +-448, sign bit kept (the conversion
 * every quantiser above applies to its fp32 quotient; FP8-RL page,
 * "Prerequisites / FP8 quantisation format").  Exposed so that the whole fp32
 * input space can be checked against an independent encoder.
 *   d_in   device, fp32 [n] (4-byte aligned)
 *   d_out  device, uint8 [n]
 * Errors: INVALID_ARG (n < 0, null pointer with n > 0), ALIGNMENT, CUDA.
 */
FP8RL_API fp8rl_status fp8rl_e4m3_encode(const float* d_in, int64_t n, uint8_t* d_out, void* stream);

/*
 * Synchronise `stream` and report the first error recorded since the last
 * call: a failed launch (CUDA), or a device-side wait that ran out (TIMEOUT).
 * Clears the recorded device error word of the current device.
 */
FP8RL_API fp8rl_status fp8rl_sync_status(void* stream);

/*
 * Test hooks for the GEMMs (no counterpart on the pages), applied to later
 * launches from any thread:
 *   key 1  tile width: 0 chooses per shape (default), 128 or 256 forces it;
 *   key 2  fault injection: the TMA producer skips K chunk `value` (negative:
 *          off), so the MMA warp's bounded wait runs out and the call reports
 *          TIMEOUT through fp8rl_sync_status (no trap, no hang);
 *   key 3  limit of every device-side wait, in nanoseconds (default 2e9);
 *   key 4  wait style, bit 0: producer and MMA threads poll instead of letting
 *          the hardware park them; bit 1: the same for the epilogue (default 0);
 *   key 5  how many K chunks beyond the shared-memory stages the TMA producer
 *          prefetches into L2 (0..64, default 0: measured slower on GB300);
 *   key 6  split-K cluster size of the dense GEMM: 0 chooses (default), 1..8
 *          forces it (reduced to what can be resident);
 *   key 7  stream-K in fp8rl_gemm_blockscaled_ws: 0 chooses per shape
 *          (default), 1 never, 2 always (m > 32);
 *   key 8  stream-K CTA count: 0 one per SM (default), else min(value, SMs),
 *          at most one per K iteration (1..1024);
 *   key 9  how data-parallel GEMM tiles are stored: 0 chooses per shape
 *          (default), 1 through shared memory and TMA stores, 2 from registers;
 *   key 10 dense GEMMs with at most 128 rows: 0 chooses (default: the
 *          swapped-operand decode kernel up to 64 rows, and up to 128 rows
 *          for fp32 scales, K >= 4096 and at most SMs / 4 blocks of 128
 *          weight rows; the 128-row-tile kernel otherwise), 1 the decode
 *          kernel up to 128 rows, 2 the 128-row-tile kernel;
 *   key 11 UE8M0 GEMMs on whole tiles (data-parallel): 0 chooses (default:
 *          the tensor cores apply the power-of-two scales, block-scaled MMA,
 *          when K >= 2048; below, the per-chunk fp32 promotion), 1 always the
 *          promotion (the fp32-scale path), 2 always the block-scaled MMA;
 *   key 12 dense data-parallel GEMMs on tensor-core pairs (256 x 256 tiles
 *          over clusters of two CTAs): 0 chooses per shape (default), 1
 *          always where the shape allows (n a multiple of 256, m > 128), 2
 *          never;
 *   key 13 overlapped launches of the activation quantiser and the decode
 *          GEMM (see the conventions above) and within fp8rl_kv_calibrate:
 *          0 on (default), 1 off;
 *   key 0  restore all defaults.
 * Every key but 0 is refused (UNSUPPORTED, nothing changes) unless the
 * process environment holds FP8RL_TEST_HOOKS=1 at the time of the call, so
 * that no production caller changes the library's behaviour by accident.
 * Errors: UNSUPPORTED (hooks not enabled), INVALID_ARG for an unknown key or
 * value.
 */
FP8RL_API fp8rl_status fp8rl_debug_set(int32_t key, int64_t value);

/*
 * MoE dispatch plan from replayed routing indices (routing-replay page,
 * "R3: Rollout Routing Replay": the rollout's recorded top-k expert indices
 * per token decide which experts a token's rows go to).  Pair p = t * topk + j
 * is token t's slot j.  Rows of expert e's segment [offsets[e], offsets[e+1])
 * hold the pairs routed to e in increasing p (the stable order; the pages fix
 * none).  An index outside [0, experts) drops its pair.
 *   d_topk          device, int32 [tokens][topk], 1 <= topk <= 32
 *   d_offsets       device, int32 [experts + 1] out (offsets[experts] = routed pairs)
 *   d_row_of_pair   device, int32 [tokens * topk] out: the row of each pair, -1 if dropped
 *   d_token_of_row  device, int32 [tokens * topk] out: the token of each row, -1 past
 *                   offsets[experts]
 *   d_workspace     device scratch of fp8rl_moe_plan_workspace_size() bytes, owned by
 *                   the caller; needs no initial contents; one call at a time per buffer
 * 1 <= experts <= 8192.  Three launches on `stream`; deterministic.
 * Errors: INVALID_ARG (sizes, null pointers, workspace too small), SHAPE
 *         (experts > 8192, tokens * topk >= 2^31 - 4096), ALIGNMENT (4 bytes), CUDA.
 */
FP8RL_API size_t fp8rl_moe_plan_workspace_size(int64_t tokens, int64_t topk, int64_t experts);
FP8RL_API fp8rl_status fp8rl_moe_plan(const int32_t* d_topk, int64_t tokens, int64_t topk, int64_t experts,
                                      int32_t* d_offsets, int32_t* d_row_of_pair, int32_t* d_token_of_row,
                                      void* d_workspace, size_t workspace_bytes, void* stream);

/*
 * MoE dispatch with 1x128 activation quantisation: for every routed pair
 * p = t * topk + j, row d_row_of_pair[p] of the grouped activation is x[t]
 * quantised exactly as fp8rl_quant_act_group quantises a row (FP8-RL page,
 * "Method steps", step 1: activations quantised dynamically in every
 * forward).  Each token row is read and quantised once and its codes and
 * scales are written to all of its rows; pairs with row -1 (dropped) or a
 * row outside [0, rows) write nothing, and rows no pair names are left as
 * they were (the grouped GEMM never reads them).
 *   x_bf16          device, bf16 [tokens][ldx], 16-byte aligned
 *   d_row_of_pair   device, int32 [tokens * topk] (fp8rl_moe_plan's output), 1 <= topk <= 32
 *   q_e4m3          device, E4M3 [rows][ldq] out, 16-byte aligned
 *   x_scale         device, [ceil(k/128)][rows] fp32 or UE8M0 bytes out
 * Errors: INVALID_ARG, SHAPE (tokens * ceil(k/128) >= 2^31 - 2^20), ALIGNMENT, CUDA.
 */
FP8RL_API fp8rl_status fp8rl_moe_dispatch_quant(const void* x_bf16, int64_t tokens, int64_t k, int64_t ldx,
                                                const int32_t* d_row_of_pair, int64_t topk, int64_t rows,
                                                void* q_e4m3, int64_t ldq, void* x_scale, fp8rl_scale_fmt fmt,
                                                void* stream);

/*
 * MoE combine: out[t] = sum over j of gate[t][j] * y[row_of_pair[t * topk + j]],
 * fp32 multiply-adds in slot order, rounded once to bf16 (nearest-even);
 * slots with row -1, or a row outside [0, rows), add nothing (a token none
 * of whose slots has a row gets zeros).  The gates are an input: the router's
 * weights of the recorded experts (replaying indices fixes which experts run,
 * not how their outputs are weighted).
 *   y_bf16          device, bf16 [rows][ldy] (the grouped GEMM's output);
 *                   may be null when rows == 0
 *   rows            y's row count (the plan's offsets[experts] is enough)
 *   d_row_of_pair   device, int32 [tokens * topk] (fp8rl_moe_plan's output)
 *   d_gate          device, fp32 [tokens][topk]
 *   out_bf16        device, bf16 [tokens][ldo]
 * 1 <= topk <= 32.  Errors: INVALID_ARG, SHAPE (rows >= 2^31, or
 *         tokens * ceil(n/8) >= 2^31 - 2^20), ALIGNMENT (element alignment), CUDA.
 */
FP8RL_API fp8rl_status fp8rl_moe_combine(const void* y_bf16, int64_t rows, int64_t n, int64_t ldy,
                                         const int32_t* d_row_of_pair,
                                         const float* d_gate, int64_t tokens, int64_t topk, void* out_bf16,
                                         int64_t ldo, void* stream);

/*
 * Token-level truncated importance sampling weights and the mismatch KL
 * estimate.  FP8-RL page, "Method steps", step 4: w = pi_theta / pi_fp8 =
 * exp(lp_train - lp_rollout), truncated at clip (C = 2 in the pages; their
 * clip to [-C, C] is min(w, C) since w > 0).  Precision-alignment page, "how
 * the gap is measured": the mean over generated tokens of lp_rollout - lp_train.
 *   d_lp_train, d_lp_rollout  device, fp32 [n] log-probabilities of the sampled tokens
 *   d_mask          device, uint8 [n] (nonzero: generated token), or null (all tokens)
 *   d_w             device, fp32 [n] out: min(expf(lp_train - lp_rollout), clip), 0 if masked out
 *   d_kl            device, double [3] out: mean (0 with no token), sum, token count
 *   d_workspace     device scratch of fp8rl_tis_workspace_size(n) bytes, owned by the
 *                   caller, 16-byte aligned; its first 16 bytes must be zero before its
 *                   first use (zero it once when allocating it); every call leaves them
 *                   zero.  One call at a time per workspace.
 * Each difference is made exact in fp32 (a TwoSum: rounded difference plus its
 * error term) and added to an fp32 (hi, lo) pair; the threads' pairs meet in a
 * fixed tree per CTA, the last CTA to finish adds the CTAs' pairs in index
 * order and converts the total to double once.  The grid, and so the order of
 * every addition, depends on n alone: the same bits on every run.  One launch.
 * Errors: INVALID_ARG (negative n, clip <= 0, null pointers, workspace too
 *         small), ALIGNMENT, CUDA.
 */
FP8RL_API size_t fp8rl_tis_workspace_size(int64_t n);
FP8RL_API fp8rl_status fp8rl_tis_weights(const float* d_lp_train, const float* d_lp_rollout, const uint8_t* d_mask,
                                         int64_t n, float clip, float* d_w, double* d_kl, void* d_workspace,
                                         size_t workspace_bytes, void* stream);

/* Static, NUL-terminated name of a status code. */
FP8RL_API const char* fp8rl_status_string(fp8rl_status s);

/* Library version as major * 10000 + minor * 100 + patch. */
FP8RL_API int32_t fp8rl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8RL_H */
