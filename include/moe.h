/*
 * moe.h -- C ABI of libmoe: the routed-expert block of a fine-grained
 * sparse-MoE decode step with 4-bit packed expert weights, on one GB300
 * (sm_103a).
 *
 * What one forward computes, per token m of a batch of M:
 *   1. router: the top_k experts with the largest logits (ties: lower expert
 *      index first; NaN orders as -inf) and a softmax over those top_k logits
 *      only ("Sovereign gpt-oss-20B (MXFP4) on Apple Silicon", section 3:
 *      top-4 routing of 32 experts; GPU top-k on the serving path in
 *      "Amortizing the per-token host-sync setup tax ...", section 3);
 *   2. per selected expert e: a = W_gu[e] x + b_gu[e] with W_gu dequantised
 *      on chip (gate rows [0, I), up rows [I, 2I)); h = silu(gate) * up with
 *      silu(g) = g / (1 + exp(-g)); y = W_d[e] h + b_d[e] (the "4 sequential
 *      experts x 2 small-block GEMVs" of the gpt-oss page, section 3);
 *   3. out[m] = r[m] + sum_s w[m][s] * y_{m,s}   (routing-weighted sum into
 *      the residual), rounded to bfloat16 (nearest even).
 *
 * Weight formats ("MXFP4 reader", gpt-oss page section 3; packed int4 with
 * on-chip dequantisation, "Single-stream int4 decode of a 30B MoE", sections
 * 1 and 6).  All matrices are row-major [N_out][K]; two 4-bit codes per byte,
 * the low nibble holding the even element:
 *   MOE_FMT_MXFP4: OCP MX v1.0 MXFP4 -- FP4 E2M1 codes, one E8M0 scale byte
 *                  (value 2^(s-127), 0xFF = NaN) per 32 consecutive elements
 *                  along K.  Scales u8 [N][K/32].
 *   MOE_FMT_INT4 : symmetric int4, W = (code - 8) * s, one fp16 scale per
 *                  `group` consecutive elements along K.  Scales fp16
 *                  [N][K/group].
 *
 * Precision: x, r and out are bfloat16; routing weights are fp32; dot
 * products are accumulated in fp32.  Denormal scales are kept (no flush to
 * zero).  How the activations reach the multiplier depends on the path:
 *   - MXFP4, M <= 4 (tensor cores, kind::mxf4): x and h' = w h enter as sums
 *     of 8 MXFP4 vectors (term j of a 32-element block has the shared
 *     exponent X0 - 2j, X0 the OCP MX exponent of the block; each term takes
 *     the nearest-even E2M1 codes of what the earlier ones left), within
 *     2^-15 of each block's largest magnitude;
 *   - MXFP4, M > 4 (batched grouped GEMMs): x and h are quantised to one
 *     MXFP4 vector each (OCP MX v1.0, nearest even);
 *   - int4: x enters as f16 after an exact power-of-two rescale, h as f16
 *     hi + lo (about 22 bits).
 *
 * Conventions:
 *   - Every call returns a moe_status (0 = MOE_OK).  Arguments are checked
 *     before anything is enqueued: a call that fails validation enqueues no
 *     work and leaves all buffers untouched.  moe_last_error() gives a
 *     message for the calling thread's last failure.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Forward calls are asynchronous on it.
 *   - Device pointers are plain CUDA device addresses (e.g. from a PyTorch
 *     tensor's data_ptr()); they are borrowed for the duration of the work
 *     enqueued by the call and never freed by the library.
 *   - A handle owns all the device memory it uses: the resident weights of
 *     every layer, a fixed workspace sized at moe_create, and a status word.
 *     No forward call allocates.
 *   - A handle is not thread-safe: use it from one host thread and one stream
 *     at a time.  Distinct handles are independent.
 *   - Failures detected on the device (a bounded wait that gave up, an index
 *     out of range) set the handle's status word; read it with
 *     moe_get_status().  Device code never traps.
 *   - A decode layer runs as one persistent launch with one CTA per SM whose
 *     CTAs wait for one another (a grid barrier before the output is summed;
 *     the pieces of a split unit exchange partial sums).  Work that other
 *     streams run at the same time can delay it; each wait gives up after
 *     about a second and reports MOE_ERR_DEVICE_TIMEOUT instead of hanging.
 */
#ifndef MOE_H
#define MOE_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_handle moe_handle;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,    /* bad pointer, size, layer, M or top_k   */
    MOE_ERR_UNSUPPORTED = -2,    /* a shape or format this build does not run */
    MOE_ERR_OOM = -3,            /* device allocation failed in moe_create */
    MOE_ERR_CUDA = -4,           /* a CUDA runtime call failed             */
    MOE_ERR_NOT_LOADED = -5,     /* forward on a layer whose experts were never loaded */
    MOE_ERR_DEVICE_TIMEOUT = -6, /* a device-side bounded wait gave up     */
    MOE_ERR_DEVICE_FAULT = -7    /* a device-side bounds check fired       */
} moe_status;

typedef enum { MOE_FMT_MXFP4 = 1, MOE_FMT_INT4 = 2 } moe_format;

typedef struct {
    int hidden;        /* H: model width, the K of gate_up and the N of down   */
    int intermediate;  /* I: expert width; gate_up has 2I rows                 */
    int num_experts;   /* E experts per layer                                  */
    int num_layers;    /* L layers held resident                               */
    int max_tokens;    /* largest M any forward will be given: 1..4 decode
                          only; 5..8192 also enables the batched path (MXFP4) */
    int max_top_k;     /* largest top_k any forward will be given (<= E)       */
    int format;        /* moe_format                                           */
    int group;         /* elements per scale along K: 32 (MXFP4) or e.g. 64 (int4) */
    int has_bias;      /* 1: bf16 biases b_gu [E][2I] and b_d [E][H] are loaded */
} moe_config;

/* Validate cfg and create a handle on the current CUDA device.  Allocates
 * the resident weight arena for all L layers plus a fixed workspace, and a
 * small pinned host staging buffer for moe_forward_host.
 * Requirements: H and I multiples of 64 and at most 3072; E in 1..256;
 * max_top_k in 1..min(E, 16); max_tokens in 1..8192, above 4 only with
 * MOE_FMT_MXFP4 (else MOE_ERR_UNSUPPORTED); MXFP4 needs group == 32; int4
 * needs group a multiple of 32 dividing both H and I.  Weights are repacked
 * at load into the layout their kernels stream, once: MXFP4 into 128-row
 * tiles whose bytes are the operands of the tensor-core MMA (gate and up rows
 * interleaved per 64), int4 into 16-row slabs of MMA fragments.  The codes,
 * scales and biases take the same bytes as in the caller layout (MXFP4 pads
 * the scales of a partial 128-row tile).  The formats are those of the
 * "MXFP4 reader" ("Sovereign gpt-oss-20B (MXFP4) on Apple Silicon", section 3)
 * and of packed int4 ("Single-stream int4 decode of a 30B MoE", section 1).
 * On success *out receives the handle; on failure *out is set to NULL and
 * nothing stays allocated. */
int moe_create(const moe_config* cfg, moe_handle** out);

/* Copy one layer's experts into the handle (the load-once tables the pages
 * build at start-up instead of per token: "Amortizing the per-token host-sync
 * setup tax ...", section 3).  Each pointer may be host or
 * device memory (any address the CUDA runtime can copy from); the caller keeps
 * ownership and may free or reuse its buffers once the call returns (the call
 * synchronises `stream`).  Layouts (E experts, caller order):
 *   gu_codes  u8 [E][2I][H/2]   gu_scales u8 [E][2I][H/32] | fp16 [E][2I][H/group]
 *   gu_bias bf16 [E][2I]        (NULL allowed only when has_bias == 0)
 *   dn_codes  u8 [E][H][I/2]    dn_scales u8 [E][H][I/32]  | fp16 [E][H][I/group]
 *   dn_bias bf16 [E][H]         (NULL allowed only when has_bias == 0)
 * A layer may be reloaded; the new weights replace the old ones. */
int moe_load_experts(moe_handle* h, int layer,
                     const void* gu_codes, const void* gu_scales, const void* gu_bias,
                     const void* dn_codes, const void* dn_scales, const void* dn_bias,
                     void* stream);

/* Checkpoint-layout flags of moe_load_experts_ex.  The pages verify the
 * MXFP4 reader's orientation against the reference checkpoint ("Sovereign
 * gpt-oss-20B (MXFP4) on Apple Silicon", section 3, "transpose orientation
 * verified"); these accept the layouts a checkpoint may use instead of the
 * caller layout above:
 *   MOE_LOAD_GATE_UP_INTERLEAVED: gate_up rows alternate, row 2j gate row j and
 *     row 2j+1 up row j (codes, scales and gu_bias alike);
 *   MOE_LOAD_TRANSPOSED: both projections stored [K][N] rather than [N][K]:
 *     codes u8 [E][K][N/2] (the element with the even index along N in the low
 *     nibble), scales [E][K/blk][N] (blk = 32 for MXFP4, group for int4); the
 *     biases are vectors and unchanged.  With both flags the transposed
 *     gate_up's N index is the alternating row order.
 * The conversion runs on the device at load time (one extra staging copy of
 * the layer); the resident layout and every forward are those of
 * moe_load_experts. */
typedef enum { MOE_LOAD_GATE_UP_INTERLEAVED = 1, MOE_LOAD_TRANSPOSED = 2 } moe_load_flags;
int moe_load_experts_ex(moe_handle* h, int layer,
                        const void* gu_codes, const void* gu_scales, const void* gu_bias,
                        const void* dn_codes, const void* dn_scales, const void* dn_bias,
                        int flags, void* stream);

/* Router weights of one layer, for calls that leave the logits to the
 * library (router_logits == NULL): logits[m][e] = b[e] + sum_h x[m][h] W[e][h]
 * over the layer's input x (the same bf16 values the experts see; in the
 * stack, the normalised residual), accumulated in fp32 -- the MoE block's
 * gate, whose top-k the pages keep on the GPU ("Amortizing the per-token
 * host-sync setup tax in fused all-layer q4 decode on Apple M1 Ultra",
 * section 3; "Sovereign gpt-oss-20B (MXFP4) on Apple Silicon", section 1,
 * top-4 of 32 experts).  w_bf16 [E][H], bias_bf16 [E] or NULL (zero); host or
 * device memory, copied before the call returns.  Summation order, the same
 * in every kernel (so the decode, int4 and batched paths give the same bits):
 * for each 8-element vector i = lane, lane + 32, ... of the row (lane =
 * 0..31), its elements in order, fused multiply-adds into the lane's sum;
 * then a butterfly over the 32 lanes; then + b[e].  The decode kernels
 * compute the logits inside the layer launch (each CTA a few experts, shared
 * through the grid-wide exchange that publishes the layer's input), so a
 * whole decode step with data-dependent routing stays one launch; the batched
 * path runs one more small kernel first.  A layer may be reloaded. */
int moe_load_router(moe_handle* h, int layer, const void* w_bf16, const void* bias_bf16);

/* One layer.  x bf16 [M][H] (the layer input, already normalised),
 * router_logits fp32 [M][E] -- or NULL: computed from x by the layer's
 * router weights (moe_load_router; MOE_ERR_NOT_LOADED without them) --,
 * out bf16 [M][H]: the residual r on entry and r + MoE(x) on return.
 * 1 <= M <= max_tokens, 1 <= top_k <= max_top_k.  x must not overlap out
 * (checked).  All three are device pointers.
 * M <= 4 runs the decode kernel (one persistent launch).  M > 4 runs the
 * batched path: per-expert grouped GEMMs on the tensor cores
 * (tcgen05.mma kind::mxf4) with x and h quantised to MXFP4 per 32 along K by
 * the OCP MX v1.0 rule (shared exponent floor(log2 amax) - 2, E2M1 nearest-
 * even with saturation); six launches (route, plan, quantise x, the gate_up
 * and down GEMMs, combine), seven when the router weights compute the
 * logits.  moe_set_batched_numerics(MOE_BATCHED_BF16) swaps the quantised
 * GEMMs for kind::f16 ones on weights dequantised to bf16.  Grouped-expert
 * GEMM batching is the lever "Sovereign gpt-oss-20B (MXFP4) on Apple
 * Silicon", section 5, names as untried; the activation quantisation is this
 * library's reading (the tensor-core instruction needs FP4 on both sides). */
int moe_forward(moe_handle* h, int layer, const void* x_bf16, const float* router_logits,
                int M, int top_k, void* out_bf16, void* stream);

/* The SwiGLU form of every forward on this handle (decode, int4, batched, the
 * stack), from the next call on:
 *   h = gc * sigmoid(alpha * gc) * (uc + beta),
 *   gc = min(g, limit), uc = clamp(u, -limit, limit),
 * with g, u the gate and up sums (bias included).  The default (1, +inf, 0)
 * is the plain silu(g) * u of the pages' layer; the expert activation of the
 * gpt-oss model in its public reference implementation is (1.702, 7, 1) --
 * the pages name the model, not these constants.  alpha and beta finite,
 * limit > 0 (+inf for no clamp); else MOE_ERR_INVALID_ARG.
 * moe_forward_noalloc always takes the plain form. */
int moe_set_swiglu(moe_handle* h, float alpha, float limit, float beta);

/* Numerics of the batched path (M > 4) on this handle:
 *   MOE_BATCHED_MXFP4 (default): tcgen05.mma kind::mxf4 -- x and h quantised
 *     to MXFP4 per 32 along K (the OCP MX rule), as that instruction needs;
 *   MOE_BATCHED_BF16: tcgen05.mma kind::f16 -- every weight dequantised to
 *     bf16 in shared memory (exactly: e2m1 * 2^(s-127) is a bf16 value), x as
 *     given and h as bf16 hi + lo (hi = bf16(h), lo = bf16(h - hi)), fp32
 *     accumulation: no activation quantisation, at the cost of the
 *     dequantisation on the CUDA cores.
 * The grouped-expert GEMM is the lever "Sovereign gpt-oss-20B (MXFP4) on
 * Apple Silicon", section 5, names as untried; the two numerics are this
 * library's.  The first switch to bf16 allocates its activation tiles.
 * MOE_ERR_UNSUPPORTED on a handle with max_tokens <= 4. */
typedef enum { MOE_BATCHED_MXFP4 = 0, MOE_BATCHED_BF16 = 1 } moe_batched_numerics;
int moe_set_batched_numerics(moe_handle* h, int numerics);

/* Debug: the router logits of the last call that computed them (the last
 * layer call of a decode launch, or the batched call), fp32 [M][E], copied to
 * the device buffer out_dev on `stream`. */
int moe_debug_router_logits(moe_handle* h, float* out_dev, int M, void* stream);

/* The same layer with host buffers (any host memory, pinned or not): packs x,
 * the residual and the logits into the handle's pinned staging buffer, which
 * is mapped into the device's address space; the layer kernel reads its
 * inputs from it and writes its result into it directly over the host-device
 * link (no separate copies).  Synchronises `stream`, then copies the result
 * into out_bf16.  Argument checks as for moe_forward; router_logits may be
 * NULL (the in-kernel router). */
int moe_forward_host(moe_handle* h, int layer, const void* x_bf16, const float* router_logits,
                     int M, int top_k, void* out_bf16, void* stream);

/* The whole L-layer expert stack for one decode step ("one command buffer per
 * decode", "Single-stream int4 decode of a 30B MoE", sections 1 and 6).  For
 * l = 0..L-1:
 *   x_l = bf16(r_l / sqrt(mean(r_l^2) + 1e-6))   (weightless RMSNorm, per token)
 *   r_{l+1} = bf16(r_l + MoE_l(x_l))
 * The pages name a residual add between layers but no coupling; the
 * normalised input is this library's reading (a literal x + MoE(x) chain
 * overflows within a few layers on these value distributions).
 * resid bf16 [M][H] holds r_0 on entry and r_L on return; logits fp32
 * [L][M][E], or NULL: each layer's logits from its router weights applied to
 * x_l (moe_load_router, every layer), so that the routing of layer l+1
 * depends on the output of layer l inside the one launch.  Layer l+1 reads
 * its logits only after layer l's output is complete.  Device pointers.  One persistent launch for all L layers (grid
 * barriers between them), both formats.  Decode sizes only: M <= 4 (else
 * MOE_ERR_UNSUPPORTED). */
int moe_forward_stack(moe_handle* h, void* resid_bf16, const float* router_logits,
                      int M, int top_k, void* stream);

/* n decode steps of the whole stack in one persistent launch (n tokens, each
 * through all L layers; P2's "all decode tokens into a single command
 * buffer"): step t runs the L layers of moe_forward_stack on its own residual
 * resid[t] (bf16 [n][M][H]: r_0 of step t on entry, its r_L on return) with
 * logits[t] (fp32 [n][L][M][E], or NULL: the in-kernel router, as for
 * moe_forward_stack), steps one after another, exactly as n
 * moe_forward_stack calls in that order would (bit-identical results).  Each
 * layer call reads its logits only after the previous call's output is
 * complete.  Device pointers, 16-byte aligned; decode sizes only (M <= 4);
 * n * L <= 2^30. */
int moe_forward_stack_steps(moe_handle* h, int n, void* resid_bf16, const float* router_logits,
                            int M, int top_k, void* stream);

/* n single-layer decode steps in sequence: step s runs resident layer
 * (layer0 + s) mod L on x[s], logits[s] and out[s] (x bf16 [n][M][H],
 * router_logits fp32 [n][M][E] or NULL for the in-kernel router, out bf16
 * [n][M][H]: the residual of each step
 * on entry, r + MoE(x) on return), exactly as n moe_forward calls in that order
 * would (bit-identical results).  Step s + 1 reads its routing and inputs only
 * after step s's output is complete.  One persistent launch for all n steps,
 * both formats ("all decode tokens in a single command buffer", "Single-stream
 * int4 decode of a 30B MoE", section 1).  Decode sizes only (M <= 4); x must
 * not overlap out; 16-byte aligned.  x, logits and out may be device memory
 * or page-locked host memory mapped into the device's address space at the
 * same address (cudaHostAlloc / cudaMallocHost, or cudaHostRegister with
 * cudaHostRegisterMapped, on a system with unified addressing): the kernel
 * then reads each step's inputs and writes each step's result over the
 * host-device link itself, and the host sees every step's result once
 * `stream` has been synchronised.  Host memory that is not mapped so is
 * rejected (MOE_ERR_INVALID_ARG).  moe_last_bytes then counts each step's
 * distinct experts (a layer run by several steps counts its last step's, n
 * times over). */
int moe_forward_steps(moe_handle* h, int n, int layer0, const void* x_bf16, const float* router_logits,
                      int M, int top_k, void* out_bf16, void* stream);

/* Measurement: the streaming floor of this GPU for decode-sized weight reads.
 * Reads the first `bytes` bytes of resident layers layer0 .. layer0 + n - 1,
 * one layer after another with a grid barrier between them (as dependent
 * decode layers are), with the copy engine and stage sizes of the decode
 * kernels (one CTA per SM, bulk copies of 32 KB, 128 KB in flight per SM) and
 * no compute.  bytes: a multiple of 16, at most one layer's arena.  Device
 * work on `stream`; errors as MOE_ERR_INVALID_ARG. */
int moe_debug_stream_weights(moe_handle* h, int layer0, int n, long long bytes, void* stream);

/* Synchronise `stream` and return (and clear) the handle's device status:
 * MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_FAULT.  After a non-OK
 * status the handle's cross-CTA counters are reset, so it can be used again.
 * (Failure detection: the pages describe none for the GPU path; every wait in
 * this library is bounded and reports here instead of hanging.) */
int moe_get_status(moe_handle* h, void* stream);

/* Debug: decode one stored expert projection to fp32, exactly (each element
 * is e2m1 * 2^(s-127) or (q - 8) * fp16 scale, rounded to fp32 once), from
 * the very bytes the forward kernels stream: MXFP4 from the tile layout, int4
 * from the slabs.  proj 0 = gate_up ([2I][H], caller row order), 1 = down
 * ([H][I]).  out_dev fp32 device buffer of N*K elements.  The bit-exact check
 * of the "MXFP4 reader" against its golden, gpt-oss page section 1. */
int moe_debug_dequant(moe_handle* h, int layer, int expert, int proj, float* out_dev,
                      void* stream);

/* Debug: the router alone.  logits fp32 [M][E] device; idx int32 [M][top_k]
 * and w fp32 [M][top_k] device outputs, selection order (largest first).
 * M up to 65536 here. */
int moe_debug_route(moe_handle* h, const float* logits, int M, int top_k, int* idx, float* w,
                    void* stream);

/* Debug: the batched path's MX quantiser on a flat fp32 vector.  in fp32 [n]
 * device, n a multiple of 32; codes u8 [n/2] (low nibble = even element) and
 * scales u8 [n/32] (E8M0) device outputs, natural order.  No handle needed.
 * in and codes 16-byte aligned. */
int moe_debug_mx_quantize(const float* in, long long n, unsigned char* codes,
                          unsigned char* scales, void* stream);

/* Debug: the quantised h of the last batched forward (M > 4) on this handle,
 * in (token, choice) order: codes u8 [M*top_k][I/2] and E8M0 scales u8
 * [M*top_k][I/32], device outputs (codes 16-byte aligned).  Choice s of token
 * m is the s-th selected expert (largest logit first). */
int moe_debug_batched_h(moe_handle* h, unsigned char* codes, unsigned char* scales, void* stream);

/* Debug: the expert stack run layer by layer with the same kernels as
 * moe_forward_stack (one launch per layer), recording the residual after
 * every layer.  resid bf16 [M][H] is updated in place as in
 * moe_forward_stack; trace bf16 [L+1][M][H] device buffer receives r_0 ..
 * r_L.  router_logits NULL: the in-kernel router, as in moe_forward_stack. */
int moe_debug_stack_trace(moe_handle* h, void* resid_bf16, const float* router_logits, int M,
                          int top_k, void* trace_bf16, void* stream);

/* Debug: moe_forward that also writes the fp32 result before its bf16
 * rounding, out_f32 fp32 [M][H] device (16-byte aligned), for checking the
 * fp32-accumulated output itself.  Everything else as moe_forward. */
int moe_debug_forward_f32(moe_handle* h, int layer, const void* x_bf16, const float* router_logits,
                          int M, int top_k, void* out_bf16, float* out_f32, void* stream);

/* Debug (failure detection): the cross-CTA waits of the MXFP4 decode layer
 * give up after `spin_limit` polls (0 restores the default, about a second),
 * and CTA `skip_cta` (-1: none) skips its arrival at the layer's grid barrier,
 * so that the other CTAs' waits run out.  Applies to moe_forward and
 * moe_debug_forward_f32 calls made after it (stack graphs already captured keep
 * the settings they were captured with).  A call whose wait ran out reports
 * MOE_ERR_DEVICE_TIMEOUT through moe_get_status, which also resets the
 * counters so the handle works again.  Every access stays inside the handle's
 * buffers; nothing traps. */
int moe_debug_set_wait(moe_handle* h, int spin_limit, int skip_cta);

/* Algorithmic expert bytes moved by the last forward call on this handle:
 * codes + scales + biases of the distinct experts selected in each layer,
 * counted once per layer (the byte counters of the pages' tracing, TinyTitan
 * tracker).  Synchronises `stream` (so the signature takes the stream and
 * returns a status, writing *bytes).  Returns MOE_OK and writes *bytes, or an
 * error. */
int moe_last_bytes(moe_handle* h, void* stream, long long* bytes);

/* Bytes of one expert (codes + scales + biases) for this handle's config. */
long long moe_expert_bytes(const moe_handle* h);

/* Number of kernel launches the last forward call enqueued (for the caller's
 * launch accounting; a graph replay counts the kernels inside it). */
int moe_last_launches(const moe_handle* h);

/* Message for the calling thread's most recent failure ("" if none). */
const char* moe_last_error(void);

/* One decode layer for callers that cannot allocate device memory.
 *
 * The pages describe no such call; it exists for users of this library whose
 * runtime forbids cudaMalloc: an inference engine that serves every buffer
 * from its own pre-sized pool, code running while a CUDA graph is captured, or
 * a plug-in that may not touch the CUDA allocator.  Such a caller cannot create
 * a moe_handle (moe_create allocates), so here every input and output is the
 * caller's memory and the call allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.
 *
 * Computes the same layer as moe_forward: out = r + sum_s w_s * y_s for the
 * top_k experts of each token.  The weights are the caller-layout tensors of
 * moe_load_experts for one layer (E experts), on the device; x bf16 [M][H],
 * router_logits fp32 [M][E] and out bf16 [M][H] (the residual on entry) are
 * device pointers; x must not overlap out.  Alignment: x, out and the code
 * and scale arrays 16-byte aligned, router_logits 4-byte, biases 2-byte
 * (else MOE_ERR_INVALID_ARG).  cfg gives H, I, E, format, group and has_bias
 * (its num_layers, max_tokens and max_top_k are ignored).
 *
 * Scratch (h, the per-slot down outputs and the output-tile counters) is one
 * file-scope __device__ array of 1,574,400 bytes that every GPU which loads the
 * library holds until the process exits.  It fixes the limits: M <= 4,
 * top_k <= 16, H and I multiples of 32 and at most 3072; larger sizes return
 * MOE_ERR_INVALID_ARG with a message.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) for that device; make that
 * first call before any stream capture.  Every call uses the same array, and
 * it keeps the contents of the last call (the tile counters are cleared at the
 * start of each call), so calls that overlap on the GPU -- on two streams, or
 * from two threads -- race and must be serialised by the caller.  Runs
 * asynchronously on `stream`. */
int moe_forward_noalloc(const moe_config* cfg, const void* gu_codes, const void* gu_scales,
                        const void* gu_bias, const void* dn_codes, const void* dn_scales,
                        const void* dn_bias, const void* x_bf16, const float* router_logits,
                        int M, int top_k, void* out_bf16, void* stream);

/* Release a handle and all device memory it owns.  NULL is a no-op. */
void moe_destroy(moe_handle* h);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
