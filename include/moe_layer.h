/*
 * moe_layer.h -- C ABI of the GB300 (sm_103a) quantized MoE decode layer.
 *
 * One handle holds one routed mixture-of-experts layer whose expert weights are
 * affine group-quantised to 4 bits (or 2, 3, 5, 6 or 8: moe_layer_config.bits; or
 * block-scaled fp4: moe_layer_config.weight_format).  moe_layer_forward() runs, for every token row,
 *
 *   router gemv -> softmax/sigmoid top-k -> (fc1_latent_proj) -> per selected
 *   expert: dequant gemv up (+gate), activation, dequant gemv down -> weighted
 *   combine in fp32 -> (fc2_latent_proj) -> + shared expert -> + residual
 *
 * in the layer order of the Bolt 74B-A9B latent MoE (TensorFold PR #1038,
 * native Metal backend, "What's in it": gate gemv -> tf_route_topk ->
 * fc1_latent_proj -> routed experts -> tf_moe_combine_rows -> fc2_latent_proj
 * -> + shared -> + residual), with the fp32 router / sigmoid top-k / per-expert
 * norm and sum of TensorFold PR #1295 (Muse Spark Open, "What this changes"),
 * and MLX-style affine int4 weights (mlx-bun decode-speed program, weight
 * format table: affine, group sizes 32/64/128, a scale and a bias per group;
 * 3- and 8-bit affine codes: the same program, section 7.2 "Freeze the
 * controls and workload matrix", weights row, and section 7.8 "Execution
 * progress and next measurements", the 3/8-bit affine dispatches).
 *
 * Every call's arithmetic runs in this library's CUDA kernels on the GPU; there
 * is no CPU fallback.  The library serves one GPU (compute capability 10.3).
 *
 * Conventions
 *   - "device pointer": memory of the GPU the handle was created on;
 *     "host pointer": ordinary or pinned host memory.
 *   - Matrices are row-major and contiguous.
 *   - Packed b-bit codes (b = bits: 2, 3, 4, 5, 6 or 8): the codes of a row form one
 *     little-endian bit stream of uint32 words -- element i occupies stream
 *     bits b*i..b*i+b-1, stream bit j is bit j%32 of word j/32, so a 3-, 5- or 6-bit code
 *     may straddle two words.  For b = 4: eight codes per uint32, element 8*w+i
 *     in bits 4*i..4*i+3 (lowest nibble first).  A weight is scale*q + bias
 *     (q unsigned, 0..2^b-1), with the scale and bias of its group of
 *     group_size consecutive elements along the input (reduction) axis.
 *   - NVFP4 experts (weight_format = MOE_WFMT_NVFP4): the codes are 4-bit
 *     E2M1 values (bit 3 sign, bits 2..1 exponent, bit 0 mantissa: magnitudes
 *     0, 0.5, 1, 1.5, 2, 3, 4, 6), packed like 4-bit affine codes; every block
 *     of 16 consecutive elements along the input axis has one E4M3 scale byte
 *     (sign, 4 exponent bits with bias 7, 3 mantissa bits; 0x7F/0xFF are NaN),
 *     and every expert matrix one fp32 scale: a weight is
 *     e2m1(q) * e4m3(block scale) * matrix scale.  The mlx-bun decode-speed
 *     program's weight-format table lists "mxfp4/nvfp4" among its supported
 *     formats; the element and scale encodings are those of the OCP
 *     Microscaling (MX) specification's FP4 E2M1 and FP8 E4M3 types.
 *   - MXFP4 experts (weight_format = MOE_WFMT_MXFP4): the same E2M1 codes with
 *     one E8M0 scale byte per 32 consecutive elements along the input axis
 *     (the power of two 2^(byte - 127); 0xFF is NaN) and no other term: a
 *     weight is e2m1(q) * 2^(s - 127) (the same specification's MXFP4).
 *   - bf16/fp16 buffers hold IEEE/bfloat16 16-bit values.
 *   - Every function returns a moe_status; MOE_OK is 0.  On error nothing that
 *     the call allocated stays allocated, and moe_layer_last_error() (where a
 *     handle exists) describes the failure.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 4

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, T out of range, overlapping x/out */
  MOE_ERR_UNSUPPORTED = 2,  /* a valid request this build does not serve */
  MOE_ERR_TOPK_GT_E = 3,    /* top_k < 1 or top_k > n_experts */
  MOE_ERR_LATENT_PROJ = 4,  /* latent layer with a missing fc1/fc2, or non-16-bit */
  MOE_ERR_SHAPE = 5,        /* sizes not multiples of the group size / 64 */
  MOE_ERR_DEVICE = 6,       /* current device is not compute capability 10.3 */
  MOE_ERR_OOM = 7,          /* device allocation failed */
  MOE_ERR_CUDA = 8,         /* a CUDA runtime call failed */
  MOE_ERR_TIMEOUT = 9,      /* a bounded device-side wait ran out */
  MOE_ERR_NONFINITE = 10,   /* a router selection key was NaN or infinite */
  MOE_ERR_INDEX = 11        /* MOE_CHECKS builds: a kernel's index check failed */
} moe_status;

typedef enum moe_act {
  MOE_ACT_SWIGLU = 0,  /* h = silu(gate x) * (up x), silu(g) = g / (1 + exp(-g)) */
  MOE_ACT_RELU2 = 1    /* h = max(up x, 0)^2 (no gate matrix) */
} moe_act;

typedef enum moe_router {
  MOE_ROUTER_SOFTMAX = 0, /* key = logit z; w = softmax over the selected ids
                             (renormalize=1) or over all experts (renormalize=0) */
  MOE_ROUTER_SIGMOID = 1  /* key = sigmoid(z) + router_bias; w = sigmoid(z),
                             divided by its sum over the selected ids when
                             renormalize=1; then times routed_scale */
} moe_router;

typedef enum moe_dtype { MOE_DTYPE_BF16 = 0, MOE_DTYPE_FP16 = 1, MOE_DTYPE_FP32 = 2 } moe_dtype;

/* Kernel schedule of a forward.
 *   GEMV     CUDA-core kernels on one stream with programmatic dependent
 *            launch: the dense pass over x (router, fc1_latent_proj, shared
 *            gate/up) with the top-k fused into a routing CTA, the expert up
 *            and down projections (the weighted combine fused into the down
 *            projection's last CTA per column range), and the output pass
 *            (fc2_latent_proj, shared down, residual).  For few token rows.
 *   GROUPED  row-grouped tcgen05 GEMMs for the experts and dense projections
 *            (many token rows per forward).
 *   AUTO     GROUPED when T >= 32 (MOE_GROUPED_MIN_T), else GEMV. */
typedef enum moe_path {
  MOE_PATH_AUTO = 0,
  MOE_PATH_GEMV = 1,
  MOE_PATH_GROUPED = 2
} moe_path;

/* Expert weight formats (moe_layer_config.weight_format). */
typedef enum moe_weight_format {
  MOE_WFMT_AFFINE = 0,   /* b-bit codes, scale and bias per group of group_size */
  MOE_WFMT_NVFP4 = 1,    /* E2M1 codes, E4M3 scale per 16, fp32 scale per matrix */
  MOE_WFMT_MXFP4 = 2     /* E2M1 codes, E8M0 scale per 32 */
} moe_weight_format;

typedef struct moe_layer_config {
  int32_t hidden;        /* H: width of x and out; multiple of 64 */
  int32_t n_experts;     /* E: routed experts, 1..1024 */
  int32_t top_k;         /* k: experts per token, 1..min(E, 16) */
  int32_t expert_ffn;    /* F: routed expert width; multiple of 64 and of group_size */
  int32_t latent;        /* L: latent width of the routed experts, 0 = none (experts on H) */
  int32_t group_size;    /* G: 32, 64 or 128 (NVFP4: 16, the scale block) */
  int32_t shared_ffn;    /* shared expert width, 0 = no shared expert */
  int32_t max_tokens;    /* largest T a forward call may pass, >= 1 */
  int32_t act;           /* moe_act (routed and shared experts alike) */
  int32_t router;        /* moe_router */
  int32_t renormalize;   /* 1: normalise weights over the selected ids */
  float routed_scale;    /* multiplies the combine weights (after normalising) */
  int32_t has_router_bias; /* sigmoid routing: per-expert fp32 selection bias */
  int32_t act_dtype;     /* BF16|FP16: x, out, fc1/fc2 and shared expert weights */
  int32_t scale_dtype;   /* BF16|FP16: expert scales and biases (ignored by NVFP4) */
  int32_t router_dtype;  /* BF16|FP16|FP32: router weight (x is widened to fp32) */
  int32_t bits;          /* code width of the routed experts: 2, 3, 4, 5, 6 or 8
                            (0 = 4).  Widths other than 4 run the GEMV schedule only: AUTO
                            selects it at every T, GROUPED is refused */
  int32_t weight_format; /* moe_weight_format (0 = affine).  NVFP4 needs bits 0
                            or 4 and group_size 16, MXFP4 bits 0 or 4 and
                            group_size 32; like 3/8-bit layers they run the
                            GEMV schedule only (the warp-MMA expert kernel) */
} moe_layer_config;

/* Weights, all DEVICE pointers owned by the caller.  moe_layer_create copies
 * them into library-owned buffers (re-laid-out for the kernels) and
 * synchronises before returning, so the caller may free them afterwards.
 * Shapes (Kin = latent if latent > 0 else hidden):
 *   router_w   [E, H]           router_dtype
 *   router_bias[E]              fp32 (has_router_bias only, else NULL)
 *   fc1_latent [L, H], fc2_latent [H, L]  act_dtype (latent layers only)
 *   gate_q, up_q [E, F, Kin*bits/32]  uint32 packed codes (gate_q: SWIGLU only)
 *   gate_s, gate_b, up_s, up_b [E, F, Kin/G]  scale_dtype
 *   down_q     [E, Kin, F*bits/32]  uint32 packed codes
 *   down_s, down_b [E, Kin, F/G] scale_dtype
 *   sh_gate, sh_up [shared_ffn, H], sh_down [H, shared_ffn]  act_dtype
 *     (sh_gate for SWIGLU only; all NULL when shared_ffn == 0)
 * NVFP4 layers: *_q as above (bits 4); *_s the E4M3 block scales, one byte per
 * 16 elements: [E, F, Kin/16] (gate, up) and [E, Kin, F/16] (down) uint8; *_b
 * the per-matrix fp32 scales [E].
 * MXFP4 layers: *_q as above; *_s the E8M0 block scales, one byte per 32
 * elements: [E, F, Kin/32] and [E, Kin, F/32] uint8; *_b unused (may be NULL). */
typedef struct moe_layer_weights {
  const void *router_w;
  const float *router_bias;
  const void *fc1_latent, *fc2_latent;
  const uint32_t *gate_q, *up_q, *down_q;
  const void *gate_s, *gate_b, *up_s, *up_b, *down_s, *down_b;
  const void *sh_gate, *sh_up, *sh_down;
} moe_layer_weights;

typedef struct moe_layer moe_layer;

/* Library ABI version (MOE_ABI_VERSION of the build). */
int32_t moe_abi_version(void);

/* How the library was built: bit MOE_BUILD_CHECKS is set in the debug build
 * (libmoe_gb300_checks.so, compiled with MOE_CHECKS=1).  There, every index a
 * kernel reads from data -- an expert id, a token-pair id or a pair range taken
 * from the route metadata -- is checked against its bound before it addresses
 * memory; a violation is recorded in the device status word (the first one
 * with its site, index and bound), the access is skipped or redirected to
 * index 0, and moe_layer_device_status() returns MOE_ERR_INDEX with the site
 * in moe_layer_last_error().  No kernel traps.  The debug build also opens
 * NVTX ranges around each forward and each of its stages (bit
 * MOE_BUILD_NVTX_DEFAULT; in either build the environment variable MOE_NVTX=1
 * or 0 at moe_layer_create turns them on or off). */
#define MOE_BUILD_CHECKS 1
#define MOE_BUILD_NVTX_DEFAULT 2
int32_t moe_build_flags(void);

/* Host-only validation of a config and of which weight pointers are present,
 * with the same refusals and codes as moe_layer_create; touches no device.
 * `w` may be NULL to check the config alone.  Refusals, in order:
 *   MOE_ERR_INVALID_ARG   null cfg, non-positive sizes, bad enum values, bits
 *                         not 0, 2, 3, 4, 5, 6 or 8 (NVFP4, MXFP4: not 0 or 4), an unknown
 *                         weight_format
 *   MOE_ERR_TOPK_GT_E     top_k < 1 or top_k > n_experts (a layer whose top-k
 *                         exceeds its own expert count is refused before any
 *                         weight is read: TensorFold PR #1038, "What's in it")
 *   MOE_ERR_LATENT_PROJ   latent > 0 with fc1/fc2 missing or act_dtype not
 *                         16-bit (missing/non-bf16 latent projections are
 *                         refused by name in the same passage)
 *   MOE_ERR_SHAPE         G not 32/64/128 (NVFP4: not 16; MXFP4: not 32), or H, F, Kin not
 *                         multiples of 64 and of G, or expert weights present
 *                         for a shape that cannot hold them
 *   MOE_ERR_UNSUPPORTED   E > 1024 or top_k > 16 or shared expert without a
 *                         weight, router_bias with softmax routing */
moe_status moe_layer_validate(const moe_layer_config *cfg, const moe_layer_weights *w);

/* Create a layer on the current CUDA device.  Validates (as above), refuses a
 * device that is not compute capability 10.3 (MOE_ERR_DEVICE), then allocates
 * and fills library-owned copies of the weights and a workspace for
 * max_tokens rows, using `stream` (a cudaStream_t, NULL = legacy default) and
 * synchronising it before returning.  On any failure every allocation made so
 * far is freed and *out is set to NULL. */
moe_status moe_layer_create(const moe_layer_config *cfg, const moe_layer_weights *w,
                            void *stream, moe_layer **out);

/* out[T, H] = layer(x[T, H]); x and out are DEVICE pointers in act_dtype,
 * row-major, must not overlap, 1 <= T <= max_tokens.  Asynchronous on
 * `stream`; no host synchronisation.  Returns launch errors only; conditions
 * found on the device (non-finite router keys) are reported by
 * moe_layer_device_status().  One handle serves one stream at a time: calls
 * on different streams must not overlap. */
moe_status moe_layer_forward(moe_layer *h, const void *x, int32_t T, void *out, void *stream);

/* As moe_layer_forward, and also writes (each may be NULL) the selected
 * expert ids topk_ids[T, k] (int32, selection order: larger key first, ties
 * to the lower index), the combine weights topk_w[T, k] (fp32) and
 * delta_f32[T, H] = out - x before the final rounding (fp32).  All DEVICE
 * pointers. */
moe_status moe_layer_forward_ex(moe_layer *h, const void *x, int32_t T, void *out, void *stream,
                                int32_t *topk_ids, float *topk_w, float *delta_f32);

/* End-to-end form for callers holding HOST buffers: copies x_host[T, H] to the
 * device, runs the forward and copies the result to out_host[T, H], all
 * queued on `stream`, then synchronises the stream.  Host buffers should be
 * pinned for asynchronous copies. */
moe_status moe_layer_forward_host(moe_layer *h, const void *x_host, int32_t T, void *out_host,
                                  void *stream);

/* Choose the routed-expert path for later forwards (A/B testing).  A path this
 * build cannot serve for the layer returns MOE_ERR_UNSUPPORTED (GROUPED for a
 * layer with a code width other than 4, NVFP4 or MXFP4 experts, or fp32
 * activations). */
moe_status moe_layer_set_path(moe_layer *h, int32_t path);

/* Synchronises `stream`, reads and clears the device status word: MOE_OK, or
 * MOE_ERR_INDEX / MOE_ERR_TIMEOUT / MOE_ERR_NONFINITE (in that precedence) for
 * conditions kernels recorded since the last call. */
moe_status moe_layer_device_status(moe_layer *h, void *stream);

/* Kernel stages of one forward, in launch order: 0 dense projections of x
 * (router gemv, fc1_latent_proj, shared gate/up), 1 routing, 2 expert up
 * (+gate, activation), 3 expert down, 4 combine + fc2_latent_proj + shared
 * down + residual. */
#define MOE_NUM_STAGES 5

/* enable != 0: later forwards record a CUDA event on their stream before each
 * stage and after the last (for per-kernel timing); 0 turns it off. */
moe_status moe_layer_profile(moe_layer *h, int32_t enable);

/* Waits for the last profiled forward and writes min(n, MOE_NUM_STAGES)
 * stage durations in milliseconds to ms[] (host pointer).  Returns
 * MOE_ERR_INVALID_ARG if profiling is off or no forward was profiled. */
moe_status moe_layer_stage_times(moe_layer *h, float *ms, int32_t n);

/* Path (moe_path, never AUTO) a forward of T rows takes on this handle, or
 * -1 for a NULL handle or T outside 1..max_tokens.  Pure host query. */
int32_t moe_layer_path_for(const moe_layer *h, int32_t T);

/* Kernel launches the handle's last forward made (0 before the first).
 * Pure host query. */
int32_t moe_layer_last_launch_count(const moe_layer *h);

/* Bytes of device memory the handle owns (weights + workspace). */
int64_t moe_layer_device_bytes(const moe_layer *h);

/* Frees everything the handle owns.  NULL is a no-op. */
moe_status moe_layer_destroy(moe_layer *h);

/* Static name of a status code. */
const char *moe_status_string(moe_status s);

/* Last error message of a handle ("" if none); NULL handle gives the last
 * error of the most recent failed create on this thread. */
const char *moe_layer_last_error(const moe_layer *h);

/* Largest T that moe_router_topk_noalloc accepts. */
#define MOE_NOALLOC_MAX_TOKENS 64

/* Router gemv + top-k selection that allocates no device memory.  (The pages
 * have no counterpart to this call; it exists for callers of this library.)
 *
 * For callers that cannot call cudaMalloc where they need the routing
 * decision -- a runtime whose device memory belongs to its own caching
 * allocator, an engine that fixes its memory plan up front, or a
 * latency-critical path where an allocation could synchronise the device.
 * Creating a moe_layer handle allocates a workspace; this call does not.  It
 * applies the top-k selection rules of moe_layer_forward_ex (the same routing
 * block, stopped after the ids and weights) to fp32 router logits from its own
 * CUDA-core router gemv of the same x, router weight, bias and routing
 * options.  (The layer computes bf16 router logits on the tensor cores, with
 * exact products and fp32 sums in another order, so the two agree on the ids
 * except at exact ties and on the weights to a few ulps.)  It writes
 *   topk_ids[T, k]  int32, selection order (larger key first, ties to the
 *                   lower index, non-finite keys last),
 *   topk_w[T, k]    fp32 combine weights,
 *   *key_status     int32, only when key_status is not NULL: 0, or bit 0 set
 *                   (value 1) when a selection key of this call was NaN or
 *                   infinite -- the condition moe_layer_device_status reports
 *                   as MOE_ERR_NONFINITE.  With key_status NULL that
 *                   condition is not reported (the keys still rank last).
 * Inputs: x[T, hidden] (x_dtype BF16|FP16), router_w[n_experts, hidden]
 * (router_dtype), router_bias[n_experts] fp32 or NULL (sigmoid routing only).
 * All pointers are DEVICE pointers owned by the caller; the call is
 * asynchronous on `stream`.
 *
 * Scratch: a fixed array in the library's device memory (the fp32 logits of
 * up to MOE_NOALLOC_MAX_TOKENS rows x 1024 experts, a counter and a status
 * word: 256 KB) that every GPU loading the library holds until the process
 * exits.  Limits: T <= MOE_NOALLOC_MAX_TOKENS, n_experts <= 1024,
 * top_k <= 16; larger sizes return MOE_ERR_UNSUPPORTED.  The first call on a
 * device looks up the array's device address and sets kernel attributes (once
 * per device, with that device current); make that first call before any
 * stream capture.  Every call shares the one array and clears what must start
 * at zero, so calls that overlap on the GPU (on different streams, or from
 * several host threads without ordering) race and must not be issued.
 * Errors: MOE_ERR_INVALID_ARG (NULL pointer, T < 1, hidden not a positive
 * multiple of 64, unknown enum), MOE_ERR_TOPK_GT_E, MOE_ERR_UNSUPPORTED,
 * MOE_ERR_DEVICE (not compute capability 10.3), MOE_ERR_CUDA (launch). */
moe_status moe_router_topk_noalloc(const void *x, int32_t T, int32_t hidden, int32_t x_dtype,
                                   const void *router_w, int32_t router_dtype,
                                   const float *router_bias, int32_t n_experts, int32_t top_k,
                                   int32_t router, int32_t renormalize, float routed_scale,
                                   int32_t *topk_ids, float *topk_w, int32_t *key_status,
                                   void *stream);

/* Device allocations currently held by all handles of this process (for leak
 * checks around refused creates). */
int64_t moe_debug_live_allocations(void);

/* Host-side fault injection for tests: make the n-th device allocation from
 * now on fail with MOE_ERR_OOM (n >= 1), or disable with n = 0. */
void moe_debug_fail_allocation(int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYER_H */
