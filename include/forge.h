/*
 * forge.h -- C ABI of the FORGE tile-fused weight-gradient + optimizer step
 * for one linear layer y = x W^T, on NVIDIA GB300 (sm_103a).
 *
 * Method: "FORGE: Fused On-Register Gradient Elimination for Memory-Efficient
 * LLM Training" (gist.science explainer), Technical Summary §2 "Core
 * Mechanism": for each tile of W the weight gradient dW = dY^T X is
 * accumulated over all tokens in FP32, the elementwise optimizer is applied to
 * that tile at once, and only the updated weights and (optionally quantised)
 * moments are written back -- no dW tensor ever reaches global memory.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers on the current CUDA device,
 *    caller-owned, row-major and contiguous, 16-byte aligned.  The library
 *    never allocates, frees or retains them beyond the call.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *    is the legacy default stream).  Arguments the host can check are checked
 *    before anything is launched; a failed check launches nothing and returns
 *    FORGE_ERR_INVALID_ARG or FORGE_ERR_UNSUPPORTED with a message available
 *    from forge_last_error_message() on the calling thread.
 *  - Errors found on the device (a bounded pipeline wait that ran out) are
 *    recorded in a per-device status word and reported by
 *    forge_get_device_status().  Kernels never trap.
 *  - Shapes: T tokens, N out-features (rows of W), K in-features.
 *    X is [T x K] bf16, dY is [T x N] bf16, W is [N x K], dX is [T x K] bf16.
 *    Requirements: N % 8 == 0, K % 8 == 0 (16-byte rows for the tensor-memory
 *    accelerator); K % 64 == 0 when states are INT8; T >= 0 (T == 0 applies
 *    the optimizer to a zero gradient).  No tile-size multiple is required:
 *    ragged edge tiles are handled.
 *  - Element index: the element W[n, k] has index n*K + k; stochastic rounding
 *    draws its random bits from Philox4x32-10 keyed by `seed` with counter
 *    (idx/8 low, idx/8 high, step low, step high), element idx%8 taking 16-bit
 *    half (idx%2) of output word (idx%8)/2.  Use a distinct seed per weight
 *    matrix.
 */
#ifndef FORGE_H_
#define FORGE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FORGE_ABI_VERSION 1

#if defined(__GNUC__)
#define FORGE_API __attribute__((visibility("default")))
#else
#define FORGE_API
#endif

typedef enum forge_status {
  FORGE_OK = 0,
  FORGE_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad enum, bad shape      */
  FORGE_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement       */
  FORGE_ERR_CUDA = 3,          /* a CUDA runtime call failed (message has details)  */
  FORGE_ERR_TIMEOUT = 4,       /* a device-side bounded wait expired                */
  FORGE_ERR_DEVICE = 5         /* any other device-side error report                */
} forge_status_t;

/* The eight elementwise rules (Technical Summary §3 "Generality").  Weight
 * decay is decoupled (w *= 1 - lr*wd) for AdamW and Lion and added to the
 * gradient (g += wd*w) for the others.  State buffers per rule:
 *   AdamW/NAdam/RAdam: s1 = first moment m, s2 = second moment v
 *   Lion: s1 = m            RMSprop: s2 = square average
 *   AdaGrad: s2 = sum of g^2   SGD-momentum: s1 = momentum buffer   SGD: none */
typedef enum forge_opt_kind {
  FORGE_ADAMW = 0, FORGE_NADAM = 1, FORGE_RADAM = 2, FORGE_LION = 3,
  FORGE_RMSPROP = 4, FORGE_ADAGRAD = 5, FORGE_SGD = 6, FORGE_SGD_MOMENTUM = 7
} forge_opt_kind_t;

/* Weight storage (§2 "Precision and Fidelity"): FP32 master weights, or BF16
 * weights written back by stochastic rounding. */
typedef enum forge_wdtype { FORGE_W_FP32 = 0, FORGE_W_BF16_SR = 1 } forge_wdtype_t;

/* State storage (§2 "Precision and Fidelity", last bullet): FP32, or INT8
 * codes in blocks of B contiguous elements of a row with one FP32 absmax per
 * block -- B = 64 is the pages' block size; 32, 128 and 256, the other widths
 * that stay inside one 256-column tile pair, exist to measure the pages'
 * block-size claim (64 against the 2048 of standard 8-bit optimizers).  s1
 * (may be negative) is int8 with codes -127..127 and value
 * code * (absmax/127); s2 (never negative) is uint8 with codes 0..255 and value
 * code * (absmax/255).  Scale arrays are [N x K/B] FP32; K % 64 == 0 and
 * K % B == 0.  With fp32 weights the fused step (T > 0) takes B = 64 only. */
typedef enum forge_sdtype {
  FORGE_STATE_FP32 = 0,      /* float32 moments                                           */
  FORGE_STATE_INT8_B64 = 1,  /* int8 / uint8 codes, float32 absmax per 64 row elements     */
  FORGE_STATE_BF16 = 2,      /* bf16 moments, rounded to nearest even after the FP32 rule; */
                             /* with fp32 weights only the optimizer-only entry points and */
                             /* T = 0 accept them (the fused kernels stage bf16 weights)    */
  FORGE_STATE_INT8_B32 = 3,  /* as INT8_B64 with one absmax per 32 row elements            */
  FORGE_STATE_INT8_B128 = 4, /* ... per 128 row elements                                    */
  FORGE_STATE_INT8_B256 = 5  /* ... per 256 row elements                                    */
} forge_sdtype_t;

/* The activations of one linear layer. */
typedef struct forge_linear {
  int64_t T, N, K;     /* tokens, out-features, in-features                    */
  const void* X;       /* bf16 [T x K] input activation                        */
  const void* dY;      /* bf16 [T x N] upstream gradient                       */
  void* dX;            /* bf16 [T x K] output, or NULL to skip the input grad  */
} forge_linear_t;

/* The parameters and optimizer state of one linear layer, updated in place. */
typedef struct forge_state {
  void* W;             /* [N x K] fp32 or bf16 (w_dtype)                        */
  int32_t w_dtype;     /* forge_wdtype_t                                        */
  int32_t s_dtype;     /* forge_sdtype_t                                        */
  void* s1;            /* [N x K] fp32 or int8, or NULL if the rule keeps none  */
  void* s2;            /* [N x K] fp32 or uint8, or NULL if the rule keeps none */
  float* s1_scale;     /* [N x K/B] fp32 absmax, INT8 only (else NULL)          */
  float* s2_scale;     /* [N x K/B] fp32 absmax, INT8 only (else NULL)          */
} forge_state_t;

/* Hyper-parameters; fields a rule does not use are ignored.
 * lr, weight_decay: all rules.  beta1, beta2: AdamW, NAdam, RAdam, Lion.
 * eps: AdamW, NAdam, RAdam, RMSprop, AdaGrad.  alpha: RMSprop.
 * momentum: SGD-momentum. */
typedef struct forge_hparams {
  float lr, beta1, beta2, eps, weight_decay, alpha, momentum;
} forge_hparams_t;

/* The fused backward step of one linear layer (Technical Summary §2 "Core
 * Mechanism" and §5 "Limitations"):
 *   1. if lin->dX != NULL: dX = dY W from the PRE-update W (bf16 operands, FP32
 *      accumulation, bf16 result; FP32 master weights enter as their nearest
 *      bf16);
 *   2. for every W tile: g = dY^T X accumulated over all T tokens in FP32 in
 *      tensor memory, then the rule `opt_kind` applied elementwise (per-step
 *      scalars formed on the host in double from `hp` and `step`), then W
 *      written back (FP32, or BF16 by stochastic rounding) and the states
 *      written back (FP32, or INT8 requantised with the new block absmax).
 * With bf16 weights, dX requested, N and K multiples of 64 and T > 0, both
 * run in ONE persistent launch (the dX tiles first; a W tile is written only
 * after every dX tile of its 256-column block has finished reading W); the
 * launch uses a library-owned counter array in device memory (cleared on
 * `stream` first), so two such calls must not run concurrently on one device
 * (order them on one stream, or call forge_set_step_fusion(0)).  The one
 * launch sizes its grid so that all of its CTA pairs fit on the device at
 * once, and a weight tile waits (bounded) for dX tiles that other pairs run,
 * so it needs all its pairs running together: before any pair writes a
 * weight, the launch checks that every one of its CTAs has started.  If a
 * kernel on another stream holds SMs for longer than the wait limit
 * (forge_set_wait_limit_ns, 2 s by default), the launch stops there: the call
 * reports FORGE_ERR_TIMEOUT (forge_get_device_status) with W, the states and
 * the scales unchanged (dX may be written) and can be repeated, for example
 * after forge_set_step_fusion(0), whose two launches wait on nothing.
 * Callers that overlap long-lived kernels (e.g. a persistent communication
 * kernel) with this step should use that form.  Otherwise
 * dX is a separate launch enqueued first on `stream`.  Both forms compute the
 * same bits.  step is 1-based (bias corrections).  Nothing is allocated; no
 * gradient tensor is written.  Returns FORGE_OK once the launches are
 * enqueued. */
FORGE_API forge_status_t forge_linear_bwd_step(const forge_linear_t* lin, const forge_state_t* state,
                                     int32_t opt_kind, const forge_hparams_t* hp,
                                     int64_t step, uint64_t seed, void* stream);

/* forge_linear_bwd_step on one row shard of a larger weight matrix: the
 * column-parallel (output-feature) split of tensor parallelism, under which
 * the pages' Technical Summary §2 "Distributed Training Compatibility" says
 * the fused step stays exact, because a shard's weight gradient
 * dW_r = dY_r^T X is complete on its own device at backward time (dY_r, the
 * shard's columns of dY, is what that device produced in the forward pass;
 * X is replicated).
 *   - lin->N is the shard's row count; W, s1, s2 and the scales hold only the
 *     shard's rows [row_offset, row_offset + N) of a matrix with K columns;
 *     lin->dY is the shard's [T x N] columns of the upstream gradient.
 *   - Every element is stepped exactly as forge_linear_bwd_step steps the same
 *     element of the whole matrix: stochastic rounding draws the bits of
 *     index (row_offset + n) * K + k, so the shards of a split matrix,
 *     stepped one by one with the same seed, reproduce the unsplit step's
 *     weights and states bit for bit.
 *   - dX (if requested) is this shard's PARTIAL input gradient dY_r W_r
 *     (pre-update W_r, bf16); the layer's dX is the sum of the shards'
 *     partials, which the caller forms (an all-reduce across the devices).
 *   - row_offset >= 0, else FORGE_ERR_INVALID_ARG; row_offset + N must fit in
 *     31 bits.  Everything else as forge_linear_bwd_step (same one-launch and
 *     two-launch forms, same concurrency rule). */
FORGE_API forge_status_t forge_linear_bwd_step_shard(const forge_linear_t* lin,
                                                     const forge_state_t* state, int32_t opt_kind,
                                                     const forge_hparams_t* hp, int64_t step,
                                                     uint64_t seed, int64_t row_offset, void* stream);

/* forge_linear_bwd_step computing the same bits, with the one-launch form's
 * scratch in a fixed, static device array of this library instead of the
 * array that forge_linear_bwd_step uses: the dX-completion counters of the
 * one launch, one 32-bit word per 256-column block of W (1024 words), and the
 * launch's two residency-gate words.  The
 * pages have no counterpart of this entry point; it exists so that a caller
 * can keep such steps off the scratch that forge_linear_bwd_step uses.
 *   - No allocation, ever; the array's device address is looked up once per
 *     device (cudaGetSymbolAddress, checked) and the counters this call uses
 *     are cleared (set to zero) on `stream` before its launch.
 *   - Requests the one launch applies to (bf16 weights, dX requested, T > 0,
 *     N and K multiples of 64) with K > 262144 return FORGE_ERR_UNSUPPORTED
 *     before any CUDA call.  Other requests, and those whose one launch
 *     cannot be resident on the device, need no scratch and run exactly as
 *     forge_linear_bwd_step's two-launch form.
 *   - Races: every call on a device uses the same array.  Two calls whose
 *     launches overlap in time (different streams, no ordering between them)
 *     corrupt each other's counters; order them on one stream or with events.
 *     Calls of this entry point and of forge_linear_bwd_step do not share
 *     scratch. */
FORGE_API forge_status_t forge_linear_bwd_step_static(const forge_linear_t* lin,
                                                      const forge_state_t* state, int32_t opt_kind,
                                                      const forge_hparams_t* hp, int64_t step,
                                                      uint64_t seed, void* stream);

/* The weight-gradient operands of one linear layer in FP8 (E4M3: 1 sign,
 * 4 exponent bits with bias 7, 3 mantissa bits; no infinity; the two codes
 * 0x7F / 0xFF are NaN; largest finite 448), one float scale per tensor:
 * X = decode(Xt)^T * x_scale, dY = decode(dYt)^T * dy_scale.  Both are stored
 * token-contiguous (transposed), T % 16 == 0 so that rows are 16-byte
 * multiples. */
typedef struct forge_linear_fp8 {
  int64_t T, N, K;     /* tokens, out-features, in-features                    */
  const void* Xt;      /* E4M3 codes [K x T] (the input activation, transposed) */
  const void* dYt;     /* E4M3 codes [N x T] (the upstream gradient, transposed) */
  float x_scale;       /* dequantisation scale of Xt                           */
  float dy_scale;      /* dequantisation scale of dYt                          */
} forge_linear_fp8_t;

/* The FORGE step (step 2 of forge_linear_bwd_step) from FP8 operands
 * (Technical Summary §4 "Composability": FORGE composes with FP8
 * quantisation; the pages give no format or scale recipe, so this is one
 * plain reading).  For every W tile, S = sum over tokens of the products of
 * the decoded codes is accumulated in FP32 in tensor memory (tcgen05 E4M3 x
 * E4M3 -> FP32), the gradient is g = S * c with c = x_scale * dy_scale
 * formed in double and rounded once to float, and the rule `opt_kind` is
 * applied exactly as in forge_linear_bwd_step.  BF16 weights (stochastic
 * rounding) only: FP32 weights return FORGE_ERR_UNSUPPORTED.  States: FP32,
 * INT8 blocks (any width) or BF16.  No dX is computed: call forge_linear_dgrad
 * first on the same stream (it reads the weights before this call updates
 * them).  T == 0 applies the rule to a zero gradient.  Requirements as in
 * the shared conventions plus T % 16 == 0 and finite scales; NaN codes
 * propagate into the updated weights.  Nothing is allocated. */
FORGE_API forge_status_t forge_linear_bwd_step_fp8(const forge_linear_fp8_t* lin,
                                                   const forge_state_t* state, int32_t opt_kind,
                                                   const forge_hparams_t* hp, int64_t step,
                                                   uint64_t seed, void* stream);

/* Whether forge_linear_bwd_step may run dX and the FORGE step in one launch
 * (non-zero, the default) or always uses two launches (0).  Process-wide. */
FORGE_API void forge_set_step_fusion(int32_t enable);

/* dX = dY W alone (step 1 above); W is fp32 or bf16 per w_dtype. */
FORGE_API forge_status_t forge_linear_dgrad(const forge_linear_t* lin, const void* W, int32_t w_dtype,
                                  void* stream);

/* Unfused schedule, pass 1 -- the "materialised gradient" the method removes
 * (Technical Summary §1): dW = dY^T X in FP32, written to the caller's
 * [N x K] fp32 buffer dW.  Same tensor-core main loop as the fused step. */
FORGE_API forge_status_t forge_unfused_wgrad(const forge_linear_t* lin, float* dW, void* stream);

/* Unfused schedule, pass 2 -- a separate optimizer kernel reading dW from
 * global memory and applying exactly the per-element arithmetic of the fused
 * step (same rule, rounding and quantisation).  dW == NULL means a zero
 * gradient. */
FORGE_API forge_status_t forge_unfused_opt_step(const float* dW, const forge_state_t* state, int64_t N,
                                      int64_t K, int32_t opt_kind, const forge_hparams_t* hp,
                                      int64_t step, uint64_t seed, void* stream);

/* INT8 state helpers (block 64 along rows; cols % 64 == 0).  quantize: x fp32
 * [rows x cols] -> codes (int8 if is_signed else uint8) and absmax
 * [rows x cols/64].  dequantize: the inverse map code * (absmax/127 or /255). */
FORGE_API forge_status_t forge_quantize_state(const float* x, void* codes, float* absmax, int64_t rows,
                                    int64_t cols, int32_t is_signed, void* stream);
FORGE_API forge_status_t forge_dequantize_state(const void* codes, const float* absmax, float* x,
                                      int64_t rows, int64_t cols, int32_t is_signed,
                                      void* stream);
/* The same two helpers for blocks of `block` (32, 64, 128 or 256) row
 * elements: absmax is [rows x cols/block]; cols % 64 == 0 and
 * cols % block == 0, else FORGE_ERR_INVALID_ARG. */
FORGE_API forge_status_t forge_quantize_state_block(const float* x, void* codes, float* absmax,
                                                    int64_t rows, int64_t cols, int32_t is_signed,
                                                    int32_t block, void* stream);
FORGE_API forge_status_t forge_dequantize_state_block(const void* codes, const float* absmax,
                                                      float* x, int64_t rows, int64_t cols,
                                                      int32_t is_signed, int32_t block,
                                                      void* stream);

/* Synchronises `stream`, then returns and clears the current device's status
 * word: FORGE_OK, FORGE_ERR_TIMEOUT (a bounded wait expired in a kernel) or
 * FORGE_ERR_CUDA (the stream reported a CUDA error). */
FORGE_API forge_status_t forge_get_device_status(void* stream);

/* Bound, in nanoseconds, on every pipeline wait inside the tensor-core
 * kernels (default 2e9).  When a wait expires the kernel records
 * FORGE_ERR_TIMEOUT, stops issuing work, releases its tensor memory and
 * returns.  0 restores the default.  Applies to later launches. */
FORGE_API forge_status_t forge_set_wait_limit_ns(uint64_t ns);

/* Test hook for the failure path: while nonzero, the tensor-core kernels'
 * load-issuing warp issues nothing, so the consumers' bounded waits expire.
 * Never set it outside tests. */
FORGE_API forge_status_t forge_debug_skip_loads(int32_t enable);

/* Static description of a status code. */
FORGE_API const char* forge_status_string(forge_status_t status);

/* Detail of the last host-side error on the calling thread ("" if none). */
FORGE_API const char* forge_last_error_message(void);

/* FORGE_ABI_VERSION of the loaded library. */
FORGE_API int32_t forge_abi_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* FORGE_H_ */
