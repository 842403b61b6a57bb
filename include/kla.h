/* kla.h — C ABI of the GB300 Kalman Linear Attention (KLA) scan library.
 *
 * The operation: "Technische Samenvatting: Kalman Linear Attention (KLA)"
 * (gist.science/nl/paper/2602.10743). Methodologie §1 "Probabilistische
 * Formulering" gives the model — an exactly discretised Ornstein–Uhlenbeck
 * prior with process noise p̄_t, tokens observed through an operator k_t with
 * value precision Λ^v_t, and a readout of the posterior mean through q_t.
 * Methodologie §2 "Parallelisatie via Möbius-transformaties" gives the filter
 * in information form: the precision is a Möbius map of the previous one,
 *     λ_t = (α λ_{t-1} + β) / (γ λ_{t-1} + δ),
 * these maps compose associatively (a prefix scan over T), and the
 * information mean follows an affine map. "Belangrijkste Bijdragen" item 1
 * fixes the diagonal structure: each head's d_k × d_v state elements are
 * independent scalar filters.
 *
 * Per head (b, h), element (i, j) and token t, with c = k_{t,i}² Λ^v_{t,j}:
 *     α = 1 + c p̄_{t,i},  β = c a_{t,i}²,  γ = p̄_{t,i},  δ = a_{t,i}²
 *     λ_pred = λ_{t-1} / (a² + p̄ λ_{t-1})
 *     λ_t = λ_pred + c                        (= the Möbius step above)
 *     η_t = (a λ_pred / λ_{t-1}) η_{t-1} + k_{t,i} Λ^v_{t,j} v_{t,j}
 *     y_{t,j} = Σ_i q_{t,i} η_{t,i,j} / λ_{t,i,j}
 * (λ0, η0) is the belief before the first token; the readout of token t uses
 * the posterior that includes token t.
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    allocates no device memory and keeps no state beyond a per-device cache
 *    of the SM count. The one exception is kla_forward_chunked_noalloc: its
 *    fixed 32 MiB scratch array lives in device memory on every GPU that
 *    loads the library, its address is cached per CUDA context, and calls of
 *    it that overlap on the GPU race (see its comment below). Work is queued
 *    on `stream` (a cudaStream_t; NULL is the legacy default stream) and the
 *    call returns without synchronising.
 *  - Layout is contiguous row-major with no strides:
 *      q, k, a, pbar : [B, H, T, d_k]     v, lam_v, y : [B, H, T, d_v]
 *      lam0, eta0, lamT, etaT : [B, H, d_k, d_v], always fp32.
 *    The I/O dtype (`io`) applies to q, k, v, lam_v, a, pbar and y.
 *  - d_k and d_v must each be one of 16, 32, 64, 128; B, H ≥ 0 and T ≥ 0
 *    (an empty batch or T = 0 is valid; T = 0 copies the initial state).
 *  - Every array pointer must be 16-byte aligned.
 *  - Arguments are validated before anything is launched; on error nothing is
 *    queued and no CUDA call has been made. An asynchronous fault of an
 *    earlier kernel is reported by a later call as KLA_ERR_CUDA.
 *  - Domain (the caller's contract): 0 < a ≤ 1, p̄ ≥ 0, Λ^v ≥ 0, λ0 > 0. The
 *    kernels raise a below 2^-40 to 2^-40 (a NaN a included) and add 2^-40 to
 *    k², which changes results only below fp32 resolution for |k| ≥ 2^-8;
 *    other violations give NaN/Inf in the elements they reach and never a
 *    trap.
 *  - Entry points are thread-safe; calls on one stream are ordered (for
 *    kla_forward_chunked_noalloc, see its comment on overlapping calls).
 */
#ifndef KLA_H_
#define KLA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kla_status {
  KLA_OK = 0,
  KLA_ERR_INVALID_ARG = 1,       /* NULL pointer, negative size, bad enum    */
  KLA_ERR_UNSUPPORTED_SHAPE = 2, /* d_k/d_v not in {16,32,64,128}, too large */
  KLA_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned          */
  KLA_ERR_WORKSPACE = 4,         /* workspace missing or smaller than needed */
  KLA_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed      */
  KLA_ERR_TIMEOUT = 6            /* reserved: a bounded device-side wait gave
                                    up. No current entry point has such a wait,
                                    so none returns this code. */
} kla_status;

typedef enum kla_dtype { KLA_F32 = 0, KLA_BF16 = 1 } kla_dtype;

/* Sequential-per-element scan over all T, or chunk-parallel over T
 * (compose per-chunk maps, carry them across chunks, re-run each chunk). */
typedef enum kla_strategy { KLA_AUTO = 0, KLA_SEQUENTIAL = 1, KLA_CHUNKED = 2 } kla_strategy;

/* Gate activations fused into the scan (the elementwise part of the layer's
 * parameterisation; Methodologie §1 of the summary: OU decay a in (0, 1),
 * process noise p̄ > 0, value precision Λ^v > 0). With a bit set, the
 * corresponding input holds a pre-activation x and the kernels use
 *   KLA_GATE_LAMV_SOFTPLUS: Λ^v = softplus(x) = log(1 + e^x)
 *   KLA_GATE_A_SIGMOID:     a = sigmoid(x) = 1 / (1 + e^-x)
 *   KLA_GATE_PBAR_SOFTPLUS: p̄ = softplus(x)
 *   KLA_GATE_PBAR_OU:       p̄ = softplus(x)·(1 − a²) — the exactly discretised
 *                           OU process with stationary variance softplus(x)
 * (at most one of the two p̄ bits). Gradients from kla_backward are then
 * with respect to the pre-activations. */
typedef enum kla_gate {
  KLA_GATE_LAMV_SOFTPLUS = 1,
  KLA_GATE_A_SIGMOID = 2,
  KLA_GATE_PBAR_SOFTPLUS = 4,
  KLA_GATE_PBAR_OU = 8
} kla_gate;

/* The coefficient pass of the sequential plan. The scan's per-row
 * coefficients of a token (from k, a, p̄, q and k of the token before) serve
 * every column of the head. When a head's columns are split over several
 * thread blocks, each block would build them again; with the pass, one
 * kernel writes them once per (token, row) into the workspace
 * (B·H·T·5·d_k fp32) and the scan blocks copy them. Results are bit for bit
 * those without the pass: it changes how kla_forward runs, not what it
 * computes (Methodologie §1–§2 of the summary cited above). kla_forward
 * only: the chunked plan, the uncertainty readout and the other entry points
 * do not use it. */
typedef enum kla_coef_pass {
  KLA_COEF_AUTO = 0, /* when a head's columns span 4 or more blocks of at most 16 columns and the
                        workspace is at most 16 GiB */
  KLA_COEF_OFF = 1,
  KLA_COEF_ON = 2    /* whenever the plan is sequential */
} kla_coef_pass;

typedef struct kla_options {
  int strategy;      /* kla_strategy */
  int chunk_len;     /* tokens per chunk for KLA_CHUNKED; 0 = automatic; multiple of 32 */
  int rows_per_lane; /* scan-kernel rows per lane: 0 = automatic, else 4 or 8 (8 needs d_k >= 64);
                        another value is INVALID_ARG. Results do not depend on it. */
  int gates;         /* kla_gate bits (0 = inputs are a, p̄, Λ^v themselves); unknown bits or both
                        p̄ bits are INVALID_ARG */
  int coef_pass;     /* kla_coef_pass; another value is INVALID_ARG. Results do not depend on it. */
} kla_options;

/* The launch plan kla_forward would use for this shape on the current device. */
typedef struct kla_plan_info {
  int strategy;           /* KLA_SEQUENTIAL or KLA_CHUNKED (never AUTO)      */
  int chunk_len;          /* tokens per chunk (T for the sequential path)    */
  int num_chunks;         /* ceil(T / chunk_len)                              */
  int cols_per_block;     /* d_v columns handled by one thread block          */
  size_t workspace_bytes; /* device workspace kla_forward needs (0 if none)   */
  int rows_per_lane;      /* d_k rows one lane of the scan kernel holds (4, 8) */
  int coef_pass;          /* 1: kla_forward runs the coefficient pass (its buffer is part of
                             workspace_bytes); 0: it does not */
} kla_plan_info;

/* Plan for the current CUDA device. Errors: INVALID_ARG (out NULL, negative
 * size, bad strategy/chunk_len), UNSUPPORTED_SHAPE, CUDA (no device). */
kla_status kla_plan(int B, int H, int T, int dk, int dv, kla_dtype io, const kla_options* opt,
                    kla_plan_info* out);

/* The same plan for a device with `num_sms` SMs (host-only; no CUDA call). */
kla_status kla_plan_for_sms(int B, int H, int T, int dk, int dv, kla_dtype io,
                            const kla_options* opt, int num_sms, kla_plan_info* out);

/* Bytes of device workspace kla_forward needs on the current device for
 * either I/O dtype; 0 when the plan needs none, (size_t)-1 if the arguments
 * are invalid or no device is available. */
size_t kla_forward_workspace_size(int B, int H, int T, int dk, int dv, const kla_options* opt);

/* Whole-sequence scan (Methodologie §1–§2 of the summary cited above).
 *   q, k, a, pbar [B,H,T,dk] and v, lam_v [B,H,T,dv] in `io`  (inputs)
 *   lam0, eta0 [B,H,dk,dv] fp32; both NULL means λ0 = 1, η0 = 0; one NULL and
 *     the other not is INVALID_ARG.
 *   y [B,H,T,dv] in `io` (output; required unless B·H·T = 0)
 *   lamT, etaT [B,H,dk,dv] fp32 final state (may be NULL; may alias lam0 /
 *     eta0 exactly for an in-place update; partial overlap is not allowed).
 *   workspace / ws_bytes: device scratch of at least
 *     kla_forward_workspace_size() bytes (may be NULL when that is 0): the
 *     chunked plan's chunk maps, or the sequential plan's coefficient pass
 *     (kla_coef_pass); the sequential plan without the pass needs none.
 *   opt: NULL means KLA_AUTO with an automatic chunk length and
 *     KLA_COEF_AUTO. */
kla_status kla_forward(const void* q, const void* k, const void* v, const void* lam_v,
                       const void* a, const void* pbar, const float* lam0, const float* eta0,
                       void* y, float* lamT, float* etaT,
                       int B, int H, int T, int dk, int dv, kla_dtype io,
                       void* workspace, size_t ws_bytes, const kla_options* opt, void* stream);

/* kla_forward plus the belief uncertainty of every readout: the variance of
 * y under the filter's posterior, y_var[t,j] = Σ_i q_{t,i}² P_{t,i,j} with
 * P = 1/λ (each element's posterior variance after token t). The summary
 * states that the layer carries an explicit belief-state uncertainty
 * (Belangrijkste Bijdragen item 3; "Expliciete Onzekerheid" under the
 * results); this readout exposes it per token. Arguments as for kla_forward, plus
 *   y_var [B,H,T,dv] in `io` (output; required unless B·H·T = 0; must not
 *   overlap y). The readout is fused into the scan: the same pass produces
 *   y and y_var (one more multiply-add per element-step and a second
 *   reduction over d_k). Where that kernel's shared memory would not fit
 *   (d_k = 128 with 32-column blocks) the library instead
 *   runs a separate pass without the mean before the main pass, so in-place
 *   λ0/η0 → λ_T/η_T updates stay correct either way. The coefficient pass
 *   (kla_coef_pass) is not used here, so the workspace this needs is at most
 *   kla_forward_workspace_size(). */
kla_status kla_forward_uncertainty(const void* q, const void* k, const void* v, const void* lam_v,
                                   const void* a, const void* pbar, const float* lam0, const float* eta0,
                                   void* y, void* y_var, float* lamT, float* etaT,
                                   int B, int H, int T, int dk, int dv, kla_dtype io,
                                   void* workspace, size_t ws_bytes, const kla_options* opt, void* stream);

/* One recurrent decode step, identical in meaning to kla_forward with T = 1
 * and the state updated in place (same summary, same sections).
 *   q, k, a, pbar [B,H,dk] and v, lam_v [B,H,dv] in `io` (one token)
 *   lam, eta [B,H,dk,dv] fp32, read and overwritten with the posterior
 *   y [B,H,dv] in `io`. */
kla_status kla_step(const void* q, const void* k, const void* v, const void* lam_v,
                    const void* a, const void* pbar, float* lam, float* eta, void* y,
                    int B, int H, int dk, int dv, kla_dtype io, void* stream);

/* kla_step with gate activations (kla_gate bits, as in kla_options.gates). */
kla_status kla_step_gated(const void* q, const void* k, const void* v, const void* lam_v,
                          const void* a, const void* pbar, float* lam, float* eta, void* y,
                          int B, int H, int dk, int dv, kla_dtype io, int gates, void* stream);

/* kla_forward on the chunk-parallel path, for callers that cannot allocate
 * device memory. (Library-side addition: the summary has no counterpart.)
 * Callers that run inside an allocator or memory-pool callback, in a loop
 * that must never take the driver's allocation lock, or under a framework
 * that owns every device allocation cannot provide kla_forward's workspace;
 * this entry point uses a fixed 32 MiB scratch array that the library keeps
 * in device memory instead, so it allocates nothing.
 *   Arguments are those of kla_forward without workspace/options; the
 *   strategy is KLA_CHUNKED with chunk_len tokens per chunk (0 = automatic,
 *   else a multiple of 32).
 *   Returns KLA_ERR_WORKSPACE, before launching anything, when the plan's
 *   workspace (kla_plan with strategy KLA_CHUNKED) exceeds 32 MiB.
 *   The first call in each CUDA context (the device's primary context, or a
 *   context the caller made current) looks up the scratch address in that
 *   context (cudaGetSymbolAddress) and caches it by context; make that first
 *   call before any stream capture. After cudaDeviceReset the device has a new
 *   primary context, so the next call looks the address up again: make it,
 *   too, outside a capture.
 *   All calls on a device share the scratch: calls whose work overlaps on the
 *   GPU (different streams, unordered host threads) race; order them. */
kla_status kla_forward_chunked_noalloc(const void* q, const void* k, const void* v, const void* lam_v,
                                       const void* a, const void* pbar, const float* lam0,
                                       const float* eta0, void* y, float* lamT, float* etaT,
                                       int B, int H, int T, int dk, int dv, kla_dtype io,
                                       int chunk_len, void* stream);

/* Context-parallel sharding over T (Methodologie §2 of the summary: the
 * per-token maps compose associatively, so a sequence can be cut into shards
 * whose composed maps are exchanged). A shard is a contiguous token range of
 * the same heads; a rank holding shard r needs only the maps of shards
 * 0..r-1 to know its start state:
 *   1. kla_shard_map composes the rank's own shard into one map per element;
 *   2. the ranks exchange their maps (an all-gather, done by the caller);
 *   3. kla_shard_start applies the maps of the earlier shards, in order, to
 *      (λ0, η0), giving the shard's start state;
 *   4. kla_forward runs the shard from that state (lam0/eta0 = the start).
 * The result equals one kla_forward over the whole sequence up to fp32
 * rounding (the same arithmetic as the KLA_CHUNKED strategy).
 *
 * kla_shard_map: the composed map of tokens [0, T) of the given inputs,
 *   per element, in homogeneous coordinates P = n/m, μ = e/m (P = 1/λ,
 *   μ = η/λ): with (A, B, C, D, E, F, G) = map[0..6], the map takes the
 *   state (P, μ) before the shard to
 *       P' = (A P + B) / (C P + D),   μ' = (E P + F + G μ) / (C P + D).
 *   The seven entries are scaled by a common power of two per element (the
 *   map is homogeneous, so the scale does not matter).
 *   Inputs as for kla_forward; gates as kla_options.gates.
 *   map: fp32 [7][B,H,dk,dv] (output; entry q at map + q·B·H·dk·dv).
 *   T = 0 writes the identity map. Errors as for kla_forward. */
kla_status kla_shard_map(const void* q, const void* k, const void* v, const void* lam_v,
                         const void* a, const void* pbar, float* map, int B, int H, int T, int dk, int dv,
                         kla_dtype io, int gates, void* stream);

/* kla_shard_start: the start state of the shard that follows n_maps shards.
 *   maps: fp32 [n_maps][7][B,H,dk,dv], the shards' maps in sequence order
 *     (as kla_shard_map writes them); n_maps = 0 gives the initial state.
 *   lam0, eta0: fp32 [B,H,dk,dv] state before the first shard (both NULL:
 *     λ0 = 1, η0 = 0).
 *   lam_start, eta_start: fp32 [B,H,dk,dv] outputs; they may alias lam0 /
 *     eta0 exactly, and must not overlap maps.
 *   Errors: INVALID_ARG (n_maps < 0, missing pointers, overlaps),
 *   UNSUPPORTED_SHAPE, MISALIGNED, CUDA. */
kla_status kla_shard_start(const float* maps, int n_maps, const float* lam0, const float* eta0,
                           float* lam_start, float* eta_start, int B, int H, int dk, int dv, void* stream);

/* Backward pass: gradients of a scalar loss L through kla_forward. It is the
 * exact reverse-mode derivative of the scan defined in Methodologie §1–§2 of
 * the summary cited above (the summary itself states the forward only).
 * A leading g names a gradient of L.
 *   Forward inputs as for kla_forward (q, k, a, pbar, v, lam_v in `io`;
 *     lam0, eta0 fp32 or both NULL for λ0 = 1, η0 = 0).
 *   gy [B,H,T,dv] in `io`: dL/dy (NULL means zero).
 *   glamT, getaT [B,H,dk,dv] fp32: dL/dλ_T, dL/dη_T (each may be NULL = zero).
 *   Outputs, in `io`, written (not accumulated): gq, gk, ga, gpbar
 *     [B,H,T,dk] and gv, glam_v [B,H,T,dv]. Required unless B·H·T = 0.
 *   glam0, geta0 [B,H,dk,dv] fp32 outputs: dL/dλ0, dL/dη0 (both NULL to
 *     skip; one NULL and the other not is INVALID_ARG). With lam0/eta0 NULL
 *     they are the gradients at λ0 = 1, η0 = 0.
 *   workspace / ws_bytes: device scratch of at least
 *     kla_backward_workspace_size() bytes (required when B·H > 0; else
 *     KLA_ERR_WORKSPACE): the forward state every 16 tokens plus, when a
 *     head's columns are split over several blocks, per-row partial sums.
 *   gates: kla_gate bits as in kla_options.gates (the forward that produced
 *     L must have used the same); ga, gpbar, glam_v are then gradients with
 *     respect to the pre-activations.
 *   Outputs must not overlap inputs or each other. Pointers 16-byte aligned
 *   (else MISALIGNED); shape rules and errors as for kla_forward. The order
 *   of the per-row and per-column sums across warps is not fixed, so the
 *   last bits of the results can differ between runs. */
size_t kla_backward_workspace_size(int B, int H, int T, int dk, int dv);

/* Launch geometry kla_backward uses. */
typedef struct kla_backward_plan_info {
  int cols_per_block;     /* d_v columns of one block of the reverse kernel   */
  int cols_per_lane;      /* 8, or 4 or 2 when eight would leave SMs with few warps */
  int threads;            /* threads per block                                 */
  int column_blocks;      /* d_v / cols_per_block                              */
  size_t workspace_bytes; /* what kla_backward_workspace_size returns          */
} kla_backward_plan_info;

/* The backward plan for a device with `num_sms` SMs (host-only; no CUDA
 * call). Errors: INVALID_ARG (out NULL, negative size, num_sms < 1),
 * UNSUPPORTED_SHAPE. B·H = 0 gives an all-zero plan. */
kla_status kla_backward_plan_for_sms(int B, int H, int T, int dk, int dv, int num_sms,
                                     kla_backward_plan_info* out);
kla_status kla_backward(const void* q, const void* k, const void* v, const void* lam_v,
                        const void* a, const void* pbar, const float* lam0, const float* eta0,
                        const void* gy, const float* glamT, const float* getaT,
                        void* gq, void* gk, void* gv, void* glam_v, void* ga, void* gpbar,
                        float* glam0, float* geta0, int B, int H, int T, int dk, int dv,
                        kla_dtype io, int gates, void* workspace, size_t ws_bytes, void* stream);

/* Causal depthwise 1-D convolution with an optional SiLU: the short
 * convolution of the Mamba-like block that the KLA layer sits in
 * (Methodologie §4 "Architectuur" of the summary: 1-D causal convolutions and
 * SiLU activations around the scan; the summary gives neither the width nor
 * the weights, so both are arguments). It maps a [B,H,T,D] stream — e.g. the
 * projections that become q, k or v, each with its own taps — channel by
 * channel (channel = (h, d)):
 *     u[t] = bias[h,d] + Σ_{k<W} weight[h,d,k] · x[t − (W−1) + k]
 *     y[t] = SiLU(u[t]) = u[t] / (1 + e^(−u[t]))   (KLA_ACT_SILU), or u[t] (KLA_ACT_NONE)
 * Tap W−1 multiplies the current token, so weight[h,d,:] is the layout of a
 * depthwise torch Conv1d weight [H·D, 1, W] with left padding. Inputs before
 * token 0 come from a carried window of the W−1 previous inputs, so a
 * sequence cut into pieces — down to one token per call for decoding — gives
 * the same result as one call.
 *   x, y [B,H,T,D] in `io`; y must not overlap any input.
 *   weight [H,D,W] fp32 (required when B·H > 0); bias [H,D] fp32 or NULL (0).
 *   window_in [B,H,W−1,D] in `io`: inputs of tokens −(W−1)…−1 (NULL: zeros).
 *   window_out [B,H,W−1,D] in `io` or NULL: the last W−1 inputs of
 *     (window_in, x), the window_in of the next call. It may be window_in
 *     itself (an in-place update) but must not overlap it otherwise, nor x or y.
 *   With W = 1 the windows are empty and their pointers are ignored.
 *   D: a multiple of 4 in [4, 512]; W in [1, 8] (else UNSUPPORTED_SHAPE);
 *   B, H, T ≥ 0 (T = 0 only copies the window). activation: kla_activation
 *   (else INVALID_ARG). Pointers 16-byte aligned (else MISALIGNED). */
typedef enum kla_activation { KLA_ACT_NONE = 0, KLA_ACT_SILU = 1 } kla_activation;

kla_status kla_conv(const void* x, const float* weight, const float* bias, const void* window_in, void* y,
                    void* window_out, int B, int H, int T, int D, int W, kla_dtype io, int activation,
                    void* stream);

/* Backward of kla_conv for a loss L, given gy = dL/dy [B,H,T,D] (`io`; NULL:
 * zero) and gwindow_out = dL/d(window_out) [B,H,W−1,D] (`io`; NULL: zero).
 *   Forward arguments (x, weight, bias, window_in, W, activation) as in the
 *   kla_conv call being differentiated.
 *   gx [B,H,T,D] in `io` (required when B·H·T > 0): dL/dx.
 *   gwindow [B,H,W−1,D] in `io` or NULL: dL/d(window_in).
 *   gweight [H,D,W] and gbias [H,D] fp32, each NULL to skip: dL/dweight and
 *     dL/dbias, summed over B and T. The sums run in a fixed order (no
 *     atomics), so repeated calls give identical bits.
 *   Outputs are written, not accumulated, and must not overlap any input or
 *   each other.
 *   workspace / ws_bytes: device scratch of at least
 *     kla_conv_backward_workspace_size() bytes when gweight or gbias is wanted
 *     (else KLA_ERR_WORKSPACE); may be NULL otherwise.
 * Shape, alignment and error rules as for kla_conv. */
size_t kla_conv_backward_workspace_size(int B, int H, int T, int D, int W);
kla_status kla_conv_backward(const void* x, const float* weight, const float* bias, const void* window_in,
                             const void* gy, const void* gwindow_out, void* gx, float* gweight, float* gbias,
                             void* gwindow, int B, int H, int T, int D, int W, kla_dtype io, int activation,
                             void* workspace, size_t ws_bytes, void* stream);

/* Static, human-readable name of a status code. */
const char* kla_status_string(kla_status s);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int kla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KLA_H_ */
