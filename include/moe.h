/*
 * moe.h -- C ABI of libmoe: the forward pass of one mixture-of-experts layer
 * on one GPU (router -> token dispatch -> grouped SwiGLU experts -> combine).
 *
 * Sources, by page title and section:
 *   [EP]       Transformers docs, "Expert parallelism" (intro): a router sends
 *              each token to a few experts and gathers the results.
 *   [EP-add]   same page, "Adding an implementation": the expert call takes
 *              (hidden_states, top_k_index, top_k_weights), runs the experts
 *              through experts_forward(tokens, expert_ids, weights), and
 *              returns each token's weighted expert output.
 *   [EP-disp]  same page, "Token dispatch": each (token, expert) pair goes to
 *              its expert, the experts run on what arrives, and the results
 *              are combined with the routing weights.
 *   [EP-impl]  same page, "Choosing an implementation": a path without host
 *              synchronisation can be captured in a CUDA graph.
 *   [TP-pack]  Transformers docs, "Tensor parallelism for inference",
 *              "Packed strategies": gate_up_proj is (num_experts, hidden,
 *              2*expert_dim), applied with a batched matmul and split with
 *              chunk(2, dim=-1) into (gate, up).
 *
 * Notation: T tokens, d hidden size, E experts, k experts per token, f expert
 * FFN width, P = T*k routed (token, expert) pairs.
 *
 * Conventions shared by every entry point:
 *   - All tensors are dense, row-major, and live in DEVICE memory unless an
 *     argument says "host".  The caller allocates and owns every buffer,
 *     including the workspace; the library never allocates or frees memory.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and never synchronises with the host, so a
 *     sequence of calls can be captured in a CUDA graph [EP-impl].
 *     moe_last_device_error() is the one call that synchronises.
 *   - Arguments are checked on the host before anything is launched; a
 *     failed check launches nothing and returns the status.  Returned
 *     statuses describe launch-time problems; problems found by a kernel
 *     (an expert id out of range, a bounded wait that ran out) are recorded
 *     in a device error word read by moe_last_device_error().
 *   - T == 0 is legal: the call returns MOE_OK and launches nothing.
 *   - An expert may receive zero pairs.
 *   - Activation dtype (x, expert weights, x_perm, h_perm, y_perm, out):
 *     MOE_BF16 (fp32 accumulation everywhere) or MOE_F32.  The router weight,
 *     logits and routing weights are always fp32.
 *   - Alignment: every pointer 16-byte aligned; d and f multiples of 8.
 *   - Limits: 1 <= k <= min(E, 32), E <= 1024, P < 2^31.
 *   - Device: the current CUDA device must be an sm_103 GPU (GB300); the
 *     library carries code for that architecture only.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,    /* null pointer, bad size, misalignment */
    MOE_ERR_UNSUPPORTED = -2,    /* shape/dtype outside the limits above, or no sm_103 device */
    MOE_ERR_WORKSPACE = -3,      /* ws_bytes smaller than the call needs */
    MOE_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed */
    MOE_ERR_DEVICE_TIMEOUT = -5, /* a kernel's bounded wait ran out (device error word) */
    MOE_ERR_BAD_ROUTING = -6     /* a kernel met an expert id outside [0, E) (device error word) */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

typedef struct {
    int64_t T;           /* tokens in the batch (>= 0) */
    int32_t d;           /* hidden size */
    int32_t E;           /* number of experts */
    int32_t k;           /* experts per token */
    int32_t f;           /* expert FFN width (gate and up each have f columns) */
    int32_t act_dtype;   /* moe_dtype_t */
    int32_t renormalize; /* 1: divide the chosen k softmax weights by their sum; 0: keep them */
    int32_t scale_inputs;  /* 0: routing weights scale the expert outputs in the combine;
                              1: they scale the expert inputs in the dispatch and the
                              combine sums unweighted (experts that receive tokens already
                              scaled by the router score [EP]; with k == E every expert
                              sees every token: the form with nothing to dispatch) */
} moe_config_t;

/* Human-readable name of a status.  Never NULL; the string is static. */
const char *moe_status_string(moe_status_t status);

/* Detail of the last failed call on this host thread (empty if none). */
const char *moe_last_error_message(void);

/*
 * Bytes of workspace moe_forward needs for `cfg` (0 when T == 0).  The same
 * buffer also satisfies moe_route and moe_dispatch.  The workspace holds the
 * router logits and scratch, routing, dispatch arrays and the permuted
 * activations h_perm, y_perm and, where moe_forward uses it, x_perm (see
 * moe_workspace_layout).  The
 * router's share depends on the current device's SM count (its K splits
 * fill one wave); with no usable device it is sized for 152 SMs.
 */
size_t moe_workspace_size(const moe_config_t *cfg);

/*
 * Where moe_forward keeps its intermediates inside its workspace: byte
 * offsets from the start of the buffer (each 256-byte aligned).  After a
 * moe_forward call has completed, these regions hold that call's router
 * logits, routing, dispatch arrays and permuted activations, so a caller can
 * read, for instance, the chosen experts and weights of every token.
 *   logits    float [T][E]   (including logit_bias)
 *   topk_idx  int32 [T][k],  topk_w float [T][k]
 *   counts    int32 [E],     offsets int32 [E+1]
 *   pos       int32 [P],     src_token int32 [P]   (as moe_dispatch defines them)
 *   x_perm    act [P][d],    h_perm act [P][f],    y_perm act [P][d]
 *   total     = moe_workspace_size(cfg)
 * Any other bytes of the workspace are library scratch.  x_perm is
 * MOE_WS_ABSENT (no such region: the workspace is that much smaller) when
 * moe_forward does not form the permuted rows: with k == E the experts read
 * x directly, and where the first grouped GEMM gathers its rows from x it
 * reads them through src_token (see moe_forward).  T == 0 gives all zeros.  Returns MOE_ERR_INVALID_ARG /
 * MOE_ERR_UNSUPPORTED for a config moe_forward would reject, or a NULL
 * `layout`.  Launches nothing (it only queries the current device's SM
 * count, as moe_workspace_size does).
 */
#define MOE_WS_ABSENT ((size_t)-1)
typedef struct {
    size_t logits, topk_idx, topk_w, counts, offsets, pos, src_token;
    size_t x_perm, h_perm, y_perm;
    size_t total;
} moe_workspace_layout_t;

moe_status_t moe_workspace_layout(const moe_config_t *cfg, moe_workspace_layout_t *layout);

/* Bytes of workspace moe_dispatch needs for `cfg`: the per-chunk expert
 * count matrix (E x chunks int32) and a 16-byte ticket counter. */
size_t moe_dispatch_workspace_size(const moe_config_t *cfg);

/*
 * Number of kernel launches one moe_forward call makes for `cfg`: the router
 * (1 to 3 launches, by path), the dispatch (2; 1 when k == E, except for
 * fp32 with scale_inputs, and 1 when it copies unscaled rows with E <= 16
 * and P <= 16384 as described at moe_dispatch), the two grouped GEMMs (2, or
 * 4 when bf16 experts average 64 to 511 rows each and are split between two
 * tile shapes) and the combine (1).  0 when T == 0; -1 for an invalid
 * configuration.  Makes no CUDA call.
 */
int moe_forward_kernel_launches(const moe_config_t *cfg);

/*
 * Bytes of workspace moe_route needs for `cfg`: 0 when the logits are
 * computed on the CUDA cores (fp32 activations, E < 64 or E > 256, E not a
 * multiple of 16, or d not a multiple of 64); otherwise the three-term bf16
 * split of Wr (E * 3d * 2 bytes) and fp32 partial logits of the K splits.
 */
size_t moe_route_workspace_size(const moe_config_t *cfg);

/*
 * Router [EP-add: the router yields top_k_index and top_k_weights].
 *   logits[t][e] = sum_i x[t][i] * Wr[e][i] + (logit_bias ? logit_bias[e] : 0),
 *     computed in fp32 and written to `logits`;
 *   topk_idx[t][j]: the j-th largest logit of row t; equal logits go to the
 *     lower expert id (+0.0 and -0.0 are equal); a NaN ranks below every
 *     number;
 *   topk_w[t][j] = p_e / (renormalize ? sum of p over the chosen k : 1) with
 *     p = softmax over all E logits of row t.
 * x          [T][d]  act dtype
 * Wr         [E][d]  fp32 (nn.Linear layout)
 * logit_bias [E]     fp32 or NULL: an additive per-expert logit offset
 * logits     [T][E]  fp32, written
 * topk_idx   [T][k]  int32, written; topk_w [T][k] fp32, written
 * ws         at least moe_route_workspace_size(cfg) bytes, 256-byte aligned
 *            (may be NULL when that size is 0)
 * The selection is made on exactly the fp32 values written to `logits`.
 * For bf16 x, d % 64 == 0 and either 64 <= E <= 256 or (8 <= E < 64 and
 * T >= 1024), with E % 8 == 0, the products are formed on the tensor cores:
 * Wr is split into three bf16 terms
 * (w = w1 + w2 + w3, ~2^-25 relative), each product with the exact bf16 x is
 * exact, and accumulation is fp32; otherwise fp32 FMAs on the CUDA cores.
 */
moe_status_t moe_route(const moe_config_t *cfg, const void *x, const float *Wr,
                       const float *logit_bias, float *logits, int32_t *topk_idx,
                       float *topk_w, void *ws, size_t ws_bytes, void *stream);

/*
 * The selection and weights of moe_route on a GIVEN fp32 logit buffer
 * [T][E] (read only).  Writes topk_idx [T][k] and topk_w [T][k].
 */
moe_status_t moe_route_from_logits(const moe_config_t *cfg, const float *logits,
                                   int32_t *topk_idx, float *topk_w, void *stream);

/*
 * Token dispatch, single-device form [EP-disp]: every (token, slot) pair is
 * given a row of the expert-contiguous order.
 *   counts[e]     = number of pairs with topk_idx == e                 [E]
 *   offsets[e]    = sum_{e' < e} counts[e'];  offsets[E] = P            [E+1]
 *   pos[t*k+j]    = row of pair (t, j): offsets[e] + the number of pairs
 *                   (t', j') with topk_idx == e and t' < t (stable, so
 *                   rows of one expert are in ascending token order)    [P]
 *   src_token[r]  = token of row r (src_token[pos[q]] == q / k)         [P]
 *   x_perm[r][:]  = x[src_token[r]][:]                                  [P][d] act dtype
 *                   (scale_inputs: topk_w[q] * x[t][:], formed in fp32 and
 *                   rounded once to the act dtype, for the pair q of row r)
 * topk_idx is [T][k] int32; each entry must lie in [0, E) -- an entry outside
 * sets MOE_ERR_BAD_ROUTING in the device error word and that pair is dropped.
 * topk_w [T][k] fp32: read only when cfg->scale_inputs (may be NULL otherwise).
 * ws: at least moe_dispatch_workspace_size(cfg) bytes, 256-byte aligned.
 * Two launches: a rank kernel (per-chunk counts, stable ranks, and, in its
 * last block, the scan that yields counts and offsets) and a kernel that
 * places every pair's row and copies it.  The rank kernel's ticket counter
 * in ws is cleared first with a 4-byte cudaMemsetAsync on `stream`.
 * One launch, with ws not touched and no memset, when E <= 16, P <= 16384,
 * the rows are not scaled and a row is k KB to 16 KB (d * element size):
 * every block of that launch counts all P ids itself and places its own
 * tokens' pairs.
 */
moe_status_t moe_dispatch(const moe_config_t *cfg, const int32_t *topk_idx,
                          const float *topk_w, const void *x, int32_t *counts,
                          int32_t *offsets, int32_t *pos, int32_t *src_token,
                          void *x_perm, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_dispatch without a caller workspace.  (The pages have no counterpart:
 * this is a deployment variant of the same dispatch.)
 *
 * For callers that cannot allocate device memory for scratch: a plugin whose
 * host framework owns all device memory and passes only the layer's inputs
 * and outputs, or a service that must not call cudaMalloc after start-up.
 * The scratch moe_dispatch would take from `ws` (its count matrix and ticket
 * counter) lives instead in a fixed 1 MiB array inside the library.  Results are
 * identical to moe_dispatch.  This call allocates nothing and calls no
 * allocating routine.
 * The array belongs to the library's device code.  With CUDA's lazy module
 * loading (the default), that code, and with it the array's 1 MiB, may be
 * loaded onto a device only when the library first uses the device; from
 * then on the device holds it until the process exits.  A service that must
 * not commit device memory once it is serving should therefore make one
 * call (any T > 0) on each device at start-up.
 *
 * Limit: moe_dispatch_workspace_size(cfg) must be <= 1 MiB (E times the
 * number of 2048-pair chunks <= 262,140: any P for E <= 256; P <= 522,240
 * for E = 1024); larger sizes return MOE_ERR_UNSUPPORTED and launch nothing.
 * Set-up: the first call with T > 0 on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current, once, and keeps
 * it; make that first call before any stream capture.  The kept address is
 * not refreshed, so a device reset (cudaDeviceReset, or a teardown and
 * re-creation of the primary context) after the first call is not
 * supported.  All calls on a device share the array, so calls whose kernels
 * overlap on the GPU race: serialise them.
 * Other arguments, errors and outputs are as for moe_dispatch.
 */
moe_status_t moe_dispatch_noalloc(const moe_config_t *cfg, const int32_t *topk_idx,
                                  const float *topk_w, const void *x, int32_t *counts,
                                  int32_t *offsets, int32_t *pos, int32_t *src_token,
                                  void *x_perm, void *stream);

/*
 * Grouped SwiGLU experts [EP-add: experts_forward; TP-pack]: for every expert
 * e and every row r in [offsets[e], offsets[e+1]):
 *   gu        = x_perm[r] @ W_gate_up[e]        (W_gate_up: [E][d][2f])
 *   h_perm[r] = silu(gu[0:f]) * gu[f:2f],  silu(z) = z / (1 + exp(-z))
 *   y_perm[r] = h_perm[r] @ W_down[e]           (W_down: [E][f][d])
 * x_perm [P][d], h_perm [P][f] (written), y_perm [P][d] (written), all in the
 * act dtype; offsets [E+1] int32 as written by moe_dispatch (P = offsets[E]).
 * bf16: fp32 accumulation on the tensor cores, h_perm and y_perm rounded to
 * bf16.  The second product reads the bf16 h_perm.
 */
moe_status_t moe_grouped_swiglu(const moe_config_t *cfg, const void *x_perm,
                                const int32_t *offsets, const void *W_gate_up,
                                const void *W_down, void *h_perm, void *y_perm,
                                void *stream);

/*
 * Weighted combine [EP-add: the weighted expert output of each token;
 * EP-disp: combined with the routing weights]:
 *   out[t][:] = sum_{j=0}^{k-1} topk_w[t][j] * y_perm[pos[t*k+j]][:]
 * summed in slot order in fp32, then rounded to the act dtype.  With
 * cfg->scale_inputs the weights were applied at dispatch: the rows are summed
 * unweighted and topk_w is not read (may be NULL).
 * y_perm [P][d], pos [P] int32, topk_w [T][k] fp32, out [T][d] (written).
 */
moe_status_t moe_combine(const moe_config_t *cfg, const void *y_perm,
                         const int32_t *pos, const float *topk_w, void *out,
                         void *stream);

/*
 * The whole layer, one stream, no host synchronisation: moe_route,
 * moe_dispatch, moe_grouped_swiglu, moe_combine.
 * When k == E every expert receives every token, so there is nothing to
 * permute [EP]: expert e's segment is rows e*T .. e*T + T-1 in token order,
 * the dispatch only writes counts, offsets, pos and src_token, and the first
 * grouped GEMM reads the rows of x itself instead of x_perm (for fp32 with
 * the weights on the inputs, the scaled rows are copied instead).
 * Otherwise, for bf16 activations with d a multiple of 64 and f <= 3072, the
 * permuted copy of x is not formed either: the dispatch writes counts,
 * offsets, pos and src_token, and the first grouped GEMM gathers row r of
 * the segments from x[src_token[r]] itself (measured faster there than
 * writing and reading x_perm; with the weights on the outputs the results
 * are bit-identical to the copying path).
 * On both paths, weights on the inputs (scale_inputs != 0, bf16) are
 * applied by the first grouped GEMM: row r's gate and up products are
 * multiplied by its pair's weight in fp32 before the SwiGLU, (w x) W =
 * w (x W), where the copying path rounds w x to bf16 first.
 * x [T][d], Wr [E][d] fp32, logit_bias [E] fp32 or NULL,
 * W_gate_up [E][d][2f], W_down [E][f][d], out [T][d] (written).
 * ws: at least moe_workspace_size(cfg) bytes, 256-byte aligned; its
 * contents after the call are the intermediates (layout internal).
 */
moe_status_t moe_forward(const moe_config_t *cfg, const void *x, const float *Wr,
                         const float *logit_bias, const void *W_gate_up,
                         const void *W_down, void *out, void *ws, size_t ws_bytes,
                         void *stream);

/*
 * moe_forward with the activations in HOST memory: copies x_host -> x_dev,
 * runs the layer into out_dev, copies out_dev -> out_host, all enqueued on
 * `stream`.  x_host / out_host ([T][d], act dtype) should be pinned for the
 * copies to be asynchronous; the caller synchronises `stream` before reading
 * out_host.  x_dev / out_dev are caller device buffers of the same size.
 */
moe_status_t moe_forward_host(const moe_config_t *cfg, const void *x_host,
                              const float *Wr, const float *logit_bias,
                              const void *W_gate_up, const void *W_down,
                              void *out_host, void *x_dev, void *out_dev,
                              void *ws, size_t ws_bytes, void *stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_BAD_ROUTING, or
 * MOE_ERR_CUDA if the synchronisation itself failed.
 */
moe_status_t moe_last_device_error(void *stream);

/*
 * Limit, in nanoseconds, on every bounded device-side wait of later launches
 * from this process (default 2e9 = 2 s; 0 restores the default).  A wait
 * that runs out records MOE_ERR_DEVICE_TIMEOUT and the kernel returns.
 * Limits below 10 ms are raised to 10 ms (unless the test hook
 * moe_debug_inject_wait_timeout is on): a CTA pair that gave up within one
 * pipeline stage could otherwise leave a copy in flight that no barrier of
 * its pair expects.
 */
void moe_set_wait_limit_ns(uint64_t ns);

/* The wait limit later launches will use, after the 10 ms floor. */
uint64_t moe_wait_limit_ns(void);

/*
 * Test hook for the failure path (no counterpart on the pages).  While
 * enabled (non-zero), every later tensor-core grouped GEMM launch first waits
 * on a barrier that nothing signals, so that wait runs out after the wait
 * limit: the kernel records MOE_ERR_DEVICE_TIMEOUT, drains its in-flight
 * copies, frees its tensor memory and returns without computing.  The
 * outputs of such a call are undefined.  Off by default.
 */
void moe_debug_inject_wait_timeout(int enable);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
