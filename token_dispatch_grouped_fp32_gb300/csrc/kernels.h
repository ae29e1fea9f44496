// kernels.h -- host-side launchers of the libmoe kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

struct Shape {
    int64_t T;
    int d, E, k, f;
    bool bf16;    // activation dtype: bf16 (else fp32)
    bool renorm;  // renormalise the chosen k weights
    bool scale_inputs;  // routing weights scale expert inputs (dispatch), not outputs
    int64_t P() const { return T * (int64_t)k; }
};

// Router: logits[T][E] = x @ Wr^T (+ bias), fp32 accumulation.  When
// router_selects_in_logits(s) and idx/w are given, the same launch also
// writes the top-k selection and weights (no separate top-k launch).
// zero_word (optional, for the selecting launches here and below): a word
// the launch sets to 0, so a later kernel in the stream finds it cleared
// (the dispatch's ticket counter).
cudaError_t launch_router_logits(const Shape &s, const void *x, const float *Wr,
                                 const float *bias, float *logits, cudaStream_t st,
                                 int32_t *idx = nullptr, float *w = nullptr,
                                 unsigned *zero_word = nullptr);
bool router_selects_in_logits(const Shape &s);
// Top-k selection and softmax weights on a given fp32 logit buffer.
cudaError_t launch_topk(const Shape &s, const float *logits, int32_t *idx, float *w,
                        cudaStream_t st, unsigned *zero_word = nullptr);
// Top-k on logits formed as sum of `splits` partial buffers [splits][T][E]
// (added in split order) plus bias; the logits are written to `logits`.
cudaError_t launch_topk_partials(const Shape &s, const float *partial, int splits,
                                 const float *bias, float *logits, int32_t *idx, float *w,
                                 cudaStream_t st, unsigned *zero_word = nullptr);

// Router logits on the tensor cores (bf16 x, fp32 Wr split into 3 bf16 terms).
struct RouterTcPlan {
    int ctas;          // 2: CTA pairs on 256-token tiles; 1: single CTAs on 128-token tiles
    int ks_total;      // pipeline stages of a row tile: d / 64 (three W' tiles each) or 3d / 64
    int ks_per_split;  // stages per CTA
    int splits;        // K splits (blockIdx.y)
};
bool router_tc_eligible(const Shape &s);
RouterTcPlan router_tc_plan(const Shape &s);
size_t router_tc_scratch_bytes(const Shape &s);  // split weight + partial logits
cudaError_t launch_router_logits_tc(const Shape &s, const void *x, const float *Wr, void *scratch,
                                    float **partial_out, int *splits_out, const DevStatus &ds,
                                    cudaStream_t st);

// Dispatch: chunking of the P pairs over the rank kernel's blocks.
struct DispatchGrid {
    int chunk;  // pairs per block (a multiple of 256)
    int blocks;  // number of blocks (>= 1 when P > 0)
};
DispatchGrid dispatch_grid(int64_t P, int E);
// A dispatch that copies unscaled rows runs as one launch (no count matrix,
// no ticket) when E <= 16, P <= 16384 and a row is k KB to 16 KB.
bool dispatch_fits_one_launch(const Shape &s);
size_t dispatch_scratch_bytes(const Shape &s);  // count matrix [E][chunks] + ticket
// The ticket counter inside the dispatch scratch `hist` (must be 0 when the
// dispatch's first launch starts; the dispatch leaves it 0).
unsigned *dispatch_ticket(const Shape &s, int32_t *hist);
// x_perm == nullptr: counts, offsets, pos and src_token only (no row gather).
// scale != nullptr: each gathered row is multiplied by its pair's weight;
// without x_perm, row_scale[row] = scale[pair] instead (if row_scale).
// in_forward: the dispatch runs inside moe_forward, after the route, whose
// last launch cleared the ticket; its launches overlap the route's by
// programmatic dependent launch.  Otherwise (a standalone call) the ticket is
// cleared here with a 4-byte cudaMemsetAsync, after which the first launch
// starts only once all earlier work in the stream is done.
cudaError_t launch_dispatch(const Shape &s, const int32_t *idx, const void *x, int32_t *counts,
                            int32_t *offsets, int32_t *pos, int32_t *src_token, void *x_perm,
                            int32_t *hist, const DevStatus &ds, cudaStream_t st,
                            const float *scale = nullptr, bool in_forward = false,
                            float *row_scale = nullptr);

// Grouped SwiGLU experts.  bf16: tcgen05 tensor-core path; fp32: SIMT path.
// Kernel launches of one launch_grouped_swiglu_tc call (2, or 4 when the
// experts are split between CTA-pair and single-CTA tiles).
int grouped_swiglu_tc_launches(const Shape &s);
// Whether launch_grouped_swiglu_tc can gather G1's rows (src_token) for s,
// and whether doing so is measured faster than reading a permuted copy.
bool grouped_swiglu_tc_gathers(const Shape &s);
bool grouped_swiglu_tc_gather_pays(const Shape &s);
// a_local: x_perm is the T token rows x, and row r of expert e's segment
// reads row r - offsets[e] (every expert receives every token, in order).
// src_token (not null): x_perm is the T token rows x, and G1 gathers row r
// of the segments from row src_token[r] (d a multiple of 64, no a_local).
// row_scale (not null): G1 multiplies row r's gate and up accumulators by
// row_scale[r] (the routing weight on the expert's input, applied after the
// product instead of to the rows).
cudaError_t launch_grouped_swiglu_tc(const Shape &s, const void *x_perm, const int32_t *offsets,
                                     const void *Wgu, const void *Wd, void *h_perm, void *y_perm,
                                     const DevStatus &ds, cudaStream_t st, bool a_local = false,
                                     const int32_t *src_token = nullptr,
                                     const float *row_scale = nullptr);
cudaError_t launch_grouped_swiglu_f32(const Shape &s, const float *x_perm, const int32_t *offsets,
                                      const float *Wgu, const float *Wd, float *h_perm,
                                      float *y_perm, cudaStream_t st, bool a_local = false);

// Dispatch when every token picks every expert (k == E): counts[e] = T,
// offsets[e] = e*T, pos[t*E+j] = idx[t][j]*T + t, src_token[e*T + t] = t.
// No rows are copied (the experts read x with a_local).  One launch.
// w, row_scale (both or neither): row_scale[idx[t][j]*T + t] = w[t][j].
cudaError_t launch_dispatch_all_experts(const Shape &s, const int32_t *idx, int32_t *counts,
                                        int32_t *offsets, int32_t *pos, int32_t *src_token,
                                        const DevStatus &ds, cudaStream_t st,
                                        const float *w = nullptr, float *row_scale = nullptr);

// Weighted combine of the expert rows back into token order (w == nullptr:
// unweighted sum).
cudaError_t launch_combine(const Shape &s, const void *y_perm, const int32_t *pos, const float *w,
                           void *out, cudaStream_t st);

// Streaming multiprocessors of the current device (queried once per device).
// Without a usable device (sizing a workspace on a host with no GPU) it is
// 152, a GB300's count; a launch always plans with the real device's count,
// and a workspace sized for fewer SMs than the device has is then reported
// as too small (MOE_ERR_WORKSPACE), never overrun.
int device_sm_count();

// Last detailed message set by a launcher (thread-local; empty if none).
void set_error_message(const char *fmt, ...);
const char *error_message();

}  // namespace moe
