// moe_api.cu -- the C ABI of libmoe (declared in include/moe.h): argument
// checks, workspace layout, and the launch sequence of the layer forward.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {

static thread_local char g_msg[512];

void set_error_message(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
}
const char *error_message() { return g_msg; }

// Per-device error word written by kernels (see moe_last_device_error).
__device__ unsigned g_device_error_word;

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s
// Floor of the wait limit outside the failure-path test hook: well above the
// time of one pipeline stage, so an abort never leaves a CTA pair with a copy
// that one CTA issued and the other never armed.
constexpr unsigned long long kMinWaitLimitNs = 10000000ull;  // 10 ms
static std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
static std::atomic<int> g_inject_wait_timeout{0};

unsigned long long effective_wait_limit_ns() {
    const unsigned long long ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    if (g_inject_wait_timeout.load(std::memory_order_relaxed)) return ns;
    return ns < kMinWaitLimitNs ? kMinWaitLimitNs : ns;
}

int device_sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();  // no usable device: clear the error so later calls do not see it
        return 152;
    }
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0) {
            cudaGetLastError();
            return 152;
        }
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

namespace {

constexpr int kMaxDevices = 64;

struct DevState {
    bool checked = false;
    bool supported = false;
    unsigned *err_word = nullptr;
};
DevState g_dev[kMaxDevices];

// First use on a device: check the architecture and fetch the error word's
// device address.  Both are cached; later calls launch without queries.
moe_status_t device_status(DevStatus *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error_message("cudaGetDevice: %s", cudaGetErrorString(e));
        return MOE_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_error_message("device ordinal %d out of range", dev);
        return MOE_ERR_UNSUPPORTED;
    }
    DevState &s = g_dev[dev];
    if (!s.checked) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        s.supported = (major == 10 && minor == 3);
        if (s.supported) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_device_error_word);
            if (e != cudaSuccess) {
                set_error_message("cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
                return MOE_ERR_CUDA;
            }
            s.err_word = static_cast<unsigned *>(p);
        } else {
            set_error_message("device %d is sm_%d%d; libmoe is built for sm_103a only", dev, major,
                              minor);
        }
        s.checked = true;
    }
    if (!s.supported) return MOE_ERR_UNSUPPORTED;
    out->err = s.err_word;
    out->wait_limit_ns = effective_wait_limit_ns();
    out->inject_wait_timeout = g_inject_wait_timeout.load(std::memory_order_relaxed);
    return MOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_cfg(const moe_config_t *cfg, Shape *s) {
    if (!cfg) {
        set_error_message("cfg is NULL");
        return MOE_ERR_INVALID_ARG;
    }
    if (cfg->T < 0 || cfg->d <= 0 || cfg->f <= 0 || cfg->E <= 0 || cfg->k < 1 || cfg->k > cfg->E) {
        set_error_message("bad sizes: T=%lld d=%d E=%d k=%d f=%d", (long long)cfg->T, cfg->d,
                          cfg->E, cfg->k, cfg->f);
        return MOE_ERR_INVALID_ARG;
    }
    if (cfg->act_dtype != MOE_F32 && cfg->act_dtype != MOE_BF16) {
        set_error_message("unknown act_dtype %d", cfg->act_dtype);
        return MOE_ERR_UNSUPPORTED;
    }
    if (cfg->d % 8 != 0 || cfg->f % 8 != 0) {
        set_error_message("d (%d) and f (%d) must be multiples of 8", cfg->d, cfg->f);
        return MOE_ERR_INVALID_ARG;
    }
    if (cfg->E > 1024 || cfg->k > 32) {
        set_error_message("unsupported E=%d k=%d (E <= 1024, k <= 32)", cfg->E, cfg->k);
        return MOE_ERR_UNSUPPORTED;
    }
    if (cfg->T * (int64_t)cfg->k >= ((int64_t)1 << 31)) {
        set_error_message("T*k = %lld must be < 2^31", (long long)(cfg->T * cfg->k));
        return MOE_ERR_INVALID_ARG;
    }
    s->T = cfg->T;
    s->d = cfg->d;
    s->E = cfg->E;
    s->k = cfg->k;
    s->f = cfg->f;
    s->bf16 = cfg->act_dtype == MOE_BF16;
    s->renorm = cfg->renormalize != 0;
    s->scale_inputs = cfg->scale_inputs != 0;
    return MOE_OK;
}

moe_status_t check_ptrs(std::initializer_list<const void *> ptrs) {
    int i = 0;
    for (const void *p : ptrs) {
        if (!p) {
            set_error_message("pointer argument %d is NULL", i);
            return MOE_ERR_INVALID_ARG;
        }
        if (!aligned16(p)) {
            set_error_message("pointer argument %d is not 16-byte aligned", i);
            return MOE_ERR_INVALID_ARG;
        }
        ++i;
    }
    return MOE_OK;
}

moe_status_t from_cuda(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return MOE_OK;
    if (error_message()[0] == 0)  // keep a launcher's more specific message
        set_error_message("%s: %s", what, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

// k == E: every expert receives every token, so moe_forward skips the
// permutation of x (see launch_dispatch_all_experts) and the experts read x
// directly.  With the weights on the inputs this needs the first GEMM to
// apply them (bf16: rows_scaled_in_gemm); the fp32 path copies scaled rows.
bool all_experts_path(const Shape &s) { return s.k == s.E && (!s.scale_inputs || s.bf16); }

// bf16 where the grouped GEMM's row gather pays
// (grouped_swiglu_tc_gather_pays): the dispatch only ranks and places the
// pairs, and the first expert GEMM gathers its rows from x through
// src_token.
bool gather_path(const Shape &s) {
    return s.bf16 && !all_experts_path(s) && grouped_swiglu_tc_gather_pays(s);
}

// Weights on the inputs with no permuted copy of x (the two paths above):
// the dispatch records each row's weight (row_scale) and the first GEMM
// multiplies the row's gate and up accumulators by it, (w x) W = w (x W).
bool rows_scaled_in_gemm(const Shape &s) {
    return s.bf16 && s.scale_inputs && (all_experts_path(s) || gather_path(s));
}

// moe_forward writes and reads x_perm unless its experts read x itself.
bool forward_uses_x_perm(const Shape &s) { return !all_experts_path(s) && !gather_path(s); }

// ----- workspace layout of moe_forward (256-byte aligned sub-buffers) -----
struct WsLayout {
    size_t logits, idx, w, counts, offsets, pos, src, hist, route, row_scale, x_perm, h_perm,
        y_perm, total;
};

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout ws_layout(const Shape &s) {
    WsLayout L;
    const size_t P = (size_t)s.P(), T = (size_t)s.T, es = s.bf16 ? 2 : 4;
    size_t o = 0;
    L.logits = o; o = up256(o + 4 * T * s.E);
    L.idx = o;    o = up256(o + 4 * P);
    L.w = o;      o = up256(o + 4 * P);
    L.counts = o; o = up256(o + 4 * (size_t)s.E);
    L.offsets = o; o = up256(o + 4 * ((size_t)s.E + 1));
    L.pos = o;    o = up256(o + 4 * P);
    L.src = o;    o = up256(o + 4 * P);
    L.hist = o;   o = up256(o + dispatch_scratch_bytes(s));
    L.route = o;  o = up256(o + router_tc_scratch_bytes(s));
    L.row_scale = o;
    if (rows_scaled_in_gemm(s)) o = up256(o + 4 * P);
    if (forward_uses_x_perm(s)) {
        L.x_perm = o;
        o = up256(o + es * P * s.d);
    } else {
        L.x_perm = MOE_WS_ABSENT;
    }
    L.h_perm = o; o = up256(o + es * P * s.f);
    L.y_perm = o; o = up256(o + es * P * s.d);
    L.total = o;
    return L;
}

template <typename T> T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

// Router: tensor-core logits (split weight, K-split partials summed by the
// top-k kernel) when the shape allows, else the SIMT logits kernel.
// zero_word (optional): cleared by the route's last launch (the dispatch's
// ticket, when moe_forward runs the dispatch next).
moe_status_t run_route(const Shape &s, const void *x, const float *Wr, const float *bias,
                       float *logits, int32_t *idx, float *w, void *route_ws,
                       const DevStatus &ds, cudaStream_t st, unsigned *zero_word = nullptr) {
    if (router_tc_eligible(s)) {
        float *partial = nullptr;
        int splits = 0;
        moe_status_t r = from_cuda(
            launch_router_logits_tc(s, x, Wr, route_ws, &partial, &splits, ds, st),
            "router logits launch");
        if (r != MOE_OK) return r;
        return from_cuda(
            launch_topk_partials(s, partial, splits, bias, logits, idx, w, st, zero_word),
            "top-k launch");
    }
    if (router_selects_in_logits(s))  // one launch: logits, selection and weights
        return from_cuda(launch_router_logits(s, x, Wr, bias, logits, st, idx, w, zero_word),
                         "router launch");
    moe_status_t r = from_cuda(launch_router_logits(s, x, Wr, bias, logits, st),
                               "router logits launch");
    if (r != MOE_OK) return r;
    return from_cuda(launch_topk(s, logits, idx, w, st, zero_word), "top-k launch");
}

// a_local: x_perm is x itself, every segment the T tokens in order (k == E).
// src_token (bf16 only): x_perm is x itself and G1 gathers its rows.
// row_scale (bf16 only): G1 scales row r's products by row_scale[r].
moe_status_t run_experts(const Shape &s, const void *x_perm, const int32_t *offsets,
                         const void *Wgu, const void *Wd, void *h_perm, void *y_perm,
                         const DevStatus &ds, cudaStream_t st, bool a_local = false,
                         const int32_t *src_token = nullptr, const float *row_scale = nullptr) {
    cudaError_t e;
    if (s.bf16)
        e = launch_grouped_swiglu_tc(s, x_perm, offsets, Wgu, Wd, h_perm, y_perm, ds, st, a_local,
                                     src_token, row_scale);
    else
        e = launch_grouped_swiglu_f32(s, static_cast<const float *>(x_perm), offsets,
                                      static_cast<const float *>(Wgu),
                                      static_cast<const float *>(Wd), static_cast<float *>(h_perm),
                                      static_cast<float *>(y_perm), st, a_local);
    return from_cuda(e, "grouped SwiGLU launch");
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(moe_status_t status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
        case MOE_ERR_BAD_ROUTING: return "MOE_ERR_BAD_ROUTING";
    }
    return "MOE_ERR_UNKNOWN";
}

const char *moe_last_error_message(void) { return error_message(); }

size_t moe_workspace_size(const moe_config_t *cfg) {
    Shape s;
    if (check_cfg(cfg, &s) != MOE_OK || s.T == 0) return 0;
    return ws_layout(s).total;
}

moe_status_t moe_workspace_layout(const moe_config_t *cfg, moe_workspace_layout_t *layout) {
    g_msg[0] = 0;
    Shape s;
    moe_status_t st = check_cfg(cfg, &s);
    if (st != MOE_OK) return st;
    if (!layout) {
        set_error_message("layout is NULL");
        return MOE_ERR_INVALID_ARG;
    }
    memset(layout, 0, sizeof(*layout));
    if (s.T == 0) return MOE_OK;
    const WsLayout L = ws_layout(s);
    layout->logits = L.logits;
    layout->topk_idx = L.idx;
    layout->topk_w = L.w;
    layout->counts = L.counts;
    layout->offsets = L.offsets;
    layout->pos = L.pos;
    layout->src_token = L.src;
    layout->x_perm = L.x_perm;
    layout->h_perm = L.h_perm;
    layout->y_perm = L.y_perm;
    layout->total = L.total;
    return MOE_OK;
}

size_t moe_route_workspace_size(const moe_config_t *cfg) {
    Shape s;
    if (check_cfg(cfg, &s) != MOE_OK || s.T == 0) return 0;
    return router_tc_scratch_bytes(s);
}

size_t moe_dispatch_workspace_size(const moe_config_t *cfg) {
    Shape s;
    if (check_cfg(cfg, &s) != MOE_OK || s.T == 0) return 0;
    return dispatch_scratch_bytes(s);
}

int moe_forward_kernel_launches(const moe_config_t *cfg) {
    Shape s;
    if (check_cfg(cfg, &s) != MOE_OK) return -1;
    if (s.T == 0) return 0;
    // the same choices as run_route: tensor cores (weight split, logits, top-k),
    // CUDA cores selecting in the logits launch, or CUDA-core logits + top-k
    const int route = router_tc_eligible(s) ? 3 : router_selects_in_logits(s) ? 1 : 2;
    const int experts = s.bf16 ? grouped_swiglu_tc_launches(s) : 2 /* G1, G2 */;
    // rank (with the count scan) and place rows, or one launch for few experts and pairs
    const int dispatch = all_experts_path(s) ||
                                 (forward_uses_x_perm(s) && !s.scale_inputs &&
                                  dispatch_fits_one_launch(s))
                             ? 1
                             : 2;
    return route + dispatch + experts + 1 /* combine */;
}

void moe_set_wait_limit_ns(uint64_t ns) {
    g_wait_limit_ns.store(ns ? ns : kDefaultWaitLimitNs, std::memory_order_relaxed);
}

uint64_t moe_wait_limit_ns(void) { return effective_wait_limit_ns(); }

void moe_debug_inject_wait_timeout(int enable) {
    g_inject_wait_timeout.store(enable ? 1 : 0, std::memory_order_relaxed);
}

moe_status_t moe_route(const moe_config_t *cfg, const void *x, const float *Wr,
                       const float *logit_bias, float *logits, int32_t *topk_idx, float *topk_w,
                       void *ws, size_t ws_bytes, void *stream) {
    g_msg[0] = 0;
    Shape s;
    moe_status_t st = check_cfg(cfg, &s);
    if (st != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;  // empty batch: nothing to check or launch
    if ((st = check_ptrs({x, Wr, logits, topk_idx, topk_w})) != MOE_OK) return st;
    if (logit_bias && !aligned16(logit_bias)) {
        set_error_message("logit_bias is not 16-byte aligned");
        return MOE_ERR_INVALID_ARG;
    }
    const size_t need = router_tc_scratch_bytes(s);
    if (need > 0) {
        if ((st = check_ptrs({ws})) != MOE_OK) return st;
        if (ws_bytes < need) {
            set_error_message("workspace %zu bytes < %zu needed", ws_bytes, need);
            return MOE_ERR_WORKSPACE;
        }
    }
    DevStatus ds;
    if ((st = device_status(&ds)) != MOE_OK) return st;
    return run_route(s, x, Wr, logit_bias, logits, topk_idx, topk_w, ws, ds,
                     static_cast<cudaStream_t>(stream));
}

moe_status_t moe_route_from_logits(const moe_config_t *cfg, const float *logits, int32_t *topk_idx,
                                   float *topk_w, void *stream) {
    g_msg[0] = 0;
    Shape s;
    moe_status_t st = check_cfg(cfg, &s);
    if (st != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;  // empty batch: nothing to check or launch
    if ((st = check_ptrs({logits, topk_idx, topk_w})) != MOE_OK) return st;
    DevStatus ds;
    if ((st = device_status(&ds)) != MOE_OK) return st;
    return from_cuda(launch_topk(s, logits, topk_idx, topk_w, static_cast<cudaStream_t>(stream)),
                     "top-k launch");
}

moe_status_t moe_dispatch(const moe_config_t *cfg, const int32_t *topk_idx, const float *topk_w,
                          const void *x, int32_t *counts, int32_t *offsets, int32_t *pos,
                          int32_t *src_token, void *x_perm, void *ws, size_t ws_bytes,
                          void *stream) {
    g_msg[0] = 0;
    Shape s;
    moe_status_t st = check_cfg(cfg, &s);
    if (st != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;  // empty batch: nothing to check or launch
    if ((st = check_ptrs({topk_idx, x, counts, offsets, pos, src_token, x_perm, ws})) != MOE_OK)
        return st;
    if (s.scale_inputs && (st = check_ptrs({topk_w})) != MOE_OK) return st;
    if (ws_bytes < dispatch_scratch_bytes(s)) {
        set_error_message("workspace %zu bytes < %zu needed", ws_bytes, dispatch_scratch_bytes(s));
        return MOE_ERR_WORKSPACE;
    }
    DevStatus ds;
    if ((st = device_status(&ds)) != MOE_OK) return st;
    return from_cuda(launch_dispatch(s, topk_idx, x, counts, offsets, pos, src_token, x_perm,
                                     static_cast<int32_t *>(ws), ds,
                                     static_cast<cudaStream_t>(stream),
                                     s.scale_inputs ? topk_w : nullptr),
                     "dispatch launch");
}

moe_status_t moe_grouped_swiglu(const moe_config_t *cfg, const void *x_perm,
                                const int32_t *offsets, const void *W_gate_up, const void *W_down,
                                void *h_perm, void *y_perm, void *stream) {
    g_msg[0] = 0;
    Shape s;
    moe_status_t st = check_cfg(cfg, &s);
    if (st != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;  // empty batch: nothing to check or launch
    if ((st = check_ptrs({x_perm, offsets, W_gate_up, W_down, h_perm, y_perm})) != MOE_OK)
        return st;
    DevStatus ds;
    if ((st = device_status(&ds)) != MOE_OK) return st;
    return run_experts(s, x_perm, offsets, W_gate_up, W_down, h_perm, y_perm, ds,
                       static_cast<cudaStream_t>(stream));
}

moe_status_t moe_combine(const moe_config_t *cfg, const void *y_perm, const int32_t *pos,
                         const float *topk_w, void *out, void *stream) {
    g_msg[0] = 0;
    Shape s;
    moe_status_t st = check_cfg(cfg, &s);
    if (st != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;  // empty batch: nothing to check or launch
    if ((st = check_ptrs({y_perm, pos, out})) != MOE_OK) return st;
    if (!s.scale_inputs && (st = check_ptrs({topk_w})) != MOE_OK) return st;
    DevStatus ds;
    if ((st = device_status(&ds)) != MOE_OK) return st;
    return from_cuda(launch_combine(s, y_perm, pos, s.scale_inputs ? nullptr : topk_w, out,
                                    static_cast<cudaStream_t>(stream)),
                     "combine launch");
}

moe_status_t moe_forward(const moe_config_t *cfg, const void *x, const float *Wr,
                         const float *logit_bias, const void *W_gate_up, const void *W_down,
                         void *out, void *ws, size_t ws_bytes, void *stream) {
    g_msg[0] = 0;
    Shape s;
    moe_status_t st = check_cfg(cfg, &s);
    if (st != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;  // empty batch: nothing to check or launch
    if ((st = check_ptrs({x, Wr, W_gate_up, W_down, out, ws})) != MOE_OK) return st;
    if (logit_bias && !aligned16(logit_bias)) {
        set_error_message("logit_bias is not 16-byte aligned");
        return MOE_ERR_INVALID_ARG;
    }
    const WsLayout L = ws_layout(s);
    if (ws_bytes < L.total) {
        set_error_message("workspace %zu bytes < %zu needed", ws_bytes, L.total);
        return MOE_ERR_WORKSPACE;
    }
    DevStatus ds;
    if ((st = device_status(&ds)) != MOE_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    float *logits = at<float>(ws, L.logits);
    int32_t *idx = at<int32_t>(ws, L.idx);
    float *w = at<float>(ws, L.w);
    int32_t *counts = at<int32_t>(ws, L.counts), *offsets = at<int32_t>(ws, L.offsets);
    int32_t *pos = at<int32_t>(ws, L.pos), *src = at<int32_t>(ws, L.src);
    void *x_perm = L.x_perm == MOE_WS_ABSENT ? nullptr : at<uint8_t>(ws, L.x_perm);
    void *h_perm = at<uint8_t>(ws, L.h_perm), *y_perm = at<uint8_t>(ws, L.y_perm);

    int32_t *hist = at<int32_t>(ws, L.hist);
    const bool all_experts = all_experts_path(s);
    const bool gather = gather_path(s);
    float *row_scale = rows_scaled_in_gemm(s) ? at<float>(ws, L.row_scale) : nullptr;
    // the route's last launch clears the dispatch's ticket counter
    if ((st = run_route(s, x, Wr, logit_bias, logits, idx, w, at<uint8_t>(ws, L.route), ds, cs,
                        all_experts ? nullptr : dispatch_ticket(s, hist))) != MOE_OK)
        return st;
    if (all_experts)
        st = from_cuda(launch_dispatch_all_experts(s, idx, counts, offsets, pos, src, ds, cs,
                                                   row_scale ? w : nullptr, row_scale),
                       "dispatch launch");
    else
        st = from_cuda(launch_dispatch(s, idx, x, counts, offsets, pos, src,
                                       gather ? nullptr : x_perm, hist, ds, cs,
                                       s.scale_inputs ? w : nullptr, /*in_forward=*/true,
                                       row_scale),
                       "dispatch launch");
    if (st != MOE_OK) return st;
    if ((st = run_experts(s, all_experts || gather ? x : x_perm, offsets, W_gate_up, W_down, h_perm,
                          y_perm, ds, cs, all_experts, gather ? src : nullptr, row_scale)) != MOE_OK)
        return st;
    return from_cuda(launch_combine(s, y_perm, pos, s.scale_inputs ? nullptr : w, out, cs),
                     "combine launch");
}

moe_status_t moe_forward_host(const moe_config_t *cfg, const void *x_host, const float *Wr,
                              const float *logit_bias, const void *W_gate_up, const void *W_down,
                              void *out_host, void *x_dev, void *out_dev, void *ws,
                              size_t ws_bytes, void *stream) {
    g_msg[0] = 0;
    Shape s;
    moe_status_t st = check_cfg(cfg, &s);
    if (st != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;  // empty batch: nothing to check or launch
    if ((st = check_ptrs({x_host, out_host, x_dev, out_dev})) != MOE_OK) return st;
    const size_t bytes = (size_t)s.T * s.d * (s.bf16 ? 2 : 4);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if ((st = from_cuda(cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, cs),
                        "host-to-device copy of x")) != MOE_OK)
        return st;
    if ((st = moe_forward(cfg, x_dev, Wr, logit_bias, W_gate_up, W_down, out_dev, ws, ws_bytes,
                          stream)) != MOE_OK)
        return st;
    return from_cuda(cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, cs),
                     "device-to-host copy of out");
}

moe_status_t moe_last_device_error(void *stream) {
    g_msg[0] = 0;
    DevStatus ds;
    moe_status_t st = device_status(&ds);
    if (st != MOE_OK) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e, "cudaStreamSynchronize");
    unsigned word = 0;
    if ((e = cudaMemcpy(&word, ds.err, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return from_cuda(e, "reading the device error word");
    const unsigned zero = 0;
    if ((e = cudaMemcpy(ds.err, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
        return from_cuda(e, "clearing the device error word");
    if (word & kErrTimeout) {
        set_error_message("a kernel's bounded wait ran out (device error word 0x%x)", word);
        return MOE_ERR_DEVICE_TIMEOUT;
    }
    if (word & kErrBadRouting) {
        set_error_message("an expert id outside [0, E) reached the dispatch (device error word 0x%x)",
                          word);
        return MOE_ERR_BAD_ROUTING;
    }
    return MOE_OK;
}

}  // extern "C"
