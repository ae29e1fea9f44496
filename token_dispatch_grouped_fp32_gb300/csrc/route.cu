// route.cu -- the router: fp32 logits, then top-k selection with softmax weights.
//
// Transformers docs "Expert parallelism", section "Adding an implementation":
// the router produces top_k_index and top_k_weights for the expert call.  The
// selection rule (larger logit first, equal logits to the lower expert id, a
// NaN below every number), softmax over all E logits and renormalisation over
// the chosen k are the router's definition.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// Router logits: C[T][E] = A[T][d] * B[E][d]^T (+ bias[E]), fp32 FFMA.
// Block tile BM x BN, K step BK; each thread owns TM x TN outputs spread with
// stride (BM/TM) rows and (BN/TN) columns so shared-memory reads are
// conflict-free.  Operand tiles are stored k-major with one word of padding.
// ---------------------------------------------------------------------------
constexpr int kLogitBK = 32;

template <typename TA, int BM, int BN, int TM, int TN>
__global__ void __launch_bounds__(256)
router_logits_kernel(const TA *__restrict__ x, const float *__restrict__ Wr,
                     const float *__restrict__ bias, float *__restrict__ logits, int64_t T, int d,
                     int E) {
    static_assert((BM / TM) * (BN / TN) == 256, "256 threads");
    constexpr int BK = kLogitBK;
    constexpr int RG = BM / TM;  // row groups
    constexpr int CG = BN / TN;  // column groups
    __shared__ float As[BK][BM + 1];
    __shared__ float Bs[BK][BN + 1];

    const int tid = threadIdx.x;
    const int tx = tid % CG, ty = tid / CG;
    const int64_t m0 = (int64_t)blockIdx.x * BM;
    const int n0 = blockIdx.y * BN;

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < d; k0 += BK) {
        for (int i = tid; i < BM * BK; i += 256) {
            int r = i / BK, c = i % BK;
            int64_t gm = m0 + r;
            int gk = k0 + c;
            float v = 0.f;
            if (gm < T && gk < d) v = Act<TA>::to_f(x[gm * d + gk]);
            As[c][r] = v;
        }
        for (int i = tid; i < BN * BK; i += 256) {
            int r = i / BK, c = i % BK;
            int gn = n0 + r, gk = k0 + c;
            float v = 0.f;
            if (gn < E && gk < d) v = Wr[(int64_t)gn * d + gk];
            Bs[c][r] = v;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = As[kk][ty + i * RG];
#pragma unroll
            for (int j = 0; j < TN; ++j) b[j] = Bs[kk][tx + j * CG];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        int64_t gm = m0 + ty + i * RG;
        if (gm >= T) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            int gn = n0 + tx + j * CG;
            if (gn < E) logits[gm * E + gn] = acc[i][j] + (bias ? bias[gn] : 0.f);
        }
    }
}

template <typename TA, int BM, int BN, int TM, int TN>
cudaError_t launch_logits_cfg(const Shape &s, const TA *x, const float *Wr, const float *bias,
                              float *logits, cudaStream_t st) {
    dim3 grid((unsigned)((s.T + BM - 1) / BM), (unsigned)((s.E + BN - 1) / BN));
    router_logits_kernel<TA, BM, BN, TM, TN><<<grid, 256, 0, st>>>(x, Wr, bias, logits, s.T, s.d, s.E);
    return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_logits_t(const Shape &s, const TA *x, const float *Wr, const float *bias,
                            float *logits, cudaStream_t st) {
    if (s.E <= 8) return launch_logits_cfg<TA, 64, 8, 2, 1>(s, x, Wr, bias, logits, st);
    if (s.E <= 16) return launch_logits_cfg<TA, 64, 16, 4, 1>(s, x, Wr, bias, logits, st);
    if (s.E <= 32) return launch_logits_cfg<TA, 64, 32, 4, 2>(s, x, Wr, bias, logits, st);
    if (s.E <= 64) return launch_logits_cfg<TA, 64, 64, 4, 4>(s, x, Wr, bias, logits, st);
    return launch_logits_cfg<TA, 64, 128, 4, 8>(s, x, Wr, bias, logits, st);
}

// ---------------------------------------------------------------------------
// Top-k: one warp per token.  Lane l holds logits l, l+32, ...; k rounds of a
// warp arg-max under the rank order pick the experts; slot j is written by
// lane j.  Weights: softmax over all E logits (max-shifted), then optional
// renormalisation over the chosen k.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib) {
    const bool an = isnan(a), bn = isnan(b);
    if (an || bn) return (an && bn) ? (ia < ib) : bn;
    if (a > b) return true;
    if (a < b) return false;
    return ia < ib;
}

constexpr int kNoExpert = 0x7fffffff;

template <int VPL>
__global__ void __launch_bounds__(256)
topk_kernel(const float *__restrict__ logits, int64_t T, int E, int k, int renorm,
            int32_t *__restrict__ idx, float *__restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;  // warp-uniform
    const float *L = logits + t * E;

    float v[VPL];
    unsigned avail = 0;  // bit i: value i of this lane is a not-yet-chosen expert
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        int e = lane + 32 * i;
        v[i] = (e < E) ? L[e] : -INFINITY;
        if (e < E) avail |= 1u << i;
    }

    float my_v = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        float bv = NAN;
        int be = kNoExpert;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (!((avail >> i) & 1u)) continue;
            int e = lane + 32 * i;
            if (be == kNoExpert || ranks_before(v[i], e, bv, be)) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (oe != kNoExpert && (be == kNoExpert || ranks_before(ov, oe, bv, be))) {
                bv = ov;
                be = oe;
            }
        }
        if (be != kNoExpert && (be & 31) == lane) avail &= ~(1u << (be >> 5));
        if (lane == j) {
            my_v = bv;
            my_e = be;
        }
    }

    // softmax over all E logits
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) m = fmaxf(m, v[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) z += expf(v[i] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);

    float p = (lane < k) ? expf(my_v - m) / z : 0.f;
    if (renorm) {
        float s = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        p = p / s;
    }
    if (lane < k) {
        idx[t * k + lane] = my_e;
        w[t * k + lane] = p;
    }
}

template <int VPL>
cudaError_t launch_topk_v(const Shape &s, const float *logits, int32_t *idx, float *w,
                          cudaStream_t st) {
    unsigned blocks = (unsigned)((s.T + 7) / 8);
    topk_kernel<VPL><<<blocks, 256, 0, st>>>(logits, s.T, s.E, s.k, s.renorm ? 1 : 0, idx, w);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits(const Shape &s, const void *x, const float *Wr, const float *bias,
                                 float *logits, cudaStream_t st) {
    if (s.bf16)
        return launch_logits_t<__nv_bfloat16>(s, static_cast<const __nv_bfloat16 *>(x), Wr, bias,
                                              logits, st);
    return launch_logits_t<float>(s, static_cast<const float *>(x), Wr, bias, logits, st);
}

cudaError_t launch_topk(const Shape &s, const float *logits, int32_t *idx, float *w,
                        cudaStream_t st) {
    if (s.E <= 32) return launch_topk_v<1>(s, logits, idx, w, st);
    if (s.E <= 64) return launch_topk_v<2>(s, logits, idx, w, st);
    if (s.E <= 128) return launch_topk_v<4>(s, logits, idx, w, st);
    if (s.E <= 256) return launch_topk_v<8>(s, logits, idx, w, st);
    if (s.E <= 512) return launch_topk_v<16>(s, logits, idx, w, st);
    return launch_topk_v<32>(s, logits, idx, w, st);
}

}  // namespace moe
