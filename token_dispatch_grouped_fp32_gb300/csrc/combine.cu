// combine.cu -- weighted combine of the expert rows back into token order.
//
// Transformers docs "Expert parallelism", sections "Adding an implementation"
// (the expert call returns each token's weighted expert output) and "Token
// dispatch" (results are combined with the routing weights):
//   out[t] = sum_{j<k} w[t][j] * y_perm[pos[t*k+j]], in slot order, fp32.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxK = 32;

// One warp per token; each lane handles 16-byte column vectors of the row.
template <typename TA>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const TA *__restrict__ y_perm, const int32_t *__restrict__ pos,
               const float *__restrict__ w, int64_t T, int k, int d, TA *__restrict__ out) {
    pdl_entry();
    constexpr int EPV = 16 / sizeof(TA);
    __shared__ int s_pos[kWarps][kMaxK];
    __shared__ float s_w[kWarps][kMaxK];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * kWarps + wid;
    if (t >= T) return;  // warp-uniform
    if (lane < k) {
        s_pos[wid][lane] = pos[t * k + lane];
        s_w[wid][lane] = w ? w[t * k + lane] : 1.f;  // no weights: plain sum
    }
    __syncwarp();
    const int nvec = d / EPV;
    constexpr int U = 4;  // 16-byte vectors per lane in flight per slot
    for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
        float acc[U][EPV];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < EPV; ++i) acc[u][i] = 0.f;
        for (int j = 0; j < k; ++j) {
            const int row = s_pos[wid][j];
            if (row < 0) continue;  // dropped pair
            const float wj = s_w[wid][j];
            const TA *yrow = y_perm + (int64_t)row * d;
            uint4 raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (v0 + 32 * u < nvec) raw[u] = ldg16(yrow + (int64_t)(v0 + 32 * u) * EPV);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (v0 + 32 * u >= nvec) continue;
                float y[EPV];
                unpack16(raw[u], y, static_cast<const TA *>(nullptr));
#pragma unroll
                for (int i = 0; i < EPV; ++i) acc[u][i] = fmaf(wj, y[i], acc[u][i]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v0 + 32 * u < nvec)
                stg16(out + t * d + (int64_t)(v0 + 32 * u) * EPV,
                      pack16(acc[u], static_cast<const TA *>(nullptr)));
    }
}

}  // namespace

cudaError_t launch_combine(const Shape &s, const void *y_perm, const int32_t *pos, const float *w,
                           void *out, cudaStream_t st) {
    const unsigned blocks = (unsigned)((s.T + kWarps - 1) / kWarps);
    if (s.bf16)
        launch_pdl(combine_kernel<__nv_bfloat16>, dim3(blocks), dim3(kThreads), 0, st,
            static_cast<const __nv_bfloat16 *>(y_perm), pos, w, s.T, s.k, s.d,
            static_cast<__nv_bfloat16 *>(out));
    else
        launch_pdl(combine_kernel<float>, dim3(blocks), dim3(kThreads), 0, st, static_cast<const float *>(y_perm), pos,
                                                          w, s.T, s.k, s.d,
                                                          static_cast<float *>(out));
    return cudaGetLastError();
}

}  // namespace moe
