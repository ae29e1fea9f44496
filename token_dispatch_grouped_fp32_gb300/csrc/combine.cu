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

// One warp per (token, column slice): a slice is a chunk of 32*U consecutive
// 16-byte vectors of the row, lane l holding vectors l, l+32, ...
// l+32*(U-1).  For each chunk the warp loads SG slots' rows at once (SG*U
// vectors per lane in flight; larger k in groups of SG slots), then adds
// them in slot order in fp32; the sum is rounded once.  Small batches
// (decode) thus spread a row over many warps instead of one.

// The chunk of token t whose lane-l vectors are v0, v0+32, ... v0+32*(U-1):
// SG slots' loads at a time, added in slot order in fp32, rounded once.
template <typename TA, int U, int SG>
__device__ __forceinline__ void combine_chunk(const TA *__restrict__ y_perm, int64_t t, int k,
                                              int d, int nvec, int v0, int my_pos, float my_w,
                                              TA *__restrict__ out) {
    constexpr int EPV = 16 / sizeof(TA);
    float acc[U][EPV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < EPV; ++i) acc[u][i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += SG) {
        uint4 raw[SG][U];
        int rows[SG];
#pragma unroll
        for (int g = 0; g < SG; ++g) {
            const int j = j0 + g;
            rows[g] = __shfl_sync(0xffffffffu, my_pos, j & 31);
            if (j >= k || rows[g] < 0) continue;  // past k, or a dropped pair
            const TA *yrow = y_perm + (int64_t)rows[g] * d;
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (v0 + 32 * u < nvec) raw[g][u] = ldg16(yrow + (int64_t)(v0 + 32 * u) * EPV);
        }
#pragma unroll
        for (int g = 0; g < SG; ++g) {
            const int j = j0 + g;
            const float wj = __shfl_sync(0xffffffffu, my_w, j & 31);
            if (j >= k || rows[g] < 0) continue;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (v0 + 32 * u >= nvec) continue;
                float y[EPV];
                unpack16(raw[g][u], y, static_cast<const TA *>(nullptr));
#pragma unroll
                for (int i = 0; i < EPV; ++i) acc[u][i] = fmaf(wj, y[i], acc[u][i]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (v0 + 32 * u < nvec)
            stg16(out + t * d + (int64_t)(v0 + 32 * u) * EPV,
                  pack16(acc[u], static_cast<const TA *>(nullptr)));
}

// One warp per (token, column slice): with WHOLE (slices == 1) the warp walks
// every 32*U-vector chunk of the row, else it does chunk `slice` only.
// Register budgets: WHOLE keeps four blocks per SM (a warp per token: a
// Mixtral-sized batch of 4096 tokens then runs in one wave), the 128-vector
// slices three.
template <typename TA, int U, int SG, bool WHOLE>
__global__ void __launch_bounds__(kThreads, WHOLE ? 4 : (U == 4 ? 3 : 2))
combine_kernel(const TA *__restrict__ y_perm, const int32_t *__restrict__ pos,
               const float *__restrict__ w, int64_t T, int k, int d, int slices,
               TA *__restrict__ out) {
    pdl_entry();
    constexpr int EPV = 16 / sizeof(TA);
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t t = gw / slices;
    if (t >= T) return;  // warp-uniform
    const int nvec = d / EPV;
    int my_pos = -1;
    float my_w = 0.f;
    if (lane < k) {
        my_pos = pos[t * k + lane];
        my_w = w ? w[t * k + lane] : 1.f;  // no weights: plain sum
    }
    if (WHOLE) {
        for (int v0 = lane; v0 - lane < nvec; v0 += 32 * U)
            combine_chunk<TA, U, SG>(y_perm, t, k, d, nvec, v0, my_pos, my_w, out);
    } else {
        combine_chunk<TA, U, SG>(y_perm, t, k, d, nvec, (int)(gw - t * slices) * 32 * U + lane,
                                 my_pos, my_w, out);
    }
}

template <typename TA, int U, int SG, bool WHOLE>
cudaError_t launch_combine_u(const Shape &s, const void *y_perm, const int32_t *pos,
                             const float *w, void *out, cudaStream_t st) {
    const int nvec = s.d / (16 / (int)sizeof(TA));
    const int slices = WHOLE ? 1 : (nvec + 32 * U - 1) / (32 * U);
    const int64_t warps = s.T * slices;
    const unsigned blocks = (unsigned)((warps + kWarps - 1) / kWarps);
    launch_pdl(combine_kernel<TA, U, SG, WHOLE>, dim3(blocks), dim3(kThreads), 0, st,
               static_cast<const TA *>(y_perm), pos, w, s.T, s.k, s.d, slices,
               static_cast<TA *>(out));
    return cudaGetLastError();
}

// Large batches: 128-vector chunks (4 vectors per lane); with k <= 2 one warp
// per token walks its whole row a slot at a time, else one warp per
// 128-vector slice with two slots' loads in flight.  Batches too small to
// fill the GPU that way: 32-vector slices (one vector per lane, many more
// warps) and up to 16 slots' loads at once.  (Interleaved A/B timing chose
// these.)
template <typename TA>
cudaError_t launch_combine_t(const Shape &s, const void *y_perm, const int32_t *pos,
                             const float *w, void *out, cudaStream_t st) {
    const int nvec = s.d / (16 / (int)sizeof(TA));
    const int64_t warps4 = s.T * ((nvec + 127) / 128);
    if (warps4 >= 152 * 32) {
        if (s.k <= 2) return launch_combine_u<TA, 4, 1, true>(s, y_perm, pos, w, out, st);
        return launch_combine_u<TA, 4, 2, false>(s, y_perm, pos, w, out, st);
    }
    if (s.k <= 4) return launch_combine_u<TA, 1, 4, false>(s, y_perm, pos, w, out, st);
    if (s.k <= 8) return launch_combine_u<TA, 1, 8, false>(s, y_perm, pos, w, out, st);
    return launch_combine_u<TA, 1, 16, false>(s, y_perm, pos, w, out, st);
}

}  // namespace

cudaError_t launch_combine(const Shape &s, const void *y_perm, const int32_t *pos, const float *w,
                           void *out, cudaStream_t st) {
    if (s.bf16) return launch_combine_t<__nv_bfloat16>(s, y_perm, pos, w, out, st);
    return launch_combine_t<float>(s, y_perm, pos, w, out, st);
}

}  // namespace moe
