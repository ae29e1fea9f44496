// gemm_f32.cu -- grouped SwiGLU experts for fp32 activations (SIMT FFMA).
//
// Transformers docs "Expert parallelism", section "Adding an implementation"
// (experts_forward runs every expert on the rows sent to it) and "Tensor
// parallelism for inference", section "Packed strategies" (gate_up_proj is
// [E][d][2f], applied as x @ gate_up_proj and split into gate = first f
// columns, up = last f columns).  For each expert e and row r of its segment
// [offsets[e], offsets[e+1]):
//   h[r] = silu(x[r] @ Wgu[e][:, :f]) * (x[r] @ Wgu[e][:, f:])
//   y[r] = h[r] @ Wd[e]
// Ragged segments: the grid covers an upper bound of the row tiles; each
// block finds its expert from the tile prefix of ceil(count/BM) and exits
// when it lies beyond the last tile.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, TM = 4, TN = 4;
constexpr int kThreads = 256;
constexpr int RG = BM / TM, CG = BN / TN;  // 16 x 16 thread grid

// Warp 0 builds s_tile[e] = sum_{e'<e} ceil(count_e'/BM), s_tile[E] = total.
__device__ void row_tile_prefix(const int32_t *__restrict__ offsets, int E, int *s_off,
                                int *s_tile) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = offsets[e];
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int local = 0;
        for (int e = e0; e < e1; ++e) local += (s_off[e + 1] - s_off[e] + BM - 1) / BM;
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        int run = incl - local;
        for (int e = e0; e < e1; ++e) {
            s_tile[e] = run;
            run += (s_off[e + 1] - s_off[e] + BM - 1) / BM;
        }
        if (lane == 31) s_tile[E] = incl;
    }
    __syncthreads();
}

// Last e with s_tile[e] <= g (the expert whose tile range holds g).
__device__ __forceinline__ int find_expert(const int *s_tile, int E, int g) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s_tile[mid] <= g) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads)
grouped_gemm_f32_kernel(const float *__restrict__ A, const int32_t *__restrict__ offsets, int E,
                        const float *__restrict__ B, int K, int Nb, int N, int f,
                        float *__restrict__ C, int a_local) {
    pdl_entry();
    extern __shared__ int s_dyn[];
    int *s_off = s_dyn;
    int *s_tile = s_dyn + (E + 1);
    __shared__ float As[BK][BM + 1];
    __shared__ float Bg[BK][BN];
    __shared__ float Bu[SWIGLU ? BK : 1][SWIGLU ? BN : 1];

    row_tile_prefix(offsets, E, s_off, s_tile);
    const int g = blockIdx.x;
    if (g >= s_tile[E]) return;  // block-uniform
    const int e = find_expert(s_tile, E, g);
    const int row0 = s_off[e] + (g - s_tile[e]) * BM;
    const int rows = min(BM, s_off[e + 1] - row0);
    // a_local: A holds one row per position of the segment (row r of expert
    // e reads A row r - offsets[e]), as when every expert sees every token
    const int arow0 = a_local ? row0 - s_off[e] : row0;
    const int n0 = blockIdx.y * BN;
    const float *Be = B + (int64_t)e * K * Nb;

    const int tid = threadIdx.x, tx = tid % CG, ty = tid / CG;
    float ag[TM][TN], au[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) ag[i][j] = au[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
        for (int r = 0; r < (BM * BK) / kThreads; ++r) {
            int i = tid + r * kThreads;
            int m = i / BK, c = i % BK;
            As[c][m] = (m < rows && k0 + c < K) ? A[(int64_t)(arow0 + m) * K + k0 + c] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < (BK * BN) / kThreads; ++r) {
            int i = tid + r * kThreads;
            int kk = i / BN, n = i % BN;
            bool ok = (k0 + kk < K) && (n0 + n < N);
            const float *brow = Be + (int64_t)(k0 + kk) * Nb;
            Bg[kk][n] = ok ? brow[n0 + n] : 0.f;
            if (SWIGLU) Bu[kk][n] = ok ? brow[f + n0 + n] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], bg[TN], bu[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = As[kk][ty + i * RG];
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                bg[j] = Bg[kk][tx + j * CG];
                if (SWIGLU) bu[j] = Bu[kk][tx + j * CG];
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    ag[i][j] = fmaf(a[i], bg[j], ag[i][j]);
                    if (SWIGLU) au[i][j] = fmaf(a[i], bu[j], au[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        int m = ty + i * RG;
        if (m >= rows) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            int n = n0 + tx + j * CG;
            if (n >= N) continue;
            float v = ag[i][j];
            if (SWIGLU) v = v / (1.f + expf(-v)) * au[i][j];
            C[(int64_t)(row0 + m) * N + n] = v;
        }
    }
}

}  // namespace

cudaError_t launch_grouped_swiglu_f32(const Shape &s, const float *x_perm, const int32_t *offsets,
                                      const float *Wgu, const float *Wd, float *h_perm,
                                      float *y_perm, cudaStream_t st, bool a_local) {
    const int64_t P = s.P();
    const int64_t mtiles = (P + BM - 1) / BM + s.E;  // upper bound of sum_e ceil(count_e / BM)
    const size_t sh = sizeof(int) * (2 * (size_t)s.E + 2);
    dim3 g1((unsigned)mtiles, (unsigned)((s.f + BN - 1) / BN));
    launch_pdl(grouped_gemm_f32_kernel<true>, dim3(g1), dim3(kThreads), sh, st, x_perm, offsets, s.E, Wgu, s.d,
                                                           2 * s.f, s.f, s.f, h_perm, a_local ? 1 : 0);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    dim3 g2((unsigned)mtiles, (unsigned)((s.d + BN - 1) / BN));
    launch_pdl(grouped_gemm_f32_kernel<false>, dim3(g2), dim3(kThreads), sh, st, h_perm, offsets, s.E, Wd, s.f, s.d,
                                                            s.d, 0, y_perm, 0);
    return cudaGetLastError();
}

}  // namespace moe
