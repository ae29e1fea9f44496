// dispatch.cu -- token dispatch on one device: per-expert histogram, exclusive
// scan, stable scatter into expert-contiguous order, and the row gather.
//
// Transformers docs "Expert parallelism", section "Token dispatch": every
// (token, expert) pair is sent to its expert and the experts run on the rows
// they receive.  On one GPU "sending" is a permutation: pair (t, j) gets row
// pos[t*k+j] of its expert's segment, segments laid out in expert order.
//
// Stability: pairs are cut into chunks of consecutive pair ids; chunk b's
// rows for expert e start at the exclusive scan of the expert-major
// [E][chunks] count matrix, and inside a chunk every warp ranks its pairs
// with __match_any_sync in pair order.  So rows of one expert are in
// ascending pair id, hence ascending token id, with no atomics deciding order.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// counts of chunk b, stored expert-major: hist[e * NB + b]
__global__ void __launch_bounds__(kThreads)
chunk_histogram_kernel(const int32_t *__restrict__ idx, int64_t P, int E, int chunk, int NB,
                       int32_t *__restrict__ hist, DevStatus ds) {
    pdl_entry();
    extern __shared__ int sh_count[];
    for (int e = threadIdx.x; e < E; e += kThreads) sh_count[e] = 0;
    __syncthreads();
    const int64_t q0 = (int64_t)blockIdx.x * chunk;
    const int64_t q1 = min(q0 + chunk, P);
#pragma unroll 8  // independent iterations: several index loads in flight
    for (int64_t q = q0 + threadIdx.x; q < q1; q += kThreads) {
        int e = idx[q];
        if ((unsigned)e < (unsigned)E)
            atomicAdd(&sh_count[e], 1);
        else
            raise_error(ds, kErrBadRouting);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) hist[(int64_t)e * NB + blockIdx.x] = sh_count[e];
}

// Single block: exclusive scan of hist[0 .. E*NB) in place (the base row of
// every (expert, chunk)), then counts[e] and offsets[0..E].  STAGED: the
// matrix (at most kScanStageMax ints) is first copied to shared memory with
// coalesced loads, scanned there and copied back, so each thread's serial
// walk over its segment reads shared memory instead of waiting on one global
// load after another.
constexpr int kScanThreads = 1024;
constexpr int kScanStageMax = 12 * 1024 - 64;  // ints: with the static arrays, under 48 KB
template <bool STAGED>
__global__ void __launch_bounds__(kScanThreads)
scan_kernel(int32_t *__restrict__ hist_g, int E, int NB, int32_t *__restrict__ counts,
            int32_t *__restrict__ offsets) {
    pdl_entry();
    __shared__ int warp_tot[kScanThreads / 32];
    __shared__ int total_s;
    extern __shared__ int sh_hist[];
    const int n = E * NB;
    int32_t *hist = hist_g;
    if (STAGED) {
        for (int i = threadIdx.x; i < n; i += kScanThreads) sh_hist[i] = hist_g[i];
        __syncthreads();
        hist = sh_hist;
    }
    const int seg = (n + kScanThreads - 1) / kScanThreads;
    const int beg = min(n, (int)threadIdx.x * seg);
    const int end = min(n, beg + seg);
    int local = 0;
    for (int i = beg; i < end; ++i) local += hist[i];
    // block exclusive scan of `local`
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int v = warp_tot[lane];
        int inc = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += u;
        }
        warp_tot[lane] = inc - v;  // exclusive warp base
        if (lane == 31) total_s = inc;
    }
    __syncthreads();
    int run = warp_tot[wid] + incl - local;
    for (int i = beg; i < end; ++i) {
        int c = hist[i];
        hist[i] = run;
        run += c;
    }
    __syncthreads();
    if (STAGED)
        for (int i = threadIdx.x; i < n; i += kScanThreads) hist_g[i] = sh_hist[i];
    const int total = total_s;
    for (int e = threadIdx.x; e < E; e += kScanThreads) {
        int b0 = hist[e * NB];
        int b1 = (e + 1 < E) ? hist[(e + 1) * NB] : total;
        offsets[e] = b0;
        counts[e] = b1 - b0;
    }
    if (threadIdx.x == 0) offsets[E] = total;
}

// Stable scatter: warp w of block b ranks pairs [q0 + w*sub, q0 + (w+1)*sub).
__global__ void __launch_bounds__(kThreads)
scatter_kernel(const int32_t *__restrict__ idx, int64_t P, int k, int E, int chunk, int NB,
               const int32_t *__restrict__ base, int32_t *__restrict__ pos,
               int32_t *__restrict__ src_token) {
    pdl_entry();
    extern __shared__ int sh_warp[];  // [kWarps][E]: per-warp counts, then running row
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kWarps * E; i += kThreads) sh_warp[i] = 0;
    __syncthreads();
    const int sub = chunk / kWarps;  // multiple of 32
    const int64_t w0 = (int64_t)blockIdx.x * chunk + (int64_t)wid * sub;
    const int64_t w1 = min(w0 + sub, P);
    int *mine = sh_warp + wid * E;
#pragma unroll 8  // independent iterations: several index loads in flight
    for (int64_t q = w0 + lane; q < w1; q += 32) {
        int e = idx[q];
        if ((unsigned)e < (unsigned)E) atomicAdd(&mine[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int run = base[(int64_t)e * NB + blockIdx.x];
        for (int w = 0; w < kWarps; ++w) {
            int c = sh_warp[w * E + e];
            sh_warp[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    // the next iteration's expert id is loaded before this one is ranked
    int e_next = (w0 + lane < w1) ? idx[w0 + lane] : -1;
    for (int64_t qb = w0; qb < w1; qb += 32) {  // warp-uniform trip count
        const int64_t q = qb + lane;
        int e = e_next;
        if (q < w1 && (unsigned)e >= (unsigned)E) e = -1;
        e_next = (q + 32 < w1) ? idx[q + 32] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt_mask);
        const int row0 = (e >= 0) ? mine[e] : 0;
        __syncwarp();
        if (q < w1) {
            if (e >= 0) {
                const int row = row0 + rank;
                pos[q] = row;
                src_token[row] = (int32_t)(q / k);
                if (lane == 31 - __clz(peers)) mine[e] = row0 + __popc(peers);
            } else {
                pos[q] = -1;  // dropped pair (expert id out of range)
            }
        }
        __syncwarp();
    }
}

// Row gather x_perm[pos[q]] = x[q / k]: one warp per pair, 16-byte vectors.
__global__ void __launch_bounds__(kThreads)
gather_rows_kernel(const uint8_t *__restrict__ x, const int32_t *__restrict__ pos, int64_t P,
                   int k, int row_vecs, uint8_t *__restrict__ x_perm) {
    pdl_entry();
    const int lane = threadIdx.x & 31;
    const int64_t q = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (q >= P) return;
    const int row = pos[q];
    if (row < 0) return;
    const int64_t t = q / k;
    const uint4 *src = reinterpret_cast<const uint4 *>(x) + t * row_vecs;
    uint4 *dst = reinterpret_cast<uint4 *>(x_perm) + (int64_t)row * row_vecs;
    int i = lane;
    for (; i + 96 < row_vecs; i += 128) {
        uint4 a = ldg16(src + i), b = ldg16(src + i + 32), c = ldg16(src + i + 64),
              d = ldg16(src + i + 96);
        stg16(dst + i, a);
        stg16(dst + i + 32, b);
        stg16(dst + i + 64, c);
        stg16(dst + i + 96, d);
    }
    for (; i < row_vecs; i += 32) stg16(dst + i, ldg16(src + i));
}

// Scaled row gather x_perm[pos[q]] = scale[q] * x[q / k], the product formed
// in fp32 and rounded once to the activation dtype.
template <typename TA>
__global__ void __launch_bounds__(kThreads)
gather_rows_scaled_kernel(const TA *__restrict__ x, const int32_t *__restrict__ pos,
                          const float *__restrict__ scale, int64_t P, int k, int d,
                          TA *__restrict__ x_perm) {
    pdl_entry();
    constexpr int EPV = 16 / sizeof(TA);
    const int lane = threadIdx.x & 31;
    const int64_t q = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (q >= P) return;
    const int row = pos[q];
    if (row < 0) return;
    const float wq = scale[q];
    const TA *src = x + (q / k) * d;
    TA *dst = x_perm + (int64_t)row * d;
    for (int v = lane; v < d / EPV; v += 32) {
        float f[EPV];
        unpack16(ldg16(src + (int64_t)v * EPV), f, static_cast<const TA *>(nullptr));
#pragma unroll
        for (int i = 0; i < EPV; ++i) f[i] *= wq;
        stg16(dst + (int64_t)v * EPV, pack16(f, static_cast<const TA *>(nullptr)));
    }
}

}  // namespace

DispatchGrid dispatch_grid(int64_t P, int E) {
    // Chunks of 2048 pairs; 256 when the E x chunks histogram stays small
    // (few experts and pairs): the histogram and scatter blocks are latency
    // bound, so more and shorter blocks finish sooner, while the single-block
    // scan over E x chunks entries must stay short (at E = 128-256 and 64K+
    // pairs, 256-pair chunks made the scan the slowest step).
    DispatchGrid g;
    g.chunk = (int64_t)E * ((P + 255) / 256) <= 4096 ? 256 : 2048;
    int64_t nb = (P + g.chunk - 1) / g.chunk;
    if (nb > 1024) {
        int64_t c = (P + 1023) / 1024;
        c = (c + 255) / 256 * 256;
        g.chunk = (int)c;
        nb = (P + c - 1) / c;
    }
    g.blocks = (int)(nb < 1 ? 1 : nb);
    return g;
}

size_t dispatch_scratch_bytes(const Shape &s) {
    DispatchGrid g = dispatch_grid(s.P(), s.E);
    return sizeof(int32_t) * (size_t)s.E * (size_t)g.blocks;
}

cudaError_t launch_dispatch(const Shape &s, const int32_t *idx, const void *x, int32_t *counts,
                            int32_t *offsets, int32_t *pos, int32_t *src_token, void *x_perm,
                            int32_t *hist, const DevStatus &ds, cudaStream_t st,
                            const float *scale) {
    const int64_t P = s.P();
    const DispatchGrid g = dispatch_grid(P, s.E);
    launch_pdl(chunk_histogram_kernel, dim3(g.blocks), dim3(kThreads), sizeof(int) * s.E, st, idx, P, s.E, g.chunk,
                                                                        g.blocks, hist, ds);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int64_t n_hist = (int64_t)s.E * g.blocks;
    if (n_hist <= kScanStageMax)
        launch_pdl(scan_kernel<true>, dim3(1), dim3(kScanThreads), sizeof(int) * (size_t)n_hist, st,
                   hist, s.E, g.blocks, counts, offsets);
    else
        launch_pdl(scan_kernel<false>, dim3(1), dim3(kScanThreads), 0, st, hist, s.E, g.blocks,
                   counts, offsets);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    const size_t sh = sizeof(int) * (size_t)kWarps * s.E;
    launch_pdl(scatter_kernel, dim3(g.blocks), dim3(kThreads), sh, st, idx, P, s.k, s.E, g.chunk, g.blocks, hist, pos,
                                                  src_token);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (!x_perm) return cudaSuccess;
    const int row_vecs = (int)((int64_t)s.d * (s.bf16 ? 2 : 4) / 16);
    const unsigned blocks = (unsigned)((P + kWarps - 1) / kWarps);
    if (scale && s.bf16)
        launch_pdl(gather_rows_scaled_kernel<__nv_bfloat16>, dim3(blocks), dim3(kThreads), 0, st,
            static_cast<const __nv_bfloat16 *>(x), pos, scale, P, s.k, s.d,
            static_cast<__nv_bfloat16 *>(x_perm));
    else if (scale)
        launch_pdl(gather_rows_scaled_kernel<float>, dim3(blocks), dim3(kThreads), 0, st,
            static_cast<const float *>(x), pos, scale, P, s.k, s.d, static_cast<float *>(x_perm));
    else
        launch_pdl(gather_rows_kernel, dim3(blocks), dim3(kThreads), 0, st, static_cast<const uint8_t *>(x), pos, P,
                                                       s.k, row_vecs,
                                                       static_cast<uint8_t *>(x_perm));
    return cudaGetLastError();
}

}  // namespace moe
