// router_tc.cu -- router logits on the sm_103a tensor cores, for bf16
// activations and 8 <= E <= 256 experts (E a multiple of 8).
//
// Transformers docs "Expert parallelism", section "Adding an implementation":
// the router produces the logits from which top_k_index and top_k_weights are
// chosen; the logits are fp32:  L[t][e] = sum_i x[t][i] * Wr[e][i].
//
// x is bf16, so it is exact as an MMA operand.  The fp32 router weight is
// split into three bf16 terms, w = w1 + w2 + w3 with w1 = bf16(w),
// w2 = bf16(w - w1), w3 = bf16(w - w1 - w2) (each difference is exact in
// fp32), which carries w to about 2^-25 relative.  Every product x * w_j is
// exact in the MMA's fp32 accumulator, so
//     L = x . w1 + x . w2 + x . w3
// is an fp32-accumulated dot product of x with w, like the SIMT kernel's,
// at a fraction of its cost.  The three terms are laid side by side along K
// (W' = [w1 | w2 | w3], E x 3d).
//
// Layout: A = x (K-major, TMA box 64 x 128 tokens), B = W' (K-major, box
// 64 x N rows with N = E rounded up to 16; rows past E read zeros).  Two
// shapes:
//  - CTA pairs (E >= 64 and T >= 512): a cluster of two CTAs owns 256
//    tokens (MMA M = 256, tcgen05.mma.cta_group::2 issued by the leader);
//    each CTA loads its own 128 tokens of x and half of the N rows of each
//    W' term, and a stage holds the x tile and the three W' half tiles of
//    the same 64 columns of d (x read once, 12 MMAs per stage).  Each SM
//    then takes in 40 KB (N = 128) or 64 KB (N = 256) per 768 / 1536 MMA
//    cycles, where one CTA with the whole of W' needs 64 KB per 768.
//  - single CTAs (M = 128 tokens): for N <= 128 a stage holds one x tile
//    and the three W' tiles; for larger N one x tile and one W' tile
//    (K' = 3d in steps of 64, x read three times).
// K is split over blockIdx.y so the grid fills the GPU; each split writes
// fp32 partial logits [split][T][E], which the top-k kernel adds in split
// order (a fixed order, so results are reproducible) before selecting.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int RBM = 128;   // tokens per tile (MMA M)
constexpr int RBK = 64;    // K elements per W' / x tile (128 bytes of bf16)
constexpr int R_MAX_STAGES = 6;
constexpr int R_A_BYTES = RBM * RBK * 2;        // 16 KB
constexpr int R_THREADS = 128;
constexpr int R_NUM_BARS = 2 * R_MAX_STAGES + 2;  // full, empty, done, drain
constexpr int R_SMEM_MAX = 210 * 1024;
constexpr int R_PAIR_STAGE_BUDGET = 200 * 1024;
constexpr int R_SMEM_PER_SM = 228 * 1024;    // shared memory of one SM (1 KB per CTA reserved)

// Shared-memory plan of one launch (host and device agree on it).
struct RouterSmem {
    int ctas;         // 1, or 2 for a CTA pair
    int n_pad;        // MMA N: E rounded up to 16
    int n_cta;        // W' rows this CTA loads per term: n_pad / ctas
    int terms;        // W' tiles per stage: 3 (pairs, or N <= 128) or 1
    int stages;
    int stage_bytes;  // one x tile + `terms` W' tiles
    int off_bar, off_tmem, off_abort, bytes;
};

inline RouterSmem router_smem(int E, int ctas) {
    RouterSmem m;
    m.ctas = ctas;
    m.n_pad = (E + 15) / 16 * 16;
    m.n_cta = m.n_pad / ctas;
    m.terms = (ctas == 2 || m.n_pad <= 128) ? 3 : 1;
    m.stage_bytes = R_A_BYTES + m.terms * m.n_cta * RBK * 2;
    // small stages: keep two CTAs per SM; large ones: one CTA with 3-6 stages
    const int budget = ctas == 2 ? R_PAIR_STAGE_BUDGET
                                 : m.stage_bytes <= 32 * 1024 ? 96 * 1024 : 192 * 1024;
    m.stages = std::max(2, std::min(R_MAX_STAGES, budget / m.stage_bytes));
    m.off_bar = m.stages * m.stage_bytes;
    m.off_tmem = m.off_bar + R_NUM_BARS * 8;
    m.off_abort = m.off_tmem + 4;
    m.bytes = m.off_abort + 4 + 1024;  // + alignment slack
    return m;
}

// W'[e][j*d + i] = j-th bf16 term of Wr[e][i], j = 0, 1, 2.  Grid: x over
// the d columns, y over the experts (no integer division per element).
__global__ void split_router_weight_kernel(const float *__restrict__ Wr, int d,
                                           __nv_bfloat16 *__restrict__ Wsplit) {
    pdl_entry();
    const int e = blockIdx.y;
    const float *src = Wr + (int64_t)e * d;
    __nv_bfloat16 *row = Wsplit + (int64_t)e * 3 * d;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d; i += gridDim.x * blockDim.x) {
        const float w = src[i];
        const __nv_bfloat16 w1 = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(w1);
        const __nv_bfloat16 w2 = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(w2);
        const __nv_bfloat16 w3 = __float2bfloat16_rn(r2);
        row[i] = w1;
        row[d + i] = w2;
        row[2 * d + i] = w3;
    }
}

struct RouterParams {
    float *partial;   // [splits][T][E]
    int64_t T;
    int d, E;
    int ks_per_split, ks_total;  // stages of this tile's K loop, per split / in all
    int n_cta, terms, stages, stage_bytes, off_bar, off_tmem, off_abort;
    uint32_t idesc;
    uint32_t tmem_cols;
    DevStatus ds;
};

// CTAS = 2: a cluster of two CTAs; blockIdx.x / 2 is the 256-token tile,
// the cluster rank picks its 128 tokens and its half of each W' tile.
template <int CTAS>
__global__ void __launch_bounds__(R_THREADS, 1)
router_logits_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmW, RouterParams p) {
    pdl_release();  // the wait for the weight split follows the set-up below
    constexpr bool PAIR = CTAS == 2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    const int S = p.stages;
    const uint32_t bar_full = base_s + p.off_bar;
    const uint32_t bar_empty = bar_full + 8 * S;
    const uint32_t bar_done = bar_empty + 8 * S;
    const uint32_t bar_drain = bar_done + 8;
    volatile uint32_t *s_tmem = reinterpret_cast<volatile uint32_t *>(base + p.off_tmem);
    volatile int *s_abort = reinterpret_cast<volatile int *>(base + p.off_abort);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_rank() : 0u;  // 0: the CTA that issues the MMAs
    const bool leader = rank == 0;
    const int64_t m0 = PAIR ? (int64_t)(blockIdx.x >> 1) * (2 * RBM) + rank * RBM
                            : (int64_t)blockIdx.x * RBM;  // this CTA's first token
    const int split = blockIdx.y;
    const int ks0 = split * p.ks_per_split;
    const int ks1 = min(ks0 + p.ks_per_split, p.ks_total);
    const uint32_t w_tile_bytes = (uint32_t)p.n_cta * RBK * 2;
    const int w_row0 = (int)rank * p.n_cta;  // first W' row this CTA loads
    // the full barriers every load signals (the leader's, in a pair)
    const uint32_t sig_full = PAIR ? map_to_rank(bar_full, 0) : bar_full;

    if (threadIdx.x == 0) {
        *s_abort = 0;
        for (int i = 0; i < S; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, 1);
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) tmem_alloc<CTAS>(base_s + p.off_tmem, p.tmem_cols);
    pdl_wait();
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // both CTAs' barriers and tensor memory are ready
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    bool mma_ok = true;

    if (warp == 0) {
        // ------------------------- TMA producer -------------------------
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0, last_par = 0;
            for (int ks = ks0; ks < ks1; ++ks) {
                if (!wait_bounded(bar_empty + 8 * s, ph ^ 1u, p.ds, s_abort)) break;
                const uint32_t fb = sig_full + 8 * s;
                const uint32_t st = base_s + (uint32_t)(s * p.stage_bytes);
                if (leader) {  // the leader's barrier expects both CTAs' bytes
                    mbar_arrive_expect_tx(bar_full + 8 * s, CTAS * (R_A_BYTES + p.terms * w_tile_bytes));
                    issued |= 1u << s;
                    last_par = (last_par & ~(1u << s)) | (ph << s);
                }
                if (p.terms == 3) {
                    // x columns [64 ks, 64 ks + 64) and the three W' tiles that meet them
                    const int kx = ks * RBK;
                    tma_load_2d<CTAS>(st, &tmX, kx, (int)m0, fb);
                    for (int j = 0; j < 3; ++j)
                        tma_load_2d<CTAS>(st + R_A_BYTES + j * w_tile_bytes, &tmW, j * p.d + kx,
                                          w_row0, fb);
                } else {  // single CTAs only
                    const int kp = ks * RBK;  // column of W' (K' = 3d)
                    tma_load_2d<CTAS>(st, &tmX, kp % p.d, (int)m0, fb);
                    tma_load_2d<CTAS>(st + R_A_BYTES, &tmW, kp, w_row0, fb);
                }
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            for (int i = 0; i < S; ++i)  // drain: every armed phase receives all its bytes
                if ((issued >> i) & 1u) {
                    volatile int never = 0;
                    if (!wait_bounded(bar_full + 8 * i, (last_par >> i) & 1u, p.ds, &never,
                                      drain_limit(p.ds)))
                        break;
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------- MMA issuer ---------------------------
        if (leader && lane == 0) {
            // A and B are both K-major: 128-byte rows, 8-row groups 1024 B
            // apart; a K step of 16 elements is 32 bytes along the row.
            const uint64_t adesc0 = smem_desc_sw128(base_s, 16, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(base_s + R_A_BYTES, 16, 1024);
            int s = 0;
            uint32_t ph = 0;
            for (int ks = ks0; ks < ks1; ++ks) {
                if (!wait_bounded(bar_full + 8 * s, ph, p.ds, s_abort)) {
                    mma_ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t a_st = adesc0 + (uint64_t)((s * p.stage_bytes) >> 4);
                const uint64_t b_st = bdesc0 + (uint64_t)((s * p.stage_bytes) >> 4);
                for (int j = 0; j < p.terms; ++j)
#pragma unroll
                    for (int kk = 0; kk < RBK / 16; ++kk)
                        mma_bf16<CTAS>(tmem, a_st + (uint64_t)((kk * 32) >> 4),
                                       b_st + (uint64_t)((j * w_tile_bytes + kk * 32) >> 4), p.idesc,
                                       (ks > ks0 || j > 0 || kk > 0) ? 1u : 0u);
                mma_commit_all<CTAS>(bar_empty + 8 * s);  // frees the stage (both CTAs)
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (mma_ok) mma_commit_all<CTAS>(bar_done);  // accumulators ready (both CTAs)
            mma_commit_local<CTAS>(bar_drain);  // drain before tensor memory is freed
            volatile int never = 0;
            wait_bounded(bar_drain, 0, p.ds, &never, drain_limit(p.ds));
        }
        __syncwarp();
    }

    // ----------------- epilogue: all four warps --------------------------
    const int good = __all_sync(0xffffffffu, wait_bounded(bar_done, 0, p.ds, s_abort));
    if (good) {
        tc_fence_after();
        const int64_t t = m0 + warp * 32 + lane;
        float *row = p.partial + ((int64_t)split * p.T + t) * p.E;
        const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
        for (int c = 0; c < p.E; c += 32) {
            uint32_t v[32];
            tmem_ld32(taddr + c, v);  // columns past N are allocated, never stored
            tmem_ld_wait();
            if (t < p.T) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (c + 4 * q < p.E)  // E is a multiple of 8
                        *reinterpret_cast<uint4 *>(row + c + 4 * q) =
                            make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal it
    tc_fence_after();
    if (warp == 0) tmem_dealloc<CTAS>(tmem, p.tmem_cols);
}

}  // namespace

bool router_tc_eligible(const Shape &s) {
    if (!s.bf16 || s.E < 8 || s.E > 256 || s.E % 8 != 0 || s.d % RBK != 0) return false;
    // up to 32 experts the CUDA-core kernel also selects in the same launch,
    // which wins for small batches
    return s.E >= 64 || s.T >= 1024;
}

bool router_tc_pair(const Shape &s) {
    // CTA pairs need at least 32 W' rows per CTA and enough tokens to fill
    // 256-token tiles
    return s.E >= 64 && s.T >= 512;
}

RouterTcPlan router_tc_plan(const Shape &s) {
    RouterTcPlan pl;
    pl.ctas = router_tc_pair(s) ? 2 : 1;
    const RouterSmem m = router_smem(s.E, pl.ctas);
    const int64_t tiles = (s.T + RBM * pl.ctas - 1) / (RBM * pl.ctas);
    pl.ks_total = (m.terms == 3 ? 1 : 3) * s.d / RBK;
    // at least 2 stages (three W' tiles each) or 4 stages (one W' tile each) per CTA
    const int min_stages = m.terms == 3 ? 2 : 4;
    const int64_t max_splits = std::max(1, pl.ks_total / min_stages);
    const int sms = device_sm_count();  // the plan fills one wave of the current device
    int64_t want;
    if (pl.ctas == 2)  // one wave of pairs: as many K splits as still fit beside the tiles
        want = std::max<int64_t>(1, (sms / 2) / tiles);
    else  // as many splits as keep the grid within one wave (CTAs per SM by shared memory)
        want = std::max<int64_t>(1, sms * std::max(1, R_SMEM_PER_SM / (m.bytes + 1024)) / tiles);
    want = std::max<int64_t>(1, std::min<int64_t>(want, max_splits));
    pl.ks_per_split = (int)((pl.ks_total + want - 1) / want);
    pl.splits = (pl.ks_total + pl.ks_per_split - 1) / pl.ks_per_split;
    return pl;
}

size_t router_tc_scratch_bytes(const Shape &s) {
    if (!router_tc_eligible(s) || s.T == 0) return 0;
    const RouterTcPlan pl = router_tc_plan(s);
    const size_t wsplit = ((size_t)s.E * 3 * s.d * 2 + 255) & ~(size_t)255;
    return wsplit + (size_t)pl.splits * (size_t)s.T * s.E * 4;
}

template <int CTAS>
cudaError_t launch_router_kernel(dim3 grid, size_t smem, cudaStream_t st, const CUtensorMap &mx,
                                 const CUtensorMap &mw, const RouterParams &p) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        if ((err = cudaFuncSetAttribute(router_logits_tc_kernel<CTAS>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        R_SMEM_MAX)) != cudaSuccess)
            return err;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(R_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CTAS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_entry
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, router_logits_tc_kernel<CTAS>, mx, mw, p);
}

cudaError_t launch_router_logits_tc(const Shape &s, const void *x, const float *Wr, void *scratch,
                                    float **partial_out, int *splits_out, const DevStatus &ds,
                                    cudaStream_t st) {
    if (!tensor_map_encoder()) {
        set_error_message("cuTensorMapEncodeTiled is not available from the driver");
        return cudaErrorNotSupported;
    }
    const RouterTcPlan pl = router_tc_plan(s);
    __nv_bfloat16 *wsplit = static_cast<__nv_bfloat16 *>(scratch);
    float *partial = reinterpret_cast<float *>(static_cast<uint8_t *>(scratch) +
                                               (((size_t)s.E * 3 * s.d * 2 + 255) & ~(size_t)255));
    launch_pdl(split_router_weight_kernel, dim3((unsigned)std::min(8, (s.d + 255) / 256), (unsigned)s.E),
               dim3(256), 0, st, Wr, s.d, wsplit);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;

    const RouterSmem m = router_smem(s.E, pl.ctas);
    CUtensorMap mx, mw;
    if (!tensor_map_rows(&mx, x, s.T, s.d, RBM) ||
        !tensor_map_rows(&mw, wsplit, s.E, 3 * (int64_t)s.d, (uint32_t)m.n_cta)) {
        set_error_message("cuTensorMapEncodeTiled rejected a router operand");
        return cudaErrorInvalidValue;
    }
    RouterParams p;
    p.partial = partial;
    p.T = s.T;
    p.d = s.d;
    p.E = s.E;
    p.ks_per_split = pl.ks_per_split;
    p.ks_total = pl.ks_total;
    p.n_cta = m.n_cta;
    p.terms = m.terms;
    p.stages = m.stages;
    p.stage_bytes = m.stage_bytes;
    p.off_bar = m.off_bar;
    p.off_tmem = m.off_tmem;
    p.off_abort = m.off_abort;
    p.idesc = idesc_bf16(RBM * pl.ctas, m.n_pad, false);
    p.tmem_cols = m.n_pad <= 32 ? 32 : m.n_pad <= 64 ? 64 : m.n_pad <= 128 ? 128 : 256;
    p.ds = ds;
    const unsigned tiles = (unsigned)((s.T + RBM * pl.ctas - 1) / (RBM * pl.ctas));
    const dim3 grid(tiles * pl.ctas, (unsigned)pl.splits);
    err = pl.ctas == 2 ? launch_router_kernel<2>(grid, m.bytes, st, mx, mw, p)
                       : launch_router_kernel<1>(grid, m.bytes, st, mx, mw, p);
    if (err != cudaSuccess) return err;
    *partial_out = partial;
    *splits_out = pl.splits;
    return cudaSuccess;
}

}  // namespace moe
