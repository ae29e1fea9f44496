// gemm_tc.cu -- grouped SwiGLU experts for bf16 activations on the sm_103a
// tensor cores (tcgen05.mma, accumulators in tensor memory, operands staged
// by TMA).
//
// Transformers docs "Expert parallelism", section "Adding an implementation"
// (experts_forward runs each expert on the rows sent to it), and "Tensor
// parallelism for inference", section "Packed strategies" (gate_up_proj is
// [E][d][2f], applied as x @ gate_up_proj and split into gate = first f
// columns, up = last f columns).  Launches of one persistent kernel compute
//   G1: h_perm[r] = silu(x_perm[r] @ Wgu[e][:, :f]) * (x_perm[r] @ Wgu[e][:, f:])
//   G2: y_perm[r] = h_perm[r] @ Wd[e]
// for every expert e and row r of its segment [offsets[e], offsets[e+1]).
// The kernel's tile list is every G1 tile, then every G2 tile, and each
// launch is given the column tiles of one product only (the other's count is
// zero), so the product is a property of the tile, not of the template.
// One launch per product when one tile shape serves every expert; two when
// the experts are split between the shapes (see tile_mode).
//
// The kernel template is grouped_gemm_tc_kernel<CTAS, GATHER, SCALE>: the
// tile shape (below), whether G1 gathers its own A rows (GATHER, below), and
// whether G1 multiplies each row's gate and up accumulators by a per-row
// weight before the SwiGLU (SCALE: routing weights on the expert inputs,
// (w x) W = w (x W)).  Each launch runs the instantiation it needs.
//
// Tiling.  Two tile shapes share the kernel template (CTAS = 1 or 2).
//  - CTAS = 2 (a cluster of 2, tcgen05.mma.cta_group::2): the pair owns a
//    256-row x 256-column tile; each CTA holds its 128 rows of A and half of
//    the 256 B columns in its own shared memory, and the leader CTA's MMA
//    (M = 256, N = 256, K = 16) reads both halves and writes each CTA's 128
//    rows into that CTA's tensor memory.  Per K step a CTA loads 16 KB of A
//    and 16 KB of B, so six stages fit; used when experts receive many rows.
//  - CTAS = 1 (tcgen05.mma.cta_group::1): a CTA owns a 128 x 256 tile and
//    loads 16 KB of A and 32 KB of B per K step (four stages).  Row tiles of
//    128 waste less on ragged segments, so it serves small per-expert batches
//    (decode), and at ~256 rows per expert the experts that 256-row tiles
//    would pad more (pair_tiles_pay), where the weight stream bounds.
// A K step is 64 elements (128 bytes: one swizzle span).  In G1 the 256
// accumulator columns are 128 gate columns and the 128 matching up columns,
// so the SwiGLU is applied in the epilogue straight from the two halves of
// one accumulator.  A (the permuted activations) is K-major; B (the weights
// as stored, [K][N] with N contiguous) is read MN-major, so no weight
// repacking is needed.
//
// Work list.  Row tiles never straddle experts: expert e owns
// ceil(count_e / tile rows) row tiles (none in a launch that serves other
// experts) and each CTA derives the prefix of those counts from `offsets` on
// the device (no host synchronisation).
// Tiles are ordered expert-major, then column tile, then row tile, so tiles
// running at the same time share the same weight tile through L2.  The grid
// is persistent (as many CTAs or pairs as fit at once) and strides over the
// tile list.
//
// Rows gathered in G1 (Params::gather, the GATHER instantiation): moe_forward
// can skip the permuted copy of x.  Two more warps then copy each stage's A
// rows from the token rows through src_token with 16-byte cp.async into the
// same swizzled layout (the TMA loads only B), and a third reports each
// stage once its rows have landed (an mbarrier that tracks the copies, a
// proxy fence, then an arrival or, in a pair, a 16-byte async copy into the
// leader whose bytes complete the stage's full barrier).
//
// Roles (192 threads per CTA; 288 with GATHER, warps 6-8 as above): one
// thread of warp 0 issues the TMA loads,
// warp 1 owns the tensor memory and one of its threads issues the MMAs and
// their commits (in a pair: the leader only, commits multicast to both CTAs,
// and every load of both CTAs signals the leader's full barrier), warps 2-5
// run the epilogue (tensor memory ->
// registers -> global), each on its 32-lane quarter of its CTA's
// accumulator.  Two accumulators (2 x 256 columns) let the epilogue of one
// tile overlap the main loop of the next.
//
// Every wait is bounded (globaltimer); a wait that runs out records a timeout
// in the device error word, raises a CTA-wide abort flag, and every role
// drains its in-flight copies/MMAs before the tensor memory is released.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;          // rows per CTA
constexpr int BN = 256;          // accumulator columns per tile (MMA N)
constexpr int BK = 64;           // K elements per stage = one 128-byte swizzle span
constexpr int UMMA_K = 16;       // K per tcgen05.mma for 16-bit operands
constexpr int A_BYTES = BM * BK * 2;          // 16 KB: this CTA's 128 rows
constexpr int B_ATOM_BYTES = BK * 128;        // 64 K-rows x 64 columns (128 B) = 8 KB
constexpr int TMEM_COLS = 2 * BN;             // two accumulators
constexpr int NUM_THREADS = 192;  // launches whose A operand arrives by TMA
// G1 launches that gather their A rows from the token rows (Params::gather)
// add kGatherWarps warps, which copy the rows of every A stage, and one warp
// that reports each stage to the MMA issuer once its rows have landed.  Two
// copying warps measured faster than one or four.
constexpr int kGatherWarps = 2;
constexpr int NUM_THREADS_GATHER = NUM_THREADS + 32 * (kGatherWarps + 1);
constexpr int kGatherRows = 128 / kGatherWarps;  // A rows per gather warp and stage
constexpr int kGatherIters = kGatherRows / 4;    // a warp instruction copies 4 rows
constexpr int MAX_E = 1024;
constexpr int kPairRowsPerExpert = 512;  // average rows per expert that selects CTA pairs

template <int CTAS> struct Cfg {
    static constexpr bool PAIR = CTAS == 2;
    static constexpr int TILE_M = BM * CTAS;              // rows per tile (MMA M)
    static constexpr int B_ATOMS = 4 / CTAS;              // 64-column B atoms per CTA
    static constexpr int B_BYTES = B_ATOMS * B_ATOM_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = PAIR ? 6 : 4;
    static constexpr int EXPECT_BYTES = STAGE_BYTES * CTAS;  // per full-barrier phase
    // shared-memory map (offsets from a 1024-byte aligned base)
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = STAGES * A_BYTES;
    static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
    // full, empty, tmem full/empty, drain, gathered (rows copied, per stage)
    static constexpr int NUM_BARS = 3 * STAGES + 2 + 2 + 1;
    // gathered stages of a pair are reported by 16-byte copies into the
    // leader's shared memory (one slot per CTA)
    static constexpr int OFF_SIGNAL = (OFF_BAR + NUM_BARS * 8 + 15) / 16 * 16;
    static constexpr int OFF_TMEM = OFF_SIGNAL + 16 * CTAS;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int OFF_OFFS = OFF_ABORT + 4;               // int[MAX_E + 1]
    static constexpr int OFF_TILE = OFF_OFFS + 4 * (MAX_E + 1);  // int[MAX_E + 1]
    static constexpr int SMEM_BYTES = OFF_TILE + 4 * (MAX_E + 1) + 1024;  // + alignment slack
    static constexpr uint32_t IDESC = idesc_bf16(TILE_M, BN, true);  // B MN-major
    static constexpr int EPI_ARRIVALS = 4 * CTAS;         // epilogue warps reporting per tile
};

// One product of the pair: [0] = G1 (gate/up + SwiGLU), [1] = G2 (down).
struct PhaseParams {
    int K;              // reduction length (d for G1, f for G2)
    int n_out;          // output columns (f for G1, d for G2)
    int n_tiles;        // column tiles per row tile
    int transpose_epi;  // epilogue store pattern (see kTransposeMaxK)
    __nv_bfloat16 *out;  // [P][n_out]
};

struct Params {
    const int32_t *offsets;
    int E;
    int f;              // column offset of the up half in Wgu
    PhaseParams g1, g2;  // a launch runs one of them: the other has n_tiles = 0
    int experts;  // which experts this launch serves: kAllExperts, kPairExperts, kSingleExperts
    // Ordering against the neighbouring launches (programmatic dependent launch).
    //  release_late: let the next launch start only after this one's own wait
    //    for its predecessor, so that by then every earlier kernel has completed.
    //  overlap_prev: this launch's tiles do not read the previous launch's
    //    output (its experts are disjoint), so it reads its inputs without
    //    waiting and waits for the previous launch only before it exits; its
    //    completion still implies the previous launch's.
    int release_late, overlap_prev;
    // B maps are the 64-column-block views (tensor_map_weight_blocks): one
    // box carries two 8 KB atoms
    int b_blocks;
    // G1's A holds one row per position of a segment: row r of expert e
    // reads A row r - offsets[e] (every expert sees every token, in order)
    int a_local;
    // G1's A rows are gathered from the token rows: row r of the segments is
    // row src_token[r] of gx ([T][K], K a multiple of 64), copied by the
    // gather warps; no permuted copy of the activations exists.  The launch
    // runs the GATHER instantiation of the kernel.
    int gather;
    const __nv_bfloat16 *gx;
    const int32_t *src_token;
    // G1 only, or nullptr: row r's gate and up accumulators are multiplied
    // by row_scale[r] before the SwiGLU (the routing weight acting on the
    // expert's input row: (w x) W = w (x W))
    const float *row_scale;
    DevStatus ds;
};

// SwiGLU in the epilogue: silu(g) * u with the fast exponential and the fast
// (approximate-reciprocal) division; both are within a few fp32 ulps, far
// below the bf16 rounding of h, and the lighter instruction stream leaves
// more issue slots to the MMA thread, which shares a scheduler with one of
// the epilogue warps.
//
// Epilogue store pattern (Params::transpose_epi): 0 = each thread stores its
// own row (16-byte stores, 32 rows per warp instruction); 1 = 16-byte chunks
// are transposed with shuffles within groups of eight lanes so each warp
// instruction stores 128 contiguous bytes of each of four rows.  The second
// costs shuffles but fewer memory transactions; it pays when epilogues are
// frequent relative to the main loop (short K).
constexpr int kTransposeMaxK = 3072;

// Lane l holds packed[i] = bf16 pair (columns 2i, 2i+1 of a 64-column block)
// of row (rbase + l): eight 16-byte chunks of 8 columns, chunk c in
// packed[4c .. 4c+3].  An 8 x 8 transpose of the chunks within each group of
// eight lanes (three butterfly steps over lane bits 4, 2, 1) leaves lane
// 8g + j with chunk j of rows 8g .. 8g+7 in chunk slots 0..7, so each store
// instruction writes 128 contiguous bytes of four rows: 48 shuffles and 8
// 16-byte stores per block.
__device__ __forceinline__ void store_rows_transposed(uint32_t (&packed)[32], __nv_bfloat16 *out,
                                                      int64_t rbase, int rows_valid, int col0,
                                                      int n_out) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (c & s) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t send = upper ? packed[4 * c + q] : packed[4 * (c + s) + q];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, s);
                if (upper) packed[4 * c + q] = recv;
                else packed[4 * (c + s) + q] = recv;
            }
        }
    }
    const int grp = lane >> 3;
    const int col = col0 + 8 * (lane & 7);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * grp + i;
        if (r < rows_valid && col + 8 <= n_out)
            stg16(out + (rbase + r) * n_out + col,
                  make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]));
    }
}

// Experts split between the two tile shapes by row count: CTA-pair tiles
// (256 rows) serve an expert when they pad its rows to no more than 1.16x
// what 128-row single-CTA tiles would (the single tile's cost per MMA row,
// measured, from its larger shared-memory fill per SM).  The predicate is
// evaluated on the device from `offsets`, identically by both launches.
constexpr int kAllExperts = 0, kPairExperts = 1, kSingleExperts = 2;
__host__ __device__ __forceinline__ bool pair_tiles_pay(int count) {
    const int pair_rows = (count + 255) / 256 * 256, single_rows = (count + 127) / 128 * 128;
    return pair_rows * 100 <= single_rows * 116;
}
__device__ __forceinline__ int expert_row_tiles(int count, int tile_m, int experts) {
    if (experts != kAllExperts && pair_tiles_pay(count) != (experts == kPairExperts)) return 0;
    return (count + tile_m - 1) / tile_m;
}

struct TileInfo {
    int e, row0, rows, n_blk;  // row0/rows: the tile's slice of expert e's segment
    bool down;                 // a G2 tile
};

// Tiles [0, total1) are G1 tiles, the rest G2 tiles; within each product the
// order is expert, then column tile, then row tile.  The expert is the last e
// with s_tile[e] <= (tile / column tiles).
__device__ __forceinline__ TileInfo decode_tile(int tile, const int *s_off, const int *s_tile,
                                                int E, int total1, int n1, int n2, int tile_m) {
    TileInfo ti;
    ti.down = tile >= total1;
    const int local = ti.down ? tile - total1 : tile;
    const int n_tiles = ti.down ? n2 : n1;
    const int g = local / n_tiles;
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s_tile[mid] <= g) lo = mid; else hi = mid - 1;
    }
    ti.e = lo;
    const int mt = s_tile[lo + 1] - s_tile[lo];
    const int r = local - s_tile[lo] * n_tiles;
    ti.n_blk = r / mt;
    ti.row0 = s_off[lo] + (r % mt) * tile_m;
    ti.rows = min(tile_m, s_off[lo + 1] - ti.row0);
    return ti;
}

// tmX / tmWgu: A and B of G1; tmH / tmWd: A and B of G2.
// SCALE: G1 multiplies each row's gate and up accumulators by
// Params::row_scale (a separate instantiation, so launches without row
// scales run the epilogue without the extra branch).
template <int CTAS, bool GATHER, bool SCALE>
__global__ void __launch_bounds__(GATHER ? NUM_THREADS_GATHER : NUM_THREADS, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmWgu,
                       const __grid_constant__ CUtensorMap tmH,
                       const __grid_constant__ CUtensorMap tmWd, Params p) {
    if (!p.release_late) pdl_release();  // the wait below follows this CTA's own set-up
    using C = Cfg<CTAS>;
    constexpr bool PAIR = C::PAIR;
    constexpr int STAGES = C::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);

    const uint32_t bar_full = base_s + C::OFF_BAR;         // [STAGES] (a pair uses the leader's)
    const uint32_t bar_empty = bar_full + 8 * STAGES;      // [STAGES]
    const uint32_t bar_tfull = bar_empty + 8 * STAGES;     // [2]
    const uint32_t bar_tempty = bar_tfull + 16;            // [2] (a pair uses the leader's)
    const uint32_t bar_drain = bar_tempty + 16;
    const uint32_t bar_gat = bar_drain + 8;                // [STAGES] (p.gather)
    volatile uint32_t *s_tmem = reinterpret_cast<volatile uint32_t *>(base + C::OFF_TMEM);
    volatile int *s_abort = reinterpret_cast<volatile int *>(base + C::OFF_ABORT);
    int *s_off = reinterpret_cast<int *>(base + C::OFF_OFFS);
    int *s_tile = reinterpret_cast<int *>(base + C::OFF_TILE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    const uint32_t rank = PAIR ? cluster_rank() : 0u;  // 0: the CTA that issues the MMAs
    const bool leader = rank == 0;
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int nunits = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    // barriers every load / epilogue signals (the leader's, in a pair)
    const uint32_t sig_full = PAIR ? map_to_rank(bar_full, 0) : bar_full;
    const uint32_t sig_tempty = PAIR ? map_to_rank(bar_tempty, 0) : bar_tempty;

    // ---- prologue: barriers and tensor memory, then (after the previous
    // kernel has completed) the row-tile prefix from `offsets` ----
    if (threadIdx.x == 0) {
        *s_abort = 0;
        // a stage is full when the leader's producer has armed it and its
        // bytes have landed; with GATHER, also once the reporting warp of
        // each CTA has seen its gathered rows land (bar_gat: one arrival per
        // gather thread) and reported them: a single CTA arrives, a pair
        // sends 16 bytes per CTA that count as transaction bytes
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(bar_full + 8 * i, GATHER && !PAIR ? 2 : 1);
            mbar_init(bar_empty + 8 * i, 1);
            mbar_init(bar_gat + 8 * i, 32 * kGatherWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_tfull + 8 * i, 1);
            mbar_init(bar_tempty + 8 * i, C::EPI_ARRIVALS);
        }
        mbar_init(bar_drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<CTAS>(base_s + C::OFF_TMEM, TMEM_COLS);
    if (!p.overlap_prev) pdl_wait();
    if (p.release_late) pdl_release();
    // through L2: with overlap_prev no grid-wide wait precedes this read
    for (int e = threadIdx.x; e <= E; e += (int)blockDim.x) s_off[e] = __ldcg(p.offsets + e);
    __syncthreads();
    if (warp == 2) {  // prefix over experts of their row tiles in this launch
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int local = 0;
        for (int e = e0; e < e1; ++e) local += expert_row_tiles(s_off[e + 1] - s_off[e], C::TILE_M, p.experts);
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        int run = incl - local;
        for (int e = e0; e < e1; ++e) {
            s_tile[e] = run;
            run += expert_row_tiles(s_off[e + 1] - s_off[e], C::TILE_M, p.experts);
        }
        if (lane == 31) s_tile[E] = incl;
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // both CTAs' barriers and tensor memory are ready
    tc_fence_after();

    const uint32_t tmem_base = *s_tmem;
    const int n1 = p.g1.n_tiles, n2 = p.g2.n_tiles;
    const int total1 = s_tile[E] * n1;
    const int total = total1 + s_tile[E] * n2;
    const int nk1 = (p.g1.K + BK - 1) / BK, nk2 = (p.g2.K + BK - 1) / BK;

    // The producer and the MMA issuer are single threads (lane 0 of warps 0
    // and 1): a warp-wide loop (a shuffle of each wait's result and a
    // reconvergence per K step) left the tensor pipe idle ~8 % of the time,
    // because the issuing thread keeps at most about one MMA queued ahead.
    if (warp == 0) {
        // ------------------------- TMA producer -------------------------
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0, last_par = 0;  // per stage armed here: ever / parity of last phase
            bool ok = true;
            for (int tile = unit; tile < total && ok; tile += nunits) {
                const TileInfo ti = decode_tile(tile, s_off, s_tile, E, total1, n1, n2, C::TILE_M);
                const CUtensorMap *tmA = ti.down ? &tmH : &tmX;
                const CUtensorMap *tmB = ti.down ? &tmWd : &tmWgu;
                // first B column of this CTA: in G1 the gate columns come first and the
                // up columns (offset f) follow; a pair splits them between its CTAs
                int n0;
                if (!ti.down) n0 = ti.n_blk * (BN / 2) + (PAIR && !leader ? p.f : 0);
                else n0 = ti.n_blk * BN + (int)rank * (BN / 2);
                const int arow = (p.a_local && !ti.down ? ti.row0 - s_off[ti.e] : ti.row0) +
                                 (int)rank * BM;
                const int nk = ti.down ? nk2 : nk1;
                for (int ks = 0; ks < nk; ++ks) {
                    if (!wait_bounded(bar_empty + 8 * s, ph ^ 1u, p.ds, s_abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = sig_full + 8 * s;
                    const int k0 = ks * BK;
                    const bool a_tma = !(GATHER && !ti.down);  // else the gather warps fill A
                    if (leader) {
                        mbar_arrive_expect_tx(bar_full + 8 * s,
                                              a_tma ? C::EXPECT_BYTES
                                                    : (C::B_BYTES + (PAIR ? 16 : 0)) * CTAS);
                        issued |= 1u << s;
                        last_par = (last_par & ~(1u << s)) | (ph << s);
                    }
                    if (a_tma) tma_load_2d<CTAS>(base_s + C::OFF_A + s * A_BYTES, tmA, k0, arow, fb);
                    const uint32_t bdst = base_s + C::OFF_B + s * C::B_BYTES;
                    if (p.b_blocks) {
                        // two atoms per box (weights viewed by 64-column blocks)
#pragma unroll
                        for (int a = 0; a < C::B_ATOMS; a += 2) {
                            int col = n0 + 64 * a;
                            if (!PAIR && !ti.down && a >= 2) col = ti.n_blk * (BN / 2) + p.f;
                            tma_load_4d<CTAS>(bdst + a * B_ATOM_BYTES, tmB, 0, k0, col >> 6, ti.e, fb);
                        }
                    } else
#pragma unroll
                    for (int a = 0; a < C::B_ATOMS; ++a) {
                        int col = n0 + 64 * a;
                        if (!PAIR && !ti.down && a >= 2) col = ti.n_blk * (BN / 2) + p.f + 64 * (a - 2);
                        tma_load_3d<CTAS>(bdst + a * B_ATOM_BYTES, tmB, col, k0, ti.e, fb);
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // drain: every phase armed here must have received all of its bytes
            if (leader) {
                for (int i = 0; i < STAGES; ++i)
                    if ((issued >> i) & 1u) {
                        volatile int never = 0;
                        if (!wait_bounded(bar_full + 8 * i, (last_par >> i) & 1u, p.ds, &never,
                                          drain_limit(p.ds)))
                            break;
                    }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------- MMA issuer ---------------------------
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            // Descriptors of stage 0, K step 0; a stage / K step only moves
            // the start address (bits 0-13, 16-byte units), so later ones are
            // adds.  A: K-major, 128-byte rows, 8-row groups 1024 B apart; a
            // K step of 16 elements is 32 bytes along the row.  B: MN-major,
            // 64-column atoms 8 KB apart (LBO), 8-row K groups 1024 B apart
            // (SBO); a K step of 16 rows is 2 KB.  In a pair the peer CTA's
            // operands sit at the same offsets in its shared memory.
            const uint64_t adesc0 = smem_desc_sw128(base_s + C::OFF_A, 16, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(base_s + C::OFF_B, B_ATOM_BYTES, 1024);
            if (p.ds.inject_wait_timeout) {
                // test hook: wait on the drain barrier, which nothing signals
                // before the issuer's own final commit, so the wait runs out
                // and the kernel takes its abort path before any MMA
                ok = wait_bounded(bar_drain, 0, p.ds, s_abort);
            }
            for (int tile = unit; tile < total && ok; tile += nunits, ++it) {
                const int acc = it & 1;
                const uint32_t aph = (uint32_t)(it >> 1) & 1u;
                const int nk = tile < total1 ? nk1 : nk2;
                if (!wait_bounded(bar_tempty + 8 * acc, aph ^ 1u, p.ds, s_abort)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int ks = 0; ks < nk; ++ks) {
                    // gathered A of a pair: the peer's rows are reported by
                    // its warps' cluster-scope arrivals
                    const bool full = PAIR && GATHER
                                          ? wait_bounded<true>(bar_full + 8 * s, ph, p.ds, s_abort)
                                          : wait_bounded(bar_full + 8 * s, ph, p.ds, s_abort);
                    if (!full) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_st = adesc0 + (uint64_t)((s * A_BYTES) >> 4);
                    const uint64_t b_st = bdesc0 + (uint64_t)((s * C::B_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        mma_bf16<CTAS>(d_tmem, a_st + (uint64_t)((kk * 32) >> 4),
                                       b_st + (uint64_t)((kk * 2048) >> 4), C::IDESC,
                                       (ks | kk) != 0 ? 1u : 0u);
                    mma_commit_all<CTAS>(bar_empty + 8 * s);  // frees the stage (both CTAs)
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_all<CTAS>(bar_tfull + 8 * acc);  // accumulators ready
            }
            // drain: every MMA issued here completes before tensor memory is freed
            mma_commit_local<CTAS>(bar_drain);
            volatile int never = 0;
            wait_bounded(bar_drain, 0, p.ds, &never, drain_limit(p.ds));
        }
        __syncwarp();
    } else if (warp < 6) {
        // --------------------------- epilogue ----------------------------
        const int quarter = warp & 3;  // tensor-memory lanes [32*quarter, 32*quarter + 32)
        const int r_in_tile = (int)rank * BM + quarter * 32 + lane;
        int it = 0;
        for (int tile = unit; tile < total; tile += nunits, ++it) {
            const TileInfo ti = decode_tile(tile, s_off, s_tile, E, total1, n1, n2, C::TILE_M);
            const bool sw = !ti.down;  // G1: SwiGLU of the gate and up halves
            __nv_bfloat16 *const out = sw ? p.g1.out : p.g2.out;
            const int n_out = sw ? p.g1.n_out : p.g2.n_out;
            const int transpose = sw ? p.g1.transpose_epi : p.g2.transpose_epi;
            const int acc = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            const int good = __all_sync(0xffffffffu,
                                        wait_bounded(bar_tfull + 8 * acc, aph, p.ds, s_abort));
            if (!good) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16);
            const bool row_ok = r_in_tile < ti.rows;
            __nv_bfloat16 *orow = out + (int64_t)(ti.row0 + r_in_tile) * n_out;
            float sc = 1.f;  // the row's weight (SCALE launches hold G1 tiles only)
            if constexpr (SCALE)
                if (row_ok) sc = __ldcg(p.row_scale + ti.row0 + r_in_tile);
            if (transpose) {
                // rows of this warp: ti.row0 + rank*BM + quarter*32 + (0..31)
                const int wrow0 = (int)rank * BM + quarter * 32;
                const int rows_valid = max(0, min(32, ti.rows - wrow0));
                const int64_t rbase = (int64_t)ti.row0 + wrow0;
                const int ncols = sw ? BN / 2 : BN;
                const int n0 = ti.n_blk * ncols;
#pragma unroll 1
                for (int c = 0; c < ncols; c += 64) {
                    uint32_t packed[32];
                    if (sw) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t g[32], u[32];
                            tmem_ld32(t_row + c + 32 * half, g);
                            tmem_ld32(t_row + BN / 2 + c + 32 * half, u);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                                float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
                                if constexpr (SCALE) {
                                    g0 *= sc;
                                    g1 *= sc;
                                    u0 *= sc;
                                    u1 *= sc;
                                }
                                __nv_bfloat162 b2 = __floats2bfloat162_rn(__fdividef(g0, 1.f + __expf(-g0)) * u0,
                                                                          __fdividef(g1, 1.f + __expf(-g1)) * u1);
                                packed[16 * half + i] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                        }
                    } else {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t y[32];
                            tmem_ld32(t_row + c + 32 * half, y);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(y[2 * i]),
                                                                          __uint_as_float(y[2 * i + 1]));
                                packed[16 * half + i] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                        }
                    }
                    store_rows_transposed(packed, out, rbase, rows_valid, n0 + c, n_out);
                }
            } else if (sw) {
                const int n0 = ti.n_blk * (BN / 2);
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 32) {
                    uint32_t g[32], u[32];
                    tmem_ld32(t_row + c, g);
                    tmem_ld32(t_row + BN / 2 + c, u);
                    tmem_ld_wait();
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                        float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
                        if constexpr (SCALE) {
                            g0 *= sc;
                            g1 *= sc;
                            u0 *= sc;
                            u1 *= sc;
                        }
                        float h0 = __fdividef(g0, 1.f + __expf(-g0)) * u0;
                        float h1 = __fdividef(g1, 1.f + __expf(-g1)) * u1;
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
                        packed[i] = *reinterpret_cast<uint32_t *>(&b2);
                    }
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int col = n0 + c + 8 * v;
                            if (col + 8 <= n_out)
                                stg16(orow + col, make_uint4(packed[4 * v], packed[4 * v + 1],
                                                             packed[4 * v + 2], packed[4 * v + 3]));
                        }
                    }
                }
            } else {
                const int n0 = ti.n_blk * BN;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t y[32];
                    tmem_ld32(t_row + c, y);
                    tmem_ld_wait();
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(y[2 * i]),
                                                                  __uint_as_float(y[2 * i + 1]));
                        packed[i] = *reinterpret_cast<uint32_t *>(&b2);
                    }
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int col = n0 + c + 8 * v;
                            if (col + 8 <= n_out)
                                stg16(orow + col, make_uint4(packed[4 * v], packed[4 * v + 1],
                                                             packed[4 * v + 2], packed[4 * v + 3]));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {  // the MMA issuer may reuse this accumulator
                if (PAIR) mbar_arrive_cluster(sig_tempty + 8 * acc);
                else mbar_arrive(bar_tempty + 8 * acc);
            }
        }
    } else if (GATHER && warp < 6 + kGatherWarps) {
        // --------------------- G1 A rows gathered (GATHER) ---------------------
        // Gather warp g fills rows [Rg, Rg + R) of this CTA's 128 A rows
        // (R = kGatherRows) in every stage: lane (j8 = lane / 8, c = lane % 8)
        // copies 16-byte chunk c of rows Rg + 4i + j8, each the K step's 64
        // columns of token row src_token[row], to where the TMA would put it
        // (row * 128 bytes, chunk c at (c ^ (row % 8)) * 16: the 128-byte
        // swizzle).  Rows past the tile's end are not copied; their
        // accumulator rows are never stored.  Every thread then has the
        // stage's bar_gat receive its arrival once its copies have landed,
        // and moves on: up to STAGES stages of copies are in flight.
        const int g = warp - 6;
        const int j8 = lane >> 3, c = lane & 7;
        const int K = p.g1.K;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int tile = unit; tile < total && ok; tile += nunits) {
            const TileInfo ti = decode_tile(tile, s_off, s_tile, E, total1, n1, n2, C::TILE_M);
            int64_t off[kGatherIters];  // element offset of this lane's chunk; -1: past the tile
#pragma unroll
            for (int i = 0; i < kGatherIters; ++i) {
                const int lr = kGatherRows * g + 4 * i + j8;  // row within this CTA's 128
                const int rt = (int)rank * BM + lr;           // row within the tile
                off[i] = rt < ti.rows ? (int64_t)__ldcg(p.src_token + ti.row0 + rt) * K + 8 * c : -1;
            }
            for (int ks = 0; ks < nk1; ++ks) {
                if (!__all_sync(0xffffffffu, wait_bounded(bar_empty + 8 * s, ph ^ 1u, p.ds, s_abort))) {
                    ok = false;
                    break;
                }
                const uint32_t dst = base_s + C::OFF_A + s * A_BYTES;
#pragma unroll
                for (int i = 0; i < kGatherIters; ++i) {
                    const int lr = kGatherRows * g + 4 * i + j8;
                    if (off[i] >= 0)
                        cp_async16(dst + lr * 128 + ((c ^ (lr & 7)) << 4), p.gx + off[i] + ks * BK);
                }
                cp_async_mbar_arrive_noinc(bar_gat + 8 * s);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        cp_async_wait_all();  // every copy lands before the shared memory is released
    } else if (GATHER) {
        // --------------- G1 gathered stages reported (GATHER) ----------------
        // Once a stage's gathered rows have landed (bar_gat), one thread
        // orders them before the tensor cores' reads (proxy fence) and
        // reports the stage on its full barrier: a single CTA arrives on its
        // own; a CTA of a pair copies 16 bytes of the stage into its slot in
        // the leader's shared memory, an async-proxy copy ordered after the
        // fence, whose completion counts as transaction bytes on the
        // leader's full barrier (an arrival with release at cluster scope,
        // once per stage, measured about twice as slow).
        const uint32_t slot = PAIR ? map_to_rank(base_s + C::OFF_SIGNAL + 16 * rank, 0) : 0u;
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int tile = unit; tile < total && ok; tile += nunits) {
                for (int ks = 0; ks < nk1; ++ks) {
                    if (!wait_bounded(bar_gat + 8 * s, ph, p.ds, s_abort)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_smem();
                    if (PAIR)
                        bulk_copy_to_cluster(slot, base_s + C::OFF_A + s * A_BYTES, 16,
                                             sig_full + 8 * s);
                    else
                        mbar_arrive(bar_full + 8 * s);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal it
    tc_fence_after();
    if (warp == 1) tmem_dealloc<CTAS>(tmem_base, TMEM_COLS);
    if (p.overlap_prev) pdl_wait();  // this grid completes only after the previous one
}

// ------------------------------ host side ----------------------------------
struct DeviceInfo {
    bool ready = false;
    int sms = 0;    // single CTAs that fit at once (one per SM)
    int pairs = 0;  // CTA pairs that fit at once
};

template <int CTAS>
cudaLaunchConfig_t launch_config(unsigned grid, cudaStream_t st, cudaLaunchAttribute *attr,
                                 int threads) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<CTAS>::SMEM_BYTES;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CTAS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_entry
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

template <int CTAS, bool GATHER, bool SCALE>
cudaError_t launch_variant(unsigned grid, const CUtensorMap &mx, const CUtensorMap &mwgu,
                           const CUtensorMap &mh, const CUtensorMap &mwd, const Params &p,
                           cudaStream_t st) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg =
        launch_config<CTAS>(grid, st, attr, GATHER ? NUM_THREADS_GATHER : NUM_THREADS);
    return cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel<CTAS, GATHER, SCALE>, mx, mwgu, mh, mwd,
                              p);
}

template <int CTAS>
cudaError_t launch(unsigned grid, const CUtensorMap &mx, const CUtensorMap &mwgu,
                   const CUtensorMap &mh, const CUtensorMap &mwd, const Params &p,
                   cudaStream_t st) {
    const bool scale = p.row_scale != nullptr;
    if (p.gather)
        return scale ? launch_variant<CTAS, true, true>(grid, mx, mwgu, mh, mwd, p, st)
                     : launch_variant<CTAS, true, false>(grid, mx, mwgu, mh, mwd, p, st);
    return scale ? launch_variant<CTAS, false, true>(grid, mx, mwgu, mh, mwd, p, st)
                 : launch_variant<CTAS, false, false>(grid, mx, mwgu, mh, mwd, p, st);
}

// Shared-memory opt-in and the clusters (or CTAs) resident at once for one
// instantiation; every instantiation fits one CTA per SM.
template <int CTAS, bool GATHER, bool SCALE> cudaError_t prepare_variant(int *resident_units) {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_tc_kernel<CTAS, GATHER, SCALE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Cfg<CTAS>::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg =
        launch_config<CTAS>(CTAS, nullptr, attr, GATHER ? NUM_THREADS_GATHER : NUM_THREADS);
    return cudaOccupancyMaxActiveClusters(resident_units,
                                          grouped_gemm_tc_kernel<CTAS, GATHER, SCALE>, &cfg);
}

// The resident count used for the grid is the smallest over the
// instantiations.
template <int CTAS> cudaError_t prepare(int *resident_units) {
    int n[4] = {0, 0, 0, 0};
    cudaError_t err;
    if ((err = prepare_variant<CTAS, false, false>(&n[0])) != cudaSuccess ||
        (err = prepare_variant<CTAS, false, true>(&n[1])) != cudaSuccess ||
        (err = prepare_variant<CTAS, true, false>(&n[2])) != cudaSuccess ||
        (err = prepare_variant<CTAS, true, true>(&n[3])) != cudaSuccess)
        return err;
    *resident_units = std::min(std::min(n[0], n[1]), std::min(n[2], n[3]));
    return cudaSuccess;
}

// Upper bound of the row tiles: sum_e ceil(count_e/TM) <= P/TM + min(E, P).
int64_t row_tiles_bound(const Shape &s, int tile_m) {
    const int64_t P = s.P();
    return (P + tile_m - 1) / tile_m + std::min<int64_t>(s.E, P);
}

// Tile shapes of a call.  Pairs when experts average >= 512 rows; 128-row
// single-CTA tiles for small per-expert batches (decode); in between, each
// expert goes to the shape that pads it less (pair_tiles_pay), in two
// launches per product.
enum TileMode { kModePairs, kModeHybrid, kModeSingles };
constexpr int kHybridRowsPerExpert = 64;  // below this average: single-CTA tiles only
TileMode tile_mode(const Shape &s) {
    if (s.P() >= (int64_t)kPairRowsPerExpert * s.E) return kModePairs;
    if (s.P() >= (int64_t)kHybridRowsPerExpert * s.E) return kModeHybrid;
    return kModeSingles;
}

// The launch of one product (G1: phase 1, G2: phase 2) over the experts
// `experts` selects, with one tile shape.
template <int CTAS>
cudaError_t launch_product(const Shape &s, int units, const CUtensorMap &mx,
                           const CUtensorMap &mwgu, const CUtensorMap &mh,
                           const CUtensorMap &mwd, const Params &both, int phase, int experts,
                           cudaStream_t st) {
    const int64_t row_tiles_max = row_tiles_bound(s, Cfg<CTAS>::TILE_M);
    Params p = both;
    p.experts = experts;
    if (phase == 1) p.g2.n_tiles = 0;
    else p.g1.n_tiles = 0;
    if (phase == 2) {
        p.gather = 0;  // G2's A (h_perm) is read by TMA
        p.row_scale = nullptr;
    }
    const int64_t n_tiles = phase == 1 ? both.g1.n_tiles : both.g2.n_tiles;
    const unsigned grid = CTAS * (unsigned)std::min<int64_t>(units, row_tiles_max * n_tiles);
    return launch<CTAS>(grid, mx, mwgu, mh, mwd, p, st);
}

// The hybrid sequence: pairs then single CTAs, per product.  The single-CTA
// launch serves other experts than the pair launch before it, so it overlaps
// that launch's last partial round (see Params::overlap_prev); the pair
// launch releases it only once every earlier kernel has completed.
template <int CTAS>
cudaError_t launch_product_ordered(const Shape &s, int units, const CUtensorMap &mx,
                                   const CUtensorMap &mwgu, const CUtensorMap &mh,
                                   const CUtensorMap &mwd, Params both, int phase, int experts,
                                   int release_late, int overlap_prev, cudaStream_t st) {
    both.release_late = release_late;
    both.overlap_prev = overlap_prev;
    return launch_product<CTAS>(s, units, mx, mwgu, mh, mwd, both, phase, experts, st);
}

}  // namespace tc

int grouped_swiglu_tc_launches(const Shape &s) {
    return tc::tile_mode(s) == tc::kModeHybrid ? 4 : 2;
}

// The row gather needs whole 64-column K steps.
bool grouped_swiglu_tc_gathers(const Shape &s) { return s.d % tc::BK == 0; }

// Gathering G1's rows saves the permuted copy of x (written once, read once)
// and costs the gather kernel's throughput (its extra warps hold the block's
// registers to 168 a thread, and its copies share the SM's intake with the
// weight tiles).  The saving per FLOP falls as 1/f.  Measured against the
// copying path: the Qwen3-30B-A3B shape (f = 768) 3-7 % faster, the
// DeepSeek-V3 shape (f = 2048) 1.4-2.7 %, gpt-oss (f = 2880) 0.9 % in short
// runs at full clock and 0.1-0.4 % slower under the power cap, the Mixtral
// shape (f = 14336) 1.3-4 % slower.
constexpr int kGatherMaxF = 3072;
bool grouped_swiglu_tc_gather_pays(const Shape &s) {
    return grouped_swiglu_tc_gathers(s) && s.f <= kGatherMaxF;
}

cudaError_t launch_grouped_swiglu_tc(const Shape &s, const void *x_perm, const int32_t *offsets,
                                     const void *Wgu, const void *Wd, void *h_perm, void *y_perm,
                                     const DevStatus &ds, cudaStream_t st, bool a_local,
                                     const int32_t *src_token, const float *row_scale) {
    using namespace tc;
    static DeviceInfo info[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!info[dev].ready) {
        int a = 0, c = 0;
        if ((err = prepare<1>(&a)) != cudaSuccess || (err = prepare<2>(&c)) != cudaSuccess)
            return err;
        info[dev].sms = a;
        info[dev].pairs = c;
        if (info[dev].sms < 1 || info[dev].pairs < 1) {
            set_error_message("the grouped GEMM does not fit on device %d", dev);
            return cudaErrorInvalidConfiguration;
        }
        info[dev].ready = true;
    }
    if (!tensor_map_encoder()) {
        set_error_message("cuTensorMapEncodeTiled is not available from the driver");
        return cudaErrorNotSupported;
    }
    const int64_t P = s.P();
    CUtensorMap mx, mwgu, mh, mwd;
    // whole 64-column blocks in both products (gate, up and down columns):
    // B boxes of two atoms; else one atom per box
    const bool blocks = s.f % 64 == 0 && s.d % 64 == 0;
    const bool maps_ok =
        blocks ? tensor_map_weight_blocks(&mwgu, Wgu, s.E, s.d, 2 * (int64_t)s.f, 2) &&
                     tensor_map_weight_blocks(&mwd, Wd, s.E, s.f, s.d, 2)
               : tensor_map_weights(&mwgu, Wgu, s.E, s.d, 2 * (int64_t)s.f) &&
                     tensor_map_weights(&mwd, Wd, s.E, s.f, s.d);
    // gather (src_token given): x_perm is the T token rows, G1's A rows are
    // gathered from them; d must be whole 64-column K steps
    const bool gather = src_token != nullptr;
    if (gather && (a_local || !grouped_swiglu_tc_gathers(s))) {
        set_error_message("the row gather needs d a multiple of %d and no local rows", BK);
        return cudaErrorInvalidValue;
    }
    // a_local: G1's A is the T token rows themselves
    if (!maps_ok || !tensor_map_rows(&mx, x_perm, a_local || gather ? s.T : P, s.d, BM) ||
        !tensor_map_rows(&mh, h_perm, P, s.f, BM)) {
        set_error_message("cuTensorMapEncodeTiled rejected an operand (alignment or size)");
        return cudaErrorInvalidValue;
    }
    const int64_t n_tiles1 = (s.f + BN / 2 - 1) / (BN / 2), n_tiles2 = (s.d + BN - 1) / BN;
    if (row_tiles_bound(s, BM) * (n_tiles1 + n_tiles2) >= (int64_t)INT32_MAX) {
        set_error_message("grouped GEMM tile count exceeds 2^31");
        return cudaErrorInvalidValue;
    }
    Params p;
    p.offsets = offsets;
    p.E = s.E;
    p.f = s.f;
    p.g1.K = s.d;
    p.g1.n_out = s.f;
    p.g1.n_tiles = (int)n_tiles1;
    p.g1.transpose_epi = s.d <= kTransposeMaxK;
    p.g1.out = static_cast<__nv_bfloat16 *>(h_perm);
    p.g2.K = s.f;
    p.g2.n_out = s.d;
    p.g2.n_tiles = (int)n_tiles2;
    p.g2.transpose_epi = s.f <= kTransposeMaxK;
    p.g2.out = static_cast<__nv_bfloat16 *>(y_perm);
    p.experts = kAllExperts;
    p.release_late = 0;
    p.overlap_prev = 0;
    p.b_blocks = blocks ? 1 : 0;
    p.a_local = a_local ? 1 : 0;
    p.gather = gather ? 1 : 0;
    p.gx = static_cast<const __nv_bfloat16 *>(x_perm);
    p.src_token = src_token;
    p.row_scale = row_scale;
    p.ds = ds;
    // G1 launches, then G2 launches (G2 reads h_perm; stream order)
    const TileMode mode = tile_mode(s);
    const int pairs = info[dev].pairs, sms = info[dev].sms;
    for (int phase = 1; phase <= 2; ++phase) {
        if (mode == kModePairs)
            err = launch_product<2>(s, pairs, mx, mwgu, mh, mwd, p, phase, kAllExperts, st);
        else if (mode == kModeSingles)
            err = launch_product<1>(s, sms, mx, mwgu, mh, mwd, p, phase, kAllExperts, st);
        else if ((err = launch_product_ordered<2>(s, pairs, mx, mwgu, mh, mwd, p, phase, kPairExperts,
                                                  1, 0, st)) == cudaSuccess)
            err = launch_product_ordered<1>(s, sms, mx, mwgu, mh, mwd, p, phase, kSingleExperts, 0, 1,
                                            st);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace moe
