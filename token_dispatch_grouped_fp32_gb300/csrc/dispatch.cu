// dispatch.cu -- token dispatch on one device: per-expert histogram, exclusive
// scan, stable scatter into expert-contiguous order, and the row gather, in
// two launches (one for a standalone dispatch of few experts and pairs).
//
// Transformers docs "Expert parallelism", section "Token dispatch": every
// (token, expert) pair is sent to its expert and the experts run on the rows
// they receive.  On one GPU "sending" is a permutation: pair (t, j) gets row
// pos[t*k+j] of its expert's segment, segments laid out in expert order.
//
// Launch 1 (rank_kernel), one block per chunk of consecutive pair ids: the
// block counts its chunk's pairs per expert, writes that column of the
// expert-major [E][chunks] count matrix, and gives every pair its rank among
// the chunk's pairs of the same expert (warps rank their pairs with
// __match_any_sync in pair order, after the counts of the warps before
// them).  The last block to finish (a ticket counter) scans the matrix into
// the first row of every (expert, chunk), which also yields counts and
// offsets, and resets the ticket for the next call.
// Launch 2 (place_rows_kernel), one warp per pair: row = first row of the
// pair's (expert, chunk) + its rank; writes pos, src_token and copies the
// token's row into x_perm.  A standalone dispatch with unscaled rows of k KB
// to 16 KB uses place_token_rows_kernel instead, a warp per token, which
// reads the token's row while launch 1 still runs.  Without x_perm (the
// experts gather the rows), place_index_kernel does the lookup alone, a
// thread per pair.  A dispatch with E <= 16 and P <= 16384 that copies
// unscaled rows of k KB to 16 KB runs as one launch instead,
// dispatch_one_launch_kernel, whose blocks each count every id.
// Stability: rows of one expert are in ascending pair id, hence ascending
// token id, and no atomic decides any order.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;      // place_rows_kernel
constexpr int kWarps = kThreads / 32;
constexpr int kTokWarps = 4;              // place_token_rows_kernel: tokens per block
constexpr int kStageRowMax = 16 * 1024;   // its largest row, staged in shared memory
constexpr int kRankThreads = 1024;  // rank_kernel for chunks of 2048 pairs and more
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kSmallRankThreads = 256;  // rank_kernel for chunks of 256 pairs
// The count matrix is staged in shared memory for the scan when it has at
// most this many entries (else the scan reads it through L2).
constexpr int kScanStageMax = 16 * 1024;
// rank_kernel packs a pair's expert id and its rank in its chunk into one
// int: (e << kRankBits) | rank.  E <= 1024 needs 10 bits; a chunk holds at
// most 2^21 pairs (P < 2^31 in at most 1024 chunks), so its ranks fit 21.
constexpr int kRankBits = 21;
constexpr int kRankMask = (1 << kRankBits) - 1;

// Exclusive scan, in place, of the expert-major count matrix hist[0 .. E*NB)
// by one block of NT threads: afterwards hist[e*NB + b] is the first row
// of expert e's pairs in chunk b, counts[e] and offsets[0..E] follow.  The
// matrix was written by other blocks of the grid, so it is read through L2;
// `stage` (shared memory for kScanStageMax ints, or nullptr) holds a copy
// while it is scanned, so the per-thread walks read shared memory.
template <int NT>
__device__ void scan_count_matrix(int32_t *__restrict__ hist_g, int E, int NB,
                                  int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                  int *stage) {
    constexpr int NW = NT / 32;
    __shared__ int warp_tot[NW];
    __shared__ int total_s;
    const int n = E * NB;
    int32_t *hist = hist_g;
    if (stage != nullptr) {
        for (int i = threadIdx.x; i < n; i += NT) stage[i] = __ldcg(hist_g + i);
        __syncthreads();
        hist = stage;
    }
    const int seg = (n + NT - 1) / NT;
    const int beg = min(n, (int)threadIdx.x * seg);
    const int end = min(n, beg + seg);
    int local = 0;
    for (int i = beg; i < end; ++i) local += stage != nullptr ? hist[i] : __ldcg(hist + i);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int v = lane < NW ? warp_tot[lane] : 0;
        int inc = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += u;
        }
        if (lane < NW) warp_tot[lane] = inc - v;  // exclusive warp base
        if (lane == 31) total_s = inc;
    }
    __syncthreads();
    int run = warp_tot[wid] + incl - local;
    for (int i = beg; i < end; ++i) {
        const int c = stage != nullptr ? hist[i] : __ldcg(hist + i);
        hist[i] = run;
        run += c;
    }
    __syncthreads();  // the block's writes above are visible to the block
    if (stage != nullptr)
        for (int i = threadIdx.x; i < n; i += NT) hist_g[i] = stage[i];
    const int total = total_s;
    for (int e = threadIdx.x; e < E; e += NT) {
        const int b0 = hist[e * NB];
        const int b1 = (e + 1 < E) ? hist[(e + 1) * NB] : total;
        offsets[e] = b0;
        counts[e] = b1 - b0;
    }
    if (threadIdx.x == 0) offsets[E] = total;
}

// Launch 1: chunk b = pairs [b*chunk, (b+1)*chunk); warp w of the block ranks
// the sub-range [q0 + w*sub, q0 + (w+1)*sub).  Writes hist[e*NB + b] (the
// chunk's count of expert e) and packed[q] = (e << kRankBits) | (the pair's
// rank among the chunk's pairs of expert e), or -1 for an expert id outside
// [0, E), which is reported and dropped.  The ticket must be 0 when the
// launch starts; the last block leaves it 0.  Dynamic shared memory:
// max(NT / 32 * E, staged count matrix) ints.
template <int NT>
__global__ void __launch_bounds__(NT)
rank_kernel(const int32_t *__restrict__ idx, int64_t P, int E, int chunk, int NB, int staged,
            int32_t *__restrict__ hist, int32_t *__restrict__ packed,
            int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
            unsigned *__restrict__ ticket, DevStatus ds) {
    pdl_entry();
    constexpr int NW = NT / 32;
    extern __shared__ int sh_warp[];  // [NW][E]: per-warp counts, then first ranks
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < NW * E; i += NT) sh_warp[i] = 0;
    __syncthreads();
    const int sub = (chunk + NW - 1) / NW;
    const int64_t cend = min((int64_t)(blockIdx.x + 1) * chunk, P);
    const int64_t w0 = min((int64_t)blockIdx.x * chunk + (int64_t)wid * sub, cend);
    const int64_t w1 = min(w0 + sub, cend);
    int *mine = sh_warp + wid * E;
#pragma unroll 4  // independent iterations: several index loads in flight
    for (int64_t q = w0 + lane; q < w1; q += 32) {
        const int e = idx[q];
        if ((unsigned)e < (unsigned)E)
            atomicAdd(&mine[e], 1);
        else
            raise_error(ds, kErrBadRouting);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += NT) {
        int run = 0;
        for (int w = 0; w < NW; ++w) {
            const int c = sh_warp[w * E + e];
            sh_warp[w * E + e] = run;
            run += c;
        }
        hist[(int64_t)e * NB + blockIdx.x] = run;
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
        const int before = __popc(peers & lt_mask);
        const int r0 = (e >= 0) ? mine[e] : 0;
        __syncwarp();
        if (q < w1) {
            packed[q] = (e >= 0) ? ((e << kRankBits) | (r0 + before)) : -1;
            if (e >= 0 && lane == 31 - __clz(peers)) mine[e] = r0 + __popc(peers);
        }
        __syncwarp();
    }
    // The last block to get here scans the count matrix.  Every thread makes
    // its count-matrix writes visible device-wide before the block takes its
    // ticket; the last block fences again before reading the others'.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1u) == (unsigned)NB - 1u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    scan_count_matrix<NT>(hist, E, NB, counts, offsets, staged ? sh_warp : nullptr);
    if (threadIdx.x == 0) *ticket = 0u;  // ready for the next call (stream order)
}

// Launch 2: one warp per pair q.  Its row is the first row of its (expert,
// chunk) plus its rank; lane 0 writes pos[q] and src_token[row], and the warp
// copies the token's row into x_perm (16-byte vectors; with SCALE, each
// element times the pair's weight, formed in fp32 and rounded once).  The
// source row is known at once, so the first vectors of the row are loaded
// before the row lookup (packed rank, then the base), whose latency they
// overlap.
template <typename TA, bool SCALE>
__global__ void __launch_bounds__(kThreads)
place_rows_kernel(const TA *__restrict__ x, const int32_t *__restrict__ hist,
                  const float *__restrict__ scale, int64_t P, int k, int d, int chunk, int NB,
                  int32_t *__restrict__ pos, int32_t *__restrict__ src_token,
                  TA *__restrict__ x_perm) {
    pdl_entry();
    constexpr int EPV = 16 / sizeof(TA);
    constexpr int U = 4;  // vectors per lane per round
    const int lane = threadIdx.x & 31;
    const int64_t q = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (q >= P) return;  // warp-uniform
    const int64_t t = q / k;
    const int nvec = x_perm != nullptr ? d / EPV : 0;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + t * d);
    uint4 first[U];  // round 0 of the copy, in flight during the lookup
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (lane + 32 * u < nvec) first[u] = ldg16(src + lane + 32 * u);
    const int v = pos[q];  // (expert << kRankBits) | rank, from launch 1
    if (v < 0) return;     // dropped pair: pos stays -1
    const int row = hist[(int64_t)(v >> kRankBits) * NB + (int)(q / chunk)] + (v & kRankMask);
    __syncwarp();  // every lane has read pos[q] before lane 0 overwrites it
    if (lane == 0) {
        pos[q] = row;
        src_token[row] = (int32_t)t;
    }
    if (nvec == 0) return;
    uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (int64_t)row * d);
    float wq = 1.f;
    if (SCALE) wq = scale[q];
    auto put = [&](int i, const uint4 &val) {
        if (SCALE) {
            float f[EPV];
            unpack16(val, f, static_cast<const TA *>(nullptr));
#pragma unroll
            for (int j = 0; j < EPV; ++j) f[j] *= wq;
            stg16(dst + i, pack16(f, static_cast<const TA *>(nullptr)));
        } else {
            stg16(dst + i, val);
        }
    };
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (lane + 32 * u < nvec) put(lane + 32 * u, first[u]);
    for (int i0 = 32 * U; i0 < nvec; i0 += 32 * U) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i0 + lane + 32 * u < nvec) buf[u] = ldg16(src + i0 + lane + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i0 + lane + 32 * u < nvec) put(i0 + lane + 32 * u, buf[u]);
    }
}

// Launch 2 of a standalone dispatch with rows copied unscaled: one warp per
// token t.  The warp copies x's row t into shared memory (cp.async) before
// it waits for launch 1, so the read overlaps the ranking.  The read is
// ordered after every earlier write of x: launch 1 follows the ticket's
// memset, so it starts only once all earlier work in the stream has
// completed; this grid starts only once every block of launch 1 has started;
// and neither launch writes x.  After
// the wait, lane j looks up pair (t, j)'s row and writes pos and src_token,
// and the warp writes the staged row to each of the token's rows of x_perm.
template <typename TA>
__global__ void __launch_bounds__(32 * kTokWarps)
place_token_rows_kernel(const TA *__restrict__ x, const int32_t *__restrict__ hist, int64_t T,
                        int k, int d, int chunk, int NB, int32_t *__restrict__ pos,
                        int32_t *__restrict__ src_token, TA *__restrict__ x_perm) {
    extern __shared__ __align__(16) unsigned char stage_raw[];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * kTokWarps + wid;
    const int nvec = d * (int)sizeof(TA) / 16;
    const uint4 *buf = reinterpret_cast<const uint4 *>(stage_raw) + (int64_t)wid * nvec;
    if (t < T) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + t * d);
        for (int i = lane; i < nvec; i += 32) tc::cp_async16(tc::smem_u32(buf + i), src + i);
        tc::cp_async_commit();
    }
    pdl_entry();
    if (t >= T) return;  // warp-uniform
    bool staged = false;
    for (int j0 = 0; j0 < k; j0 += 32) {
        int row = -1;
        if (j0 + lane < k) {
            const int64_t q = t * k + j0 + lane;
            const int v = pos[q];  // (expert << kRankBits) | rank, from launch 1
            if (v >= 0) {          // else a dropped pair: pos stays -1
                row = hist[(int64_t)(v >> kRankBits) * NB + (int)(q / chunk)] + (v & kRankMask);
                pos[q] = row;
                src_token[row] = (int32_t)t;
            }
        }
        if (!staged) {  // each lane reads back only the vectors it copied
            tc::cp_async_wait_all();
            staged = true;
        }
        const int nj = min(32, k - j0);
        for (int jj = 0; jj < nj; ++jj) {
            const int r = __shfl_sync(0xffffffffu, row, jj);
            if (r < 0) continue;  // warp-uniform
            uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (int64_t)r * d);
#pragma unroll 4
            for (int i = lane; i < nvec; i += 32) stg16(dst + i, buf[i]);
        }
    }
}

// A dispatch with few experts and few pairs in ONE launch (the limits
// below; rows unscaled, of k KB to 16 KB).  Block b owns the contiguous
// tokens [b*T/G, (b+1)*T/G) of a grid of G = min(SMs, T) blocks, one warp
// per token (up to 32 warps; a warp takes a further token each round when
// the block owns more tokens than its warps).  Each warp first copies its
// token row into shared memory with cp.async, so the reads of all the
// block's rows (27 rows of 8 KB each on the Mixtral layer's shape) overlap
// the ranking.  Every block then reads all P expert ids (at most 64 KB, L2
// hits after the first block) and counts them per expert in two parts: the
// pairs before its first pair, and the rest.  The totals give counts and
// offsets; the first part gives the row at which the block's pairs of each
// expert start.  So no block waits for another, and no count matrix or
// ticket is needed.  Per-thread counts are 8-bit fields of two 64-bit words
// (experts 0-7 and 8-15); the launcher checks that no thread sees more than
// 255 ids.  The block's pairs are then ranked in pair order (a warp's 32
// pairs with __match_any_sync, after the warps before it, as rank_kernel
// does) and each staged row is written to its k rows.
// Standalone (STAGE_FIRST), the launch carries no programmatic-serialisation
// attribute, so it starts only after all earlier work in the stream has
// completed (x and the ids included), and the rows are staged at once; its
// pdl_entry() then only lets a following kernel be scheduled.  Inside
// moe_forward it is launched like the layer's other kernels and stages
// nothing before its wait (x may be the output of a kernel still running).
constexpr int kOneMaxE = 16;
constexpr int kOneMaxP = 16384;
constexpr int kOneMaxWarps = 32;            // per block: a warp per token
constexpr int kOneStageBytes = 216 * 1024;  // staged rows per block
constexpr int kOneBlockPairs = 1024;        // pairs one block may own

template <typename TA, bool STAGE_FIRST>
__global__ void __launch_bounds__(32 * kOneMaxWarps)
dispatch_one_launch_kernel(const int32_t *__restrict__ idx, const TA *__restrict__ x, int64_t T,
                           int k, int E, int d, int32_t *__restrict__ counts,
                           int32_t *__restrict__ offsets, int32_t *__restrict__ pos,
                           int32_t *__restrict__ src_token, TA *__restrict__ x_perm,
                           DevStatus ds) {
    extern __shared__ __align__(16) unsigned char stage_raw[];
    __shared__ int s_part[kOneMaxWarps][kOneMaxE];  // per-warp counts (before, then rank bases)
    __shared__ int s_all[kOneMaxWarps][kOneMaxE];   // per-warp counts of all pairs
    __shared__ int s_base[kOneMaxE];                // next row of each expert in this block
    __shared__ int s_pair[kOneBlockPairs];          // the block's expert ids, then their rows
    const int nthr = blockDim.x, nw = nthr >> 5;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * T / gridDim.x;
    const int64_t t1 = (int64_t)(blockIdx.x + 1) * T / gridDim.x;
    const int64_t P = T * k, p0 = t0 * k, p1 = t1 * k;
    const int nvec = d * (int)sizeof(TA) / 16;
    uint4 *buf = reinterpret_cast<uint4 *>(stage_raw) + (int64_t)wid * nvec;
    auto stage = [&](int64_t t) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + t * d);
        for (int i = lane; i < nvec; i += 32) tc::cp_async16(tc::smem_u32(buf + i), src + i);
        tc::cp_async_commit();
    };
    if (STAGE_FIRST && t0 + wid < t1) stage(t0 + wid);
    pdl_entry();
    if (!STAGE_FIRST && t0 + wid < t1) stage(t0 + wid);

    // 8-bit field e & 7 of word lo (e < 8) or hi (8 <= e < 16); other ids add 0
    auto field = [E](int e) -> uint64_t {
        return (unsigned)e < (unsigned)E ? 1ull << ((e & 7) << 3) : 0ull;
    };
    uint64_t pre_lo = 0, pre_hi = 0, rest_lo = 0, rest_hi = 0;
    auto tally = [&](int64_t i, int e) {
        const uint64_t inc = field(e);
        const uint64_t lo = e < 8 ? inc : 0ull, hi = e < 8 ? 0ull : inc;
        if (i < p0) {
            pre_lo += lo;
            pre_hi += hi;
        } else {
            rest_lo += lo;
            rest_hi += hi;
            if (i < p1) s_pair[i - p0] = e;  // the block's own pairs, for the ranking
        }
    };
    int64_t scalar_from = 0;
    if ((reinterpret_cast<uintptr_t>(idx) & 15u) == 0) {  // 16-byte loads of four ids
        const int64_t nv = P >> 2;
        const int4 *v4 = reinterpret_cast<const int4 *>(idx);
#pragma unroll 4
        for (int64_t v = threadIdx.x; v < nv; v += nthr) {
            const int4 e4 = v4[v];
            tally(4 * v, e4.x);
            tally(4 * v + 1, e4.y);
            tally(4 * v + 2, e4.z);
            tally(4 * v + 3, e4.w);
        }
        scalar_from = nv << 2;
    }
    for (int64_t i = scalar_from + threadIdx.x; i < P; i += nthr) tally(i, idx[i]);
    for (int e = 0; e < E; ++e) {
        const int sh = (e & 7) << 3;
        const unsigned pv = (unsigned)(((e < 8 ? pre_lo : pre_hi) >> sh) & 255u);
        const unsigned rv = (unsigned)(((e < 8 ? rest_lo : rest_hi) >> sh) & 255u);
        const int ps = (int)__reduce_add_sync(0xffffffffu, pv);
        const int rs = (int)__reduce_add_sync(0xffffffffu, rv);
        if (lane == 0) {
            s_part[wid][e] = ps;
            s_all[wid][e] = ps + rs;
        }
    }
    __syncthreads();
    if (wid == 0) {  // lane e: expert e's total, its offset and the block's first row
        int tot = 0, pre = 0;
        if (lane < E)
            for (int w = 0; w < nw; ++w) {
                tot += s_all[w][lane];
                pre += s_part[w][lane];
            }
        int incl = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);  // lanes >= E add 0
        if (lane < E) s_base[lane] = incl - tot + pre;
        if (blockIdx.x == 0) {
            if (lane < E) {
                counts[lane] = tot;
                offsets[lane] = incl - tot;
            }
            if (lane == 0) offsets[E] = total;
        }
    }
    __syncthreads();

    // Rank the block's pairs [p0, p1) in pair order, nthr at a time.
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int64_t qb = p0; qb < p1; qb += nthr) {
        const int64_t q = qb + threadIdx.x;
        int e = -1;
        if (q < p1) {
            e = s_pair[q - p0];
            if ((unsigned)e >= (unsigned)E) {
                raise_error(ds, kErrBadRouting);  // the pair is dropped
                e = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int before = __popc(peers & lt_mask);
        if (lane < E) s_part[wid][lane] = 0;
        __syncwarp();
        if (e >= 0 && lane == 31 - __clz(peers)) s_part[wid][e] = __popc(peers);
        __syncthreads();
        if (threadIdx.x < E) {  // per expert: the warps' bases, in warp order
            int run = s_base[threadIdx.x];
            for (int w = 0; w < nw; ++w) {
                const int c = s_part[w][threadIdx.x];
                s_part[w][threadIdx.x] = run;
                run += c;
            }
            s_base[threadIdx.x] = run;
        }
        __syncthreads();
        if (q < p1) {
            const int row = e >= 0 ? s_part[wid][e] + before : -1;
            s_pair[q - p0] = row;  // this thread alone read that entry
            pos[q] = row;
            if (row >= 0) src_token[row] = (int32_t)(q / k);
        }
        __syncthreads();  // the rows are complete; s_part may be reused
    }

    // Each warp writes its staged token rows to their k rows of x_perm.  A
    // lane reads back only the vectors it staged, so the next token's
    // cp.async into the same buffer follows that lane's own reads.
    for (int64_t t = t0 + wid; t < t1; t += nw) {
        if (t != t0 + wid) stage(t);
        tc::cp_async_wait_all();
        const int b = (int)((t - t0) * k);
        for (int j = 0; j < k; ++j) {
            const int r = s_pair[b + j];
            if (r < 0) continue;  // warp-uniform: a dropped pair
            uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (int64_t)r * d);
#pragma unroll 4
            for (int i = lane; i < nvec; i += 32) stg16(dst + i, buf[i]);
        }
    }
}

// Launch 2 when no row moves (x_perm == nullptr: the experts gather the rows
// themselves): a thread per pair, the same row lookup as place_rows_kernel.
// With row_scale, also row_scale[row] = w[q] (the weight the experts apply
// to the row's products).
__global__ void __launch_bounds__(kThreads)
place_index_kernel(const int32_t *__restrict__ hist, int64_t P, int k, int chunk, int NB,
                   int32_t *__restrict__ pos, int32_t *__restrict__ src_token,
                   const float *__restrict__ w, float *__restrict__ row_scale) {
    pdl_entry();
    const int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (q >= P) return;
    const int v = pos[q];  // (expert << kRankBits) | rank, from launch 1
    if (v < 0) return;     // dropped pair: pos stays -1
    const int row = hist[(int64_t)(v >> kRankBits) * NB + (int)(q / chunk)] + (v & kRankMask);
    pos[q] = row;
    src_token[row] = (int32_t)(q / k);
    if (row_scale != nullptr) row_scale[row] = w[q];
}

// Every token picks every expert (k == E), each once, so expert e's segment
// is the T tokens in order: the row of pair q = (t, j) is idx[q] * T + t.
__global__ void __launch_bounds__(kThreads)
dispatch_all_experts_kernel(const int32_t *__restrict__ idx, int64_t T, int E,
                            int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                            int32_t *__restrict__ pos, int32_t *__restrict__ src_token,
                            const float *__restrict__ w, float *__restrict__ row_scale,
                            DevStatus ds) {
    pdl_entry();
    const int64_t P = T * E;
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += kThreads) {
            offsets[e] = (int32_t)(e * T);
            if (e < E) counts[e] = (int32_t)T;
        }
    }
    for (int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x; q < P;
         q += (int64_t)gridDim.x * kThreads) {
        const int e = idx[q];
        const int64_t t = q / E;
        if ((unsigned)e >= (unsigned)E) {
            raise_error(ds, kErrBadRouting);
            pos[q] = -1;
            continue;
        }
        const int64_t row = (int64_t)e * T + t;
        pos[q] = (int32_t)row;
        src_token[row] = (int32_t)t;
        if (row_scale != nullptr) row_scale[row] = w[q];
    }
}

// place_token_rows_kernel with up to kTokWarps x 16 KB of shared memory; the
// carveout favours shared memory, since the kernel uses no L1 caching.
template <typename TA>
cudaError_t launch_token_rows(const void *x, const int32_t *hist, const Shape &s,
                              const DispatchGrid &g, int32_t *pos, int32_t *src_token,
                              void *x_perm, unsigned blocks, size_t smem, cudaStream_t st) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        if ((err = cudaFuncSetAttribute(place_token_rows_kernel<TA>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kTokWarps * kStageRowMax)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(place_token_rows_kernel<TA>,
                                        cudaFuncAttributePreferredSharedMemoryCarveout,
                                        (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return err;
        attr_set[dev] = true;
    }
    launch_pdl(place_token_rows_kernel<TA>, dim3(blocks), dim3(32 * kTokWarps), smem, st,
               static_cast<const TA *>(x), hist, s.T, s.k, s.d, g.chunk, g.blocks, pos, src_token,
               static_cast<TA *>(x_perm));
    return cudaGetLastError();
}

// dispatch_one_launch_kernel where dispatch_fits_one_launch(s), the block
// count leaves at most kOneBlockPairs pairs per block and no thread counts
// more than 255 ids (both hold on a GPU of up to 1024 SMs).  *launched says
// whether it launched; otherwise it returns cudaSuccess.
template <typename TA>
cudaError_t launch_dispatch_one(const Shape &s, const int32_t *idx, const void *x,
                                int32_t *counts, int32_t *offsets, int32_t *pos,
                                int32_t *src_token, void *x_perm, const DevStatus &ds,
                                cudaStream_t st, bool in_forward, bool *launched) {
    *launched = false;
    static bool attr_set[64] = {};
    static int sms[64] = {};
    const int64_t row_bytes = (int64_t)s.d * (int64_t)sizeof(TA);
    if (!dispatch_fits_one_launch(s)) return cudaSuccess;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        if ((err = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev)) !=
                cudaSuccess ||
            (err = cudaFuncSetAttribute(dispatch_one_launch_kernel<TA, true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kOneStageBytes)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(dispatch_one_launch_kernel<TA, false>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kOneStageBytes)) != cudaSuccess)
            return err;
        attr_set[dev] = true;
    }
    const int64_t P = s.P();
    const int64_t blocks = std::min<int64_t>(sms[dev], s.T);
    const int64_t tok = (s.T + blocks - 1) / blocks;  // most tokens a block owns
    const int nw = (int)std::min<int64_t>(std::min<int64_t>(kOneMaxWarps, tok),
                                          kOneStageBytes / row_bytes);
    const int64_t nthr = 32 * (int64_t)nw;
    if (blocks < 1 || tok * s.k > kOneBlockPairs || (P + nthr - 1) / nthr + 5 > 255)
        return cudaSuccess;
    *launched = true;
    const size_t smem = (size_t)nw * (size_t)row_bytes;
    if (in_forward)
        launch_pdl(dispatch_one_launch_kernel<TA, false>, dim3((unsigned)blocks), dim3(32 * nw),
                   smem, st, idx, static_cast<const TA *>(x), s.T, s.k, s.E, s.d, counts,
                   offsets, pos, src_token, static_cast<TA *>(x_perm), ds);
    else
        dispatch_one_launch_kernel<TA, true><<<(unsigned)blocks, 32 * nw, smem, st>>>(
            idx, static_cast<const TA *>(x), s.T, s.k, s.E, s.d, counts, offsets, pos, src_token,
            static_cast<TA *>(x_perm), ds);
    return cudaGetLastError();
}

}  // namespace

bool dispatch_fits_one_launch(const Shape &s) {
    const int64_t row_bytes = (int64_t)s.d * (s.bf16 ? 2 : 4);
    return s.E <= kOneMaxE && s.P() <= kOneMaxP && row_bytes <= kStageRowMax &&
           (int64_t)s.k * 1024 <= row_bytes;
}

cudaError_t launch_dispatch_all_experts(const Shape &s, const int32_t *idx, int32_t *counts,
                                        int32_t *offsets, int32_t *pos, int32_t *src_token,
                                        const DevStatus &ds, cudaStream_t st, const float *w,
                                        float *row_scale) {
    const int64_t P = s.P();
    const unsigned blocks = (unsigned)std::min<int64_t>((P + kThreads - 1) / kThreads, 4096);
    launch_pdl(dispatch_all_experts_kernel, dim3(blocks), dim3(kThreads), 0, st, idx, s.T, s.E,
               counts, offsets, pos, src_token, w, row_scale, ds);
    return cudaGetLastError();
}

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

// The count matrix [E][chunks] and, after it, the rank kernel's ticket.
size_t dispatch_scratch_bytes(const Shape &s) {
    DispatchGrid g = dispatch_grid(s.P(), s.E);
    return sizeof(int32_t) * (size_t)s.E * (size_t)g.blocks + 16;
}

unsigned *dispatch_ticket(const Shape &s, int32_t *scratch) {
    DispatchGrid g = dispatch_grid(s.P(), s.E);
    return reinterpret_cast<unsigned *>(scratch + (size_t)s.E * (size_t)g.blocks);
}

cudaError_t launch_dispatch(const Shape &s, const int32_t *idx, const void *x, int32_t *counts,
                            int32_t *offsets, int32_t *pos, int32_t *src_token, void *x_perm,
                            int32_t *hist, const DevStatus &ds, cudaStream_t st,
                            const float *scale, bool in_forward, float *row_scale) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {  // E = 1024: 32 warps x 1024 counts = 128 KB
        if ((err = cudaFuncSetAttribute(rank_kernel<kRankThreads>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kRankWarps * 1024 * (int)sizeof(int))) != cudaSuccess ||
            (err = cudaFuncSetAttribute(rank_kernel<kSmallRankThreads>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kScanStageMax * (int)sizeof(int))) != cudaSuccess)
            return err;
        attr_set[dev] = true;
    }
    const int64_t P = s.P();
    if (scale == nullptr && x_perm != nullptr) {
        bool one = false;
        err = s.bf16 ? launch_dispatch_one<__nv_bfloat16>(s, idx, x, counts, offsets, pos,
                                                          src_token, x_perm, ds, st, in_forward,
                                                          &one)
                     : launch_dispatch_one<float>(s, idx, x, counts, offsets, pos, src_token,
                                                  x_perm, ds, st, in_forward, &one);
        if (err != cudaSuccess || one) return err;
    }
    const DispatchGrid g = dispatch_grid(P, s.E);
    unsigned *ticket = dispatch_ticket(s, hist);
    if (!in_forward && (err = cudaMemsetAsync(ticket, 0, sizeof(unsigned), st)) != cudaSuccess)
        return err;
    const int64_t n_hist = (int64_t)s.E * g.blocks;
    const int staged = n_hist <= kScanStageMax ? 1 : 0;
    // chunks of 256 pairs: one warp per 32 of them (a block of 1024 threads
    // would leave most lanes idle, and its per-expert walk over 32 warps'
    // counts is serial)
    const bool small = g.chunk == kSmallRankThreads;
    const int nw = small ? kSmallRankThreads / 32 : kRankWarps;
    const size_t sh = sizeof(int) * (size_t)std::max<int64_t>((int64_t)nw * s.E,
                                                               staged ? n_hist : 0);
    if (small)
        launch_pdl(rank_kernel<kSmallRankThreads>, dim3(g.blocks), dim3(kSmallRankThreads), sh, st,
                   idx, P, s.E, g.chunk, g.blocks, staged, hist, pos, counts, offsets, ticket, ds);
    else
        launch_pdl(rank_kernel<kRankThreads>, dim3(g.blocks), dim3(kRankThreads), sh, st, idx, P,
                   s.E, g.chunk, g.blocks, staged, hist, pos, counts, offsets, ticket, ds);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (x_perm == nullptr) {  // pos and src_token only (moe_forward's gathered-row path)
        launch_pdl(place_index_kernel, dim3((unsigned)((P + kThreads - 1) / kThreads)),
                   dim3(kThreads), 0, st, static_cast<const int32_t *>(hist), P, s.k, g.chunk,
                   g.blocks, pos, src_token, scale, scale != nullptr ? row_scale : nullptr);
        return cudaGetLastError();
    }
    const unsigned blocks = (unsigned)((P + kWarps - 1) / kWarps);
    const int32_t *chist = hist;
    const int64_t row_bytes = (int64_t)s.d * (s.bf16 ? 2 : 4);
    if (!in_forward && scale == nullptr && row_bytes <= kStageRowMax &&
        (int64_t)s.k * 1024 <= row_bytes) {
        const unsigned tblocks = (unsigned)((s.T + kTokWarps - 1) / kTokWarps);
        const size_t tsh = (size_t)kTokWarps * (size_t)row_bytes;
        if (s.bf16)
            return launch_token_rows<__nv_bfloat16>(x, chist, s, g, pos, src_token, x_perm,
                                                    tblocks, tsh, st);
        return launch_token_rows<float>(x, chist, s, g, pos, src_token, x_perm, tblocks, tsh, st);
    }
    if (s.bf16) {
        using T = __nv_bfloat16;
        const T *xt = static_cast<const T *>(x);
        T *xp = static_cast<T *>(x_perm);
        if (scale && x_perm)
            launch_pdl(place_rows_kernel<T, true>, dim3(blocks), dim3(kThreads), 0, st, xt, chist,
                       scale, P, s.k, s.d, g.chunk, g.blocks, pos, src_token, xp);
        else
            launch_pdl(place_rows_kernel<T, false>, dim3(blocks), dim3(kThreads), 0, st, xt, chist,
                       (const float *)nullptr, P, s.k, s.d, g.chunk, g.blocks, pos, src_token, xp);
    } else {
        const float *xt = static_cast<const float *>(x);
        float *xp = static_cast<float *>(x_perm);
        if (scale && x_perm)
            launch_pdl(place_rows_kernel<float, true>, dim3(blocks), dim3(kThreads), 0, st, xt,
                       chist, scale, P, s.k, s.d, g.chunk, g.blocks, pos, src_token, xp);
        else
            launch_pdl(place_rows_kernel<float, false>, dim3(blocks), dim3(kThreads), 0, st, xt,
                       chist, (const float *)nullptr, P, s.k, s.d, g.chunk, g.blocks, pos,
                       src_token, xp);
    }
    return cudaGetLastError();
}

}  // namespace moe
