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
// Router logits, warp-split form (used for E <= 32, and for larger E when the
// batch is small).  A block owns TPW tokens x EP experts (TPW * EP = 32;
// EP = E rounded up to a power of two, or 32-expert groups along blockIdx.y
// when E > 32).  Its 8 warps split the hidden dimension: warp w, lane l
// walks 8-element chunks q = 32w + l, q + 256, ... with 16-byte loads of x
// and two float4 loads per expert of Wr, keeping 32 partial sums.  A
// butterfly reduce-scatter (31 shuffles) leaves partial i of every warp in
// lane i; warp 0 then adds the 8 warps' values in warp order (a fixed order,
// so results are reproducible) and lane i writes logit (token i/EP, expert
// e0 + i%EP).
// ---------------------------------------------------------------------------
template <typename TA> struct Chunk8;
template <> struct Chunk8<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&v)[8]) {
        unpack16(ldg16(p), v, static_cast<const __nv_bfloat16 *>(nullptr));
    }
};
template <> struct Chunk8<float> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[8]) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

// After the call lane l holds the warp-wide sum of v[l] in v[0].
__device__ __forceinline__ void warp_reduce_scatter32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int half = 16; half >= 1; half >>= 1) {
        const bool upper = (lane & half) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float send = upper ? v[j] : v[j + half];
            const float recv = __shfl_xor_sync(0xffffffffu, send, half);
            v[j] = (upper ? v[j + half] : v[j]) + recv;
        }
    }
}

constexpr int kSplitWarps = 8;

constexpr int kNoExpert = 0x7fffffff;  // "no candidate" in a warp arg-max

// Rank order of the selection: a larger logit first; equal logits (+0.0 and
// -0.0 are equal) to the lower expert id; a NaN below every number.
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib) {
    const bool an = isnan(a), bn = isnan(b);
    if (an || bn) return (an && bn) ? (ia < ib) : bn;
    if (a > b) return true;
    if (a < b) return false;
    return ia < ib;
}

// Top-k selection and softmax weights inside EP-lane segments of a warp:
// lane tt*EP + e holds the logit v of expert e of the segment's token
// (valid: e is one of its experts).  Every lane of the warp must call it.
// Slot j of the token's selection ends in lane tt*EP + j, which stores it
// to idx_row[j] and w_row[j] when `store`.
template <int EP>
__device__ __forceinline__ void select_in_segment(float v, int e, bool valid, int k, int renorm,
                                                  bool store, int32_t *idx_row, float *w_row) {
    bool avail = valid;
    float my_v = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        float bv = avail ? v : NAN;
        int be = avail ? e : kNoExpert;
#pragma unroll
        for (int off = EP / 2; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (oe != kNoExpert && (be == kNoExpert || ranks_before(ov, oe, bv, be))) {
                bv = ov;
                be = oe;
            }
        }
        if (be == e) avail = false;
        if (e == j) {
            my_v = bv;
            my_e = be;
        }
    }
    float m = valid ? v : -INFINITY;
#pragma unroll
    for (int off = EP / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float z = valid ? expf(v - m) : 0.f;
#pragma unroll
    for (int off = EP / 2; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    float pr = (e < k) ? expf(my_v - m) / z : 0.f;
    if (renorm) {
        float sum = pr;
#pragma unroll
        for (int off = EP / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        pr = pr / sum;
    }
    if (e < k && store) {
        idx_row[e] = my_e;
        w_row[e] = pr;
    }
}

template <typename TA, int EP>
__global__ void __launch_bounds__(256)
router_logits_split_kernel(const TA *__restrict__ x, const float *__restrict__ Wr,
                           const float *__restrict__ bias, float *__restrict__ logits,
                           int64_t T, int d, int E, int k, int renorm,
                           int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                           unsigned *__restrict__ zero_word) {
    pdl_entry();
    if (zero_word != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        *zero_word = 0u;
    constexpr int TPW = 32 / EP;
    __shared__ float red[kSplitWarps][32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * TPW;
    const int e0 = blockIdx.y * EP;
    const int ne = min(EP, E - e0);  // experts of this block's group
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    const TA *xr[TPW];
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt) xr[tt] = x + min(t0 + tt, T - 1) * d;
    const float *wr = Wr + (int64_t)e0 * d;
    for (int c = (wid * 32 + lane) * 8; c < d; c += 32 * kSplitWarps * 8) {
        if constexpr (EP > TPW) {
            // hold the TPW token chunks, stream the experts
            float xv[TPW][8];
#pragma unroll
            for (int tt = 0; tt < TPW; ++tt) Chunk8<TA>::load(xr[tt] + c, xv[tt]);
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                if (e < ne) {
                    float wv[8];
                    Chunk8<float>::load(wr + (int64_t)e * d + c, wv);
#pragma unroll
                    for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            acc[tt * EP + e] = fmaf(xv[tt][i], wv[i], acc[tt * EP + e]);
                }
            }
        } else {
            // hold the EP expert chunks, stream the tokens
            float wv[EP][8];
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                if (e < ne) Chunk8<float>::load(wr + (int64_t)e * d + c, wv[e]);
                else
#pragma unroll
                    for (int i = 0; i < 8; ++i) wv[e][i] = 0.f;
            }
#pragma unroll
            for (int tt = 0; tt < TPW; ++tt) {
                float xv[8];
                Chunk8<TA>::load(xr[tt] + c, xv);
#pragma unroll
                for (int e = 0; e < EP; ++e)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[tt * EP + e] = fmaf(xv[i], wv[e][i], acc[tt * EP + e]);
            }
        }
    }
    warp_reduce_scatter32(acc);
    red[wid][lane] = acc[0];
    __syncthreads();
    if (wid == 0) {
        float v = red[0][lane];
#pragma unroll
        for (int w = 1; w < kSplitWarps; ++w) v += red[w][lane];
        const int tt = lane / EP, e = lane % EP;
        const int64_t t = t0 + tt;
        v += bias ? bias[e0 + min(e, ne - 1)] : 0.f;
        if (e < ne && t < T) logits[t * E + e0 + e] = v;
        // E <= 32: select and weigh here, on exactly the values just written.
        // Token tt's logits sit in the EP-lane segment of lanes tt*EP + e.
        if (topk_idx != nullptr) {  // warp-uniform: every lane joins the shuffles
            const int64_t tr = t < T ? t : 0;
            select_in_segment<EP>(v, e, e < ne, k, renorm, t < T, topk_idx + tr * k,
                                  topk_w + tr * k);
        }
    }
}

// ---------------------------------------------------------------------------
// Router logits, larger E: C[T][E] = A[T][d] * B[E][d]^T (+ bias[E]), fp32
// FFMA.  Block tile BM x BN, K step BK; each thread owns TM x TN outputs
// spread with stride (BM/TM) rows and (BN/TN) columns so shared-memory reads
// are conflict-free.  Operand tiles are stored k-major with one word of
// padding and double-buffered: the next K step is fetched into registers
// while the current one is multiplied.
// ---------------------------------------------------------------------------
constexpr int kLogitBK = 16;

template <typename TA, int BM, int BN, int TM, int TN>
__global__ void __launch_bounds__(256)
router_logits_kernel(const TA *__restrict__ x, const float *__restrict__ Wr,
                     const float *__restrict__ bias, float *__restrict__ logits, int64_t T, int d,
                     int E) {
    pdl_entry();
    static_assert((BM / TM) * (BN / TN) == 256, "256 threads");
    constexpr int BK = kLogitBK;
    constexpr int RG = BM / TM;  // row groups
    constexpr int CG = BN / TN;  // column groups
    constexpr int AL = BM * BK / 256, BL = BN * BK / 256;  // loads per thread
    __shared__ float As[2][BK][BM + 1];
    __shared__ float Bs[2][BK][BN + 1];

    const int tid = threadIdx.x;
    const int tx = tid % CG, ty = tid / CG;
    const int64_t m0 = (int64_t)blockIdx.x * BM;
    const int n0 = blockIdx.y * BN;

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    float ra[AL], rb[BL];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int l = 0; l < AL; ++l) {
            const int i = tid + l * 256, r = i / BK, c = i % BK;
            const int64_t gm = m0 + r;
            const int gk = k0 + c;
            ra[l] = (gm < T && gk < d) ? Act<TA>::to_f(x[gm * d + gk]) : 0.f;
        }
#pragma unroll
        for (int l = 0; l < BL; ++l) {
            const int i = tid + l * 256, r = i / BK, c = i % BK;
            const int gn = n0 + r, gk = k0 + c;
            rb[l] = (gn < E && gk < d) ? Wr[(int64_t)gn * d + gk] : 0.f;
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int l = 0; l < AL; ++l) {
            const int i = tid + l * 256;
            As[buf][i % BK][i / BK] = ra[l];
        }
#pragma unroll
        for (int l = 0; l < BL; ++l) {
            const int i = tid + l * 256;
            Bs[buf][i % BK][i / BK] = rb[l];
        }
    };

    const int nk = (d + BK - 1) / BK;
    fetch(0);
    stash(0);
    __syncthreads();
    for (int kt = 0; kt < nk; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < nk) fetch((kt + 1) * BK);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = As[buf][kk][ty + i * RG];
#pragma unroll
            for (int j = 0; j < TN; ++j) b[j] = Bs[buf][kk][tx + j * CG];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (kt + 1 < nk) stash(buf ^ 1);
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
    launch_pdl(router_logits_kernel<TA, BM, BN, TM, TN>, dim3(grid), dim3(256), 0, st, x, Wr, bias, logits, s.T, s.d, s.E);
    return cudaGetLastError();
}

template <typename TA, int EP>
cudaError_t launch_logits_split(const Shape &s, const TA *x, const float *Wr, const float *bias,
                                float *logits, int32_t *idx, float *w, cudaStream_t st,
                                unsigned *zero_word) {
    constexpr int TPW = 32 / EP;
    dim3 grid((unsigned)((s.T + TPW - 1) / TPW), (unsigned)((s.E + EP - 1) / EP));
    // with a single expert group (E <= 32) the kernel also selects; larger E
    // leaves the selection to the top-k kernel
    const bool fused = grid.y == 1 && idx != nullptr;
    launch_pdl(router_logits_split_kernel<TA, EP>, dim3(grid), dim3(256), 0, st,
        x, Wr, bias, logits, s.T, s.d, s.E, s.k, s.renorm ? 1 : 0, fused ? idx : nullptr,
        fused ? w : nullptr, fused ? zero_word : nullptr);
    return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_logits_t(const Shape &s, const TA *x, const float *Wr, const float *bias,
                            float *logits, int32_t *idx, float *w, cudaStream_t st,
                            unsigned *zero_word) {
    if (s.E <= 1) return launch_logits_split<TA, 1>(s, x, Wr, bias, logits, idx, w, st, zero_word);
    if (s.E <= 2) return launch_logits_split<TA, 2>(s, x, Wr, bias, logits, idx, w, st, zero_word);
    if (s.E <= 4) return launch_logits_split<TA, 4>(s, x, Wr, bias, logits, idx, w, st, zero_word);
    if (s.E <= 8) return launch_logits_split<TA, 8>(s, x, Wr, bias, logits, idx, w, st, zero_word);
    if (s.E <= 16) return launch_logits_split<TA, 16>(s, x, Wr, bias, logits, idx, w, st, zero_word);
    if (s.E <= 32) return launch_logits_split<TA, 32>(s, x, Wr, bias, logits, idx, w, st, zero_word);
    // larger E: the tiled kernel re-reads Wr far less per token, but needs
    // enough row tiles to fill the GPU; small batches use 32-expert groups.
    if (s.T < 2048) return launch_logits_split<TA, 32>(s, x, Wr, bias, logits, idx, w, st, zero_word);
    if (s.E <= 64) return launch_logits_cfg<TA, 64, 64, 4, 4>(s, x, Wr, bias, logits, st);
    return launch_logits_cfg<TA, 64, 128, 4, 8>(s, x, Wr, bias, logits, st);
}

// ---------------------------------------------------------------------------
// Top-k: one warp per token.  Lane l holds logits l, l+32, ...; k rounds of a
// warp arg-max under the rank order pick the experts; slot j is written by
// lane j.  Each round is two warp reductions (redux.sync): the maximum of the
// values' order-preserving 32-bit images, then the minimum expert id among
// the still-available values that reach it (the lower id wins ties).  With
// SORTED (up to 8 values a lane, E <= 256, and batches large enough that the
// kernel is bound by instruction issue rather than latency) the lane sorts
// its values once, so a round looks at each lane's head only.
// Weights: softmax over all E logits (max-shifted), then optional
// renormalisation over the chosen k.
// ---------------------------------------------------------------------------

// Order-preserving unsigned image of a logit: a > b as floats exactly when
// rank_bits(a) > rank_bits(b), with +0.0 and -0.0 alike and a NaN lowest (0;
// no number maps to 0).  With the lower expert id breaking ties this is the
// order ranks_before defines.
__device__ __forceinline__ uint32_t rank_bits(float v) {
    if (isnan(v)) return 0u;
    const uint32_t b = __float_as_uint(v == 0.f ? 0.f : v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float rank_value(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// With nparts > 0 the logits are first formed as the sum of nparts partial
// buffers (stride T*E, added in buffer order) plus bias, and written to
// `logits`; the selection then uses exactly the written values.
template <int VPL, bool SORTED>
__global__ void __launch_bounds__(256)
topk_kernel(float *__restrict__ logits, const float *__restrict__ partial, int nparts,
            const float *__restrict__ bias, int64_t T, int E, int k, int renorm,
            int32_t *__restrict__ idx, float *__restrict__ w, unsigned *__restrict__ zero_word) {
    pdl_entry();
    if (zero_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *zero_word = 0u;
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;  // warp-uniform
    float *L = logits + t * E;

    float v[VPL];
    unsigned avail = 0;  // bit i: value i of this lane is a not-yet-chosen expert
    const float *src = nparts > 0 ? partial + t * E : L;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? src[e] : 0.f;
        if (e < E) avail |= 1u << i;
    }
    if (nparts > 0) {
        // remaining partial buffers, each added to all VPL values at once, in
        // buffer order; unrolled so that the loads of several buffers are in
        // flight together (the adds stay in order)
#pragma unroll 4
        for (int q = 1; q < nparts; ++q) {
            const float *pq = partial + (int64_t)q * T * E + t * E;
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E) v[i] += pq[e];
            }
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                if (bias) v[i] += bias[e];
                L[e] = v[i];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (!((avail >> i) & 1u)) v[i] = -INFINITY;

    uint32_t ord[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) ord[i] = rank_bits(v[i]);
    float my_v = 0.f;
    int my_e = 0;
    uint32_t top = 0u;  // the first round's maximum: the largest logit
    if constexpr (SORTED) {
        // Each lane first sorts its values (rank image descending, expert id
        // ascending among equal images), so a round compares the lanes'
        // heads only, and the lane whose head is chosen shifts its list.
        // Entries past E rank lowest with the largest id: a valid expert
        // (a NaN logit included) always wins over them.
        uint32_t key[VPL], id[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const bool ok = (avail >> i) & 1u;
            key[i] = ok ? ord[i] : 0u;
            id[i] = ok ? (uint32_t)(lane + 32 * i) : 0xFFFFFFFFu;
        }
#pragma unroll
        for (int pass = 0; pass < VPL; ++pass) {  // odd-even transposition sort
#pragma unroll
            for (int i = pass & 1; i + 1 < VPL; i += 2) {
                const bool swap = key[i] < key[i + 1] || (key[i] == key[i + 1] && id[i] > id[i + 1]);
                const uint32_t k0 = key[i], i0 = id[i];
                key[i] = swap ? key[i + 1] : k0;
                id[i] = swap ? id[i + 1] : i0;
                key[i + 1] = swap ? k0 : key[i + 1];
                id[i + 1] = swap ? i0 : id[i + 1];
            }
        }
        for (int j = 0; j < k; ++j) {
            const uint32_t omax = __reduce_max_sync(0xffffffffu, key[0]);
            const uint32_t be = __reduce_min_sync(0xffffffffu, key[0] == omax ? id[0] : 0xFFFFFFFFu);
            if (id[0] == be) {  // this lane's head was chosen: drop it
#pragma unroll
                for (int i = 0; i + 1 < VPL; ++i) {
                    key[i] = key[i + 1];
                    id[i] = id[i + 1];
                }
                key[VPL - 1] = 0u;
                id[VPL - 1] = 0xFFFFFFFFu;
            }
            if (j == 0) top = omax;
            if (lane == j) {
                my_v = rank_value(omax);
                my_e = (int)be;
            }
        }
    } else
    for (int j = 0; j < k; ++j) {
        // every round has an available value somewhere in the warp (j < k <= E)
        uint32_t lmax = 0u;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if ((avail >> i) & 1u) lmax = ord[i] > lmax ? ord[i] : lmax;
        const uint32_t omax = __reduce_max_sync(0xffffffffu, lmax);
        uint32_t le = 0xFFFFFFFFu;  // this lane's lowest available expert at the maximum
#pragma unroll
        for (int i = VPL - 1; i >= 0; --i)
            if (((avail >> i) & 1u) && ord[i] == omax) le = (uint32_t)(lane + 32 * i);
        const int be = (int)__reduce_min_sync(0xffffffffu, le);
        if ((be & 31) == lane) avail &= ~(1u << (be >> 5));
        if (j == 0) top = omax;
        if (lane == j) {
            my_v = rank_value(omax);
            my_e = be;
        }
    }

    // softmax over all E logits, shifted by their maximum (-inf if every
    // logit is NaN, as a max that skips NaNs would give)
    const float m = top != 0u ? rank_value(top) : -INFINITY;
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

// Sorted heads pay from about this many tokens (measured: T = 4096-16384
// 1-9 % faster routes; T = 64 1.7 us slower, where the kernel is latency bound).
constexpr int64_t kTopkSortedMinT = 1024;

template <int VPL>
cudaError_t launch_topk_v(const Shape &s, float *logits, const float *partial, int nparts,
                          const float *bias, int32_t *idx, float *w, cudaStream_t st,
                          unsigned *zero_word) {
    unsigned blocks = (unsigned)((s.T + 7) / 8);
    if (VPL <= 8 && s.T >= kTopkSortedMinT)
        launch_pdl(topk_kernel<VPL, (VPL <= 8)>, dim3(blocks), dim3(256), 0, st, logits, partial,
                   nparts, bias, s.T, s.E, s.k, s.renorm ? 1 : 0, idx, w, zero_word);
    else
        launch_pdl(topk_kernel<VPL, false>, dim3(blocks), dim3(256), 0, st, logits, partial, nparts,
                   bias, s.T, s.E, s.k, s.renorm ? 1 : 0, idx, w, zero_word);
    return cudaGetLastError();
}

cudaError_t launch_topk_any(const Shape &s, float *logits, const float *partial, int nparts,
                            const float *bias, int32_t *idx, float *w, cudaStream_t st,
                            unsigned *zero_word) {
    if (s.E <= 32) return launch_topk_v<1>(s, logits, partial, nparts, bias, idx, w, st, zero_word);
    if (s.E <= 64) return launch_topk_v<2>(s, logits, partial, nparts, bias, idx, w, st, zero_word);
    if (s.E <= 128) return launch_topk_v<4>(s, logits, partial, nparts, bias, idx, w, st, zero_word);
    if (s.E <= 256) return launch_topk_v<8>(s, logits, partial, nparts, bias, idx, w, st, zero_word);
    if (s.E <= 512) return launch_topk_v<16>(s, logits, partial, nparts, bias, idx, w, st, zero_word);
    return launch_topk_v<32>(s, logits, partial, nparts, bias, idx, w, st, zero_word);
}

}  // namespace

cudaError_t launch_router_logits(const Shape &s, const void *x, const float *Wr, const float *bias,
                                 float *logits, cudaStream_t st, int32_t *idx, float *w,
                                 unsigned *zero_word) {
    if (s.bf16)
        return launch_logits_t<__nv_bfloat16>(s, static_cast<const __nv_bfloat16 *>(x), Wr, bias,
                                              logits, idx, w, st, zero_word);
    return launch_logits_t<float>(s, static_cast<const float *>(x), Wr, bias, logits, idx, w, st,
                                  zero_word);
}

bool router_selects_in_logits(const Shape &s) { return s.E <= 32; }

cudaError_t launch_topk(const Shape &s, const float *logits, int32_t *idx, float *w,
                        cudaStream_t st, unsigned *zero_word) {
    // nparts == 0: the kernel only reads `logits`
    return launch_topk_any(s, const_cast<float *>(logits), nullptr, 0, nullptr, idx, w, st,
                           zero_word);
}

cudaError_t launch_topk_partials(const Shape &s, const float *partial, int splits,
                                 const float *bias, float *logits, int32_t *idx, float *w,
                                 cudaStream_t st, unsigned *zero_word) {
    return launch_topk_any(s, logits, partial, splits, bias, idx, w, st, zero_word);
}

}  // namespace moe
