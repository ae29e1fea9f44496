// common.cuh -- small device helpers shared by the libmoe kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Bits of the per-device error word (see moe_last_device_error).
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrBadRouting = 2u;

// Runtime parameters every kernel that can fail receives.
struct DevStatus {
    unsigned *err;          // device error word (never null)
    unsigned long long wait_limit_ns;  // bound on each device-side wait
    int inject_wait_timeout;  // test hook: the GEMM waits on a barrier nothing signals
};

__device__ __forceinline__ void raise_error(const DevStatus &st, unsigned bit) {
    atomicOr(st.err, bit);
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

// Activation element <-> float.
template <typename T> struct Act;
template <> struct Act<float> {
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Act<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// 16-byte vector of activations: 8 bf16 or 4 fp32.
template <typename T> struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
};

__device__ __forceinline__ void unpack16(const uint4 &v, float (&o)[8], const __nv_bfloat16 *) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void unpack16(const uint4 &v, float (&o)[4], const float *) {
    o[0] = __uint_as_float(v.x);
    o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z);
    o[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ uint4 pack16(const float (&o)[8], const __nv_bfloat16 *) {
    uint4 v;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
    return v;
}
__device__ __forceinline__ uint4 pack16(const float (&o)[4], const float *) {
    return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                      __float_as_uint(o[3]));
}

// Streaming 16-byte global load / store helpers.
__device__ __forceinline__ uint4 ldg16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void stg16(void *p, const uint4 &v) {
    *reinterpret_cast<uint4 *>(p) = v;
}

// Programmatic dependent launch.  Every kernel of the layer starts with
// pdl_entry(): it lets the next kernel in the stream be scheduled (once all
// of this grid's blocks have started, so a dependent never takes SMs from
// this grid's own blocks), then waits until the previous kernel in the
// stream has completed and its writes are visible.  Nothing is read from
// earlier kernels before that wait.  Launched without the attribute (or
// after a copy), both instructions are no-ops.
__device__ __forceinline__ void pdl_release() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_entry() {
    pdl_release();
    pdl_wait();
}

// Launch with programmatic stream serialization (see pdl_entry); extra
// attributes (a cluster shape) may be appended.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace moe
