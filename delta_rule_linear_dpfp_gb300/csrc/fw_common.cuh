// fw_common.cuh -- small device helpers shared by the sm_103a kernels of the
// fast-weight layer core.  Nothing here is specific to one kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define FW_DEV __device__ __forceinline__

namespace fw {

// Bit values of the device-side status word (see fw_device_status).
enum : unsigned { kStatusTimeout = 1u };

// ---------------------------------------------------------------- dtype I/O
template <typename T> struct io;

template <> struct io<float> {
    static FW_DEV float load(const float *p) { return __ldcg(p); }
    static FW_DEV float to_f(float x) { return x; }
    static FW_DEV float from_f(float x) { return x; }
    static FW_DEV void store(float *p, float x) { *p = x; }
};

template <> struct io<__nv_bfloat16> {
    static FW_DEV float load(const __nv_bfloat16 *p) { return __bfloat162float(__ldcg(p)); }
    static FW_DEV float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static FW_DEV __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
    static FW_DEV void store(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};

// Load 8 consecutive elements (16-byte aligned for bf16, 32-byte for fp32)
// and widen them to fp32.
FW_DEV void load8(const float *p, float (&o)[8]) {
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldcg(reinterpret_cast<const float4 *>(p) + 1);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

FW_DEV void load8(const __nv_bfloat16 *p, float (&o)[8]) {
    const uint4 u = __ldcg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Round 8 fp32 values to the output type and store them (16-byte aligned for
// bf16, 32-byte for fp32).
FW_DEV void store8(float *p, const float (&v)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

FW_DEV uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

FW_DEV void store8(__nv_bfloat16 *p, const float (&v)[8]) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4 *>(p) = u;
}

// Warm L2 with `bytes` from global memory (16-byte aligned address, a
// multiple of 16 bytes): no data reaches the issuing thread, and L2 is the
// point of coherence, so it is safe on data another kernel is still writing.
FW_DEV void l2_prefetch(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// -------------------------------------------- programmatic dependent launch
// The next kernel on the stream may start launching (it still waits in
// griddep_wait before touching what this kernel writes).
FW_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Block until the preceding kernel on the stream has completed and its memory
// operations are visible (returns at once when the launch did not overlap).
FW_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// A pointer read after griddep_wait: its value passes through an opaque step
// placed after the wait, so the compiler cannot schedule a load through it
// (a read-only or cache-hinted load included) ahead of the wait.  Loads of
// data another kernel may have written use the coherent L2 path (__ldcg),
// not the read-only path, whose contract is data constant for the kernel's
// whole lifetime -- which an overlapped launch does not give.
template <class T> FW_DEV T *after_wait(T *p) {
    asm volatile("" : "+l"(p)::"memory");
    return p;
}

// Launch with programmatic stream serialization: the kernel's CTAs may be
// scheduled while the preceding kernel on the stream finishes, so the launch
// latency is hidden behind its tail.  Every kernel launched this way calls
// griddep_wait before its first global access.  Because each kernel lets its
// successor launch early, a kernel may start while kernels two or more places
// before it still run: a load before griddep_wait would race with them (the
// one exception, the forward's scan reading W0, is made safe by its
// predecessor triggering only after its own wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
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
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

FW_DEV float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

FW_DEV void record_status(unsigned *status, unsigned bits) {
    if (status)
        atomicOr(status, bits);
}

} // namespace fw
