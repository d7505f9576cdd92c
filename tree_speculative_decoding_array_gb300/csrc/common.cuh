// Shared helpers of the tsv CUDA library: error reporting, device status
// words, storage conversions and small PTX wrappers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <utility>

#include "../../include/tsv.h"

namespace tsv {

// Programmatic dependent launch.  Every kernel of the library is launched with launch_pdl() and begins with
// griddep_begin(): griddepcontrol.wait returns once the kernel before it on the stream has completed and its
// memory is visible (at once when there is no such kernel), and launch_dependents then lets the next kernel's
// CTAs be scheduled while this one runs, so that launches and ramp-ups overlap the tails of their predecessors.
// Nothing a kernel reads or writes in global memory, and no TMEM allocation, comes before the wait: a waiting
// CTA holds no resource that the kernel it waits for could need.
__device__ __forceinline__ void griddep_begin() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              A&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Records the reason of a failed call for tsv_last_error() (per host thread).
tsv_status fail(tsv_status st, const char* fmt, ...);
// Clears the per-thread error string (called at the start of every entry point).
void clear_error();
// Maps a CUDA error after enqueueing to TSV_ECUDA with its name.
tsv_status check_launch(const char* what);
// SM count of the current device (cached per device).
int sm_count();

// First device error wins; words 1..2 record where it happened.
__device__ __forceinline__ void dev_fail(int32_t* st, int code, int a, int b) {
    if (st == nullptr) return;
    if (atomicCAS(st, 0, code) == 0) {
        st[1] = a;
        st[2] = b;
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t u) { return __uint_as_float(((uint32_t)u) << 16); }
__device__ __forceinline__ float f16_bits_to_f32(uint16_t u) { return __half2float(__ushort_as_half(u)); }
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t u) {
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

// Monotone map of fp32 to uint32 (larger float -> larger integer), used to pack
// (logit, index) into one 64-bit key for an atomic maximum.
__device__ __forceinline__ uint32_t orderable(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unorderable(uint32_t o) {
    uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}
// Larger key = larger logit, ties -> smaller index.
__device__ __forceinline__ unsigned long long pack_best(float v, uint32_t idx) {
    return ((unsigned long long)orderable(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

// 16-byte streaming load that does not allocate in L1 (weights read once).
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

}  // namespace tsv
