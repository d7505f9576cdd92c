// Device-side fill of synthetic input tensors (input generation, not the
// verify step).  Element i of a tensor's logical row-major index gets
// dist(splitmix64(key, i)), exactly as the host generator in synth/rng.py and
// synth/tensors.py computes it, so large tensors can be written straight into
// GPU memory and any slice regenerated on the host for checking.
//
// SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): output n of the stream
// with state s is mix64(s + n * 0x9E3779B97F4A7C15).  Floating-point steps are
// single IEEE fp32 operations with round-to-nearest-even (this file is
// compiled with -fmad=false), so they match numpy's fp32 arithmetic bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t idx) {
    return mix64(key + (idx + 1ull) * 0x9E3779B97F4A7C15ull);
}

__device__ __forceinline__ float normal_f32(uint64_t h) {
    const int64_t s = (int64_t)((h & 0xFFFFull) + ((h >> 16) & 0xFFFFull) + ((h >> 32) & 0xFFFFull) + (h >> 48));
    const float c = (float)(s - 131070);  // exact (|c| < 2^18)
    return __fmul_rn(c, __uint_as_float(0x37DDB3D7u));
}

__device__ __forceinline__ float uniform_f32(uint64_t h, float lo, float width) {
    const float u = __fmul_rn((float)(uint32_t)(h >> 40), 5.9604644775390625e-08f);  // 2^-24, exact
    return __fadd_rn(__fmul_rn(u, width), lo);
}

__device__ __forceinline__ uint32_t int_below(uint64_t h, uint32_t n) {
    return (uint32_t)(((h >> 32) * (uint64_t)n) >> 32);
}

enum Dist {
    NORMAL_F16 = 0,
    NORMAL_BF16 = 1,
    INT8_CODE = 2,
    UNIFORM_F16 = 3,
    UNIFORM_BF16 = 4,
    Q4_PACKED = 5,
    Q4_BIAS = 6,
};

__global__ void fill_kernel(void* __restrict__ dst, int dist, uint64_t key, uint64_t key2, int64_t n1, int64_t n2,
                            int64_t n3, int64_t nrows, int64_t s0, int64_t s1, int64_t s2, float p0, float p1,
                            float p2, float p3) {
    for (int64_t row = blockIdx.x; row < nrows; row += gridDim.x) {
        const int64_t i2 = row % n2;
        const int64_t t = row / n2;
        const int64_t i1 = t % n1;
        const int64_t i0 = t / n1;
        const int64_t dbase = i0 * s0 + i1 * s1 + i2 * s2;
        const uint64_t lbase = (uint64_t)row * (uint64_t)n3;
        for (int64_t i3 = threadIdx.x; i3 < n3; i3 += blockDim.x) {
            const uint64_t idx = lbase + (uint64_t)i3;
            const int64_t o = dbase + i3;
            switch (dist) {
                case NORMAL_F16:
                    reinterpret_cast<__half*>(dst)[o] = __float2half_rn(__fmul_rn(normal_f32(draw(key, idx)), p0));
                    break;
                case NORMAL_BF16:
                    reinterpret_cast<__nv_bfloat16*>(dst)[o] =
                        __float2bfloat16_rn(__fmul_rn(normal_f32(draw(key, idx)), p0));
                    break;
                case INT8_CODE:
                    reinterpret_cast<int8_t*>(dst)[o] = (int8_t)((int)int_below(draw(key, idx), 255) - 127);
                    break;
                case UNIFORM_F16:
                    reinterpret_cast<__half*>(dst)[o] = __float2half_rn(uniform_f32(draw(key, idx), p0, p1));
                    break;
                case UNIFORM_BF16:
                    reinterpret_cast<__nv_bfloat16*>(dst)[o] = __float2bfloat16_rn(uniform_f32(draw(key, idx), p0, p1));
                    break;
                case Q4_PACKED: {  // byte idx packs elements 2 idx (low nibble) and 2 idx + 1 (high nibble)
                    const uint32_t lo = int_below(draw(key, 2 * idx), 16);
                    const uint32_t hi = int_below(draw(key, 2 * idx + 1), 16);
                    reinterpret_cast<uint8_t*>(dst)[o] = (uint8_t)(lo | (hi << 4));
                    break;
                }
                case Q4_BIAS: {  // -(U(p0, p0 + p1) * bf16(U(p2, p2 + p3))) with the scale's own stream key2
                    const float s = __bfloat162float(__float2bfloat16_rn(uniform_f32(draw(key2, idx), p2, p3)));
                    const float t = uniform_f32(draw(key, idx), p0, p1);
                    reinterpret_cast<__nv_bfloat16*>(dst)[o] = __float2bfloat16_rn(-__fmul_rn(t, s));
                    break;
                }
                default:
                    break;
            }
        }
    }
}

}  // namespace

// Fills a tensor of logical shape [n0, n1, n2, n3] whose destination strides
// (in elements) are s0, s1, s2 for the outer dims and 1 for the innermost.
// Returns 0 on success, else the CUDA error code of the launch.
extern "C" int tsv_synth_fill(void* dst, int dist, uint64_t key, uint64_t key2, int64_t n0, int64_t n1, int64_t n2,
                              int64_t n3, int64_t s0, int64_t s1, int64_t s2, float p0, float p1, float p2, float p3,
                              cudaStream_t stream) {
    if (!dst || n0 <= 0 || n1 <= 0 || n2 <= 0 || n3 <= 0) return (int)cudaErrorInvalidValue;
    const int64_t nrows = n0 * n1 * n2;
    int threads = n3 >= 256 ? 256 : (n3 >= 128 ? 128 : 64);
    int64_t blocks = nrows < 65536 * 8 ? nrows : 65536 * 8;
    fill_kernel<<<(unsigned)blocks, threads, 0, stream>>>(dst, dist, key, key2, n1, n2, n3, nrows, s0, s1, s2, p0, p1,
                                                          p2, p3);
    return (int)cudaGetLastError();
}

// Restores workload buffers between benchmark rounds: table[3 * i .. 3 * i + 2]
// = (source address, destination address, bytes) of n independent copies, all
// done by one launch (one CTA per copy, 16-byte words when both ends allow).
namespace {
__global__ void copy_table_kernel(const int64_t* __restrict__ table, int n) {
    const int i = blockIdx.x;
    if (i >= n) return;
    const char* src = reinterpret_cast<const char*>(table[3 * i]);
    char* dst = reinterpret_cast<char*>(table[3 * i + 1]);
    const int64_t bytes = table[3 * i + 2];
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | (uintptr_t)bytes) & 15) == 0) {
        const uint4* s = reinterpret_cast<const uint4*>(src);
        uint4* d = reinterpret_cast<uint4*>(dst);
        for (int64_t k = threadIdx.x; k < bytes / 16; k += blockDim.x) d[k] = s[k];
    } else {
        for (int64_t k = threadIdx.x; k < bytes; k += blockDim.x) dst[k] = src[k];
    }
}
}  // namespace

extern "C" int tsv_synth_copy_table(const int64_t* table, int n, cudaStream_t stream) {
    if (n <= 0) return 0;
    copy_table_kernel<<<n, 256, 0, stream>>>(table, n);
    return (int)cudaGetLastError();
}
