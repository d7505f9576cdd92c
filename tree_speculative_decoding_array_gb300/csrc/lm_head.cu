// tsv_lm_head_argmax: LM-head projection fused with a greedy argmax.
//
// mlxcel issue #1185, "Phase 2" item 2a: at temperature 0 the vocabulary-wide
// logits are only needed for their argmax, so a fused projection + argmax
// never writes them out.  "Phase 3" and the cost-model table: the head may be
// affine group-64 4-bit (weight, scales, biases).
//
// Weight-streaming GEMV: the head is read exactly once per call (per group of
// up to 8 hidden rows), with 16-byte streaming loads that bypass L1.  Hidden
// rows sit in shared memory; each warp owns whole vocabulary rows, reduces
// the dot products with shuffles and keeps a running best (logit, index) per
// hidden row.  Bests are merged with 64-bit atomic maxima on a packed key
// (orderable fp32 logit << 32 | ~index), so ties go to the lowest index
// regardless of the order in which CTAs finish.  A last tiny kernel unpacks.
#include "common.cuh"

namespace tsv {

constexpr int kLmThreads = 256;

__device__ __forceinline__ float dot8_bf16w(uint4 w, uint4 h) {
    float a = bf16_lo(w.x) * bf16_lo(h.x);
    a = fmaf(bf16_hi(w.x), bf16_hi(h.x), a);
    a = fmaf(bf16_lo(w.y), bf16_lo(h.y), a);
    a = fmaf(bf16_hi(w.y), bf16_hi(h.y), a);
    a = fmaf(bf16_lo(w.z), bf16_lo(h.z), a);
    a = fmaf(bf16_hi(w.z), bf16_hi(h.z), a);
    a = fmaf(bf16_lo(w.w), bf16_lo(h.w), a);
    a = fmaf(bf16_hi(w.w), bf16_hi(h.w), a);
    return a;
}

__device__ __forceinline__ float dot8_f16w(uint4 w, uint4 h) {
    float2 w0 = f16x2_to_f32x2(w.x), w1 = f16x2_to_f32x2(w.y), w2 = f16x2_to_f32x2(w.z), w3 = f16x2_to_f32x2(w.w);
    float a = w0.x * bf16_lo(h.x);
    a = fmaf(w0.y, bf16_hi(h.x), a);
    a = fmaf(w1.x, bf16_lo(h.y), a);
    a = fmaf(w1.y, bf16_hi(h.y), a);
    a = fmaf(w2.x, bf16_lo(h.z), a);
    a = fmaf(w2.y, bf16_hi(h.z), a);
    a = fmaf(w3.x, bf16_lo(h.w), a);
    a = fmaf(w3.y, bf16_hi(h.w), a);
    return a;
}

template <int R>
__device__ __forceinline__ void warp_sum(float (&acc)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[r] += __shfl_xor_sync(0xFFFFFFFFu, acc[r], o);
}

// Merge per-warp bests (held by lane 0 of every warp) into the global keys.
template <int R>
__device__ __forceinline__ void merge_best(const unsigned long long (&mine)[R], unsigned long long* s_best,
                                           unsigned long long* best, int r0, int rows) {
    const int lane = threadIdx.x & 31;
    if (lane == 0)
#pragma unroll
        for (int r = 0; r < R; ++r) atomicMax(&s_best[r], mine[r]);
    __syncthreads();
    if (threadIdx.x < R && r0 + (int)threadIdx.x < rows) atomicMax(&best[r0 + threadIdx.x], s_best[threadIdx.x]);
}

// Every logit to logits[row][v] (sampled verification): lane r writes hidden row r0 + r of vocabulary rows v
// (a0) and v + 1 (a1, when has1); warp_sum left the sums in every lane.
template <int R>
__device__ __forceinline__ void store_logits(float* logits, const float (&a0)[R], const float (&a1)[R], bool has1,
                                             int v, int V, int r0, int rows, int lane) {
#pragma unroll
    for (int r = 0; r < R; ++r)
        if (lane == r && r0 + r < rows) {
            logits[(size_t)(r0 + r) * V + v] = a0[r];
            if (has1) logits[(size_t)(r0 + r) * V + v + 1] = a1[r];
        }
}

// fp16 / bf16 weights [V, H]; hidden rows r0 .. r0 + R - 1.  H % 256 == 0.
template <int R, bool BF16W>
__global__ void __launch_bounds__(kLmThreads, R <= 4 ? 3 : 2) lm_gemv16_kernel(const uint16_t* __restrict__ hidden, int rows, int H,
                                                               int V, const uint16_t* __restrict__ W,
                                                               unsigned long long* __restrict__ best, int r0,
                                                               float* __restrict__ logits) {
    griddep_begin();
    extern __shared__ uint4 smem[];
    __shared__ unsigned long long s_best[8];
    uint4* hs = smem;  // [R][H/8]
    const int nvec = H >> 3;
    for (int e = threadIdx.x; e < R * nvec; e += blockDim.x) {
        const int r = e / nvec, c = e % nvec;
        hs[e] = (r0 + r < rows) ? reinterpret_cast<const uint4*>(hidden + (size_t)(r0 + r) * H)[c] : make_uint4(0, 0, 0, 0);
    }
    if (threadIdx.x < 8) s_best[threadIdx.x] = 0ull;
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    unsigned long long mine[R];
#pragma unroll
    for (int r = 0; r < R; ++r) mine[r] = 0ull;

    constexpr int U = 4;
    for (int v0 = 2 * gw; v0 < V; v0 += 2 * warps) {
        const bool has1 = v0 + 1 < V;
        const uint4* w0p = reinterpret_cast<const uint4*>(W + (size_t)v0 * H);
        const uint4* w1p = reinterpret_cast<const uint4*>(W + (size_t)(has1 ? v0 + 1 : v0) * H);
        float a0[R], a1[R];
#pragma unroll
        for (int r = 0; r < R; ++r) a0[r] = a1[r] = 0.f;
        for (int base = 0; base < nvec; base += 32 * U) {
            uint4 x0[U], x1[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = base + u * 32 + lane;
                if (i < nvec) {
                    x0[u] = ldg_stream16(w0p + i);
                    x1[u] = ldg_stream16(w1p + i);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = base + u * 32 + lane;
                if (i < nvec) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint4 hv = hs[r * nvec + i];
                        if (BF16W) {
                            a0[r] += dot8_bf16w(x0[u], hv);
                            a1[r] += dot8_bf16w(x1[u], hv);
                        } else {
                            a0[r] += dot8_f16w(x0[u], hv);
                            a1[r] += dot8_f16w(x1[u], hv);
                        }
                    }
                }
            }
        }
        warp_sum<R>(a0);
        warp_sum<R>(a1);
        if (logits) store_logits<R>(logits, a0, a1, has1, v0, V, r0, rows, lane);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                unsigned long long k0 = pack_best(a0[r], (uint32_t)v0);
                if (k0 > mine[r]) mine[r] = k0;
                if (has1) {
                    unsigned long long k1 = pack_best(a1[r], (uint32_t)(v0 + 1));
                    if (k1 > mine[r]) mine[r] = k1;
                }
            }
        }
    }
    merge_best<R>(mine, s_best, best, r0, rows);
}

// 4-bit affine weights: packed [V, H/2], scales/biases bf16 [V, H/64].
// A 16-byte vector holds 32 codes = half a group, so
//   sum_k (s q_k + b) h_k = s * sum_k q_k h_k + b * sum_k h_k
// with the per-half-group sums of h precomputed once in shared memory.
template <int R>
__global__ void __launch_bounds__(kLmThreads, R <= 4 ? 3 : 2) lm_gemv_q4_kernel(const uint16_t* __restrict__ hidden, int rows, int H,
                                                                int V, const uint8_t* __restrict__ Wq,
                                                                const uint16_t* __restrict__ scales,
                                                                const uint16_t* __restrict__ biases,
                                                                unsigned long long* __restrict__ best, int r0,
                                                                float* __restrict__ logits) {
    griddep_begin();
    extern __shared__ uint4 smem[];
    __shared__ unsigned long long s_best[8];
    const int nvec = H >> 5;  // 32-code vectors per row
    uint4* hs = smem;         // [R][H/8] bf16 hidden
    float* hsum = reinterpret_cast<float*>(smem + R * (H >> 3));  // [R][nvec]
    const int hv8 = H >> 3;
    for (int e = threadIdx.x; e < R * hv8; e += blockDim.x) {
        const int r = e / hv8, c = e % hv8;
        hs[e] = (r0 + r < rows) ? reinterpret_cast<const uint4*>(hidden + (size_t)(r0 + r) * H)[c] : make_uint4(0, 0, 0, 0);
    }
    if (threadIdx.x < 8) s_best[threadIdx.x] = 0ull;
    __syncthreads();
    for (int e = threadIdx.x; e < R * nvec; e += blockDim.x) {
        const int r = e / nvec, c = e % nvec;
        const uint32_t* hw = reinterpret_cast<const uint32_t*>(hs + r * hv8 + c * 4);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) s += bf16_lo(hw[k]) + bf16_hi(hw[k]);
        hsum[e] = s;
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int ng = H >> 6;
    unsigned long long mine[R];
#pragma unroll
    for (int r = 0; r < R; ++r) mine[r] = 0ull;

    for (int v = gw; v < V; v += warps) {
        const uint4* wp = reinterpret_cast<const uint4*>(Wq + (size_t)v * (H >> 1));
        float acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = 0.f;
        for (int i = lane; i < nvec; i += 32) {
            const uint4 q = ldg_stream16(wp + i);
            const float s = bf16_bits_to_f32(scales[(size_t)v * ng + (i >> 1)]);
            const float bb = bf16_bits_to_f32(biases[(size_t)v * ng + (i >> 1)]);
            const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t* hw = reinterpret_cast<const uint32_t*>(hs + r * hv8 + i * 4);
                float d = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // byte m of word j holds elements 8j + 2m (low nibble) and 8j + 2m + 1 (high)
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t byte = (qw[j] >> (8 * m)) & 0xFFu;
                        const uint32_t hpair = hw[4 * j + m];
                        d = fmaf((float)(byte & 0xFu), bf16_lo(hpair), d);
                        d = fmaf((float)(byte >> 4), bf16_hi(hpair), d);
                    }
                }
                acc[r] = fmaf(s, d, fmaf(bb, hsum[r * nvec + i], acc[r]));
            }
        }
        warp_sum<R>(acc);
        if (logits) store_logits<R>(logits, acc, acc, false, v, V, r0, rows, lane);
        if (lane == 0)
#pragma unroll
            for (int r = 0; r < R; ++r) {
                unsigned long long k = pack_best(acc[r], (uint32_t)v);
                if (k > mine[r]) mine[r] = k;
            }
    }
    merge_best<R>(mine, s_best, best, r0, rows);
}

// best[0 .. rows) = 0, the neutral element of the packed-key maximum (a kernel, not a memset, so that the
// launches around it keep their programmatic overlap).
__global__ void lm_zero_best_kernel(unsigned long long* __restrict__ best, int rows) {
    griddep_begin();
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) best[r] = 0ull;
}

__global__ void lm_unpack_kernel(const unsigned long long* __restrict__ best, int rows, int32_t* __restrict__ argmax,
                                 float* __restrict__ maxlogit) {
    griddep_begin();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const unsigned long long k = best[r];
    argmax[r] = (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
    if (maxlogit) maxlogit[r] = unorderable((uint32_t)(k >> 32));
}

template <int R>
static void launch_group(int grid_unused, cudaStream_t st, const uint16_t* hidden, int rows, int H, int V,
                         int w_dtype, const void* W, const void* scales, const void* biases, unsigned long long* best,
                         int r0, float* logits) {
    (void)grid_unused;
    // one wave: the resident CTAs per SM the launch bounds allow (3 up to 4 rows, 2 for 8)
    const int grid = sm_count() * (R <= 4 ? 3 : 2);
    if (w_dtype == TSV_Q4_G64) {
        const size_t sm = (size_t)R * (H >> 3) * 16 + (size_t)R * (H >> 5) * 4;
        cudaFuncSetAttribute(lm_gemv_q4_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        launch_pdl(lm_gemv_q4_kernel<R>, grid, kLmThreads, sm, st, hidden, rows, H, V, (const uint8_t*)W,
                                                           (const uint16_t*)scales, (const uint16_t*)biases, best, r0,
                                                           logits);
    } else {
        const size_t sm = (size_t)R * (H >> 3) * 16;
        if (w_dtype == TSV_BF16) {
            cudaFuncSetAttribute(lm_gemv16_kernel<R, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            launch_pdl(lm_gemv16_kernel<R, true>, grid, kLmThreads, sm, st, hidden, rows, H, V, (const uint16_t*)W, best, r0,
                                                                    logits);
        } else {
            cudaFuncSetAttribute(lm_gemv16_kernel<R, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            launch_pdl(lm_gemv16_kernel<R, false>, grid, kLmThreads, sm, st, hidden, rows, H, V, (const uint16_t*)W, best, r0,
                                                                     logits);
        }
    }
}

}  // namespace tsv

namespace tsv {
// Defined in lm_head_tc.cu.
size_t lm_tc_extra_bytes(int rows, int H, int w_dtype);
bool lm_tc_applies(int rows, int H, int V, int w_dtype);
tsv_status launch_lm_tc(const void* hidden, int rows, int H, int V, int w_dtype, const void* W, const void* scales,
                        const void* biases, unsigned long long* best, float* logits, void* extra, cudaStream_t stream);
static size_t best_bytes(int rows) { return ((size_t)rows * sizeof(unsigned long long) + 255) & ~(size_t)255; }
}  // namespace tsv

extern "C" size_t tsv_lm_head_workspace_size(int32_t rows, int32_t H, int32_t V, int32_t w_dtype) {
    using namespace tsv;
    if (rows < 1 || H < 1 || V < 1) return 0;
    size_t n = best_bytes(rows);
    if (lm_tc_applies(rows, H, V, w_dtype)) n += lm_tc_extra_bytes(rows, H, w_dtype);
    return n;
}

namespace tsv {

// Shared body of tsv_lm_head_argmax (argmax != NULL) and tsv_lm_head_logits (logits != NULL).
static tsv_status lm_head_run(const char* name, const void* hidden, int32_t rows, int32_t H, int32_t V,
                              int32_t w_dtype, const void* W, const void* scales, const void* biases, int32_t* argmax,
                              float* maxlogit, float* logits, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    if (rows < 1 || V < 1 || H < 64) return fail(TSV_EINVAL, "%s: rows=%d V=%d H=%d", name, rows, V, H);
    if (!hidden || !W || !(argmax || logits) || !workspace) return fail(TSV_EINVAL, "%s: null pointer argument", name);
    if (w_dtype != TSV_F16 && w_dtype != TSV_BF16 && w_dtype != TSV_Q4_G64)
        return fail(TSV_EUNSUPPORTED, "%s: weight format %d (fp16, bf16 or 4-bit group-64 only)", name, w_dtype);
    if (w_dtype == TSV_Q4_G64) {
        if (H % 64) return fail(TSV_EINVAL, "%s: H=%d not a multiple of the 64-wide group", name, H);
        if (!scales || !biases) return fail(TSV_EINVAL, "%s: 4-bit head without scales/biases", name);
    } else if (H % 256) {
        return fail(TSV_EINVAL, "%s: H=%d not a multiple of 256", name, H);
    }
    if ((size_t)H * 17 > 200 * 1024) return fail(TSV_ECAPACITY, "%s: H=%d above the supported 12,000", name, H);
    if (((uintptr_t)hidden | (uintptr_t)W) & 15) return fail(TSV_EINVAL, "%s: hidden/W not 16-byte aligned", name);
    if (ws_bytes < best_bytes(rows))
        return fail(TSV_ECAPACITY, "%s: workspace %zu < %zu bytes", name, ws_bytes, best_bytes(rows));
    unsigned long long* best = (unsigned long long*)workspace;
    launch_pdl(lm_zero_best_kernel, std::min((rows + 255) / 256, sm_count()), 256, 0, stream, best, rows);
    // The tensor-core kernels where they apply (every 4-bit head; a 16-bit head with more rows than one GEMV
    // pass serves), when the workspace also holds what they need.
    const bool sb_aligned = w_dtype != TSV_Q4_G64 || ((((uintptr_t)scales | (uintptr_t)biases) & 15) == 0);
    if (lm_tc_applies(rows, H, V, w_dtype) && sb_aligned &&
        ws_bytes >= best_bytes(rows) + lm_tc_extra_bytes(rows, H, w_dtype)) {
        tsv_status st = launch_lm_tc(hidden, rows, H, V, w_dtype, W, scales, biases, best, logits,
                                     (char*)workspace + best_bytes(rows), stream);
        if (st != TSV_OK || !argmax) return st;
        launch_pdl(lm_unpack_kernel, (rows + 127) / 128, 128, 0, stream, best, rows, argmax, maxlogit);
        return check_launch(name);
    }
    const int grid = sm_count() * 4;
    const uint16_t* hb = (const uint16_t*)hidden;
    for (int r0 = 0; r0 < rows;) {
        const int left = rows - r0;
        if (left >= 8) { launch_group<8>(grid, stream, hb, rows, H, V, w_dtype, W, scales, biases, best, r0, logits); r0 += 8; }
        else if (left >= 4) { launch_group<4>(grid, stream, hb, rows, H, V, w_dtype, W, scales, biases, best, r0, logits); r0 += 4; }
        else if (left == 3) { launch_group<3>(grid, stream, hb, rows, H, V, w_dtype, W, scales, biases, best, r0, logits); r0 += 3; }
        else if (left == 2) { launch_group<2>(grid, stream, hb, rows, H, V, w_dtype, W, scales, biases, best, r0, logits); r0 += 2; }
        else { launch_group<1>(grid, stream, hb, rows, H, V, w_dtype, W, scales, biases, best, r0, logits); r0 += 1; }
        tsv_status st = check_launch(name);
        if (st != TSV_OK) return st;
    }
    if (!argmax) return TSV_OK;
    launch_pdl(lm_unpack_kernel, (rows + 127) / 128, 128, 0, stream, best, rows, argmax, maxlogit);
    return check_launch(name);
}

}  // namespace tsv

extern "C" tsv_status tsv_lm_head_argmax(const void* hidden, int32_t rows, int32_t H, int32_t V, int32_t w_dtype,
                                         const void* W, const void* scales, const void* biases, int32_t* argmax,
                                         float* maxlogit, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (!argmax) return fail(TSV_EINVAL, "lm_head_argmax: null pointer argument");
    return lm_head_run("lm_head_argmax", hidden, rows, H, V, w_dtype, W, scales, biases, argmax, maxlogit, nullptr,
                       workspace, ws_bytes, stream);
}

extern "C" tsv_status tsv_lm_head_logits(const void* hidden, int32_t rows, int32_t H, int32_t V, int32_t w_dtype,
                                         const void* W, const void* scales, const void* biases, float* logits,
                                         void* workspace, size_t ws_bytes, cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (!logits) return fail(TSV_EINVAL, "lm_head_logits: null pointer argument");
    return lm_head_run("lm_head_logits", hidden, rows, H, V, w_dtype, W, scales, biases, nullptr, nullptr, logits,
                       workspace, ws_bytes, stream);
}

// ---------------------------------------------------------------------------
// tsv_lm_head_argmax_noalloc: the same projection + argmax for callers that
// cannot hand the library a workspace.  Its scratch (one 64-bit running best
// per hidden row) lives in a fixed array in this library's device image
// instead of caller memory; every GPU that loads the library keeps the array
// until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace tsv {

static __device__ __align__(256) unsigned long long g_lm_noalloc_best[TSV_NOALLOC_MAX_ROWS];

// Device address of the scratch array on the current device, looked up once
// per device with that device current.  The array's name in host code is only
// a host-side handle, never a device address, so it is never passed to a
// kernel directly.
static tsv_status noalloc_scratch(void** out) {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(TSV_ECUDA, "lm_head_argmax_noalloc: cudaGetDevice: %s", cudaGetErrorName(e));
    if (dev < 0 || dev >= 64) return fail(TSV_EUNSUPPORTED, "lm_head_argmax_noalloc: device ordinal %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_lm_noalloc_best);
        if (e != cudaSuccess || p == nullptr)
            return fail(TSV_ECUDA, "lm_head_argmax_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorName(e));
        addr[dev] = p;
    }
    *out = addr[dev];
    return TSV_OK;
}

}  // namespace tsv

extern "C" tsv_status tsv_lm_head_argmax_noalloc(const void* hidden, int32_t rows, int32_t H, int32_t V,
                                                 int32_t w_dtype, const void* W, const void* scales,
                                                 const void* biases, int32_t* argmax, float* maxlogit,
                                                 cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (rows > TSV_NOALLOC_MAX_ROWS)
        return fail(TSV_ECAPACITY, "lm_head_argmax_noalloc: rows=%d exceeds the fixed scratch of %d rows "
                                   "(use tsv_lm_head_argmax with a workspace)", rows, TSV_NOALLOC_MAX_ROWS);
    if (rows < 1) return fail(TSV_EINVAL, "lm_head_argmax_noalloc: rows=%d", rows);
    void* scratch = nullptr;
    tsv_status st = noalloc_scratch(&scratch);
    if (st != TSV_OK) return st;
    // The workspace call clears the rows' entries on the stream before use.
    return tsv_lm_head_argmax(hidden, rows, H, V, w_dtype, W, scales, biases, argmax, maxlogit, scratch,
                              sizeof(g_lm_noalloc_best), stream);
}
