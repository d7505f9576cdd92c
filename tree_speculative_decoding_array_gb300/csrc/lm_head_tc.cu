// Tensor-core (tcgen05) path of tsv_lm_head_argmax for many hidden rows.
//
// Same operation as the CUDA-core GEMV in lm_head.cu (mlxcel issue #1185,
// "Phase 2" item 2a: projection fused with the argmax, logits never written;
// "Phase 3": affine group-64 4-bit weights), for row counts where streaming
// the head once per 8 rows would make the CUDA-core path compute-bound.
//
// Swap-AB: one MMA tile is D[128 vocabulary rows x NP hidden rows] =
// W_tile[128 x 64] . hidden_chunk[NP x 64]^T, accumulated over H / 64
// k-blocks in TMEM (two 256-column buffers, so the argmax of one vocabulary
// tile overlaps the MMAs of the next).  Warps:
//   0-3   epilogue: TMEM lane = vocabulary row; per hidden row (column) a
//         warp-shuffle max of the packed (logit, ~index) key, then a shared
//         atomic max; the CTA's bests go to global memory once at the end.
//   4     TMA producer (W block [128 x 64] swizzled, or the raw 4-bit block
//         [128 x 32 bytes]; hidden block [NP x 64] swizzled) into a ring of
//         as many stages (up to 16) as shared memory holds for this NP, so
//         that narrow hidden chunks still keep ~100 KB per SM in flight.
//   5     TMEM allocation and MMA issue.
//   6-13  (4-bit heads) converter: w = scale * q + bias evaluated in fp16
//         with one rounding (q exact via the 1024 + q trick), written into
//         a separate 3-stage ring of swizzled A blocks.  The hidden rows arrive as fp16 too (a copy
//         made by a small kernel into the workspace); fp16 keeps the
//         dequantised weights within 2^-11 relative.
// A CTA keeps one chunk of hidden rows and walks vocabulary tiles strided
// by the number of CTAs per chunk, so CTAs working on one tile run together
// and the tile's second and later reads hit L2.
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace tsv {

constexpr int kLmM = 128;
constexpr int kLmKB = 64;
constexpr int kLmEpi = 128;
constexpr int kLmConv = 256;

struct LmTcParams {
    CUtensorMap wmap;
    CUtensorMap hmap;
    const uint16_t* scales;
    const uint16_t* biases;
    unsigned long long* best;
    int rows, H, V, NP, nchunks, vtiles, mma_bf16, stages, stage_bytes;
    int sb_vec;  // scales/biases 16-byte aligned with H / 64 a multiple of 8: 8 groups per vector load
};

constexpr int kLmMaxStages = 16;
constexpr int kLmConvStages = 3;
constexpr int kLmSmem = 224 * 1024;     // dynamic shared memory requested
constexpr int kLmUsable = kLmSmem - 1024 - 4096;  // minus alignment slack and the tail (bests + barriers)

template <bool Q4>
struct LmLayout {
    static constexpr int kW = Q4 ? 4096 : 16384;  // per stage: raw 4-bit block [128 x 32 B] or W block [128 x 64]
    static constexpr int kConv = Q4 ? kLmConvStages * 16384 : 0;  // dequantised fp16 A blocks
    static constexpr int kThreads = Q4 ? kLmEpi + 64 + kLmConv : kLmEpi + 64;
};

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int o) {
    const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)v, o);
    const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), o);
    return ((uint64_t)hi << 32) | lo;
}

// Shared memory: [conv ring (4-bit)] [TMA ring: stages x (W or raw block | hidden block)] ... [bests | barriers]
template <bool Q4>
__global__ void __launch_bounds__(LmLayout<Q4>::kThreads, 1) lm_tc_kernel(const __grid_constant__ LmTcParams p) {
    using L = LmLayout<Q4>;
    const int S = p.stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* conv = sm;                // [kLmConvStages][128 x 64] fp16 (4-bit heads)
    uint8_t* ring = sm + L::kConv;     // [S][stage_bytes]
    uint8_t* tail = sm + kLmUsable;
    unsigned long long* s_best = reinterpret_cast<unsigned long long*>(tail);  // [256]
    uint64_t* bars = reinterpret_cast<uint64_t*>(tail + 2048);
    uint64_t* full = bars;                       // [16]
    uint64_t* empty = bars + 16;                 // [16]
    uint64_t* conv_full = bars + 32;             // [3]
    uint64_t* conv_empty = bars + 35;            // [3]
    uint64_t* acc_full = bars + 38;              // [2]
    uint64_t* acc_empty = bars + 40;             // [2]
    uint64_t* drain = bars + 42;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 43);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 44);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x % p.nchunks;
    const int group = blockIdx.x / p.nchunks;
    const int groups = gridDim.x / p.nchunks;
    const int KB = p.H / kLmKB;
    const int nrows = min(p.NP, p.rows - chunk * p.NP);  // real hidden rows of this chunk
    if (group >= p.vtiles || nrows <= 0) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], Q4 ? 1 + kLmConv / 32 : 1);
        }
        for (int s = 0; s < kLmConvStages; ++s) {
            tc::mbar_init(&conv_full[s], kLmConv / 32);
            tc::mbar_init(&conv_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&acc_full[s], 1);
            tc::mbar_init(&acc_empty[s], kLmEpi / 32);
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    for (int c = threadIdx.x; c < 256; c += blockDim.x) s_best[c] = 0ull;
    if (warp == 5) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t b_bytes = (uint32_t)p.NP * 128;

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tc::tma_prefetch_desc(&p.wmap);
            tc::tma_prefetch_desc(&p.hmap);
            int g = 0, issued = 0;
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups) {
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const int st = g % S;
                    if (g >= S && !tc::mbar_wait(&empty[st], ((g / S) - 1) & 1, abort_flag)) { ok = false; break; }
                    uint8_t* stage = ring + st * p.stage_bytes;
                    tc::mbar_expect_tx(&full[st], L::kW + b_bytes);
                    if (Q4) tc::tma_load_2d(stage, &p.wmap, &full[st], kb * 32, vt * kLmM);
                    else tc::tma_load_2d(stage, &p.wmap, &full[st], kb * kLmKB, vt * kLmM);
                    tc::tma_load_2d(stage + L::kW, &p.hmap, &full[st], kb * kLmKB, chunk * p.NP);
                    issued = g + 1;
                }
            }
            if (*abort_flag)
                for (int q = max(0, issued - S); q < issued; ++q) {
                    const uint64_t t0 = tc::globaltimer();
                    while (!tc::mbar_try_wait(&full[q % S], (q / S) & 1))
                        if (tc::globaltimer() - t0 > 200000000ull) break;
                }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16(p.mma_bf16 != 0, false, false, kLmM, p.NP);
            const uint32_t rbase = tc::smem_u32(ring), cbase = tc::smem_u32(conv);
            int g = 0, it = 0;
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups, ++it) {
                const int buf = it & 1;
                if (it >= 2 && !tc::mbar_wait_spin(&acc_empty[buf], ((it >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const int st = g % S, cs = g % kLmConvStages;
                    if (!tc::mbar_wait_spin(&full[st], (g / S) & 1, abort_flag)) { ok = false; break; }
                    if (Q4 && !tc::mbar_wait_spin(&conv_full[cs], (g / kLmConvStages) & 1, abort_flag)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t sa = Q4 ? cbase + cs * 16384 : rbase + st * p.stage_bytes;
                    const uint32_t sb = rbase + st * p.stage_bytes + L::kW;
#pragma unroll
                    for (int kk = 0; kk < kLmKB / 16; ++kk)
                        tc::mma_f16(tmem + buf * 256, tc::sdesc_sw128(sa + kk * 32, 16, 1024),
                                    tc::sdesc_sw128(sb + kk * 32, 16, 1024), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    tc::mma_commit(&empty[st]);
                    if (Q4) tc::mma_commit(&conv_empty[cs]);
                }
                if (ok) tc::mma_commit(&acc_full[buf]);
            }
            tc::mma_commit(drain);
            const uint64_t t0 = tc::globaltimer();
            while (!tc::mbar_try_wait(drain, 0))
                if (tc::globaltimer() - t0 > 200000000ull) break;
        }
    } else if (Q4 && warp >= 6) {
        // ------------------------------------------------------------ 4-bit converter
        const int ct = threadIdx.x - (kLmEpi + 64);
        const int row = ct >> 1, half = ct & 1;
        const int ng = p.H >> 6;
        const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
        // Scales and biases of this thread's row, 8 groups per 16-byte load, fetched one group of 8 ahead.
        const bool vec = p.sb_vec != 0;
        uint4 s_cur = make_uint4(0, 0, 0, 0), b_cur = s_cur, s_nxt = s_cur, b_nxt = s_cur;
        auto fetch8 = [&](int vt_, int kb_) {
            const int v_ = vt_ * kLmM + row;
            if (vt_ < p.vtiles && v_ < p.V && kb_ < KB) {
                s_nxt = *reinterpret_cast<const uint4*>(p.scales + (size_t)v_ * ng + kb_);
                b_nxt = *reinterpret_cast<const uint4*>(p.biases + (size_t)v_ * ng + kb_);
            }
        };
        if (vec) fetch8(group, 0);
        int g = 0;
        bool ok = true;
        for (int vt = group; ok && vt < p.vtiles; vt += groups) {
            const int v = vt * kLmM + row;
            const bool vok = v < p.V;
            for (int kb = 0; kb < KB; ++kb, ++g) {
                const int st = g % S, cs = g % kLmConvStages;
                float sc, bi;
                if (vec) {
                    if ((kb & 7) == 0) {
                        s_cur = s_nxt;
                        b_cur = b_nxt;
                        if (kb + 8 < KB) fetch8(vt, kb + 8);
                        else fetch8(vt + groups, 0);
                    }
                    const int e = kb & 7, wsel = e >> 1;
                    const uint32_t sw = wsel == 0 ? s_cur.x : wsel == 1 ? s_cur.y : wsel == 2 ? s_cur.z : s_cur.w;
                    const uint32_t bw = wsel == 0 ? b_cur.x : wsel == 1 ? b_cur.y : wsel == 2 ? b_cur.z : b_cur.w;
                    sc = vok ? ((e & 1) ? bf16_hi(sw) : bf16_lo(sw)) : 0.f;
                    bi = vok ? ((e & 1) ? bf16_hi(bw) : bf16_lo(bw)) : 0.f;
                } else {
                    sc = vok ? bf16_bits_to_f32(p.scales[(size_t)v * ng + kb]) : 0.f;
                    bi = vok ? bf16_bits_to_f32(p.biases[(size_t)v * ng + kb]) : 0.f;
                }
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&full[st], (g / S) & 1, abort_flag))) { ok = false; break; }
                if (g >= kLmConvStages &&
                    !__all_sync(0xFFFFFFFFu, tc::mbar_wait(&conv_empty[cs], ((g / kLmConvStages) - 1) & 1, abort_flag))) { ok = false; break; }
                const uint4 raw = *reinterpret_cast<const uint4*>(ring + st * p.stage_bytes + row * 32 + half * 16);
                const __half2 s2 = __floats2half2_rn(sc, sc), b2 = __floats2half2_rn(bi, bi);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                uint32_t out[16];
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int by = 0; by < 4; ++by) {
                        const uint32_t x = w[k] >> (8 * by);
                        uint32_t h = (x & 0xFu) | ((x & 0xF0u) << 12) | 0x64006400u;  // (1024 + lo, 1024 + hi)
                        __half2 q = __hsub2(*reinterpret_cast<__half2*>(&h), k1024);
                        __half2 r = __hfma2(q, s2, b2);
                        out[4 * k + by] = *reinterpret_cast<uint32_t*>(&r);
                    }
                uint8_t* arow = conv + cs * 16384 + row * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int chk = half * 4 + q;
                    *reinterpret_cast<uint4*>(arow + ((chk ^ (row & 7)) << 4)) =
                        make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&empty[st]);
                    tc::mbar_arrive(&conv_full[cs]);
                }
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ argmax epilogue
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        int it = 0;
        for (int vt = group; vt < p.vtiles; vt += groups, ++it) {
            const int buf = it & 1;
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&acc_full[buf], (it >> 1) & 1, abort_flag))) break;
            tc::tc_fence_after();
            const int v = vt * kLmM + warp * 32 + lane;
            for (int c0 = 0; c0 < nrows; c0 += 32) {
                uint32_t d[32];
                tc::tmem_ld32(tmem + lane_base + buf * 256 + c0, d);
                tc::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    if (c0 + k < nrows) {  // uniform across the warp
                        uint64_t key = v < p.V ? pack_best(__uint_as_float(d[k]), (uint32_t)v) : 0ull;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const uint64_t other = shfl_xor_u64(key, o);
                            key = other > key ? other : key;
                        }
                        if (lane == 0) atomicMax(&s_best[c0 + k], (unsigned long long)key);
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
        }
    }

    __syncthreads();
    if (!*abort_flag)
        for (int c = threadIdx.x; c < nrows; c += blockDim.x)
            if (s_best[c]) atomicMax(&p.best[chunk * p.NP + c], s_best[c]);
    if (warp == 5) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// bf16 hidden rows -> fp16 copy (operand type of the fp16 MMA).
__global__ void hidden_to_f16_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n / 2; i += (size_t)gridDim.x * blockDim.x) {
        const uint32_t w = reinterpret_cast<const uint32_t*>(in)[i];
        __half2 h = __floats2half2_rn(bf16_lo(w), bf16_hi(w));
        reinterpret_cast<uint32_t*>(out)[i] = *reinterpret_cast<uint32_t*>(&h);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*LmEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static LmEncodeFn lm_encode_fn() {
    static LmEncodeFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<LmEncodeFn>(f);
    }
    return fn;
}

static bool map2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box0, uint32_t box1, bool swizzle) {
    LmEncodeFn enc = lm_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box0, box1};
    cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bytes of workspace the tensor-core path needs beyond the per-row bests
// (the fp16 copy of hidden when the MMA runs in fp16).
size_t lm_tc_extra_bytes(int rows, int H, int w_dtype) {
    return w_dtype == TSV_BF16 ? 0 : (((size_t)rows * H * 2 + 255) & ~(size_t)255);
}

bool lm_tc_applies(int rows, int H, int V, int w_dtype) {
    return rows > 8 && H % 64 == 0 && V >= 1 && (w_dtype == TSV_Q4_G64 || H % 64 == 0);
}

tsv_status launch_lm_tc(const void* hidden, int rows, int H, int V, int w_dtype, const void* W, const void* scales,
                        const void* biases, unsigned long long* best, void* extra, cudaStream_t stream) {
    static thread_local LmTcParams prm;
    const bool q4 = w_dtype == TSV_Q4_G64;
    const int nchunks = (rows + 255) / 256;
    int NP = (rows + nchunks - 1) / nchunks;
    NP = ((NP + 15) / 16) * 16;
    const void* hsrc = hidden;
    if (w_dtype != TSV_BF16) {  // fp16 MMA: fp16 copy of hidden
        const size_t n = (size_t)rows * H;
        hidden_to_f16_kernel<<<sm_count() * 4, 256, 0, stream>>>((const uint16_t*)hidden, (uint16_t*)extra, n);
        tsv_status st = check_launch("lm_head_argmax(hidden fp16)");
        if (st != TSV_OK) return st;
        hsrc = extra;
    }
    bool ok;
    if (q4)
        ok = map2d(&prm.wmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)H / 2, (uint64_t)V, (uint64_t)H / 2, 32,
                   kLmM, false);
    else
        ok = map2d(&prm.wmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, 64, kLmM,
                   true);
    ok = ok && map2d(&prm.hmap, hsrc, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)H, (uint64_t)rows, (uint64_t)H * 2, 64,
                     (uint32_t)NP, true);
    if (!ok) return fail(TSV_ECUDA, "lm_head_argmax: tensor map encoding failed");
    prm.scales = (const uint16_t*)scales;
    prm.sb_vec = q4 && (H / 64) % 8 == 0 && (((uintptr_t)scales | (uintptr_t)biases) & 15) == 0;
    prm.biases = (const uint16_t*)biases;
    prm.best = best;
    prm.rows = rows;
    prm.H = H;
    prm.V = V;
    prm.NP = NP;
    prm.nchunks = nchunks;
    prm.vtiles = (V + kLmM - 1) / kLmM;
    prm.mma_bf16 = w_dtype == TSV_BF16;
    const int wbytes = q4 ? LmLayout<true>::kW : LmLayout<false>::kW;
    const int conv_bytes = q4 ? LmLayout<true>::kConv : 0;
    prm.stage_bytes = wbytes + NP * 128;  // multiples of 1024: every block stays 1024-aligned
    int stages = (kLmUsable - conv_bytes) / prm.stage_bytes;
    prm.stages = stages > kLmMaxStages ? kLmMaxStages : stages;
    if (prm.stages < 2) return fail(TSV_EUNSUPPORTED, "lm_head_argmax: hidden chunk too wide for the pipeline");
    const int sms = sm_count();
    const int groups = sms / nchunks > 0 ? sms / nchunks : 1;
    const int grid = groups * nchunks;
    if (q4) {
        cudaFuncSetAttribute(lm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLmSmem);
        lm_tc_kernel<true><<<grid, LmLayout<true>::kThreads, kLmSmem, stream>>>(prm);
    } else {
        cudaFuncSetAttribute(lm_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLmSmem);
        lm_tc_kernel<false><<<grid, LmLayout<false>::kThreads, kLmSmem, stream>>>(prm);
    }
    return check_launch("lm_head_argmax(tcgen05)");
}

}  // namespace tsv
