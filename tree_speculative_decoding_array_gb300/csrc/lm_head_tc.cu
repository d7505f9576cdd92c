// Tensor-core (tcgen05) paths of tsv_lm_head_argmax for many hidden rows.
//
// Same operation as the CUDA-core GEMV in lm_head.cu (mlxcel issue #1185,
// "Phase 2" item 2a: projection fused with the argmax, logits never written;
// "Phase 3": affine group-64 4-bit weights), for every 4-bit head and for
// 16-bit heads with more rows than one pass of the CUDA-core GEMV serves: there
// the GEMV would be bound by its arithmetic or stream the head more than once.
//
// Swap-AB: one MMA tile is D[128 vocabulary rows x NP hidden rows] =
// W_tile[128 x 64] . hidden_chunk[NP x 64]^T, accumulated over H / 64
// k-blocks in TMEM (two accumulator buffers, so the argmax of one vocabulary
// tile overlaps the MMAs of the next).  A CTA keeps one chunk of hidden rows
// and walks vocabulary tiles strided by the number of CTAs per chunk, so CTAs
// working on one tile run together and the tile's second and later reads hit
// L2.  The epilogue (warps 0-3, TMEM lane = vocabulary row) finds, per hidden
// row, the warp's largest logit with a 32-bit warp maximum and the lowest lane
// holding it, and merges the packed (logit, ~index) key with a shared atomic
// maximum; the CTA's bests go to global memory once at the end.
//
// 16-bit heads (lm_tc_kernel): warp 4 streams W blocks [128 x 64] from HBM
// through a ring of up to 16 stages, warp 6 the hidden blocks [NP x 64] (L2
// hits after the first vocabulary tile) through a ring of 3-4 (both 128-byte
// swizzled): the W ring carries the DRAM latency, so it gets the shared
// memory; warp 5 issues the MMAs from shared memory.
//
// 4-bit heads (lm_q4_kernel): the dequantised weights never touch shared
// memory.  Warp 4 streams the raw codes of 8 k-blocks plus their scales and
// biases per stage, warp 22 the hidden blocks, through separate rings;
// 16 converter warps (6-21) evaluate w = scale * q + bias in fp16 with one
// rounding (q exact via the 1024 + q bit trick) and store the A operand
// straight into TMEM slots with tcgen05.st; warp 5 issues MMAs whose A
// operand is read from TMEM.  The converter emits a code word's 8 features in
// the order (0,4,1,5,2,6,3,7) (one mask per pair of features); the fp16 copy
// of the hidden rows is written in the same order, so both operands agree.
// fp16 keeps the dequantised weights within 2^-11 relative.
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace tsv {

constexpr int kLmM = 128;
constexpr int kLmKB = 64;
constexpr int kLmEpi = 128;
constexpr int kLmSmem = 224 * 1024;               // dynamic shared memory requested
constexpr int kLmUsable = kLmSmem - 1024 - 4096;  // minus alignment slack and the tail (bests + barriers)

// ------------------------------------------------------------------ shared pieces
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Argmax of one accumulator tile over this warp's 32 vocabulary rows, for each of the nrows hidden rows (TMEM
// columns starting at taddr).  v = this lane's vocabulary row; rows >= V never win; ties go to the lowest row.
// With logits != NULL every logit is also written to logits[row0 + column][v] (sampled verification).  Each warp
// keeps a best per hidden row in its own row of wbest (no atomics, no divergent branch): per 32 columns the 32
// warp maxima and ballots first (independent of each other), then lane k takes column k's result and updates
// wbest[c0 + k] with a plain compare and store; the CTA merges its warps' rows at the end.  A shared 64-bit atomic
// per column behind a lane-0 branch, four warps contending, had made this epilogue slower than a 256-column
// tile's MMAs.
template <bool LOGITS>
__device__ __forceinline__ void lm_epilogue_warp(uint32_t taddr, int nrows, int v, int V, unsigned long long* wbest,
                                                 int lane, float* logits, int row0) {
    const uint32_t v0 = (uint32_t)(v - lane);
    for (int c0 = 0; c0 < nrows; c0 += 32) {
        uint32_t d[32];
        tc::tmem_ld32(taddr + c0, d);
        tc::tmem_wait_ld();
        uint32_t my_mx = 0u, my_who = 0u;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (LOGITS && v < V && c0 + k < nrows) logits[(size_t)(row0 + c0 + k) * V + v] = __uint_as_float(d[k]);
            const uint32_t o = v < V ? orderable(__uint_as_float(d[k])) : 0u;
            const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, o);
            const uint32_t who = __ballot_sync(0xFFFFFFFFu, o == mx);
            if (k == lane) {  // a predicated move: k is a constant of the unrolled loop
                my_mx = mx;
                my_who = who;
            }
        }
        const int c = c0 + lane;
        if (c < nrows && my_mx != 0u) {
            const uint32_t idx = v0 + (uint32_t)(__ffs(my_who) - 1);
            const unsigned long long key = ((unsigned long long)my_mx << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
            if (key > wbest[c]) wbest[c] = key;
        }
    }
}

// lm_epilogue_warp over the sum (fp32) of NI accumulators (columns taddr + i * DC), CW columns at a time (lanes
// 0 .. CW - 1 take the columns; CW = 8 or 16, which the 4-bit few-row kernel's register budget allows).
template <bool LOGITS, int NI, int CW>
__device__ __forceinline__ void lm_epilogue_sum_warp(uint32_t taddr, int DC, int nrows, int v, int V,
                                                     unsigned long long* wbest, int lane, float* logits, int row0) {
    const uint32_t v0 = (uint32_t)(v - lane);
    for (int c0 = 0; c0 < nrows; c0 += CW) {
        float acc[CW];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            uint32_t d[CW];
            if constexpr (CW == 8) tc::tmem_ld8(taddr + (uint32_t)(i * DC) + c0, d);
            else tc::tmem_ld16(taddr + (uint32_t)(i * DC) + c0, d);
            tc::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < CW; ++k) acc[k] = i == 0 ? __uint_as_float(d[k]) : acc[k] + __uint_as_float(d[k]);
        }
        uint32_t my_mx = 0u, my_who = 0u;
#pragma unroll
        for (int k = 0; k < CW; ++k) {
            if (LOGITS && v < V && c0 + k < nrows) logits[(size_t)(row0 + c0 + k) * V + v] = acc[k];
            const uint32_t o = v < V ? orderable(acc[k]) : 0u;
            const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, o);
            const uint32_t who = __ballot_sync(0xFFFFFFFFu, o == mx);
            if (k == lane) {
                my_mx = mx;
                my_who = who;
            }
        }
        const int c = c0 + lane;
        if (lane < CW && c < nrows && my_mx != 0u) {
            const uint32_t idx = v0 + (uint32_t)(__ffs(my_who) - 1);
            const unsigned long long key = ((unsigned long long)my_mx << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
            if (key > wbest[c]) wbest[c] = key;
        }
    }
}

// Bounded wait used only while draining after an abort.
__device__ __forceinline__ void lm_drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(bar, parity))
        if (tc::globaltimer() - t0 > 200000000ull) break;  // 200 ms
}

// ------------------------------------------------------------------ 16-bit heads
constexpr int kLmMaxStages = 16;
constexpr int kLmUsable16 = kLmUsable - 6144;  // the 16-bit kernel's rings end here: per-warp bests [4][256] follow
constexpr int kLmHStages256 = 4;  // hidden stages at 256 rows (32 KB each)
constexpr uint32_t kLmProdSleep = 256;  // producers' longest sleep between polls (ns)
constexpr int kLmThreads16 = kLmEpi + 96;

struct LmTcParams {
    CUtensorMap wmap;
    CUtensorMap hmap;
    unsigned long long* best;
    float* logits;  // NULL, or [rows][V] fp32 written by the epilogue
    int rows, H, V, NP, nchunks, vtiles, mma_bf16;
    int stages, hstages;  // W ring stages (16 KB each), hidden ring stages (NP x 128 B each)
};

// Shared memory: [W ring: stages x 16 KB] [hidden ring: hstages x NP*128 B] ... [bests | barriers]
template <bool LOGITS>
__global__ void __launch_bounds__(kLmThreads16, 1) lm_tc_kernel(const __grid_constant__ LmTcParams p) {
    griddep_begin();
    const int S = p.stages, HS = p.hstages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* ring = sm;                  // [S][16 KB]
    uint8_t* hring = sm + S * 16384;     // [HS][NP * 128]
    uint8_t* tail = sm + kLmUsable;
    // each epilogue warp's best per hidden row: [4][256], the last 2 KB in the tail's best slot
    unsigned long long* wbest = reinterpret_cast<unsigned long long*>(sm + kLmUsable16);
    uint64_t* bars = reinterpret_cast<uint64_t*>(tail + 2048);
    // One barrier pair per k-block serves both rings: full[g % S] completes when both producers have armed it
    // for k-block g (two arrivals, each with its own byte count) and its W and hidden blocks have landed,
    // empty[g % S] when its MMAs are done.  The hidden producer refills slot g % HS after the MMAs of k-block
    // g - HS (HS <= S, so it arms full[g % S] only after the phase of k-block g - S has completed).  The MMA
    // thread waits once and commits once per k-block.
    uint64_t* full = bars;            // [16] W and hidden blocks landed
    uint64_t* empty = bars + 16;      // [16] MMAs done with both
    uint64_t* acc_full = bars + 48;   // [2]
    uint64_t* acc_empty = bars + 50;  // [2]
    uint64_t* drain = bars + 52;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 53);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 54);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x % p.nchunks;
    const int group = blockIdx.x / p.nchunks;
    const int groups = gridDim.x / p.nchunks;
    const int KB = p.H / kLmKB;
    const int nrows = min(p.NP, p.rows - chunk * p.NP);  // real hidden rows of this chunk
    if (group >= p.vtiles || nrows <= 0) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(&full[s], 2);
            tc::mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&acc_full[s], 1);
            tc::mbar_init(&acc_empty[s], kLmEpi / 32);
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    for (int c = threadIdx.x; c < 4 * 256; c += blockDim.x) wbest[c] = 0ull;
    if (warp == 5) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t b_bytes = (uint32_t)p.NP * 128;

    if (warp == 4) {
        // ------------------------------------------------------------ W producer
        if (lane == 0) {
            tc::tma_prefetch_desc(&p.wmap);
            int g = 0, issued = 0, st = 0;
            uint32_t fill = 0;  // parity of stage st's current use
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups) {
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    if (g >= S && !tc::mbar_wait(&empty[st], fill ^ 1u, abort_flag, kLmProdSleep)) { ok = false; break; }
                    tc::mbar_expect_tx(&full[st], 16384u);
                    tc::tma_load_2d(ring + st * 16384, &p.wmap, &full[st], kb * kLmKB, vt * kLmM);
                    issued = g + 1;
                    if (++st == S) { st = 0; fill ^= 1u; }
                }
            }
            if (*abort_flag)
                for (int q = max(0, issued - S); q < issued; ++q) lm_drain_wait(&full[q % S], (q / S) & 1);
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ hidden producer (a warp of its own: a lane
        // that sleeps in its wait would hold up the W producer)
        if (lane == 0) {
            tc::tma_prefetch_desc(&p.hmap);
            int g = 0, hs = 0, fs = 0, es = 0;  // k-block, hidden slot, its full[] index, empty[] index of g - HS
            uint32_t eph = 0;                    // parity of that empty[] phase
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups) {
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    if (g >= HS) {
                        if (!tc::mbar_wait(&empty[es], eph, abort_flag, kLmProdSleep)) { ok = false; break; }
                        if (++es == S) { es = 0; eph ^= 1u; }
                    }
                    tc::mbar_expect_tx(&full[fs], b_bytes);
                    tc::tma_load_2d(hring + hs * b_bytes, &p.hmap, &full[fs], kb * kLmKB, chunk * p.NP);
                    if (++hs == HS) hs = 0;
                    if (++fs == S) fs = 0;
                }
            }
            // at most HS copies are in flight: let them land (bounded waits) before the CTA goes away
            if (*abort_flag)
                for (int q = max(0, g - HS); q < g; ++q) lm_drain_wait(&full[q % S], (q / S) & 1);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16(p.mma_bf16 != 0, false, false, kLmM, p.NP);
            const uint64_t dW0 = tc::sdesc_sw128(tc::smem_u32(ring), 16, 1024);
            const uint64_t dH0 = tc::sdesc_sw128(tc::smem_u32(hring), 16, 1024);
            int it = 0, st = 0, hs = 0;
            uint32_t ph = 0;  // phase parity of the W ring
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups, ++it) {
                const int buf = it & 1;
                if (it >= 2 && !tc::mbar_wait_spin(&acc_empty[buf], ((it >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                for (int kb = 0; kb < KB; ++kb) {
                    if (!tc::mbar_wait_spin(&full[st], ph, abort_flag)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint64_t da = tc::sdesc_add(dW0, (uint32_t)st * 16384u);
                    const uint64_t db = tc::sdesc_add(dH0, (uint32_t)hs * b_bytes);
#pragma unroll
                    for (int kk = 0; kk < kLmKB / 16; ++kk)
                        tc::mma_f16(tmem + buf * 256, tc::sdesc_add(da, kk * 32), tc::sdesc_add(db, kk * 32), idesc,
                                    (kb > 0 || kk > 0) ? 1u : 0u);
                    tc::mma_commit(&empty[st]);
                    if (++st == S) { st = 0; ph ^= 1u; }
                    if (++hs == HS) hs = 0;
                }
                if (ok) tc::mma_commit(&acc_full[buf]);
            }
            tc::mma_commit(drain);
            lm_drain_wait(drain, 0);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ argmax epilogue
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        int it = 0;
        for (int vt = group; vt < p.vtiles; vt += groups, ++it) {
            const int buf = it & 1;
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&acc_full[buf], (it >> 1) & 1, abort_flag, 1024))) break;
            tc::tc_fence_after();
            lm_epilogue_warp<LOGITS>(tmem + lane_base + buf * 256, nrows, vt * kLmM + warp * 32 + lane, p.V,
                                     wbest + warp * 256, lane, p.logits, chunk * p.NP);
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(&acc_empty[buf]);
        }
    }

    __syncthreads();
    if (!*abort_flag)
        for (int c = threadIdx.x; c < nrows; c += blockDim.x) {
            unsigned long long b = wbest[c];
#pragma unroll
            for (int w = 1; w < 4; ++w) b = wbest[w * 256 + c] > b ? wbest[w * 256 + c] : b;
            if (b) atomicMax(&p.best[chunk * p.NP + c], b);
        }
    if (warp == 5) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ 4-bit heads
constexpr int kQ4Sets = 4;                            // converter sets; a set = 4 warps, one per TMEM lane quarter
constexpr int kQ4Conv = kQ4Sets * 128;                // converter warps 6 .. 6 + 4 * kQ4Sets - 1
constexpr int kQ4HWarp = 6 + kQ4Conv / 32;            // the hidden-block producer's warp
constexpr int kQ4Threads = kLmEpi + 64 + kQ4Conv + 32;
constexpr int kQ4KBPerStage = 8;                      // k-blocks of 64 features per W stage
constexpr int kQ4WStages = 3;                         // lm_q4_kernel: at most 3 W stages (p.WS)
constexpr int kQ4WStage = 2 * 16384 + 2 * 2048;       // codes [128 rows x 256 B] as two swizzled boxes, scales, biases
constexpr int kQ4MaxHStages = 16;
constexpr int kQ4MaxAGroups = 8;
constexpr int kQ4MaxNP = 128;

struct LmQ4Params {
    CUtensorMap wmap;  // codes, UINT8 [V][H/2], box {128 B, 128 rows}, 128-byte swizzle
    CUtensorMap smap;  // scales, UINT16 [V][H/64], box {8, 128}
    CUtensorMap bmap;  // biases, same
    CUtensorMap hmap;  // fp16 hidden copy in converter feature order, UINT16 [rows][H], box {64, NP}, swizzled
    unsigned long long* best;
    float* logits;     // NULL, or [rows][V] fp32 written by the epilogue
    int rows, H, V, NP, DC, NA, HS, nchunks, vtiles;
    int GK;            // k-blocks per A-slot group and per hidden stage (1, 2 or 4): one wait and one commit each
    int WS;            // W stages
};

// One 32-bit word of codes (features 8j..8j+7, feature 8j+i in bits 4i..4i+3) -> four fp16 pairs
// (8j+m, 8j+m+4), m = 0..3, each w = scale * q + bias with a single rounding.  A code in the low nibble of its
// byte becomes the fp16 1024 + q under the mask (1024 + q - 1024 = q exactly); one in the high nibble becomes
// 1024 + 16 q without a shift, and (1024 + 16 q) / 16 - 64 = q exactly in one fma; one shift of the word by 8
// serves codes m = 2, 3.
__device__ __forceinline__ void q4_word(uint32_t x, __half2 s2, __half2 b2, __half2 k1024, uint32_t* out) {
    const __half2 k16th = __floats2half2_rn(0.0625f, 0.0625f), km64 = __floats2half2_rn(-64.f, -64.f);
    const uint32_t x8 = x >> 8;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t src = m < 2 ? x : x8;
        uint32_t h = (src & ((m & 1) ? 0x00F000F0u : 0x000F000Fu)) | 0x64006400u;
        const __half2 hv = *reinterpret_cast<__half2*>(&h);
        const __half2 q = (m & 1) ? __hfma2(hv, k16th, km64) : __hsub2(hv, k1024);  // (q_m, q_{m+4}), exact
        const __half2 w = __hfma2(q, s2, b2);
        out[m] = *reinterpret_cast<const uint32_t*>(&w);
    }
}

__device__ __forceinline__ uint32_t u4_word(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Row r (= this thread's TMEM lane) of k-block kk of a landed W stage: 64 codes -> 32 fp16 pairs
// w = scale * q + bias, stored to TMEM columns [taddr, taddr + 32) (HALVES: as two stores of 16 columns,
// which keeps fewer registers live).  The caller waits for the store.
template <bool HALVES = false>
__device__ __forceinline__ void q4_convert_row(const uint8_t* st, int r, int kk, float sf, float bf, __half2 k1024,
                                               uint32_t taddr) {
    const __half2 s2 = __floats2half2_rn(sf, sf), b2 = __floats2half2_rn(bf, bf);
    // this row's 32 bytes of codes: 16-byte chunks c0, c0 + 1 of box kk / 4 (128-byte swizzle)
    const uint8_t* rowp = st + (kk >> 2) * 16384 + r * 128;
    const int c0 = (kk & 3) * 2;
    const uint4 lo = *reinterpret_cast<const uint4*>(rowp + ((c0 ^ (r & 7)) << 4));
    const uint4 hi = *reinterpret_cast<const uint4*>(rowp + (((c0 + 1) ^ (r & 7)) << 4));
    if (HALVES) {
        uint32_t h[16];
        q4_word(lo.x, s2, b2, k1024, h + 0);
        q4_word(lo.y, s2, b2, k1024, h + 4);
        q4_word(lo.z, s2, b2, k1024, h + 8);
        q4_word(lo.w, s2, b2, k1024, h + 12);
        tc::tmem_st16(taddr, h);
        q4_word(hi.x, s2, b2, k1024, h + 0);
        q4_word(hi.y, s2, b2, k1024, h + 4);
        q4_word(hi.z, s2, b2, k1024, h + 8);
        q4_word(hi.w, s2, b2, k1024, h + 12);
        tc::tmem_st16(taddr + 16, h);
        return;
    }
    uint32_t out[32];
    q4_word(lo.x, s2, b2, k1024, out + 0);
    q4_word(lo.y, s2, b2, k1024, out + 4);
    q4_word(lo.z, s2, b2, k1024, out + 8);
    q4_word(lo.w, s2, b2, k1024, out + 12);
    q4_word(hi.x, s2, b2, k1024, out + 16);
    q4_word(hi.y, s2, b2, k1024, out + 20);
    q4_word(hi.z, s2, b2, k1024, out + 24);
    q4_word(hi.w, s2, b2, k1024, out + 28);
    tc::tmem_st32(taddr, out);
}

template <bool HALVES = false>
__device__ __forceinline__ void q4_convert_kblock(const uint8_t* st, int r, int kk, const uint4& sc8, const uint4& bi8,
                                                  __half2 k1024, uint32_t taddr) {
    const uint32_t sw = u4_word(sc8, kk >> 1), bw = u4_word(bi8, kk >> 1);
    q4_convert_row<HALVES>(st, r, kk, (kk & 1) ? bf16_hi(sw) : bf16_lo(sw), (kk & 1) ? bf16_hi(bw) : bf16_lo(bw), k1024,
                           taddr);
}

// Shared memory: [W ring: 3 x 36 KB] [hidden ring: HS x NP*128 B] ... [bests | barriers].
// TMEM: accumulators [0, DC) and [DC, 2 DC); from 2 DC, NA groups of GK A slots of 32 columns (one k-block
// each).  Hidden stages hold GK k-blocks too, so the MMA thread waits, fences and commits once per GK k-blocks
// (each M=128 MMA occupies the tensor pipe ~100 cycles at these N; per-k-block barrier traffic would double it).
template <bool LOGITS>
__global__ void __launch_bounds__(kQ4Threads, 1) lm_q4_kernel(const __grid_constant__ LmQ4Params p) {
    griddep_begin();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* wring = sm;
    const int WSt = p.WS;  // W stages: 2 or 3
    uint8_t* hring = sm + WSt * kQ4WStage;
    uint8_t* tail = sm + kLmUsable;
    // each epilogue warp's best per hidden row: [4][128], ending in the tail's best slot
    unsigned long long* wbest = reinterpret_cast<unsigned long long*>(tail - 2048);
    uint64_t* bars = reinterpret_cast<uint64_t*>(tail + 2048);
    uint64_t* wfull = bars;           // [3] codes, scales and biases of a stage landed
    uint64_t* wempty = bars + 3;      // [3] every converter warp is done with the stage
    uint64_t* hfull = bars + 6;       // [16] hidden block landed
    uint64_t* hempty = bars + 22;     // [16] MMAs done with the hidden block
    uint64_t* afull = bars + 38;      // [8] A-slot group written (the converter warps that contribute to it)
    uint64_t* aempty = bars + 52;     // [8] MMAs done with the A-slot group
    uint64_t* acc_full = bars + 66;   // [2]
    uint64_t* acc_empty = bars + 68;  // [2]
    uint64_t* drain = bars + 70;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 71);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 72);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x % p.nchunks;
    const int group = blockIdx.x / p.nchunks;
    const int groups = gridDim.x / p.nchunks;
    const int KB = p.H / kLmKB;
    const int NSt = KB / kQ4KBPerStage;  // W stages per vocabulary tile
    const int NA = p.NA, HS = p.HS, GK = p.GK;  // A-slot groups, hidden stages, k-blocks per group
    const int nrows = min(p.NP, p.rows - chunk * p.NP);
    if (group >= p.vtiles || nrows <= 0) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WSt; ++s) {
            tc::mbar_init(&wfull[s], 1);
            tc::mbar_init(&wempty[s], kQ4Conv / 32);
        }
        for (int s = 0; s < HS; ++s) {
            tc::mbar_init(&hfull[s], 1);
            tc::mbar_init(&hempty[s], 1);
        }
        for (int s = 0; s < NA; ++s) {
            tc::mbar_init(&afull[s], 4 * GK);  // one set (4 warps) converts each k-block of the group
            tc::mbar_init(&aempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&acc_full[s], 1);
            tc::mbar_init(&acc_empty[s], kLmEpi / 32);
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    for (int c = threadIdx.x; c < 4 * kQ4MaxNP; c += blockDim.x) wbest[c] = 0ull;
    if (warp == 5) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t a_col = 2u * (uint32_t)p.DC;
    const uint32_t h_bytes = (uint32_t)p.NP * 128;

    if (warp == 4) {
        if (lane == 0) {
            // -------------------------------------------------------- W stages: codes, scales, biases of 8 k-blocks
            // (each producer has a warp of its own: a lane that sleeps in its wait holds up the other lanes)
            tc::tma_prefetch_desc(&p.wmap);
            tc::tma_prefetch_desc(&p.smap);
            tc::tma_prefetch_desc(&p.bmap);
            int c = 0, issued = 0, s = 0;
            uint32_t fill = 0;  // parity of stage s's current fill
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups) {
                for (int i = 0; i < NSt; ++i, ++c) {
                    if (c >= WSt && !tc::mbar_wait(&wempty[s], fill ^ 1u, abort_flag, 512)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = wring + s * kQ4WStage;
                    tc::mbar_expect_tx(&wfull[s], kQ4WStage);
                    tc::tma_load_2d(st, &p.wmap, &wfull[s], i * 256, vt * kLmM);
                    tc::tma_load_2d(st + 16384, &p.wmap, &wfull[s], i * 256 + 128, vt * kLmM);
                    tc::tma_load_2d(st + 32768, &p.smap, &wfull[s], i * kQ4KBPerStage, vt * kLmM);
                    tc::tma_load_2d(st + 34816, &p.bmap, &wfull[s], i * kQ4KBPerStage, vt * kLmM);
                    issued = c + 1;
                    if (++s == WSt) { s = 0; fill ^= 1u; }
                }
            }
            if (*abort_flag)
                for (int q = max(0, issued - WSt); q < issued; ++q)
                    lm_drain_wait(&wfull[q % WSt], (q / WSt) & 1);
        }
    } else if (warp == kQ4HWarp) {
        if (lane == 0) {
            // -------------------------------------------------------- hidden blocks, GK k-blocks per stage
            tc::tma_prefetch_desc(&p.hmap);
            int g = 0, issued = 0, s = 0;
            uint32_t fill = 0;
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups) {
                for (int kb = 0; kb < KB; kb += GK, ++g) {
                    if (g >= HS && !tc::mbar_wait(&hempty[s], fill ^ 1u, abort_flag, 512)) { ok = false; break; }
                    tc::mbar_expect_tx(&hfull[s], h_bytes * GK);
                    for (int u = 0; u < GK; ++u)
                        tc::tma_load_2d(hring + (s * GK + u) * h_bytes, &p.hmap, &hfull[s], (kb + u) * kLmKB, chunk * p.NP);
                    issued = g + 1;
                    if (++s == HS) { s = 0; fill ^= 1u; }
                }
            }
            if (*abort_flag)
                for (int q = max(0, issued - HS); q < issued; ++q) lm_drain_wait(&hfull[q % HS], (q / HS) & 1);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer: A from TMEM, hidden from smem
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16(false, false, false, kLmM, p.NP);
            const uint64_t hdesc0 = tc::sdesc_sw128(tc::smem_u32(hring), 16, 1024);
            int it = 0, as = 0, hs = 0;
            uint32_t aph = 0, hph = 0;  // phase parities of the A-slot and hidden rings
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups, ++it) {
                const int buf = it & 1;
                if (it >= 2 && !tc::mbar_wait_spin(&acc_empty[buf], ((it >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                for (int kb = 0; kb < KB; kb += GK) {  // one group of GK k-blocks: one wait each, one commit each
                    // short sleeps between polls: this thread shares its SM sub-partition with two converter warps
                    if (!tc::mbar_wait(&afull[as], aph, abort_flag, 64)) { ok = false; break; }
                    if (!tc::mbar_wait(&hfull[hs], hph, abort_flag, 64)) { ok = false; break; }
                    tc::tc_fence_after();
                    for (int u = 0; u < GK; ++u) {
                        const uint32_t a = tmem + a_col + (uint32_t)(as * GK + u) * 32;
                        const uint64_t b = tc::sdesc_add(hdesc0, (uint32_t)(hs * GK + u) * h_bytes);
#pragma unroll
                        for (int kk = 0; kk < kLmKB / 16; ++kk)
                            tc::mma_f16_ts(tmem + buf * p.DC, a + kk * 8, tc::sdesc_add(b, kk * 32), idesc,
                                           (kb + u > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(&aempty[as]);
                    tc::mma_commit(&hempty[hs]);
                    if (++as == NA) { as = 0; aph ^= 1u; }
                    if (++hs == HS) { hs = 0; hph ^= 1u; }
                }
                if (ok) tc::mma_commit(&acc_full[buf]);
            }
            tc::mma_commit(drain);
            lm_drain_wait(drain, 0);
        }
    } else if (warp >= 6) {
        // ------------------------------------------------------------ converters: codes -> fp16 A slots in TMEM
        // Set `par` converts the k-blocks g with g % kQ4Sets == par (k-blocks par and par + 4 of every W stage);
        // its four warps cover the four lane quarters.  k-block g goes to A-slot group g / GK, slot g % GK of it;
        // a set's consecutive k-blocks are kQ4Sets / GK groups apart, and NA is a multiple of that step, so a
        // set's group index advances by the step and wraps at NA, flipping the parity of its slots' reuse.
        const int par = (warp - 6) >> 2, quad = warp & 3;
        const int r = quad * 32 + lane;  // vocabulary row within the tile = TMEM lane
        const uint32_t a_lane = tmem + ((uint32_t)(quad * 32) << 16) + a_col + (uint32_t)(par % GK) * 32;
        const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
        const int step = kQ4Sets / GK;
        int as = par / GK, n = 0, ws = 0;  // A-slot group, k-blocks converted, W stage
        uint32_t use = 0, wph = 0;         // parity of the group's current use; of stage ws's fill
        bool ok = true;
        for (int vt = group; ok && vt < p.vtiles; vt += groups) {
            for (int i = 0; ok && i < NSt; ++i) {
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&wfull[ws], wph, abort_flag, 256))) {
                    ok = false;
                    break;
                }
                const uint8_t* st = wring + ws * kQ4WStage;
                const uint16_t* scr = reinterpret_cast<const uint16_t*>(st + 32768 + r * 16);
                const uint16_t* bir = reinterpret_cast<const uint16_t*>(st + 34816 + r * 16);
#pragma unroll
                for (int h = 0; h < kQ4KBPerStage / kQ4Sets; ++h) {
                    const int kk = par + kQ4Sets * h;
                    // the group's previous use (n * step >= NA) must have been read by its MMAs
                    if (n * step >= NA &&
                        !__all_sync(0xFFFFFFFFu, tc::mbar_wait(&aempty[as], use ^ 1u, abort_flag, 256))) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    q4_convert_row(st, r, kk, __uint_as_float((uint32_t)scr[kk] << 16),
                                   __uint_as_float((uint32_t)bir[kk] << 16), k1024, a_lane + (uint32_t)(as * GK) * 32);
                    tc::tmem_wait_st();
                    tc::tc_fence_before();
                    __syncwarp();
                    tc::mbar_arrive_one(&afull[as]);
                    ++n;
                    as += step;
                    if (as >= NA) { as -= NA; use ^= 1u; }
                }
                __syncwarp();
                tc::mbar_arrive_one(&wempty[ws]);
                if (++ws == WSt) { ws = 0; wph ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------------------ argmax epilogue
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        int it = 0;
        for (int vt = group; vt < p.vtiles; vt += groups, ++it) {
            const int buf = it & 1;
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&acc_full[buf], (it >> 1) & 1, abort_flag, 1024))) break;
            tc::tc_fence_after();
            lm_epilogue_warp<LOGITS>(tmem + lane_base + buf * p.DC, nrows, vt * kLmM + warp * 32 + lane, p.V,
                                     wbest + warp * kQ4MaxNP, lane, p.logits, chunk * p.NP);
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(&acc_empty[buf]);
        }
    }

    __syncthreads();
    if (!*abort_flag)
        for (int c = threadIdx.x; c < nrows; c += blockDim.x) {
            unsigned long long b = wbest[c];
#pragma unroll
            for (int w = 1; w < 4; ++w) b = wbest[w * kQ4MaxNP + c] > b ? wbest[w * kQ4MaxNP + c] : b;
            if (b) atomicMax(&p.best[chunk * p.NP + c], b);
        }
    if (warp == 5) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ 4-bit heads, few hidden rows
// An M = 128 MMA holds its issuing thread for ~44 cycles whatever N is up to 64, while at N = 16 the tensor
// pipe needs ~8, and one thread issuing every MMA of a tile (4 per k-block) falls behind the converters.
// Here every converter set has an issuer warp of its own (warps 6 .. 6 + NI - 1, each on its own SM
// sub-partition) and each issuer its own accumulator: the k-blocks of a tile are split NI ways and the
// epilogue adds the NI partial sums (fp32) before the argmax.  Set par converts the k-blocks kb = par mod 4
// into a ring of NAS A slots of its own; issuer i takes the sets par = i mod NI.  Hidden stages hold 4
// k-blocks, one per set.
constexpr int kQ4sMaxNP = 32;
constexpr int kQ4sKBPerHStage = kQ4Sets;
constexpr int kQ4sMaxWStages = 8;
constexpr int kQ4sMinHStages = 4;  // the rest of shared memory goes to W stages: they carry the DRAM latency
// polls before the first sleep: every poll is an issue slot taken from the converters
constexpr uint32_t kQ4sConvSpins = 2, kQ4sIssSpins = 4;

template <int NI>
struct Q4s {
    static constexpr int kConv0 = 6 + NI;                        // first converter warp
    static constexpr int kThreads = kLmEpi + 64 + NI * 32 + kQ4Conv;
};

// Shared memory: [W ring: WS x 36 KB] [hidden ring: HS stages of 4 k-blocks] ... [bests | barriers]; the W ring
// takes all but kQ4sMinHStages hidden stages, since its stages carry the DRAM latency (~5 us from TMA issue to
// landing under full load) while the hidden blocks come from L2.  TMEM: accumulators [buf][issuer] of DC
// columns from 0, then 4 x NAS A slots of 32 columns (set par owns slots par * NAS .. par * NAS + NAS - 1).
template <bool LOGITS, int NI>
__global__ void __launch_bounds__(Q4s<NI>::kThreads, 1) lm_q4s_kernel(const __grid_constant__ LmQ4Params p) {
    griddep_begin();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* wring = sm;
    uint8_t* hring = sm + p.WS * kQ4WStage;
    uint8_t* tail = sm + kLmUsable;
    unsigned long long* wbest = reinterpret_cast<unsigned long long*>(tail);  // [4 warps][kQ4sMaxNP] bests
    uint64_t* bars = reinterpret_cast<uint64_t*>(tail + 2048);
    uint64_t* wfull = bars;           // [8]
    uint64_t* wempty = bars + 8;      // [8] every converter warp is done with the stage
    uint64_t* hfull = bars + 16;      // [16]
    uint64_t* hempty = bars + 32;     // [16] the MMAs of all 4 k-blocks of the stage are done
    uint64_t* afull = bars + 48;      // [16] slot written by its set's 4 warps
    uint64_t* aempty = bars + 64;     // [16] MMAs done with the slot
    uint64_t* acc_full = bars + 80;   // [2] every issuer's MMAs of the tile are done
    uint64_t* acc_empty = bars + 82;  // [2]
    uint64_t* drain = bars + 84;      // [4] one per issuer
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 88);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 89);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x % p.nchunks;
    const int group = blockIdx.x / p.nchunks;
    const int groups = gridDim.x / p.nchunks;
    const int KB = p.H / kLmKB;
    const int NSt = KB / kQ4KBPerStage;
    const int NAS = p.NA, HS = p.HS, DC = p.DC, WS = p.WS;  // A slots per set, hidden and W stages, accumulator columns
    const int nrows = min(p.NP, p.rows - chunk * p.NP);
    if (group >= p.vtiles || nrows <= 0) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WS; ++s) {
            tc::mbar_init(&wfull[s], 1);
            tc::mbar_init(&wempty[s], kQ4Conv / 32);
        }
        for (int s = 0; s < HS; ++s) {
            tc::mbar_init(&hfull[s], 1);
            tc::mbar_init(&hempty[s], kQ4sKBPerHStage);
        }
        for (int s = 0; s < kQ4Sets * NAS; ++s) {
            tc::mbar_init(&afull[s], 4);
            tc::mbar_init(&aempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&acc_full[s], NI);
            tc::mbar_init(&acc_empty[s], kLmEpi / 32);
        }
        for (int s = 0; s < NI; ++s) tc::mbar_init(&drain[s], 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    for (int c = threadIdx.x; c < 4 * kQ4sMaxNP; c += blockDim.x) wbest[c] = 0ull;
    if (warp == 5) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t a_col = 2u * (uint32_t)(NI * DC);
    const uint32_t h_bytes = (uint32_t)p.NP * 128;

    if (warp == 4) {
        if (lane == 0) {
            // -------------------------------------------------------- W stages: codes, scales, biases of 8 k-blocks
            tc::tma_prefetch_desc(&p.wmap);
            tc::tma_prefetch_desc(&p.smap);
            tc::tma_prefetch_desc(&p.bmap);
            int c = 0, issued = 0, s = 0;
            uint32_t fill = 0;  // parity of stage s's current fill
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups) {
                for (int i = 0; i < NSt; ++i, ++c) {
                    if (c >= WS && !tc::mbar_wait(&wempty[s], fill ^ 1u, abort_flag, 512)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = wring + s * kQ4WStage;
                    tc::mbar_expect_tx(&wfull[s], kQ4WStage);
                    tc::tma_load_2d(st, &p.wmap, &wfull[s], i * 256, vt * kLmM);
                    tc::tma_load_2d(st + 16384, &p.wmap, &wfull[s], i * 256 + 128, vt * kLmM);
                    tc::tma_load_2d(st + 32768, &p.smap, &wfull[s], i * kQ4KBPerStage, vt * kLmM);
                    tc::tma_load_2d(st + 34816, &p.bmap, &wfull[s], i * kQ4KBPerStage, vt * kLmM);
                    issued = c + 1;
                    if (++s == WS) { s = 0; fill ^= 1u; }
                }
            }
            if (*abort_flag)
                for (int q = max(0, issued - WS); q < issued; ++q)
                    lm_drain_wait(&wfull[q % WS], (q / WS) & 1);
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // -------------------------------------------------------- hidden blocks, 4 k-blocks per stage
            tc::tma_prefetch_desc(&p.hmap);
            int g = 0, issued = 0, s = 0;
            uint32_t fill = 0;
            bool ok = true;
            for (int vt = group; ok && vt < p.vtiles; vt += groups) {
                for (int kb = 0; kb < KB; kb += kQ4sKBPerHStage, ++g) {
                    if (g >= HS && !tc::mbar_wait(&hempty[s], fill ^ 1u, abort_flag, 512)) { ok = false; break; }
                    tc::mbar_expect_tx(&hfull[s], h_bytes * kQ4sKBPerHStage);
                    for (int u = 0; u < kQ4sKBPerHStage; ++u)
                        tc::tma_load_2d(hring + (s * kQ4sKBPerHStage + u) * h_bytes, &p.hmap, &hfull[s], (kb + u) * kLmKB,
                                        chunk * p.NP);
                    issued = g + 1;
                    if (++s == HS) { s = 0; fill ^= 1u; }
                }
            }
            if (*abort_flag)
                for (int q = max(0, issued - HS); q < issued; ++q) lm_drain_wait(&hfull[q % HS], (q / HS) & 1);
        }
    } else if (warp >= 6 && warp < Q4s<NI>::kConv0) {
        // ------------------------------------------------------------ issuer iss: k-blocks of sets iss, iss + NI, ...
        // The whole warp runs the loop (warp-uniform operands); lane 0 issues the MMAs and commits.
        const int iss = warp - 6;
        const uint32_t idesc = tc::idesc_f16(false, false, false, kLmM, p.NP);
        const uint64_t hdesc0 = tc::sdesc_sw128(tc::smem_u32(hring), 16, 1024);
        int it = 0, hs = 0, slot = 0;  // hidden stage; A slot (the same in every set: one k-block per stage each)
        uint32_t hph = 0, aph = 0;
        bool ok = true;
        for (int vt = group; ok && vt < p.vtiles; vt += groups, ++it) {
            const int buf = it & 1;
            if (it >= 2 && !__all_sync(0xFFFFFFFFu, tc::mbar_wait_spin(&acc_empty[buf], ((it >> 1) - 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t d = tmem + (uint32_t)((buf * NI + iss) * DC);
            for (int kb0 = 0; ok && kb0 < KB; kb0 += kQ4sKBPerHStage) {
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&hfull[hs], hph, abort_flag, 64, kQ4sIssSpins))) { ok = false; break; }
                for (int u = iss; u < kQ4sKBPerHStage; u += NI) {  // set u converts k-block kb0 + u
                    const int sl = u * NAS + slot;
                    if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&afull[sl], aph, abort_flag, 64, kQ4sIssSpins))) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t a = tmem + a_col + (uint32_t)sl * 32;
                    const uint64_t b = tc::sdesc_add(hdesc0, (uint32_t)(hs * kQ4sKBPerHStage + u) * h_bytes);
                    const uint32_t first = (kb0 == 0 && u == iss) ? 0u : 1u;
                    tc::mma_f16_ts_lane0(d, a, b, idesc, first);
                    tc::mma_f16_ts_lane0(d, a + 8, tc::sdesc_add(b, 32), idesc, 1u);
                    tc::mma_f16_ts_lane0(d, a + 16, tc::sdesc_add(b, 64), idesc, 1u);
                    tc::mma_f16_ts_lane0(d, a + 24, tc::sdesc_add(b, 96), idesc, 1u);
                    tc::mma_commit_lane0(&aempty[sl]);
                    tc::mma_commit_lane0(&hempty[hs]);
                }
                if (++slot == NAS) { slot = 0; aph ^= 1u; }
                if (++hs == HS) { hs = 0; hph ^= 1u; }
            }
            if (ok) tc::mma_commit_lane0(&acc_full[buf]);
        }
        tc::mma_commit_lane0(&drain[iss]);
        lm_drain_wait(&drain[iss], 0);
    } else if (warp >= Q4s<NI>::kConv0) {
        // ------------------------------------------------------------ converters: codes -> fp16 A slots in TMEM
        // Set par converts k-blocks par and par + 4 of every W stage into its own ring of NAS slots; every
        // index and parity advances by increments (no division on this path), and warp-level arrivals are
        // predicated on one elected lane.
        const int cw = warp - Q4s<NI>::kConv0;
        const int par = cw >> 2, quad = warp & 3;
        const int r = quad * 32 + lane;  // vocabulary row within the tile = TMEM lane
        const uint32_t a_set = tmem + ((uint32_t)(quad * 32) << 16) + a_col + (uint32_t)(par * NAS) * 32;
        uint64_t* afull_set = afull + par * NAS;
        uint64_t* aempty_set = aempty + par * NAS;
        const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
        int ws = 0, slot = 0, n = 0;  // W stage, A slot, k-blocks converted
        uint32_t wph = 0, use = 0;    // parity of stage ws's fill; parity of slot's current use
        bool ok = true;
        for (int vt = group; ok && vt < p.vtiles; vt += groups) {
            for (int i = 0; ok && i < NSt; ++i) {
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&wfull[ws], wph, abort_flag, 256, kQ4sConvSpins))) {
                    ok = false;
                    break;
                }
                const uint8_t* st = wring + ws * kQ4WStage;
                const uint16_t* scr = reinterpret_cast<const uint16_t*>(st + 32768 + r * 16);
                const uint16_t* bir = reinterpret_cast<const uint16_t*>(st + 34816 + r * 16);
#pragma unroll
                for (int h = 0; h < kQ4KBPerStage / kQ4Sets; ++h) {
                    const int kk = par + kQ4Sets * h;
                    if (n >= NAS && !__all_sync(0xFFFFFFFFu, tc::mbar_wait(&aempty_set[slot], use ^ 1u, abort_flag, 256,
                                                                           kQ4sConvSpins))) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    q4_convert_row<true>(st, r, kk, __uint_as_float((uint32_t)scr[kk] << 16),
                                         __uint_as_float((uint32_t)bir[kk] << 16), k1024, a_set + (uint32_t)slot * 32);
                    tc::tmem_wait_st();
                    tc::tc_fence_before();
                    __syncwarp();
                    tc::mbar_arrive_one(&afull_set[slot]);
                    ++n;
                    if (++slot == NAS) { slot = 0; use ^= 1u; }
                }
                __syncwarp();
                tc::mbar_arrive_one(&wempty[ws]);
                if (++ws == WS) { ws = 0; wph ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------------------ argmax epilogue (warps 0-3)
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        int it = 0;
        for (int vt = group; vt < p.vtiles; vt += groups, ++it) {
            const int buf = it & 1;
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&acc_full[buf], (it >> 1) & 1, abort_flag, 1024))) break;
            tc::tc_fence_after();
            lm_epilogue_sum_warp<LOGITS, NI, LOGITS ? 8 : 16>(tmem + lane_base + (uint32_t)(buf * NI * DC), DC, nrows,
                                             vt * kLmM + warp * 32 + lane, p.V, wbest + warp * kQ4sMaxNP, lane, p.logits,
                                             chunk * p.NP);
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
        }
    }

    __syncthreads();
    if (!*abort_flag)
        for (int c = threadIdx.x; c < nrows; c += blockDim.x) {
            unsigned long long b = wbest[c];
#pragma unroll
            for (int w = 1; w < 4; ++w) b = wbest[w * kQ4sMaxNP + c] > b ? wbest[w * kQ4sMaxNP + c] : b;
            if (b) atomicMax(&p.best[chunk * p.NP + c], b);
        }
    if (warp == 5) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// bf16 hidden rows -> fp16 copy (operand type of the fp16 MMA).
__global__ void hidden_to_f16_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, size_t n) {
    griddep_begin();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n / 2; i += (size_t)gridDim.x * blockDim.x) {
        const uint32_t w = reinterpret_cast<const uint32_t*>(in)[i];
        __half2 h = __floats2half2_rn(bf16_lo(w), bf16_hi(w));
        reinterpret_cast<uint32_t*>(out)[i] = *reinterpret_cast<uint32_t*>(&h);
    }
}

// bf16 hidden rows -> fp16 copy with every 8 features in the 4-bit converter's order (0,4,1,5,2,6,3,7).
__global__ void hidden_to_f16_q4order_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, size_t n8) {
    griddep_begin();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        const uint4 w = in[i];
        const __half2 a = __floats2half2_rn(bf16_lo(w.x), bf16_lo(w.z));  // features 0, 4
        const __half2 b = __floats2half2_rn(bf16_hi(w.x), bf16_hi(w.z));  // 1, 5
        const __half2 c = __floats2half2_rn(bf16_lo(w.y), bf16_lo(w.w));  // 2, 6
        const __half2 d = __floats2half2_rn(bf16_hi(w.y), bf16_hi(w.w));  // 3, 7
        out[i] = make_uint4(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b),
                            *reinterpret_cast<const uint32_t*>(&c), *reinterpret_cast<const uint32_t*>(&d));
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

// Bytes of workspace the tensor-core paths need beyond the per-row bests
// (the fp16 copy of hidden when the MMA runs in fp16).
size_t lm_tc_extra_bytes(int rows, int H, int w_dtype) {
    return w_dtype == TSV_BF16 ? 0 : (((size_t)rows * H * 2 + 255) & ~(size_t)255);
}

// Shape conditions of the tensor-core paths.  The 4-bit path reads scales and biases 8 groups of a row at a
// time, so H must be a multiple of 512 and (checked by the caller) both pointers 16-byte aligned.  Row counts:
// a 4-bit head takes the tensor-core kernels at every count: the CUDA-core GEMV runs below the HBM rate even at
// one row and dequantises each weight again for every row (248,320 x 5120 head: 0.32 ms at 1 row, 0.82 at 3,
// 2.1 at 8, against 0.19 ms for the few-row kernel at 1 to 16 rows, the rows padded to the MMA's 16); a 16-bit head
// stays on the GEMV while one pass of it serves every row (up to kLmGemvRows16 rows, at the HBM rate: 0.35-0.37
// ms for 2.54 GB), above that the GEMV streams the head twice (0.73 ms at 8 rows, against 0.39 ms for the
// tensor-core kernel).
constexpr int kLmGemvRows16 = 4;
bool lm_tc_applies(int rows, int H, int V, int w_dtype) {
    if (rows < 1 || V < 1) return false;
    if (w_dtype == TSV_Q4_G64) return H % (kLmKB * kQ4KBPerStage) == 0;
    return rows > kLmGemvRows16 && H % kLmKB == 0;
}

static tsv_status launch_lm_q4(const void* hidden, int rows, int H, int V, const void* W, const void* scales,
                               const void* biases, unsigned long long* best, float* logits, void* extra,
                               cudaStream_t stream) {
    static thread_local LmQ4Params prm;
    const int nchunks = (rows + kQ4MaxNP - 1) / kQ4MaxNP;
    int NP = (rows + nchunks - 1) / nchunks;
    NP = ((NP + 15) / 16) * 16;
    const int DC = ((NP + 31) / 32) * 32;
    // W stages: 3 when each CTA streams its W tiles from DRAM alone, 2 when several row chunks walk the same
    // vocabulary tiles together (the later ones read them from L2): that leaves room for hidden stages of 4
    // k-blocks, so the MMA thread issues 16 MMAs per wait (2,048 rows: 6.22 -> 5.03 ms; an issuer that waits
    // between short bursts lets the tensor pipe drain every burst).
    const int WS = nchunks >= 2 ? 2 : kQ4WStages;
    // k-blocks per group: the largest of 4, 2, 1 that leaves at least 2 hidden stages and 2 A-slot groups
    int GK = 4, NA = 0, HS = 0;
    for (; GK >= 1; GK >>= 1) {
        NA = (512 - 2 * DC) / (32 * GK);
        NA = NA > kQ4MaxAGroups ? kQ4MaxAGroups : NA;
        // a slot group must always be refilled by the same converter sets (its previous use then completed
        // before they wait again): NA a multiple of kQ4Sets / GK
        NA -= NA % (kQ4Sets / GK);
        HS = (kLmUsable - 2048 - WS * kQ4WStage) / (NP * 128 * GK);  // per-warp bests take the last 2 KB
        HS = HS > kQ4MaxHStages ? kQ4MaxHStages : HS;
        if (NA >= 2 && HS >= 2) break;
    }
    if (GK < 1) return fail(TSV_EUNSUPPORTED, "lm_head_argmax: hidden chunk too wide for the 4-bit pipeline");

    const size_t n8 = (size_t)rows * H / 8;
    launch_pdl(hidden_to_f16_q4order_kernel, sm_count() * 4, 256, 0, stream, (const uint4*)hidden, (uint4*)extra, n8);
    tsv_status st = check_launch("lm_head_argmax(hidden fp16)");
    if (st != TSV_OK) return st;

    bool ok = map2d(&prm.wmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)H / 2, (uint64_t)V, (uint64_t)H / 2, 128,
                    kLmM, true);
    ok = ok && map2d(&prm.smap, scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)H / 64, (uint64_t)V,
                     (uint64_t)H / 64 * 2, kQ4KBPerStage, kLmM, false);
    ok = ok && map2d(&prm.bmap, biases, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)H / 64, (uint64_t)V,
                     (uint64_t)H / 64 * 2, kQ4KBPerStage, kLmM, false);
    ok = ok && map2d(&prm.hmap, extra, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)H, (uint64_t)rows, (uint64_t)H * 2,
                     64, (uint32_t)NP, true);
    if (!ok) return fail(TSV_ECUDA, "lm_head_argmax: tensor map encoding failed");
    prm.best = best;
    prm.logits = logits;
    prm.rows = rows;
    prm.H = H;
    prm.V = V;
    prm.NP = NP;
    prm.DC = DC;
    prm.NA = NA;
    prm.HS = HS;
    prm.GK = GK;
    prm.WS = WS;
    prm.nchunks = nchunks;
    prm.vtiles = (V + kLmM - 1) / kLmM;
    const int sms = sm_count();
    const int groups = sms / nchunks > 0 ? sms / nchunks : 1;
    if (NP <= kQ4sMaxNP) {
        // few hidden rows: one issuer and one accumulator per converter set
        constexpr int NI = kQ4Sets;
        prm.DC = NP;
        prm.NA = (512 - 2 * NI * NP) / 32 / kQ4Sets;
        prm.NA = prm.NA > 4 ? 4 : prm.NA;
        const int hst = NP * 128 * kQ4sKBPerHStage;
        const int ws = (kLmUsable - kQ4sMinHStages * hst) / kQ4WStage;
        prm.WS = ws > kQ4sMaxWStages ? kQ4sMaxWStages : ws;
        const int hs = (kLmUsable - prm.WS * kQ4WStage) / hst;
        prm.HS = hs > kQ4MaxHStages ? kQ4MaxHStages : hs;
        if (prm.WS < 2 || prm.HS < 2 || prm.NA < 1)  // the rings index stages modulo their counts
            return fail(TSV_EUNSUPPORTED, "lm_head_argmax: shared memory too small for the 4-bit pipeline");
        if (logits) {
            cudaFuncSetAttribute(lm_q4s_kernel<true, NI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLmSmem);
            launch_pdl(lm_q4s_kernel<true, NI>, groups * nchunks, Q4s<NI>::kThreads, kLmSmem, stream, prm);
        } else {
            cudaFuncSetAttribute(lm_q4s_kernel<false, NI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLmSmem);
            launch_pdl(lm_q4s_kernel<false, NI>, groups * nchunks, Q4s<NI>::kThreads, kLmSmem, stream, prm);
        }
        return check_launch("lm_head_argmax(tcgen05, 4-bit, few rows)");
    }
    if (logits) {
        cudaFuncSetAttribute(lm_q4_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLmSmem);
        launch_pdl(lm_q4_kernel<true>, groups * nchunks, kQ4Threads, kLmSmem, stream, prm);
    } else {
        cudaFuncSetAttribute(lm_q4_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLmSmem);
        launch_pdl(lm_q4_kernel<false>, groups * nchunks, kQ4Threads, kLmSmem, stream, prm);
    }
    return check_launch("lm_head_argmax(tcgen05, 4-bit)");
}

tsv_status launch_lm_tc(const void* hidden, int rows, int H, int V, int w_dtype, const void* W, const void* scales,
                        const void* biases, unsigned long long* best, float* logits, void* extra, cudaStream_t stream) {
    if (w_dtype == TSV_Q4_G64) return launch_lm_q4(hidden, rows, H, V, W, scales, biases, best, logits, extra, stream);
    static thread_local LmTcParams prm;
    const int nchunks = (rows + 255) / 256;
    int NP = (rows + nchunks - 1) / nchunks;
    NP = ((NP + 15) / 16) * 16;
    const void* hsrc = hidden;
    if (w_dtype != TSV_BF16) {  // fp16 MMA: fp16 copy of hidden
        const size_t n = (size_t)rows * H;
        launch_pdl(hidden_to_f16_kernel, sm_count() * 4, 256, 0, stream, (const uint16_t*)hidden, (uint16_t*)extra, n);
        tsv_status st = check_launch("lm_head_argmax(hidden fp16)");
        if (st != TSV_OK) return st;
        hsrc = extra;
    }
    bool ok = map2d(&prm.wmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, 64, kLmM,
                    true);
    ok = ok && map2d(&prm.hmap, hsrc, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)H, (uint64_t)rows, (uint64_t)H * 2, 64,
                     (uint32_t)NP, true);
    if (!ok) return fail(TSV_ECUDA, "lm_head_argmax: tensor map encoding failed");
    prm.best = best;
    prm.logits = logits;
    prm.rows = rows;
    prm.H = H;
    prm.V = V;
    prm.NP = NP;
    prm.nchunks = nchunks;
    prm.vtiles = (V + kLmM - 1) / kLmM;
    prm.mma_bf16 = w_dtype == TSV_BF16;
    // hidden blocks (NP x 128 B, multiples of 1024: every block stays 1024-aligned) come from L2 after the first
    // tile: 3 stages at 256 rows, 4 below; the W ring takes the rest
    prm.hstages = NP >= 256 ? kLmHStages256 : NP >= 128 ? 5 : 4;
    const int stages = (kLmUsable16 - prm.hstages * NP * 128) / 16384;
    prm.stages = stages > kLmMaxStages ? kLmMaxStages : stages;
    if (prm.stages < 2 || prm.stages < prm.hstages)  // the two rings share one barrier pair per W stage
        return fail(TSV_EUNSUPPORTED, "lm_head_argmax: hidden chunk too wide for the pipeline");
    const int sms = sm_count();
    const int groups = sms / nchunks > 0 ? sms / nchunks : 1;
    if (logits) {
        cudaFuncSetAttribute(lm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLmSmem);
        launch_pdl(lm_tc_kernel<true>, groups * nchunks, kLmThreads16, kLmSmem, stream, prm);
    } else {
        cudaFuncSetAttribute(lm_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLmSmem);
        launch_pdl(lm_tc_kernel<false>, groups * nchunks, kLmThreads16, kLmSmem, stream, prm);
    }
    return check_launch("lm_head_argmax(tcgen05)");
}

}  // namespace tsv
