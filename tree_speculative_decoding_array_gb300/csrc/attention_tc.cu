// Tensor-core (tcgen05) path of tsv_tree_verify_attention for 16-bit caches
// with head dimension 256.
//
// Same operation as the CUDA-core path (see attention.cu): per (layer,
// sequence, kv head) unit, the G*T query rows (node i, head g of the GQA
// group) attend the S cached positions in full and the block positions of
// their ancestors, split over key ranges with fp32 partials (Splash issue
// #728, "Earlier shader evidence": split-KV tree attention with fp32 partials
// and statistics; mlxcel issue #1204, "What this needs" item 1).
//
// One CTA = one 128-row tile of one unit and one key range; 352 threads:
//   warps 0-3  softmax, first half: lane r of warp q owns query row
//              32 q + r = TMEM lane.  Stores Q into TMEM, reads its 32 of
//              the tile's 64 S columns from TMEM, applies the scale and the
//              ancestor bits, runs the online softmax (fp32, log2 domain,
//              lazy rescale of O when the max grows by > 2^8), writes its
//              P columns as 16-bit pairs back over the S tile in TMEM,
//              finally reads out its half of O.
//   warps 7-10 softmax, second half: the other 32 columns of the same rows;
//              each pair of warps on one lane quarter exchanges its row
//              maxima (and at the end its row sums) through shared memory.
//   warp 4, 6  TMA producers (4: K, 6: V; one lane each): tiles of 64 keys x
//              256, 128-byte swizzled, each in its own 3-stage ring (a K
//              stage frees after Q K^T, a V stage after P V).
//   warp 5     allocates TMEM (512 columns: Q 128 as 16-bit pairs, S 2 x 64,
//              O 256) and issues the MMAs from an event loop:
//              S = Q K^T (M=128, N=64, K=256, A read from TMEM) and
//              O += P V (M=128, N=256, K=64, A = P read from TMEM, V read
//              MN-major).  An S buffer is reused once the P V of the P
//              written over it is done, so the softmax of tile j + 1 never
//              waits for the P V of tile j (except to rescale O).
// Int8 caches (Int8 codes with fp16 per-token scales) use 640 threads: warps
// 6-9 convert K tiles, warps 10-13 convert V tiles, warp 14 is the V
// producer, warps 15-18 the softmax's second half; warp 5 issues only the
// Q K^T MMAs and warp 19 the P V MMAs (an issuing thread is held for each
// MMA's whole pipe time, so one thread issuing both would make a ready P V
// wait behind the next Q K^T).  TMEM then holds Q, one S tile (released as
// soon as both softmax halves have read it, so the next Q K^T never waits
// for a P V), two P buffers of 32 columns and O.  TMA brings the raw int8
// tiles (128-byte swizzled halves) into 2-stage staging rings; each converter
// thread owns one key of every tile and writes its codes times its scale
// (fp16, one rounding; the scale fetched a tile ahead) into 2-stage operand
// rings, so the softmax does no scale work.
// Warp-collective roles take every wait decision warp-uniformly (__all_sync),
// so that tcgen05.ld / __syncwarp never see a partial warp.
// Every mbarrier wait is bounded in time: on expiry the CTA raises a shared
// abort flag, records TSV_DEV_TIMEOUT, drains its own MMAs and copies and
// frees TMEM before returning.
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace tsv {

constexpr int kTcRows = 128;
constexpr int kTcBK = 64;
constexpr int kTcD = 256;
constexpr int kTcThreads16 = 256;  // 128-key kernel: + warp 6: V producer, warp 7: P V issuer
// 64-key kernel: 16-bit: warp 6 V producer, warps 7-10 the softmax's second half; Int8: warps 6-9 K converters,
// 10-13 V converters, warp 14 V producer, warps 15-18 the softmax's second half, warp 19 issues the P V MMAs
constexpr int kTc64Threads16 = 352;
constexpr int kTcThreadsI8 = 640;
constexpr int kTcSmem = 1024 + 215040 + 512;
constexpr uint32_t kTileBytes = kTcBK * kTcD * 2;  // one K (or V) tile: 32 KiB

struct TcParams {
    CUtensorMap kmap[TSV_MAX_LAYERS];
    CUtensorMap vmap[TSV_MAX_LAYERS];
    const uint16_t* q[TSV_MAX_LAYERS];
    void* o[TSV_MAX_LAYERS];
    const uint16_t* ks[TSV_MAX_LAYERS];
    const uint16_t* vs[TSV_MAX_LAYERS];
    const int32_t* kv_len;
    const uint64_t* anc;
    float* ws_o;
    float* ws_ml;
    int32_t* status;
    int window[TSV_MAX_LAYERS];  // per layer sliding window, 0 = full attention
    int64_t s_cap;
    int B, T, HQ, HKV, G, R, mtiles, splits, chunk, max_kv_len, mma_bf16;
};

__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __half2 h = __floats2half2_rn(bf16_lo(w[k]), bf16_hi(w[k]));
        w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf) {
    if (bf) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Bounded wait that ignores the abort flag (used only while draining).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(bar, parity))
        if (tc::globaltimer() - t0 > 200000000ull) break;  // 200 ms
}

// Int8 -> fp16 for 16 codes (one 16-byte chunk): exact, via 1024 + (code + 128) - 1152.
__device__ __forceinline__ void i8x16_to_f16x16(uint4 in, uint32_t (&out)[8]) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    const __half2 bias = __floats2half2_rn(1152.f, 1152.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t x = w[k] ^ 0x80808080u;
        uint32_t lo = __byte_perm(x, 0x64646464u, 0x5140);
        uint32_t hi = __byte_perm(x, 0x64646464u, 0x7362);
        __half2 a = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
        __half2 c = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
        out[2 * k] = *reinterpret_cast<uint32_t*>(&a);
        out[2 * k + 1] = *reinterpret_cast<uint32_t*>(&c);
    }
}

// Raw int8 tile [64 keys x 256] as TMA lands it: two 128-byte-swizzled halves [2][64 keys][128 B] (16-byte
// chunk c of key k's half h at h * 8192 + k * 128 + ((c ^ (k & 7)) << 4)) -> fp16 operand tile in the
// 128-byte-swizzled layout (4 blocks of [64 keys x 64]); keys >= nk become 0.  A quarter-warp takes one chunk
// column of 8 consecutive keys, so its 16-byte loads and stores each hit 8 distinct bank groups.
__device__ __forceinline__ void convert_i8_tile(const uint8_t* raw, uint8_t* dst, int nk, int ct) {
    const int key = ct & 63, k7 = key & 7;  // chunk q of the 256-byte row: 2 s + (ct >> 6)
    uint4 in[8];  // all eight 16-byte loads in flight before the first conversion
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int q = 2 * s + (ct >> 6);
        in[s] = key < nk ? *reinterpret_cast<const uint4*>(raw + (q >> 3) * 8192 + key * 128 + (((q & 7) ^ k7) << 4))
                         : make_uint4(0, 0, 0, 0);
    }
    uint8_t* row = dst + key * 128;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int q = 2 * s + (ct >> 6);
        uint32_t w[8];
        i8x16_to_f16x16(in[s], w);
        if (key >= nk) {
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = 0;
        }
        // features 16 q .. 16 q + 15: fp16 block q >> 2, 16-byte chunks (q & 3) * 2 and the next
        const int cc0 = (q & 3) * 2;
        uint8_t* rb = row + (q >> 2) * 8192;
        *reinterpret_cast<uint4*>(rb + ((cc0 ^ k7) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(rb + (((cc0 + 1) ^ k7) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// The same 16 codes times a per-token scale: fp16(code) exact, then one rounding of code * scale.
__device__ __forceinline__ void i8x16_to_f16x16_scaled(uint4 in, __half2 s2, uint32_t (&out)[8]) {
    i8x16_to_f16x16(in, out);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const __half2 w = __hmul2(*reinterpret_cast<const __half2*>(&out[k]), s2);
        out[k] = *reinterpret_cast<const uint32_t*>(&w);
    }
}

// convert_i8_tile with every key's codes multiplied by its scale (scale2: this thread's key, both halves).
__device__ __forceinline__ void convert_i8_tile_scaled(const uint8_t* raw, uint8_t* dst, int nk, int ct, __half2 scale2) {
    const int key = ct & 63, k7 = key & 7;
    uint4 in[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int q = 2 * s + (ct >> 6);
        in[s] = key < nk ? *reinterpret_cast<const uint4*>(raw + (q >> 3) * 8192 + key * 128 + (((q & 7) ^ k7) << 4))
                         : make_uint4(0, 0, 0, 0);
    }
    uint8_t* row = dst + key * 128;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int q = 2 * s + (ct >> 6);
        uint32_t w[8];
        i8x16_to_f16x16_scaled(in[s], scale2, w);
        if (key >= nk) {
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = 0;
        }
        const int cc0 = (q & 3) * 2;
        uint8_t* rb = row + (q >> 2) * 8192;
        *reinterpret_cast<uint4*>(rb + ((cc0 ^ k7) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(rb + (((cc0 + 1) ^ k7) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

constexpr int kNS = 3;  // stages of the K ring and of the V ring

template <bool I8>
__global__ void __launch_bounds__(I8 ? kTcThreadsI8 : kTc64Threads16, 1) attn_tc_kernel(const __grid_constant__ TcParams p) {
    griddep_begin();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // Q, S and P live in TMEM.  16-bit caches: K stages [3 x 32K] at 0, V stages [3 x 32K] at 96K.
    // Int8 caches: fp16 K tiles [2 x 32K] at 0, fp16 V tiles [2 x 32K] at 64K, raw K stages [2 x 16K] at 128K,
    // raw V stages [2 x 16K] at 160K.  Both: the softmax halves' exchange [2 slots x 2 halves x 128 rows] fp32
    // at 192K.
    constexpr int NS = I8 ? 2 : kNS;  // stages of the TMA rings
    constexpr int kSoftB = I8 ? 15 : 7;  // first warp of the softmax's second half
    uint8_t* sK = sm;
    uint8_t* sV = sm + (I8 ? 65536 : 98304);
    uint8_t* sRawK = sm + 131072;
    uint8_t* sRawV = sm + 163840;
    float* xv = reinterpret_cast<float*>(sm + 196608);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 215040);
    uint64_t* kfull = bars + 0;      // [3] K tile (16-bit) / raw K tile (Int8) landed
    uint64_t* kempty = bars + 3;     // [3] stage free again: after Q K^T (16-bit) / after conversion (Int8)
    uint64_t* vfull = bars + 6;      // [3] V tile / raw V tile landed
    uint64_t* vempty = bars + 9;     // [3] stage free again: after P V (16-bit) / after conversion (Int8)
    uint64_t* s_full = bars + 12;    // [2] S tile b written by Q K^T
    uint64_t* sp_free = bars + 14;   // [2] P V of the P held in S buffer b done: buffer b and O free again
    uint64_t* p_full = bars + 16;    // [2] P written over S buffer b
    uint64_t* o_done = bars + 18;
    uint64_t* q_full = bars + 19;
    uint64_t* drain = bars + 20;
    uint64_t* kc_full = bars + 21;   // Int8: [2] fp16 K tile written
    uint64_t* vc_full = bars + 25;   // Int8: [2] fp16 V tile written
    uint64_t* drain_pv = bars + 29;  // Int8: every MMA of the P V issuer done (abort path)
    uint64_t* s_free = bars + 30;    // Int8: every softmax warp has read the S tile
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 33);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 34);
    uint64_t* xch = bars + 36;       // [4 lane quarters][2 parities] both softmax halves posted their value
    // TMEM columns.  16-bit caches: Q [0, 128) as 16-bit pairs, S [128, 192) and [192, 256) (P, 16-bit pairs,
    // over the first 32 columns of its S tile once the softmax has read it), O [256, 512).  Int8 caches: Q, one
    // S tile [128, 192) (freed as soon as both softmax halves have read it, so Q K^T of the next tile never
    // waits for a P V), P [192, 224) and [224, 256) for tiles j & 1, O [256, 512).
    constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256, kColP8 = 192;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int item = blockIdx.x;
    const int mt = item % p.mtiles;
    item /= p.mtiles;
    const int split = item % p.splits;
    const int unit = item / p.splits;
    const int kvh = unit % p.HKV;
    const int b = (unit / p.HKV) % p.B;
    const int layer = unit / (p.HKV * p.B);
    const int T = p.T;
    const int kvl = p.kv_len[b];
    if (kvl < T || kvl > p.max_kv_len || (int64_t)kvl > p.s_cap) {
        if (split == 0 && mt == 0 && kvh == 0 && layer == 0 && threadIdx.x == 0)
            dev_fail(p.status, TSV_DEV_BAD_KV_LEN, b, kvl);
        return;
    }
    const int S = kvl - T;
    const int row0 = mt * kTcRows;
    const int k_end = min(kvl, split * p.chunk + p.chunk);
    // Sliding-window layer: node i keeps keys c >= S + i - window + 1.  lo_first / lo_last are that bound for
    // the first and last real row of this tile; key tiles below lo_first are skipped (64-key steps from the
    // range start), tiles at or above lo_last need no band test.
    const int win = p.window[layer];
    const int lo_first = win > 0 ? S + row0 / p.G - win + 1 : INT_MIN;
    const int lo_last = win > 0 ? S + (min(p.R, row0 + kTcRows) - 1) / p.G - win + 1 : INT_MIN;
    int k_begin = split * p.chunk;
    if (lo_first > k_begin) k_begin += ((lo_first - k_begin) / kTcBK) * kTcBK;
    const int ntiles = k_end > k_begin ? (k_end - k_begin + kTcBK - 1) / kTcBK : 0;

    // A CTA of this launch already timed out: do not start (keeps a broken launch short).
    if (p.status != nullptr && *reinterpret_cast<volatile int32_t*>(p.status) == TSV_DEV_TIMEOUT) return;

    if (ntiles == 0) {  // an empty key range contributes nothing to the combine
        if (threadIdx.x < kTcRows && row0 + (int)threadIdx.x < p.R) {
            const size_t slot = ((size_t)unit * p.splits + split) * p.R + row0 + threadIdx.x;
            p.ws_ml[2 * slot] = -INFINITY;
            p.ws_ml[2 * slot + 1] = 0.f;
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(&kfull[s], 1);
            tc::mbar_init(&kempty[s], I8 ? 4 : 1);
            tc::mbar_init(&vfull[s], 1);
            tc::mbar_init(&vempty[s], I8 ? 4 : 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&s_full[s], 1);
            tc::mbar_init(&sp_free[s], 1);
            tc::mbar_init(&p_full[s], 8);  // both softmax halves
            tc::mbar_init(&kc_full[s], 4);
            tc::mbar_init(&vc_full[s], 4);
        }
        for (int s = 0; s < 8; ++s) tc::mbar_init(&xch[s], 2);
        tc::mbar_init(o_done, 1);
        tc::mbar_init(q_full, 4);
        tc::mbar_init(drain, 1);
        tc::mbar_init(drain_pv, 1);
        tc::mbar_init(s_free, 8);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 5) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int vwarp = I8 ? 14 : 6;
    if (warp == 4 || warp == vwarp) {
        // ------------------------------------------------------------ TMA producers: warp 4 K, the last warp V
        // (a warp each: a lane that sleeps in its wait would hold up the other producer)
        if (lane == 0) {
            const bool isK = warp == 4;
            const CUtensorMap* m = isK ? &p.kmap[layer] : &p.vmap[layer];
            uint64_t* fullb = isK ? kfull : vfull;
            uint64_t* emptyb = isK ? kempty : vempty;
            tc::tma_prefetch_desc(m);
            const int rowbase = (int)(((int64_t)b * p.HKV + kvh) * p.s_cap + k_begin);
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int st = j % NS;
                if (j >= NS && !tc::mbar_wait(&emptyb[st], ((j / NS) - 1) & 1, abort_flag, 256)) break;
                const int row = rowbase + j * kTcBK;
                if (I8) {  // two 128-byte-wide swizzled halves of the 256-byte rows
                    tc::mbar_expect_tx(&fullb[st], kTcBK * kTcD);
                    uint8_t* dst = (isK ? sRawK : sRawV) + st * 16384;
                    tc::tma_load_2d(dst, m, &fullb[st], 0, row);
                    tc::tma_load_2d(dst + 8192, m, &fullb[st], 128, row);
                } else {
                    tc::mbar_expect_tx(&fullb[st], kTileBytes);
                    uint8_t* dst = (isK ? sK : sV) + st * kTileBytes;
#pragma unroll
                    for (int db = 0; db < 4; ++db) tc::tma_load_2d(dst + db * 8192, m, &fullb[st], db * 64, row);
                }
                issued = j + 1;
            }
            if (*abort_flag) {  // let our own copies land before the CTA goes away
                for (int j = max(0, issued - NS); j < issued; ++j) drain_wait(&fullb[j % NS], (j / NS) & 1);
            }
        }
    } else if (I8 && (warp == 5 || warp == 19)) {
        // ------------------------------------------------------------ Int8: two MMA issuers
        // warp 5: S = Q K^T once the fp16 K tile is written and both softmax halves have read the previous S;
        // warp 19: O += P V (A = P buffer j & 1) once both halves wrote P and the fp16 V tile is written.  O is
        // only written by warp 19, in tile order.  Their commits free the operand slots too: s_full[j & 1]
        // (Q K^T of tile j done) frees fp16 K slot j & 1, sp_free[j & 1] (P V of tile j done) fp16 V slot and P
        // buffer j & 1.
        if (lane == 0) {
            const bool qk = warp == 5;
            const uint32_t id_qk = tc::idesc_f16(false, false, false, kTcRows, kTcBK);
            const uint32_t id_pv = tc::idesc_f16(false, false, true, kTcRows, kTcD);
            const uint64_t dK0 = tc::sdesc_sw128(tc::smem_u32(sK), 16, 1024);
            const uint64_t dV0 = tc::sdesc_sw128(tc::smem_u32(sV), 8192, 1024);
            bool ok = !qk || tc::mbar_wait_spin(q_full, 0, abort_flag);
            if (ok) tc::tc_fence_after();
            for (int j = 0; ok && j < ntiles; ++j) {
                const int b2 = j & 1;
                if (qk) {
                    ok = tc::mbar_wait(&kc_full[b2], (j >> 1) & 1, abort_flag, 32, 64);
                    if (ok && j >= 1) ok = tc::mbar_wait(s_free, (j - 1) & 1, abort_flag, 32, 64);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint64_t kdesc = tc::sdesc_add(dK0, (uint32_t)b2 * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kTcD / 16; ++kk) {
                        const uint64_t db = tc::sdesc_add(kdesc, (kk >> 2) * 8192 + (kk & 3) * 32);
                        tc::mma_f16_ts(tmem + kColS, tmem + kColQ + kk * 8, db, id_qk, kk > 0);
                    }
                    tc::mma_commit(&s_full[b2]);
                } else {
                    ok = tc::mbar_wait(&p_full[b2], (j >> 1) & 1, abort_flag, 32, 64);
                    if (ok) ok = tc::mbar_wait(&vc_full[b2], (j >> 1) & 1, abort_flag, 32, 64);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint64_t vdesc = tc::sdesc_add(dV0, (uint32_t)b2 * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kTcBK / 16; ++kk) {  // A = P, 16-bit pairs in P buffer b2
                        const uint64_t db = tc::sdesc_add(vdesc, kk * 2048);
                        tc::mma_f16_ts(tmem + kColO, tmem + kColP8 + b2 * 32 + kk * 8, db, id_pv,
                                       (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(&sp_free[b2]);
                }
            }
            if (ok) {
                if (!qk) tc::mma_commit(o_done);
            } else {  // wait for every MMA this thread issued before TMEM is freed
                uint64_t* dr = qk ? drain : drain_pv;
                tc::mma_commit(dr);
                drain_wait(dr, 0);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        // Event loop: issue whichever of the next P V and the next Q K^T is ready (P V first), so that a P V
        // never waits behind a K tile that is still in flight.  Q K^T reads Q from TMEM.
        if (lane == 0) {
            const bool bf = p.mma_bf16 != 0;
            const uint32_t id_qk = tc::idesc_f16(bf, false, false, kTcRows, kTcBK);
            const uint32_t id_pv = tc::idesc_f16(bf, false, true, kTcRows, kTcD);
            const uint64_t dK0 = tc::sdesc_sw128(tc::smem_u32(sK), 16, 1024);
            const uint64_t dV0 = tc::sdesc_sw128(tc::smem_u32(sV), 8192, 1024);
            bool ok = tc::mbar_wait_spin(q_full, 0, abort_flag);
            if (ok) tc::tc_fence_after();
            int sj = 0, pj = 0;
            uint32_t idle = 0;
            uint64_t t_idle = 0;
            while (ok && pj < ntiles) {
                bool prog = false;
                // P V first: it is on the critical path (the softmax waits for it before writing the next P);
                // an issued Q K^T would hold the tensor pipe for its whole duration in front of it.
                if (pj < sj) {
                    const int st = pj % NS, cb = pj & 1;
                    bool ready = tc::mbar_test(&p_full[cb], (pj >> 1) & 1);
                    if (ready) ready = tc::mbar_test(&vfull[st], (pj / NS) & 1);
                    if (ready) {
                        tc::tc_fence_after();
                        const uint64_t vdesc = tc::sdesc_add(dV0, (uint32_t)st * kTileBytes);
#pragma unroll
                        for (int kk = 0; kk < kTcBK / 16; ++kk) {  // A = P, 16-bit pairs over S buffer cb
                            const uint64_t db = tc::sdesc_add(vdesc, kk * 2048);
                            tc::mma_f16_ts(tmem + kColO, tmem + kColS + cb * kTcBK + kk * 8, db, id_pv,
                                           (pj > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc::mma_commit(&sp_free[cb]);
                        tc::mma_commit(&vempty[st]);
                        ++pj;
                        prog = true;
                    }
                }
                if (sj < ntiles) {
                    const int sb = sj & 1, st = sj % NS;
                    bool ready = tc::mbar_test(&kfull[st], (sj / NS) & 1);
                    if (ready && sj >= 2) ready = tc::mbar_test(&sp_free[sb], ((sj >> 1) - 1) & 1);
                    if (ready) {
                        tc::tc_fence_after();
                        const uint64_t kdesc = tc::sdesc_add(dK0, (uint32_t)st * kTileBytes);
#pragma unroll
                        for (int kk = 0; kk < kTcD / 16; ++kk) {
                            const uint64_t db = tc::sdesc_add(kdesc, (kk >> 2) * 8192 + (kk & 3) * 32);
                            tc::mma_f16_ts(tmem + kColS + sb * kTcBK, tmem + kColQ + kk * 8, db, id_qk, kk > 0);
                        }
                        tc::mma_commit(&s_full[sb]);
                        tc::mma_commit(&kempty[st]);
                        ++sj;
                        prog = true;
                    }
                }
                if (prog) {
                    idle = 0;
                } else if ((++idle & 63) == 1) {  // bounded: give up after kWaitNs without progress
                    const uint64_t now = tc::globaltimer();
                    if (idle == 1) t_idle = now;
                    if (*abort_flag || now - t_idle > tc::kWaitNs) {
                        *abort_flag = 1;
                        ok = false;
                    }
                }
            }
            if (ok) {
                tc::mma_commit(o_done);
            } else {  // wait for every MMA this thread issued before TMEM is freed
                tc::mma_commit(drain);
                drain_wait(drain, 0);
            }
        }
    } else if (I8 && warp >= 10 && warp < 14) {
        // ------------------------------------------------------------ Int8 V converters
        // each thread converts key ct & 63 of every tile and multiplies its codes by that key's scale; the scale
        // is fetched one tile ahead so that the global load's latency overlaps the previous tile's work
        const int ct = threadIdx.x - 320;
        const uint16_t* vsrc = p.vs[layer] + ((size_t)b * p.HKV + kvh) * (size_t)p.s_cap + k_begin + (ct & 63);
        auto vscale = [&](int jj) -> uint16_t {
            return (jj < ntiles && k_begin + jj * kTcBK + (ct & 63) < k_end) ? vsrc[jj * kTcBK] : (uint16_t)0;
        };
        uint16_t sc_next = vscale(0);
        for (int j = 0; j < ntiles; ++j) {
            const int st = j % NS, cb = j & 1;
            const __half sh = __ushort_as_half(sc_next);
            sc_next = vscale(j + 1);
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&vfull[st], (j / NS) & 1, abort_flag))) break;
            const int nk = min(kTcBK, k_end - (k_begin + j * kTcBK));
            // fp16 V slot cb free once P V of tile j - 2 is done
            if (j >= 2 && !__all_sync(0xFFFFFFFFu, tc::mbar_wait(&sp_free[cb], ((j >> 1) - 1) & 1, abort_flag))) break;
            convert_i8_tile_scaled(sRawV + st * 16384, sV + cb * kTileBytes, nk, ct, __halves2half2(sh, sh));
            tc::fence_proxy_async_smem();
            __syncwarp();
            tc::mbar_arrive_one(&vempty[st]);
            tc::mbar_arrive_one(&vc_full[cb]);
        }
    } else if (I8 && warp >= 6 && warp < 10) {
        // ------------------------------------------------------------ Int8 K converters
        // as the V converters: key ct & 63 of every tile, times its scale, fetched one tile ahead
        const int ct = threadIdx.x - 192;
        const uint16_t* ksrc = p.ks[layer] + ((size_t)b * p.HKV + kvh) * (size_t)p.s_cap + k_begin + (ct & 63);
        auto kscale = [&](int jj) -> uint16_t {
            return (jj < ntiles && k_begin + jj * kTcBK + (ct & 63) < k_end) ? ksrc[jj * kTcBK] : (uint16_t)0;
        };
        uint16_t sc_next = kscale(0);
        for (int j = 0; j < ntiles; ++j) {
            const int st = j % NS, cb = j & 1;
            const __half sh = __ushort_as_half(sc_next);
            sc_next = kscale(j + 1);
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&kfull[st], (j / NS) & 1, abort_flag))) break;
            const int nk = min(kTcBK, k_end - (k_begin + j * kTcBK));
            // fp16 K slot cb free once Q K^T of tile j - 2 is done
            if (j >= 2 && !__all_sync(0xFFFFFFFFu, tc::mbar_wait(&s_full[cb], ((j >> 1) - 1) & 1, abort_flag))) break;
            convert_i8_tile_scaled(sRawK + st * 16384, sK + cb * kTileBytes, nk, ct, __halves2half2(sh, sh));
            tc::fence_proxy_async_smem();
            __syncwarp();
            tc::mbar_arrive_one(&kempty[st]);
            tc::mbar_arrive_one(&kc_full[cb]);
        }
    } else if (warp < 4 || warp >= kSoftB) {
        // ------------------------------------------------------------ softmax, in two halves
        // Half 0 (warps 0-3) takes key columns 0-31 of every tile, half 1 (the last four warps) columns 32-63,
        // of the same rows.  The two warps owning one TMEM lane quarter exchange their row maxima (and at the
        // end their row sums) through shared memory, one mbarrier per warp pair and tile parity, so both take
        // the same lazy-rescale decisions; each rescales and reads out its 128 columns of O and writes its 16
        // columns of P.  16-bit caches: half 1 writes P over S columns that half 0 reads, so only after the
        // exchange, which half 0 enters once its scores are in registers.  Int8 caches: P goes to its own
        // buffer, and the S tile is released right after it is read.
        const int h = warp < 4 ? 0 : 1;
        const int qd = warp & 3;
        const int r = qd * 32 + lane;  // row within the tile == TMEM lane
        const int gr = row0 + r;
        const bool row_ok = gr < p.R;
        const int node = row_ok ? gr / p.G : 0;
        const int head = kvh * p.G + (row_ok ? gr % p.G : 0);
        const uint64_t anc = row_ok ? p.anc[(size_t)b * T + node] : 0ull;
        const int lo_row = win > 0 ? S + node - win + 1 : INT_MIN;  // sliding band of this row
        const bool bf = p.mma_bf16 != 0;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        if (h == 0) {  // Q row -> TMEM lane r, 16-bit pairs (rounded to fp16 when the MMA runs in fp16)
            const uint4* src = reinterpret_cast<const uint4*>(p.q[layer] + ((size_t)(b * T + node) * p.HQ + head) * kTcD);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint4 v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = row_ok ? src[half * 16 + i] : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t w[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint4 x = v[c2 * 8 + i];
                        if (!bf) x = bf16x8_to_f16x8(x);
                        w[4 * i] = x.x;
                        w[4 * i + 1] = x.y;
                        w[4 * i + 2] = x.z;
                        w[4 * i + 3] = x.w;
                    }
                    tc::tmem_st32(tmem + lane_base + kColQ + (half * 2 + c2) * 32, w);
                }
            }
            tc::tmem_wait_st();
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(q_full);
        }
        // exchange number jj (one per tile, then one for the row sums): xv[(jj & 1) * 2 + half][row]
        auto exchange = [&](int jj, float mine, float& other) -> bool {
            const int slot = jj & 1;
            xv[(slot * 2 + h) * kTcRows + r] = mine;
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(&xch[qd * 2 + slot]);
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&xch[qd * 2 + slot], (jj >> 1) & 1, abort_flag))) return false;
            tc::tc_fence_after();
            other = xv[(slot * 2 + (h ^ 1)) * kTcRows + r];
            return true;
        };
        const float qk_scale = 1.4426950408889634f * 0.0625f;  // log2(e) / sqrt(256)
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int sb = j & 1;
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag))) { ok = false; break; }
            tc::tc_fence_after();
            uint32_t sc[32];
            tc::tmem_ld32(tmem + lane_base + kColS + (I8 ? 0 : sb * kTcBK) + h * 32, sc);
            tc::tmem_wait_ld();
            if (I8) {  // the S tile is free for the next Q K^T
                tc::tc_fence_before();
                __syncwarp();
                tc::mbar_arrive_one(s_free);
            }

            const int ct = k_begin + j * kTcBK;  // first key of the tile
            const int c0 = ct + h * 32;          // first key of this half
            // Raw scores (Int8: the K scales are in the fp16 copy of K); masked keys become -inf.  Tiles whose 64
            // keys are all history keys inside the range need no mask (padding rows past the unit's G*T rows take
            // it too: their Q is zero and their results are dropped).  The maximum is taken on the raw scores (the
            // scale is positive) and every p is ex2(s * scale - m) in one fused multiply-add, in the log2 domain.
            float x[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(sc[c]);
            if (!(ct + kTcBK <= k_end && ct + kTcBK <= S && ct >= lo_last)) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int key = c0 + c;
                    bool v = row_ok && key < k_end && key >= lo_row;
                    if (key >= S) v = v && ((anc >> ((key - S) & 63)) & 1ull);
                    if (!v) x[c] = -INFINITY;
                }
            }
            float mx[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) mx[c] = fmaxf(x[c], x[c + 16]);
#pragma unroll
            for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
            float mo;
            if (!exchange(j, mx[0], mo)) { ok = false; break; }
            const float mt_ = fmaxf(mx[0], mo) * qk_scale;  // the row's tile maximum, the same in both halves
            float alpha = 1.f;
            bool resc = false;
            if (mt_ > m_ref + 8.f) {  // also when m_ref is still -inf
                alpha = tc::ex2_approx(m_ref - mt_);
                m_ref = mt_;
                resc = true;
            }
            // m_ref == -inf only while every score so far was masked (then every p below is 0)
            const float msub = m_ref == -INFINITY ? 0.f : m_ref;
            uint32_t pk[16];
            float sm2[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
                const float p0 = tc::ex2_approx(fmaf(x[c], qk_scale, -msub));
                const float p1 = tc::ex2_approx(fmaf(x[c + 1], qk_scale, -msub));
                sm2[c >> 1] = p0 + p1;
                pk[c >> 1] = pack2(p0, p1, I8 ? false : bf);
            }
#pragma unroll
            for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                for (int c = 0; c < w; ++c) sm2[c] += sm2[c + w];
            l = l * alpha + sm2[0];  // this half's part of the row sum

            // O *= alpha for this warp's rows and half of the columns, once P V of tile j - 1 is done with O.  Its
            // buffer's barrier has completed the phase before (P V of tile j - 3, which Q K^T of tile j - 1 waited
            // for) and cannot complete the one after (P V of tile j + 1) before this P is written.
            if (j >= 1 && __any_sync(0xFFFFFFFFu, resc)) {
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&sp_free[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t o[32];
                    tc::tmem_ld32(tmem + lane_base + kColO + (h * 4 + ch) * 32, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tc::tmem_st32(tmem + lane_base + kColO + (h * 4 + ch) * 32, o);
                }
                tc::tmem_wait_st();
            }
            const bool zero_v = !I8 && h == 0 && ct + kTcBK > k_end;
            if (zero_v) {  // last tile: zero V rows past the key range (their bytes are not ours)
                const int st = j % NS;
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&vfull[st], (j / NS) & 1, abort_flag))) { ok = false; break; }
                const int nk = k_end - ct;
                uint8_t* vb = sV + st * kTileBytes;
                for (int e = r; e < (kTcBK - nk) * 32; e += kTcRows) {
                    const int row = nk + e / 32, chunk = e % 32;
                    *reinterpret_cast<uint4*>(vb + (chunk >> 3) * 8192 + row * 128 + (chunk & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            // Int8: P buffer sb is free once P V of tile j - 2 is done (the phase before, P V of tile j - 4, was
            // waited for at tile j - 2; the one after needs this P)
            if (I8 && j >= 2 && !__all_sync(0xFFFFFFFFu, tc::mbar_wait(&sp_free[sb], ((j >> 1) - 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            // this half's 32 keys of P, 16-bit pairs (the A operand of P V): 16-bit caches over S columns
            // [16 h, 16 h + 16) of its S tile, Int8 columns [16 h, 16 h + 16) of P buffer sb
            tc::tmem_st16(tmem + lane_base + (I8 ? kColP8 + sb * 32 : kColS + sb * kTcBK) + h * 16, pk);
            tc::tmem_wait_st();
            if (zero_v) tc::fence_proxy_async_smem();  // the zeroed V rows
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(&p_full[sb]);
        }
        if (ok) {  // the row sum of both halves
            float lo;
            if (exchange(ntiles, l, lo)) l += lo;
            else ok = false;
        }
        if (ok && __all_sync(0xFFFFFFFFu, tc::mbar_wait(o_done, 0, abort_flag))) {
            tc::tc_fence_after();
            const size_t slot = ((size_t)unit * p.splits + split) * p.R + gr;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int ch = h * 4; ch < h * 4 + 4; ++ch) {
                uint32_t o[32];
                tc::tmem_ld32(tmem + lane_base + kColO + ch * 32, o);
                tc::tmem_wait_ld();
                if (!row_ok) continue;
                if (p.splits == 1) {
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o[layer]) +
                                                          ((size_t)(b * T + node) * p.HQ + head) * kTcD + ch * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack2(__uint_as_float(o[8 * k + 2 * e]) * inv, __uint_as_float(o[8 * k + 2 * e + 1]) * inv, true);
                        dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * kTcD + ch * 32);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                             __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
                }
            }
            if (h == 0 && row_ok && p.splits > 1) {
                p.ws_ml[2 * slot] = m_ref;
                p.ws_ml[2 * slot + 1] = l;
            }
        }
    }
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) dev_fail(p.status, TSV_DEV_TIMEOUT, b, blockIdx.x);
    if (warp == 5) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ 16-bit caches: 128-key score tiles
// Q K^T over 128 keys per MMA (N = 128): an MMA occupies the tensor pipe for about 100 cycles whatever N <= 128
// is, so 128-key tiles halve the Q K^T issue cost per key of the 64-key design above.  P V still runs over
// 64-key halves (V stages of 64 keys, P written half by half, so P V of the first half starts while the
// second is being written).  TMEM: Q [0, 128), S [128, 256) (one buffer: the softmax frees it right after
// reading it), O [256, 512).  Shared memory: K stages [2 x 64 KB] at 0 (layout [64-dim block][128 keys][128 B]),
// V stages [2 x 32 KB] at 128 KB, P [2 halves x 16 KB] at 192 KB, barriers at 224 KB.  Warp 5 issues Q K^T and
// warp 7 P V, so a P V never waits behind the next tile's Q K^T.
constexpr int kWK = 128;
constexpr uint32_t kWKTile = kWK * kTcD * 2;  // 64 KiB
constexpr int kWSmem = 1024 + 229376 + 512;

__global__ void __launch_bounds__(kTcThreads16, 1) attn_tcw_kernel(const __grid_constant__ TcParams p) {
    griddep_begin();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = sm;
    uint8_t* sV = sm + 131072;
    uint8_t* sP = sm + 196608;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 229376);
    uint64_t* kfull = bars + 0;   // [2] 128-key K tile landed
    uint64_t* kempty = bars + 2;  // [2] Q K^T done with it
    uint64_t* vfull = bars + 4;   // [2] 64-key V half landed
    uint64_t* vempty = bars + 6;  // [2] P V done with it
    uint64_t* s_full = bars + 8;
    uint64_t* s_free = bars + 9;
    uint64_t* p_full = bars + 10;  // [2] P half written (4 softmax warps)
    uint64_t* p_free = bars + 12;  // [2] P V done with the P half
    uint64_t* o_done = bars + 14;
    uint64_t* q_full = bars + 15;
    uint64_t* drain = bars + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 18);
    uint64_t* drain_pv = bars + 19;  // every MMA of the P V issuer done (abort path)
    constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int item = blockIdx.x;
    const int mt = item % p.mtiles;
    item /= p.mtiles;
    const int split = item % p.splits;
    const int unit = item / p.splits;
    const int kvh = unit % p.HKV;
    const int b = (unit / p.HKV) % p.B;
    const int layer = unit / (p.HKV * p.B);
    const int T = p.T;
    const int kvl = p.kv_len[b];
    if (kvl < T || kvl > p.max_kv_len || (int64_t)kvl > p.s_cap) {
        if (split == 0 && mt == 0 && kvh == 0 && layer == 0 && threadIdx.x == 0)
            dev_fail(p.status, TSV_DEV_BAD_KV_LEN, b, kvl);
        return;
    }
    const int S = kvl - T;
    const int row0 = mt * kTcRows;
    const int k_end = min(kvl, split * p.chunk + p.chunk);
    const int win = p.window[layer];
    const int lo_first = win > 0 ? S + row0 / p.G - win + 1 : INT_MIN;
    const int lo_last = win > 0 ? S + (min(p.R, row0 + kTcRows) - 1) / p.G - win + 1 : INT_MIN;
    int k_begin = split * p.chunk;
    if (lo_first > k_begin) k_begin += ((lo_first - k_begin) / kWK) * kWK;
    const int ntiles = k_end > k_begin ? (k_end - k_begin + kWK - 1) / kWK : 0;  // 128-key tiles
    const int nhalves = 2 * ntiles;

    if (p.status != nullptr && *reinterpret_cast<volatile int32_t*>(p.status) == TSV_DEV_TIMEOUT) return;
    if (ntiles == 0) {
        if (threadIdx.x < kTcRows && row0 + (int)threadIdx.x < p.R) {
            const size_t slot = ((size_t)unit * p.splits + split) * p.R + row0 + threadIdx.x;
            p.ws_ml[2 * slot] = -INFINITY;
            p.ws_ml[2 * slot + 1] = 0.f;
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&kfull[s], 1);
            tc::mbar_init(&kempty[s], 1);
            tc::mbar_init(&vfull[s], 1);
            tc::mbar_init(&vempty[s], 1);
            tc::mbar_init(&p_full[s], 4);
            tc::mbar_init(&p_free[s], 1);
        }
        tc::mbar_init(s_full, 1);
        tc::mbar_init(s_free, 4);
        tc::mbar_init(o_done, 1);
        tc::mbar_init(q_full, 4);
        tc::mbar_init(drain, 1);
        tc::mbar_init(drain_pv, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 5) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4 || warp == 6) {
        // ------------------------------------------------------------ TMA producers: warp 4 K tiles, warp 6 V halves
        if (lane == 0) {
            const bool isK = warp == 4;
            const CUtensorMap* m = isK ? &p.kmap[layer] : &p.vmap[layer];
            uint64_t* fullb = isK ? kfull : vfull;
            uint64_t* emptyb = isK ? kempty : vempty;
            tc::tma_prefetch_desc(m);
            const int rowbase = (int)(((int64_t)b * p.HKV + kvh) * p.s_cap + k_begin);
            const int n = isK ? ntiles : nhalves;
            int issued = 0;
            for (int j = 0; j < n; ++j) {
                const int st = j & 1;
                if (j >= 2 && !tc::mbar_wait(&emptyb[st], ((j >> 1) - 1) & 1, abort_flag, 256)) break;
                if (isK) {  // 128 keys: two 64-row boxes per 64-dim block
                    tc::mbar_expect_tx(&fullb[st], kWKTile);
                    uint8_t* dst = sK + st * kWKTile;
#pragma unroll
                    for (int db = 0; db < 4; ++db) {
                        tc::tma_load_2d(dst + db * 16384, m, &fullb[st], db * 64, rowbase + j * kWK);
                        tc::tma_load_2d(dst + db * 16384 + 8192, m, &fullb[st], db * 64, rowbase + j * kWK + 64);
                    }
                } else {
                    tc::mbar_expect_tx(&fullb[st], kTileBytes);
                    uint8_t* dst = sV + st * kTileBytes;
#pragma unroll
                    for (int db = 0; db < 4; ++db) tc::tma_load_2d(dst + db * 8192, m, &fullb[st], db * 64, rowbase + j * kTcBK);
                }
                issued = j + 1;
            }
            if (*abort_flag)
                for (int j = max(0, issued - 2); j < issued; ++j) drain_wait(&fullb[j & 1], (j >> 1) & 1);
        }
    } else if (warp == 5 || warp == 7) {
        // ------------------------------------------------------------ MMA issuers: warp 5 Q K^T, warp 7 P V
        // One issuing thread is held for each MMA's whole pipe time, so a P V whose P is ready would otherwise
        // wait behind the 16 MMAs of the next tile's Q K^T.
        if (lane == 0) {
            const bool qk = warp == 5;
            const bool bf = p.mma_bf16 != 0;
            const uint32_t id_qk = tc::idesc_f16(bf, false, false, kTcRows, kWK);
            const uint32_t id_pv = tc::idesc_f16(bf, false, true, kTcRows, kTcD);
            // descriptors built once; each MMA adds its byte offset to the address field
            const uint64_t dK0 = tc::sdesc_sw128(tc::smem_u32(sK), 16, 1024);
            const uint64_t dV0 = tc::sdesc_sw128(tc::smem_u32(sV), 8192, 1024);
            const uint64_t dP0 = tc::sdesc_sw128(tc::smem_u32(sP), 16, 1024);
            bool ok = !qk || tc::mbar_wait_spin(q_full, 0, abort_flag);
            if (ok) tc::tc_fence_after();
            if (qk) {
                for (int sj = 0; ok && sj < ntiles; ++sj) {  // S = Q K^T once K is there and S was read
                    const int st = sj & 1;
                    ok = tc::mbar_wait(&kfull[st], (sj >> 1) & 1, abort_flag, 32, 64);
                    if (ok && sj >= 1) ok = tc::mbar_wait(s_free, (sj - 1) & 1, abort_flag, 32, 64);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint64_t dk = tc::sdesc_add(dK0, st * kWKTile);
#pragma unroll
                    for (int kk = 0; kk < kTcD / 16; ++kk) {
                        const uint64_t db = tc::sdesc_add(dk, (kk >> 2) * 16384 + (kk & 3) * 32);
                        tc::mma_f16_ts(tmem + kColS, tmem + kColQ + kk * 8, db, id_qk, kk > 0);
                    }
                    tc::mma_commit(s_full);
                    tc::mma_commit(&kempty[st]);
                }
            } else {
                for (int pq = 0; ok && pq < nhalves; ++pq) {  // O += P V over 64-key half pq
                    const int h = pq & 1, j = pq >> 1, st = pq & 1;
                    ok = tc::mbar_wait(&p_full[h], j & 1, abort_flag, 32, 64);
                    if (ok) ok = tc::mbar_wait(&vfull[st], (pq >> 1) & 1, abort_flag, 32, 64);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint64_t dv = tc::sdesc_add(dV0, st * kTileBytes), dp = tc::sdesc_add(dP0, h * 16384);
#pragma unroll
                    for (int kk = 0; kk < kTcBK / 16; ++kk) {
                        const uint64_t da = tc::sdesc_add(dp, kk * 32);
                        const uint64_t db = tc::sdesc_add(dv, kk * 2048);
                        tc::mma_f16(tmem + kColO, da, db, id_pv, (pq > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(&p_free[h]);
                    tc::mma_commit(&vempty[st]);
                }
            }
            if (ok) {
                if (!qk) tc::mma_commit(o_done);
            } else {  // wait for every MMA this thread issued before TMEM is freed
                uint64_t* dr = qk ? drain : drain_pv;
                tc::mma_commit(dr);
                drain_wait(dr, 0);
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ softmax warpgroup
        const int r = threadIdx.x;
        const int gr = row0 + r;
        const bool row_ok = gr < p.R;
        const int node = row_ok ? gr / p.G : 0;
        const int head = kvh * p.G + (row_ok ? gr % p.G : 0);
        const uint64_t anc = row_ok ? p.anc[(size_t)b * T + node] : 0ull;
        const int lo_row = win > 0 ? S + node - win + 1 : INT_MIN;
        const bool bf = p.mma_bf16 != 0;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        {  // Q row -> TMEM lane r, 16-bit pairs (rounded to fp16 when the MMA runs in fp16)
            const uint4* src = reinterpret_cast<const uint4*>(p.q[layer] + ((size_t)(b * T + node) * p.HQ + head) * kTcD);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint4 v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = row_ok ? src[half * 16 + i] : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t w[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint4 x = v[c2 * 8 + i];
                        if (!bf) x = bf16x8_to_f16x8(x);
                        w[4 * i] = x.x;
                        w[4 * i + 1] = x.y;
                        w[4 * i + 2] = x.z;
                        w[4 * i + 3] = x.w;
                    }
                    tc::tmem_st32(tmem + lane_base + kColQ + (half * 2 + c2) * 32, w);
                }
            }
            tc::tmem_wait_st();
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(q_full);
        }
        const float qk_scale = 1.4426950408889634f * 0.0625f;  // log2(e) / sqrt(256)
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(s_full, j & 1, abort_flag))) { ok = false; break; }
            tc::tc_fence_after();
            float x[128];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t sv[32];
                tc::tmem_ld32(tmem + lane_base + kColS + q4 * 32, sv);
                tc::tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) x[q4 * 32 + c] = __uint_as_float(sv[c]);
            }
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(s_free);

            const int c0 = k_begin + j * kWK;
            // Raw scores; masked keys become -inf.  The tile maximum is taken on the raw scores (the scale is
            // positive, eight independent chains) and every p is ex2(s * scale - m) in one fused multiply-add.
            if (!(c0 + kWK <= k_end && c0 + kWK <= S && c0 >= lo_last)) {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const int key = c0 + c;
                    bool v = row_ok && key < k_end && key >= lo_row;
                    if (key >= S) v = v && ((anc >> ((key - S) & 63)) & 1ull);
                    if (!v) x[c] = -INFINITY;
                }
            }
            float mx[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = x[k];
#pragma unroll
            for (int c = 8; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], x[c]);
#pragma unroll
            for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                for (int k = 0; k < w; ++k) mx[k] = fmaxf(mx[k], mx[k + w]);
            const float mt_ = mx[0] * qk_scale;
            float alpha = 1.f;
            bool resc = false;
            if (mt_ > m_ref + 8.f) {
                alpha = tc::ex2_approx(m_ref - mt_);
                m_ref = mt_;
                resc = true;
            }
            const float msub = m_ref == -INFINITY ? 0.f : m_ref;
            if (j >= 1 && __any_sync(0xFFFFFFFFu, resc)) {  // P V of the previous tile done with O: rescale it
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&p_free[1], (j - 1) & 1, abort_flag))) { ok = false; break; }
                tc::tc_fence_after();
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t o[32];
                    tc::tmem_ld32(tmem + lane_base + kColO + ch * 32, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tc::tmem_st32(tmem + lane_base + kColO + ch * 32, o);
                }
                tc::tmem_wait_st();
            }
            float ps = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // P half h of the previous tile no longer read (P V of that half done)
                if (j >= 1 && !__all_sync(0xFFFFFFFFu, tc::mbar_wait(&p_free[h], (j - 1) & 1, abort_flag))) { ok = false; break; }
                const int ch0 = c0 + h * kTcBK;
                if (ch0 + kTcBK > k_end) {  // zero V rows past the key range in this half's stage (not our bytes)
                    const int q = 2 * j + h, st = q & 1;
                    if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&vfull[st], (q >> 1) & 1, abort_flag))) { ok = false; break; }
                    const int nk = max(0, k_end - ch0);
                    uint8_t* vb = sV + st * kTileBytes;
                    for (int e = r; e < (kTcBK - nk) * 32; e += kTcRows) {
                        const int row = nk + e / 32, chunk = e % 32;
                        *reinterpret_cast<uint4*>(vb + (chunk >> 3) * 8192 + row * 128 + (chunk & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                uint32_t pk[32];
                float sm4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const float p0 = tc::ex2_approx(fmaf(x[h * 64 + c], qk_scale, -msub));
                    const float p1 = tc::ex2_approx(fmaf(x[h * 64 + c + 1], qk_scale, -msub));
                    sm4[(c >> 1) & 3] += p0 + p1;
                    pk[c >> 1] = pack2(p0, p1, bf);
                }
                ps += (sm4[0] + sm4[1]) + (sm4[2] + sm4[3]);
                uint8_t* ph = sP + h * 16384;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4*>(ph + r * 128 + ((ch ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                __syncwarp();
                tc::mbar_arrive_one(&p_full[h]);
            }
            if (!ok) break;
            l = l * alpha + ps;
        }
        if (ok && __all_sync(0xFFFFFFFFu, tc::mbar_wait(o_done, 0, abort_flag))) {
            tc::tc_fence_after();
            const size_t slot = ((size_t)unit * p.splits + split) * p.R + gr;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t o[32];
                tc::tmem_ld32(tmem + lane_base + kColO + ch * 32, o);
                tc::tmem_wait_ld();
                if (!row_ok) continue;
                if (p.splits == 1) {
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o[layer]) +
                                                          ((size_t)(b * T + node) * p.HQ + head) * kTcD + ch * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack2(__uint_as_float(o[8 * k + 2 * e]) * inv, __uint_as_float(o[8 * k + 2 * e + 1]) * inv, true);
                        dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * kTcD + ch * 32);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                             __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
                }
            }
            if (row_ok && p.splits > 1) {
                p.ws_ml[2 * slot] = m_ref;
                p.ws_ml[2 * slot + 1] = l;
            }
        }
    }

    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) dev_fail(p.status, TSV_DEV_TIMEOUT, b, blockIdx.x);
    if (warp == 5) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ Int8 caches: 128-key score tiles
// The same 128-key Q K^T (N = 128) for Int8 caches.  TMEM as in attn_tcw_kernel: Q [0, 128), S [128, 256) (one
// buffer, freed as soon as the softmax has read it), O [256, 512).  An fp16 K tile of 128 keys (64 KB) does
// not fit twice beside the other rings, so K moves in dim quarters (128 keys x 64 dims): TMA lands a raw quarter
// (8 KB, 64-byte swizzle) in a 3-stage ring, the K converters write its fp16 copy (16 KB, 128-byte swizzle) into
// a 4-slot ring -- slot q holds quarter q of the current tile -- and Q K^T issues the quarter's MMAs as soon as
// it is there.  V moves in 64-key halves (raw halves, fp16 halves); P goes to shared memory in two 64-key
// halves, one per softmax half, and P V reads A from there.
// The converters fold each token's scale into its fp16 row (code exact, then one rounding of code * scale), and
// Q is stored pre-multiplied by log2(e) / sqrt(256), so S arrives in the log2 domain and the softmax multiplies
// nothing but P.
// Two issuing threads: warp 4 issues Q K^T a quarter (four MMAs) at a time as each fp16 K quarter is written,
// warp 19 P V a half (four MMAs) at a time as each P half and fp16 V half are written; one issuing thread is held
// for each MMA's whole pipe time, so one thread issuing both serialises them.
// 640 threads (96 registers each: a softmax thread holds its 64 scores):
//   warps 0-3, 7-10  softmax halves 0 and 1 (key columns 64 h .. 64 h + 63 of the tile; lane quarter = warp & 3);
//                    half 0 also stores Q into TMEM
//   warp 4           TMEM allocation and the Q K^T issuer
//   warp 5, 6        TMA producers: raw K quarters, raw V halves
//   warps 11-14      K converters (thread = key of the quarter)
//   warps 15-18      V converters
//   warp 19          the P V issuer
constexpr int kW8Threads = 640;

// Keys c0 .. c0 + 63 as a bit mask (bit c = key c0 + c) of what one query row sees: keys below k_end and at or
// above lo_row (the sliding band), history keys (< S) in full, block keys S + i where bit i of anc is set.
__device__ __forceinline__ uint64_t visible64(int c0, int k_end, int lo_row, int S, uint64_t anc, bool row_ok) {
    if (!row_ok) return 0ull;
    const int n_end = min(max(k_end - c0, 0), 64);                              // keys < k_end
    uint64_t m = n_end >= 64 ? ~0ull : ((1ull << n_end) - 1ull);
    if (lo_row > c0) m &= lo_row - c0 >= 64 ? 0ull : (~0ull << (lo_row - c0));  // keys >= lo_row
    const int sh = S - c0;                                                       // first block key's bit
    if (sh <= 0) m &= -sh >= 64 ? 0ull : (anc >> (-sh));
    else if (sh < 64) m &= ((1ull << sh) - 1ull) | (anc << sh);
    return m;
}

constexpr int kW8KR = 3;                          // raw K quarter stages
constexpr uint32_t kW8OffKh = 0;                  // 4 x 16 KB fp16 K quarters [128 keys][128 B]
constexpr uint32_t kW8OffKr = 65536;              // 3 x 8 KB raw K quarters [128 keys][64 B], 64-byte swizzle
constexpr uint32_t kW8OffVh = 90112;              // 2 x 32 KB fp16 V halves [4 dim blocks][64 keys][128 B]
constexpr uint32_t kW8OffVr = 155648;             // 2 x 16 KB raw V halves [2][64 keys][128 B]
constexpr uint32_t kW8OffP = 188416;              // 2 x 16 KB P halves [128 rows][128 B]
constexpr uint32_t kW8OffX = 221184;              // softmax halves' exchange [2 slots][2 halves][128 rows] fp32
constexpr uint32_t kW8OffBar = 223232;            // barriers, TMEM slot, abort flag
constexpr int kW8Smem = 1024 + 223232 + 512;
constexpr float kLog2eOverSqrtD = 1.4426950408889634f * 0.0625f;


__global__ void __launch_bounds__(kW8Threads, 1) attn_tcw8_kernel(const __grid_constant__ TcParams p) {
    griddep_begin();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sKh = sm + kW8OffKh;
    uint8_t* sKr = sm + kW8OffKr;
    uint8_t* sVh = sm + kW8OffVh;
    uint8_t* sVr = sm + kW8OffVr;
    uint8_t* sP = sm + kW8OffP;
    float* xv = reinterpret_cast<float*>(sm + kW8OffX);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kW8OffBar);
    uint64_t* kr_full = bars + 0;    // [3] raw K quarter landed
    uint64_t* kr_empty = bars + 3;   // [3] the K converters are done with it
    uint64_t* kq_full = bars + 6;    // [4] fp16 K quarter written
    uint64_t* kq_empty = bars + 10;  // [4] Q K^T done with it
    uint64_t* vr_full = bars + 14;   // [2] raw V half landed
    uint64_t* vr_empty = bars + 16;  // [2] the V converters are done with it
    uint64_t* vh_full = bars + 18;   // [2] fp16 V half written
    uint64_t* vh_empty = bars + 20;  // [2] P V done with it
    uint64_t* s_full = bars + 22;    // Q K^T of a tile done
    uint64_t* s_free = bars + 23;    // both softmax halves read S (8 warps)
    uint64_t* p_full = bars + 24;    // [2] P half written (4 warps)
    uint64_t* p_free = bars + 26;    // [2] P V done with the P half
    uint64_t* xch = bars + 28;       // [4 lane quarters][2 parities] both halves posted their value
    uint64_t* q_full = bars + 36;
    uint64_t* o_done = bars + 37;
    uint64_t* drain = bars + 38;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 39);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 40);
    uint64_t* drain_pv = bars + 41;  // every MMA of the P V issuer done (abort path)
    constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int item = blockIdx.x;
    const int mt = item % p.mtiles;
    item /= p.mtiles;
    const int split = item % p.splits;
    const int unit = item / p.splits;
    const int kvh = unit % p.HKV;
    const int b = (unit / p.HKV) % p.B;
    const int layer = unit / (p.HKV * p.B);
    const int T = p.T;
    const int kvl = p.kv_len[b];
    if (kvl < T || kvl > p.max_kv_len || (int64_t)kvl > p.s_cap) {
        if (split == 0 && mt == 0 && kvh == 0 && layer == 0 && threadIdx.x == 0)
            dev_fail(p.status, TSV_DEV_BAD_KV_LEN, b, kvl);
        return;
    }
    const int S = kvl - T;
    const int row0 = mt * kTcRows;
    const int k_end = min(kvl, split * p.chunk + p.chunk);
    const int win = p.window[layer];
    const int lo_first = win > 0 ? S + row0 / p.G - win + 1 : INT_MIN;
    const int lo_last = win > 0 ? S + (min(p.R, row0 + kTcRows) - 1) / p.G - win + 1 : INT_MIN;
    int k_begin = split * p.chunk;
    if (lo_first > k_begin) k_begin += ((lo_first - k_begin) / kWK) * kWK;
    const int ntiles = k_end > k_begin ? (k_end - k_begin + kWK - 1) / kWK : 0;  // 128-key tiles
    const int nhalves = 2 * ntiles;

    if (p.status != nullptr && *reinterpret_cast<volatile int32_t*>(p.status) == TSV_DEV_TIMEOUT) return;
    if (ntiles == 0) {
        if (threadIdx.x < kTcRows && row0 + (int)threadIdx.x < p.R) {
            const size_t slot = ((size_t)unit * p.splits + split) * p.R + row0 + threadIdx.x;
            p.ws_ml[2 * slot] = -INFINITY;
            p.ws_ml[2 * slot + 1] = 0.f;
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kW8KR; ++s) {
            tc::mbar_init(&kr_full[s], 1);
            tc::mbar_init(&kr_empty[s], 4);
        }
        for (int s = 0; s < 4; ++s) {
            tc::mbar_init(&kq_full[s], 4);
            tc::mbar_init(&kq_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&vr_full[s], 1);
            tc::mbar_init(&vr_empty[s], 4);
            tc::mbar_init(&vh_full[s], 4);
            tc::mbar_init(&vh_empty[s], 1);
            tc::mbar_init(&p_full[s], 4);
            tc::mbar_init(&p_free[s], 1);
        }
        for (int s = 0; s < 8; ++s) tc::mbar_init(&xch[s], 2);
        tc::mbar_init(s_full, 1);
        tc::mbar_init(s_free, 8);
        tc::mbar_init(q_full, 4);
        tc::mbar_init(o_done, 1);
        tc::mbar_init(drain, 1);
        tc::mbar_init(drain_pv, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 4) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int rowbase = (int)(((int64_t)b * p.HKV + kvh) * p.s_cap + k_begin);
    const size_t seq_row = ((size_t)b * p.HKV + kvh) * (size_t)p.s_cap;

    if (warp == 5 || warp == 6) {
        // ------------------------------------------------------------ TMA producers (lane 0 of each warp)
        if (lane == 0) {
            const bool isK = warp == 5;
            const CUtensorMap* m = isK ? &p.kmap[layer] : &p.vmap[layer];
            tc::tma_prefetch_desc(m);
            const int n = isK ? 4 * ntiles : nhalves;
            const int NS = isK ? kW8KR : 2;
            uint64_t* fullb = isK ? kr_full : vr_full;
            uint64_t* emptyb = isK ? kr_empty : vr_empty;
            int issued = 0;
            for (int g = 0; g < n; ++g) {
                const int st = g % NS;
                if (g >= NS && !tc::mbar_wait(&emptyb[st], ((g / NS) - 1) & 1, abort_flag, 256)) break;
                if (isK) {  // quarter g & 3 of tile g >> 2: 128 keys x 64 bytes
                    tc::mbar_expect_tx(&fullb[st], 8192);
                    tc::tma_load_2d(sKr + st * 8192, m, &fullb[st], (g & 3) * 64, rowbase + (g >> 2) * kWK);
                } else {    // 64 keys x 256 bytes as two 128-byte-wide halves
                    tc::mbar_expect_tx(&fullb[st], 16384);
                    uint8_t* dst = sVr + st * 16384;
                    tc::tma_load_2d(dst, m, &fullb[st], 0, rowbase + g * kTcBK);
                    tc::tma_load_2d(dst + 8192, m, &fullb[st], 128, rowbase + g * kTcBK);
                }
                issued = g + 1;
            }
            if (*abort_flag)
                for (int g = max(0, issued - NS); g < issued; ++g) drain_wait(&fullb[g % NS], (g / NS) & 1);
        }
    } else if (warp == 4 || warp == 19) {
        // ------------------------------------------------------------ MMA issuers: warp 4 Q K^T, warp 19 P V
        if (lane == 0) {
            const bool qk = warp == 4;
            const uint32_t id_qk = tc::idesc_f16(false, false, false, kTcRows, kWK);
            const uint32_t id_pv = tc::idesc_f16(false, false, true, kTcRows, kTcD);
            // one descriptor per operand ring; every MMA below is a constant offset from one of them
            const uint64_t dK = tc::sdesc_sw128(tc::smem_u32(sKh), 16, 1024);
            const uint64_t dV = tc::sdesc_sw128(tc::smem_u32(sVh), 8192, 1024);
            const uint64_t dP = tc::sdesc_sw128(tc::smem_u32(sP), 16, 1024);
            const uint32_t tS = tmem + kColS, tO = tmem + kColO;
            bool ok = !qk || tc::mbar_wait_spin(q_full, 0, abort_flag);
            if (ok) tc::tc_fence_after();
            if (qk) {
                for (int g = 0; ok && g < 4 * ntiles; ++g) {  // quarter g & 3 of tile g >> 2
                    const int sj = g >> 2, sq = g & 3;
                    if (sq == 0 && sj > 0) ok = tc::mbar_wait(s_free, (sj - 1) & 1, abort_flag, 32, 64);
                    if (ok) ok = tc::mbar_wait(&kq_full[sq], sj & 1, abort_flag, 32, 64);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint64_t bk = tc::sdesc_add(dK, sq * 16384);
                    const uint32_t aq = tmem + kColQ + sq * 32;  // Q columns of features 64 sq ..
                    tc::mma_f16_ts(tS, aq, bk, id_qk, sq > 0 ? 1u : 0u);
                    tc::mma_f16_ts(tS, aq + 8, tc::sdesc_add(bk, 32), id_qk, 1u);
                    tc::mma_f16_ts(tS, aq + 16, tc::sdesc_add(bk, 64), id_qk, 1u);
                    tc::mma_f16_ts(tS, aq + 24, tc::sdesc_add(bk, 96), id_qk, 1u);
                    tc::mma_commit(&kq_empty[sq]);
                    if (sq == 3) tc::mma_commit(s_full);
                }
            } else {
                for (int pq = 0; ok && pq < nhalves; ++pq) {  // P V of half pq: P written, fp16 V half there
                    const int h = pq & 1, jt = pq >> 1;
                    ok = tc::mbar_wait(&p_full[h], jt & 1, abort_flag, 32, 64);
                    if (ok) ok = tc::mbar_wait(&vh_full[h], jt & 1, abort_flag, 32, 64);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint64_t a = tc::sdesc_add(dP, h * 16384), bv = tc::sdesc_add(dV, h * 32768);
                    tc::mma_f16(tO, a, bv, id_pv, pq > 0 ? 1u : 0u);
                    tc::mma_f16(tO, tc::sdesc_add(a, 32), tc::sdesc_add(bv, 2048), id_pv, 1u);
                    tc::mma_f16(tO, tc::sdesc_add(a, 64), tc::sdesc_add(bv, 4096), id_pv, 1u);
                    tc::mma_f16(tO, tc::sdesc_add(a, 96), tc::sdesc_add(bv, 6144), id_pv, 1u);
                    tc::mma_commit(&p_free[h]);
                    tc::mma_commit(&vh_empty[h]);
                }
            }
            if (ok) {
                if (!qk) tc::mma_commit(o_done);
            } else {  // wait for every MMA this thread issued before TMEM is freed
                uint64_t* dr = qk ? drain : drain_pv;
                tc::mma_commit(dr);
                drain_wait(dr, 0);
            }
        }
    } else if (warp >= 11 && warp < 15) {
        // ------------------------------------------------------------ K converters: thread = key of the quarter
        const int key = threadIdx.x - 352;
        const uint16_t* ksg = p.ks[layer] + seq_row;
        auto scale_of = [&](int jj) -> float {  // this thread's key of tile jj; keys past the range: 0
            const int k = k_begin + jj * kWK + key;
            return (jj < ntiles && k < k_end) ? f16_bits_to_f32(ksg[k]) : 0.f;
        };
        float sc_cur = scale_of(0), sc_nxt = 0.f;
        __half2 s2 = __floats2half2_rn(sc_cur, sc_cur);
        for (int g = 0; g < 4 * ntiles; ++g) {
            const int rs = g % kW8KR, q = g & 3;
            if (q == 0) {  // a new tile: this key's scale, and the next tile's fetched ahead
                s2 = __floats2half2_rn(sc_cur, sc_cur);
                sc_nxt = scale_of((g >> 2) + 1);
            }
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&kr_full[rs], (g / kW8KR) & 1, abort_flag))) break;
            if (g >= 4 &&
                !__all_sync(0xFFFFFFFFu, tc::mbar_wait(&kq_empty[q], ((g >> 2) - 1) & 1, abort_flag)))
                break;
            // raw row: 64 bytes, 16-byte chunk c at ((c ^ ((key >> 1) & 3)) << 4) (64-byte swizzle)
            const uint8_t* raw = sKr + rs * 8192 + key * 64;
            uint4 in[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) in[c] = *reinterpret_cast<const uint4*>(raw + ((c ^ ((key >> 1) & 3)) << 4));
            uint8_t* row = sKh + q * 16384 + key * 128;  // fp16 row: chunk c at ((c ^ (key & 7)) << 4)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[8];
                i8x16_to_f16x16_scaled(in[c], s2, w);
                *reinterpret_cast<uint4*>(row + (((2 * c) ^ (key & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(row + (((2 * c + 1) ^ (key & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            tc::mbar_arrive_one(&kr_empty[rs]);
            tc::mbar_arrive_one(&kq_full[q]);
            if (q == 3) sc_cur = sc_nxt;
        }
    } else if (warp >= 15 && warp < 19) {
        // ------------------------------------------------------------ V converters: 64-key halves
        const int ct = threadIdx.x - 480;
        const uint16_t* vsg = p.vs[layer] + seq_row;
        auto scale_of = [&](int hh) -> float {  // key ct & 63 of half hh; keys past the range: 0
            const int k = k_begin + hh * kTcBK + (ct & 63);
            return (hh < nhalves && k < k_end) ? f16_bits_to_f32(vsg[k]) : 0.f;
        };
        float sc_cur = scale_of(0);
        for (int hh = 0; hh < nhalves; ++hh) {
            const int st = hh & 1;
            const __half2 s2 = __floats2half2_rn(sc_cur, sc_cur);
            const float sc_nxt = scale_of(hh + 1);
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&vr_full[st], (hh >> 1) & 1, abort_flag))) break;
            if (hh >= 2 &&
                !__all_sync(0xFFFFFFFFu, tc::mbar_wait(&vh_empty[st], ((hh >> 1) - 1) & 1, abort_flag)))
                break;
            const int nk = min(kTcBK, k_end - (k_begin + hh * kTcBK));  // keys >= nk (past the range) become 0
            convert_i8_tile_scaled(sVr + st * 16384, sVh + st * 32768, nk, ct, s2);
            tc::fence_proxy_async_smem();
            __syncwarp();
            tc::mbar_arrive_one(&vr_empty[st]);
            tc::mbar_arrive_one(&vh_full[st]);
            sc_cur = sc_nxt;
        }
    } else {
        // ------------------------------------------------------------ softmax halves (warps 0-3 and 7-10)
        const int h = warp < 4 ? 0 : 1;
        const int qd = warp & 3;
        const int r = qd * 32 + lane;  // row within the tile == TMEM lane
        const int gr = row0 + r;
        const bool row_ok = gr < p.R;
        const int node = row_ok ? gr / p.G : 0;
        const int head = kvh * p.G + (row_ok ? gr % p.G : 0);
        const uint64_t anc = row_ok ? p.anc[(size_t)b * T + node] : 0ull;
        const int lo_row = win > 0 ? S + node - win + 1 : INT_MIN;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        if (h == 0) {  // Q row x log2(e)/16 -> TMEM lane r as fp16 pairs, 64 features (32 columns) at a time
            const uint4* src = reinterpret_cast<const uint4*>(p.q[layer] + ((size_t)(b * T + node) * p.HQ + head) * kTcD);
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 v = row_ok ? src[c4 * 8 + i] : make_uint4(0, 0, 0, 0);
                    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __half2 hh2 = __floats2half2_rn(bf16_lo(in[e]) * kLog2eOverSqrtD,
                                                             bf16_hi(in[e]) * kLog2eOverSqrtD);
                        w[4 * i + e] = *reinterpret_cast<const uint32_t*>(&hh2);
                    }
                }
                tc::tmem_st32(tmem + lane_base + kColQ + c4 * 32, w);
            }
            tc::tmem_wait_st();
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(q_full);
        }
        auto exchange = [&](int jj, float mine, float& other) -> bool {
            const int slot = jj & 1;
            xv[(slot * 2 + h) * kTcRows + r] = mine;
            __syncwarp();
            tc::mbar_arrive_one(&xch[qd * 2 + slot]);
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&xch[qd * 2 + slot], (jj >> 1) & 1, abort_flag))) return false;
            other = xv[(slot * 2 + (h ^ 1)) * kTcRows + r];
            return true;
        };
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(s_full, j & 1, abort_flag))) { ok = false; break; }
            tc::tc_fence_after();
            float x[64];  // scores of this half, already in the log2 domain
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t sv[32];
                tc::tmem_ld32(tmem + lane_base + kColS + h * 64 + c2 * 32, sv);
                tc::tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c2 * 32 + c] = __uint_as_float(sv[c]);
            }
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(s_free);
            const int ct = k_begin + j * kWK;  // first key of the tile
            const int c0 = ct + h * 64;        // first key of this half
            if (!(ct + kWK <= k_end && ct + kWK <= S && ct >= lo_last)) {  // some key of the tile is masked
                const uint64_t vis = visible64(c0, k_end, lo_row, S, anc, row_ok);  // bit c: key c0 + c
#pragma unroll
                for (int c = 0; c < 64; ++c) x[c] = ((vis >> c) & 1ull) ? x[c] : -INFINITY;
            }
            float mx = x[0];
#pragma unroll
            for (int c = 1; c < 64; ++c) mx = fmaxf(mx, x[c]);
            float mo;
            if (!exchange(j, mx, mo)) { ok = false; break; }
            const float mt_ = fmaxf(mx, mo);
            float alpha = 1.f;
            bool resc = false;
            if (mt_ > m_ref + 8.f) {
                alpha = tc::ex2_approx(m_ref - mt_);
                m_ref = mt_;
                resc = true;
            }
            const float msub = m_ref == -INFINITY ? 0.f : m_ref;
            if (j >= 1) {  // P V of the previous tile done: the P halves are free again and O is stable
                if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&p_free[1], (j - 1) & 1, abort_flag))) { ok = false; break; }
                tc::tc_fence_after();
            }
            float ps = 0.f;
            uint8_t* prow = sP + h * 16384 + r * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {  // 8 keys per 16-byte chunk of this row's P half
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = ch * 8 + 2 * e;
                    const float p0 = tc::ex2_approx(x[c] - msub);
                    const float p1 = tc::ex2_approx(x[c + 1] - msub);
                    ps += p0 + p1;
                    pk[e] = pack2(p0, p1, false);
                }
                *reinterpret_cast<uint4*>(prow + ((ch ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            // O *= alpha, all 256 columns, by half 0 alone: the P V over the first 64 keys, which writes every
            // column of O, waits only for half 0's P (both halves take the same rescale decision)
            if (h == 0 && j >= 1 && __any_sync(0xFFFFFFFFu, resc)) {
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t o[32];
                    tc::tmem_ld32(tmem + lane_base + kColO + ch * 32, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tc::tmem_st32(tmem + lane_base + kColO + ch * 32, o);
                }
                tc::tmem_wait_st();
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            __syncwarp();
            tc::mbar_arrive_one(&p_full[h]);
            l = l * alpha + ps;
        }
        if (ok) {  // the row sum of both halves
            float lo;
            if (exchange(ntiles, l, lo)) l += lo;
            else ok = false;
        }
        if (ok && __all_sync(0xFFFFFFFFu, tc::mbar_wait(o_done, 0, abort_flag))) {
            tc::tc_fence_after();
            const size_t slot = ((size_t)unit * p.splits + split) * p.R + gr;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int ch = h * 4; ch < h * 4 + 4; ++ch) {
                uint32_t o[32];
                tc::tmem_ld32(tmem + lane_base + kColO + ch * 32, o);
                tc::tmem_wait_ld();
                if (!row_ok) continue;
                if (p.splits == 1) {
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o[layer]) +
                                                          ((size_t)(b * T + node) * p.HQ + head) * kTcD + ch * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack2(__uint_as_float(o[8 * k + 2 * e]) * inv, __uint_as_float(o[8 * k + 2 * e + 1]) * inv, true);
                        dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * kTcD + ch * 32);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                             __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
                }
            }
            if (h == 0 && row_ok && p.splits > 1) {  // the row's maximum and sum in the log2 domain, for the combine
                p.ws_ml[2 * slot] = m_ref;
                p.ws_ml[2 * slot + 1] = l;
            }
        }
    }
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) dev_fail(p.status, TSV_DEV_TIMEOUT, b, blockIdx.x);
    if (warp == 4) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// 2-D map over all (sequence, kv head, position) rows of one cache buffer:
// [B * HKV * s_cap rows, 256 columns].  16-bit caches: boxes of 64 columns x
// 64 rows with the 128-byte swizzle the MMA operands use.  Int8 caches:
// boxes of 128 bytes x 64 rows, 128-byte swizzled too (bank-conflict-free
// reads for the converter, which re-lays them out as fp16 operand tiles).
// quarters = true (Int8 K for the 128-key kernel): boxes of 64 bytes x 128 rows (one dim quarter of a 128-key
// tile) with the 64-byte swizzle.
static bool make_kv_map(CUtensorMap* m, const void* base, long long rows, bool i8, bool quarters = false) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kTcD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kTcD * (i8 ? 1 : 2)};
    cuuint32_t box[2] = {quarters ? 64u : (i8 ? 128u : 64u), quarters ? (cuuint32_t)kWK : (cuuint32_t)kTcBK};
    cuuint32_t es[2] = {1, 1};
    return enc(m, i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               quarters ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_supported(const tsv_attn_desc* d) {
    return d->D == kTcD && (d->kv_dtype == TSV_F16 || d->kv_dtype == TSV_BF16 || d->kv_dtype == TSV_I8_SCALED) &&
           (long long)d->B * d->HKV * d->s_cap < (1LL << 31) - kTcBK;
}

int tc_mtiles(const tsv_attn_desc* d) { return ((d->HQ / d->HKV) * d->T + kTcRows - 1) / kTcRows; }

// 128-key score tiles or 64-key ones.  TSV_ATTN_TCGEN05_64 / _128 choose; otherwise the 128-key kernel for
// 16-bit caches when a unit has more than one 128-row tile of query rows (there the halved Q K^T issue cost wins;
// with a single, mostly empty row tile the deeper 64-key pipeline is faster).  Int8 caches take the 64-key
// kernel: on the 16- and 64-node workloads the 128-key Int8 kernel measured level with it or up to 2 % slower.
bool tc_wide(const tsv_attn_desc* d) {
    if (d->path == TSV_ATTN_TCGEN05_64) return false;
    if (d->path == TSV_ATTN_TCGEN05_128) return true;
    return d->kv_dtype != TSV_I8_SCALED && tc_mtiles(d) >= 2;
}

tsv_status launch_tc(const tsv_attn_desc* d, int splits, int chunk, float* ws_o, float* ws_ml, int32_t* status,
                     cudaStream_t stream) {
    static thread_local TcParams prm;
    const bool i8 = d->kv_dtype == TSV_I8_SCALED;
    const bool wide = tc_wide(d);
    const long long rows = (long long)d->B * d->HKV * d->s_cap;
    for (int l = 0; l < d->n_layers; ++l) {
        if (!make_kv_map(&prm.kmap[l], d->k[l], rows, i8, i8 && wide) || !make_kv_map(&prm.vmap[l], d->v[l], rows, i8))
            return fail(TSV_ECUDA, "tree_verify_attention: tensor map encoding failed for layer %d", l);
        prm.q[l] = reinterpret_cast<const uint16_t*>(d->q[l]);
        prm.o[l] = d->o[l];
        prm.ks[l] = reinterpret_cast<const uint16_t*>(d->k_scale[l]);
        prm.vs[l] = reinterpret_cast<const uint16_t*>(d->v_scale[l]);
    }
    for (int l = 0; l < d->n_layers; ++l) prm.window[l] = d->window[l];
    prm.kv_len = d->kv_len;
    prm.anc = d->anc;
    prm.ws_o = ws_o;
    prm.ws_ml = ws_ml;
    prm.status = status;
    prm.s_cap = d->s_cap;
    prm.B = d->B;
    prm.T = d->T;
    prm.HQ = d->HQ;
    prm.HKV = d->HKV;
    prm.G = d->HQ / d->HKV;
    prm.R = prm.G * d->T;
    prm.mtiles = tc_mtiles(d);
    prm.splits = splits;
    prm.chunk = chunk;
    prm.max_kv_len = d->max_kv_len;
    prm.mma_bf16 = d->kv_dtype == TSV_BF16;
    const long long items = (long long)d->n_layers * d->B * d->HKV * splits * prm.mtiles;
    if (items > 0x7FFFFFFFLL) return fail(TSV_ECAPACITY, "tree_verify_attention: too many work items");
    if (i8 && wide) {
        cudaFuncSetAttribute(attn_tcw8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kW8Smem);
        launch_pdl(attn_tcw8_kernel, (unsigned)items, kW8Threads, kW8Smem, stream, prm);
    } else if (i8) {
        cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        launch_pdl(attn_tc_kernel<true>, (unsigned)items, kTcThreadsI8, kTcSmem, stream, prm);
    } else if (wide) {
        cudaFuncSetAttribute(attn_tcw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
        launch_pdl(attn_tcw_kernel, (unsigned)items, kTcThreads16, kWSmem, stream, prm);
    } else {
        cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        launch_pdl(attn_tc_kernel<false>, (unsigned)items, kTc64Threads16, kTcSmem, stream, prm);
    }
    return check_launch("tree_verify_attention(tcgen05)");
}

}  // namespace tsv
