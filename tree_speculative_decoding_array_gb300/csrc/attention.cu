// tsv_tree_verify_attention: tree-masked GQA attention of the verify block.
//
// mlxcel issue #1204, "What this needs" item 1 and "Increment 3"; PR #1212's
// history-mask commit (every node attends the cached history in full; inside
// the block a node sees its ancestors and itself) and verify commit (blocked
// entries must never make a row all-masked); Splash issue #728, "Earlier
// shader evidence" (split-KV tree attention with fp32 partials and
// statistics; 16 nodes x 24 heads x D256 over histories up to 8192).
//
// Split-KV flash decode.  A CTA owns up to 16 query rows of one
// (layer, sequence, kv head) unit - rows are (node i, head g of the GQA group)
// so every row of the CTA shares one K/V stream - and one key range.  Keys
// stream through shared memory in tiles of 32, dequantised to fp32 on the way
// in (Int8 codes times their per-token fp16 scale).  The tree mask is the
// per-node 64-bit ancestor word in shared memory, consulted only for keys at
// or past the block start S; no dense mask exists anywhere.  Online softmax
// in the log2 domain keeps fp32 running max / sum per row.  With more than
// one split, partial (unnormalised O, max, sum) go to the workspace and a
// combine kernel merges them.
#include <math.h>

#include "common.cuh"

namespace tsv {

constexpr int kRB = 16;   // query rows per CTA
constexpr int kBK = 32;   // keys per tile
constexpr int kAttThreads = 256;

struct AttnGeom {
    int units, rgs, splits, chunk, rows_unit, path;
};

// Defined in attention_tc.cu.
bool tc_supported(const tsv_attn_desc* d);
int tc_mtiles(const tsv_attn_desc* d);
bool tc_wide(const tsv_attn_desc* d);
tsv_status launch_tc(const tsv_attn_desc* d, int splits, int chunk, float* ws_o, float* ws_ml, int32_t* status,
                     cudaStream_t stream);

static AttnGeom attn_geom(const tsv_attn_desc* d) {
    AttnGeom g;
    g.rows_unit = (d->HQ / d->HKV) * d->T;
    g.units = d->n_layers * d->B * d->HKV;
    g.rgs = (g.rows_unit + kRB - 1) / kRB;
    g.path = (d->path >= TSV_ATTN_TCGEN05 || (d->path == TSV_ATTN_AUTO && tc_supported(d))) ? TSV_ATTN_TCGEN05
                                                                                           : TSV_ATTN_SIMT;
    // key tiles: 128 for the tcgen05 128-key kernel, 64 for its 64-key kernels, kBK for the CUDA cores
    const int key_tile = g.path == TSV_ATTN_TCGEN05 ? (tc_wide(d) ? 128 : 64) : kBK;
    int s = d->splits;
    if (s <= 0) {
        const int cap_s = (d->max_kv_len + 255) / 256 < 64 ? (d->max_kv_len + 255) / 256 : 64;
        if (g.path == TSV_ATTN_TCGEN05) {
            // One CTA per SM.  Estimated time of s splits: waves(s) x (fixed CTA cost + tiles per split x tile
            // cost), with the fixed cost (TMEM, Q tile, pipeline fill, partial write) worth about 8 tiles.
            const long long base = (long long)g.units * tc_mtiles(d);
            const long long slots = sm_count();
            const long long tiles = (d->max_kv_len + 63) / 64;
            bool sliding = false;
            for (int l = 0; l < d->n_layers; ++l) sliding = sliding || d->window[l] > 0;
            double best = 1e300;
            s = 1;
            for (int c = 1; c <= (cap_s > 1 ? cap_s : 1); ++c) {
                double t;
                if (!sliding) {
                    const long long waves = (base * c + slots - 1) / slots;
                    t = (double)waves * (8.0 + (double)((tiles + c - 1) / c)) + (c > 1 ? 2.0 : 0.0);
                } else {
                    // Sliding-window layers only keep the key ranges that meet their band; their other CTAs
                    // return at once.  Estimate: total work over the SMs, but never below the longest CTA.
                    const long long chunk = ((d->max_kv_len + c - 1) / c + 63) / 64 * 64;
                    const long long per_layer = base / d->n_layers;  // (sequence, kv head, m-tile) items
                    double work = 0.0, longest = 0.0;
                    for (int l = 0; l < d->n_layers; ++l) {
                        const long long w = d->window[l];
                        const long long len = w > 0 ? (w + d->T - 1 < d->max_kv_len ? w + d->T - 1 : d->max_kv_len)
                                                    : d->max_kv_len;
                        const long long first = (d->max_kv_len - len) / chunk, last = (d->max_kv_len - 1) / chunk;
                        const long long active = last - first + 1;
                        const double tl = 8.0 + (double)(((len < chunk ? len : chunk) + 63) / 64 + (w > 0 ? 1 : 0));
                        work += (double)per_layer * ((double)active * tl + 0.5 * (double)(c - active));
                        longest = longest > tl ? longest : tl;
                    }
                    t = (work / (double)slots > longest ? work / (double)slots : longest) + (c > 1 ? 2.0 : 0.0);
                }
                if (t < best * 0.98) {
                    best = t;
                    s = c;
                }
            }
        } else {
            const long long base = (long long)g.units * g.rgs;
            const long long target = 4LL * sm_count();
            s = (int)((target + base - 1) / base);
            if (s > cap_s) s = cap_s;
        }
    }
    if (s < 1) s = 1;
    int chunk = (d->max_kv_len + s - 1) / s;
    chunk = ((chunk + key_tile - 1) / key_tile) * key_tile;
    if (chunk < key_tile) chunk = key_tile;
    g.splits = s;
    g.chunk = chunk;
    return g;
}

__device__ __forceinline__ bool kv_len_ok(int kvl, int T, int max_kv_len, int64_t s_cap) {
    return kvl >= T && kvl <= max_kv_len && (int64_t)kvl <= s_cap;
}

// Loads 8 consecutive stored K/V elements as fp32 (Int8: times the token's scale).
__device__ __forceinline__ void load8(const void* base, size_t elem, int dtype, float scale, float* out) {
    if (dtype == TSV_I8_SCALED) {
        const uint2 w = *reinterpret_cast<const uint2*>(reinterpret_cast<const int8_t*>(base) + elem);
        const int8_t* c = reinterpret_cast<const int8_t*>(&w);
#pragma unroll
        for (int k = 0; k < 8; ++k) out[k] = (float)c[k] * scale;
    } else {
        const uint4 w = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(base) + elem);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        if (dtype == TSV_BF16) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                out[2 * k] = bf16_lo(u[k]);
                out[2 * k + 1] = bf16_hi(u[k]);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = f16x2_to_f32x2(u[k]);
                out[2 * k] = f.x;
                out[2 * k + 1] = f.y;
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kAttThreads) attn_simt_kernel(const __grid_constant__ tsv_attn_desc d, int splits,
                                                                int chunk, float* __restrict__ ws_o,
                                                                float* __restrict__ ws_ml, int32_t* status) {
    griddep_begin();
    constexpr int KS = D + 4;                   // padded K row stride (floats)
    constexpr int RPT = kRB * D / 4 / kAttThreads;  // output rows per thread in PV
    static_assert(RPT >= 1, "tile too small");
    extern __shared__ float sm[];
    float* q_s = sm;                 // [kRB][D]
    float* k_s = q_s + kRB * D;      // [kBK][KS]
    float* v_s = k_s + kBK * KS;     // [kBK][D]
    float* p_s = v_s + kBK * D;      // [kRB][kBK]
    __shared__ uint64_t anc_s[kRB];
    __shared__ int lo_s[kRB];  // sliding-window layers: smallest key position each row keeps
    __shared__ float m_s[kRB], l_s[kRB], alpha_s[kRB];

    const int unit = blockIdx.z;
    const int kvh = unit % d.HKV;
    const int b = (unit / d.HKV) % d.B;
    const int layer = unit / (d.HKV * d.B);
    const int rg = blockIdx.y, s = blockIdx.x;
    const int G = d.HQ / d.HKV, T = d.T;
    const int rows_unit = G * T;
    const int row0 = rg * kRB;
    const int kvl = d.kv_len[b];
    if (!kv_len_ok(kvl, T, d.max_kv_len, d.s_cap)) {
        if (s == 0 && rg == 0 && kvh == 0 && layer == 0 && threadIdx.x == 0) dev_fail(status, TSV_DEV_BAD_KV_LEN, b, kvl);
        return;
    }
    const int S = kvl - T;
    const int win = d.window[layer];
    int k_begin = s * chunk;
    const int k_end = min(kvl, k_begin + chunk);
    // Sliding-window layer: node i keeps keys c >= S + i - win + 1; key tiles below the first row's bound are
    // skipped (whole tiles from the range start).
    const int lo_first = win > 0 ? S + row0 / G - win + 1 : INT_MIN;
    if (lo_first > k_begin) k_begin += ((lo_first - k_begin) / kBK) * kBK;
    const float qscale = 1.4426950408889634f * rsqrtf((float)D);  // log2(e) / sqrt(D)

    // Q rows (fp32, pre-scaled into the log2 domain) and their ancestor words
    const uint16_t* Q = reinterpret_cast<const uint16_t*>(d.q[layer]);
    for (int e = threadIdx.x; e < kRB * D; e += blockDim.x) {
        const int r = e / D, c = e % D, gr = row0 + r;
        float x = 0.f;
        if (gr < rows_unit) {
            const int i = gr / G, h = kvh * G + gr % G;
            x = bf16_bits_to_f32(Q[((size_t)(b * T + i) * d.HQ + h) * D + c]) * qscale;
        }
        q_s[e] = x;
    }
    if (threadIdx.x < kRB) {
        const int gr = row0 + threadIdx.x;
        anc_s[threadIdx.x] = gr < rows_unit ? d.anc[(size_t)b * T + gr / G] : 0ull;
        lo_s[threadIdx.x] = (win > 0 && gr < rows_unit) ? S + gr / G - win + 1 : INT_MIN;
        m_s[threadIdx.x] = -INFINITY;
        l_s[threadIdx.x] = 0.f;
    }

    const size_t seq0 = ((size_t)b * d.HKV + kvh) * (size_t)d.s_cap;  // first cache row of this unit
    const void* Kp = d.k[layer];
    const void* Vp = d.v[layer];
    const uint16_t* KSc = reinterpret_cast<const uint16_t*>(d.k_scale[layer]);
    const uint16_t* VSc = reinterpret_cast<const uint16_t*>(d.v_scale[layer]);

    const int dq = threadIdx.x % (D / 4);     // output column quad
    const int rq = threadIdx.x / (D / 4);     // output row group
    float acc[RPT][4];
#pragma unroll
    for (int r = 0; r < RPT; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;

    for (int kt = k_begin; kt < k_end; kt += kBK) {
        const int nk = min(kBK, k_end - kt);
        __syncthreads();
        for (int e = threadIdx.x; e < kBK * (D / 8); e += blockDim.x) {
            const int j = e / (D / 8), c8 = (e % (D / 8)) * 8;
            float kf[8], vf[8];
            if (j < nk) {
                const size_t row = seq0 + kt + j;
                const float ks = d.kv_dtype == TSV_I8_SCALED ? f16_bits_to_f32(KSc[row]) : 1.f;
                const float vs = d.kv_dtype == TSV_I8_SCALED ? f16_bits_to_f32(VSc[row]) : 1.f;
                load8(Kp, row * D + c8, d.kv_dtype, ks, kf);
                load8(Vp, row * D + c8, d.kv_dtype, vs, vf);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) kf[k] = vf[k] = 0.f;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                k_s[j * KS + c8 + k] = kf[k];
                v_s[j * D + c8 + k] = vf[k];
            }
        }
        __syncthreads();
        // scores: thread -> key j, rows r and r + 8
        {
            const int j = threadIdx.x % kBK;
            const int r0 = threadIdx.x / kBK;  // 0..7
            float s0 = 0.f, s1 = 0.f;
            const float4* kr = reinterpret_cast<const float4*>(k_s + j * KS);
            const float4* q0 = reinterpret_cast<const float4*>(q_s + r0 * D);
            const float4* q1 = reinterpret_cast<const float4*>(q_s + (r0 + 8) * D);
#pragma unroll 8
            for (int c = 0; c < D / 4; ++c) {
                const float4 kk = kr[c], a = q0[c], bb = q1[c];
                s0 = fmaf(kk.x, a.x, fmaf(kk.y, a.y, fmaf(kk.z, a.z, fmaf(kk.w, a.w, s0))));
                s1 = fmaf(kk.x, bb.x, fmaf(kk.y, bb.y, fmaf(kk.z, bb.z, fmaf(kk.w, bb.w, s1))));
            }
            const int c = kt + j;
            bool v0 = j < nk && c >= lo_s[r0], v1 = j < nk && c >= lo_s[r0 + 8];
            if (c >= S) {
                const int node = c - S;
                v0 = v0 && ((anc_s[r0] >> node) & 1ull);
                v1 = v1 && ((anc_s[r0 + 8] >> node) & 1ull);
            }
            p_s[r0 * kBK + j] = v0 ? s0 : -INFINITY;
            p_s[(r0 + 8) * kBK + j] = v1 ? s1 : -INFINITY;
        }
        __syncthreads();
        // online softmax: warp w -> rows 2w, 2w + 1; lane -> key
        {
            const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = 2 * w + rr;
                const float x = p_s[r * kBK + lane];
                float mt = x;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, o));
                const float m_old = m_s[r];
                const float m_new = fmaxf(m_old, mt);
                float p = 0.f, alpha = 1.f;
                if (m_new != -INFINITY) {
                    p = exp2f(x - m_new);
                    alpha = exp2f(m_old - m_new);
                }
                float ps = p;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, o);
                p_s[r * kBK + lane] = p;
                __syncwarp();
                if (lane == 0) {
                    l_s[r] = l_s[r] * alpha + ps;
                    m_s[r] = m_new;
                    alpha_s[r] = alpha;
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr) {
            const int r = rq * RPT + rr;
            const float a = alpha_s[r];
            float4 o = make_float4(acc[rr][0] * a, acc[rr][1] * a, acc[rr][2] * a, acc[rr][3] * a);
            for (int j = 0; j < nk; ++j) {
                const float p = p_s[r * kBK + j];
                const float4 vv = reinterpret_cast<const float4*>(v_s + j * D)[dq];
                o.x = fmaf(p, vv.x, o.x);
                o.y = fmaf(p, vv.y, o.y);
                o.z = fmaf(p, vv.z, o.z);
                o.w = fmaf(p, vv.w, o.w);
            }
            acc[rr][0] = o.x;
            acc[rr][1] = o.y;
            acc[rr][2] = o.z;
            acc[rr][3] = o.w;
        }
    }
    __syncthreads();

#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
        const int r = rq * RPT + rr, gr = row0 + r;
        if (gr >= rows_unit) continue;
        if (splits == 1) {
            const int i = gr / G, h = kvh * G + gr % G;
            const float inv = l_s[r] > 0.f ? 1.f / l_s[r] : 0.f;
            __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(d.o[layer]) + ((size_t)(b * T + i) * d.HQ + h) * D;
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[rr][0] * inv, acc[rr][1] * inv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[rr][2] * inv, acc[rr][3] * inv);
            reinterpret_cast<__nv_bfloat162*>(O + 4 * dq)[0] = lo;
            reinterpret_cast<__nv_bfloat162*>(O + 4 * dq)[1] = hi;
        } else {
            const size_t slot = ((size_t)unit * splits + s) * rows_unit + gr;
            reinterpret_cast<float4*>(ws_o + slot * D)[dq] = make_float4(acc[rr][0], acc[rr][1], acc[rr][2], acc[rr][3]);
            if (dq == 0) {
                ws_ml[2 * slot] = m_s[r];
                ws_ml[2 * slot + 1] = l_s[r];
            }
        }
    }
}

// Merge split partials: O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.  One warp per query row: the lanes
// take the splits' weights (each computed once per row, kept in shared memory), then 4 columns each per pass
// with 16-byte loads of the partials.
constexpr int kCombRows = 4;  // rows (warps) per block
constexpr int kCombMaxSplits = 64;
__global__ void __launch_bounds__(kCombRows * 32) attn_combine_kernel(const __grid_constant__ tsv_attn_desc d, int splits,
                                                                      const float* __restrict__ ws_o,
                                                                      const float* __restrict__ ws_ml) {
    griddep_begin();
    __shared__ float sw[kCombRows][kCombMaxSplits];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows_unit = (d.HQ / d.HKV) * d.T;
    const int unit = blockIdx.y;
    const int gr = blockIdx.x * kCombRows + warp;
    const int kvh = unit % d.HKV;
    const int b = (unit / d.HKV) % d.B;
    const int layer = unit / (d.HKV * d.B);
    if (gr >= rows_unit || !kv_len_ok(d.kv_len[b], d.T, d.max_kv_len, d.s_cap)) return;  // whole warps
    const int G = d.HQ / d.HKV, D = d.D;
    const size_t slot0 = (size_t)unit * splits * rows_unit + gr;  // split s: slot0 + s * rows_unit
    float M = -INFINITY;
    for (int s = lane; s < splits; s += 32) M = fmaxf(M, ws_ml[2 * (slot0 + (size_t)s * rows_unit)]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    float L = 0.f;
    for (int s = lane; s < splits; s += 32) {
        const size_t sl = slot0 + (size_t)s * rows_unit;
        const float m = ws_ml[2 * sl];
        const float w = m != -INFINITY ? exp2f(m - M) : 0.f;
        sw[warp][s] = w;
        L += w * ws_ml[2 * sl + 1];
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
    __syncwarp();
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int i = gr / G, h = kvh * G + gr % G;
    __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(d.o[layer]) + ((size_t)(b * d.T + i) * d.HQ + h) * D;
    for (int c = lane * 4; c < D; c += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < splits; ++s) {
            const float w = sw[warp][s];
            if (w != 0.f) {
                const float4 v = *reinterpret_cast<const float4*>(ws_o + (slot0 + (size_t)s * rows_unit) * D + c);
                acc.x += w * v.x;
                acc.y += w * v.y;
                acc.z += w * v.z;
                acc.w += w * v.w;
            }
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(O + c) = pk;
    }
}

template <int D>
static size_t simt_smem() {
    return (size_t)(kRB * D + kBK * (D + 4) + kBK * D + kRB * kBK) * sizeof(float);
}

template <int D>
static void launch_simt(const tsv_attn_desc* d, const AttnGeom& g, float* ws_o, float* ws_ml, int32_t* status,
                        cudaStream_t stream) {
    const size_t sm = simt_smem<D>();
    cudaFuncSetAttribute(attn_simt_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    dim3 grid(g.splits, g.rgs, g.units);
    launch_pdl(attn_simt_kernel<D>, grid, kAttThreads, sm, stream, *d, g.splits, g.chunk, ws_o, ws_ml, status);
}

static size_t ws_bytes_for(const tsv_attn_desc* d, const AttnGeom& g) {
    if (g.splits <= 1) return 0;
    const size_t slots = (size_t)g.units * g.splits * g.rows_unit;
    const size_t o = (slots * d->D * sizeof(float) + 255) & ~(size_t)255;
    const size_t ml = (slots * 2 * sizeof(float) + 255) & ~(size_t)255;
    return o + ml;
}

static tsv_status check_desc(const tsv_attn_desc* d) {
    if (!d) return fail(TSV_EINVAL, "tree_verify_attention: null descriptor");
    if (d->n_layers < 1 || d->n_layers > TSV_MAX_LAYERS)
        return fail(TSV_ECAPACITY, "tree_verify_attention: n_layers=%d outside [1, %d]", d->n_layers, TSV_MAX_LAYERS);
    if (d->T < 1 || d->T > TSV_MAX_T)
        return fail(TSV_ECAPACITY, "tree_verify_attention: T=%d outside [1, %d]", d->T, TSV_MAX_T);
    if (d->B < 0 || d->HKV < 1 || d->HQ < 1 || d->HQ % d->HKV)
        return fail(TSV_EINVAL, "tree_verify_attention: B=%d HQ=%d HKV=%d", d->B, d->HQ, d->HKV);
    if (d->D != 64 && d->D != 128 && d->D != 256)
        return fail(TSV_EUNSUPPORTED, "tree_verify_attention: head dim %d is not 64, 128 or 256", d->D);
    if (d->kv_dtype != TSV_F16 && d->kv_dtype != TSV_BF16 && d->kv_dtype != TSV_I8_SCALED)
        return fail(TSV_EUNSUPPORTED, "tree_verify_attention: cache format %d", d->kv_dtype);
    if (d->max_kv_len < d->T || (int64_t)d->max_kv_len > d->s_cap)
        return fail(TSV_EINVAL, "tree_verify_attention: max_kv_len=%d must be in [T, s_cap=%lld]", d->max_kv_len,
                    (long long)d->s_cap);
    if (d->splits < 0) return fail(TSV_EINVAL, "tree_verify_attention: splits=%d < 0", d->splits);
    if (d->splits > kCombMaxSplits)
        return fail(TSV_ECAPACITY, "tree_verify_attention: splits=%d > %d", d->splits, kCombMaxSplits);
    for (int l = 0; l < d->n_layers; ++l)
        if (d->window[l] < 0) return fail(TSV_EINVAL, "tree_verify_attention: layer %d window=%d < 0", l, d->window[l]);
    if (d->path < TSV_ATTN_AUTO || d->path > TSV_ATTN_TCGEN05_128)
        return fail(TSV_EINVAL, "tree_verify_attention: path=%d", d->path);
    if (d->path >= TSV_ATTN_TCGEN05 && !tc_supported(d))
        return fail(TSV_EUNSUPPORTED, "tree_verify_attention: the tcgen05 kernel needs D == 256 and an fp16 or bf16 "
                                      "cache of fewer than 2^31 rows");
    if (d->B == 0) return TSV_OK;  // an empty batch: no pointer is read
    if (!d->kv_len || !d->anc) return fail(TSV_EINVAL, "tree_verify_attention: kv_len and anc must be non-null");
    const int G = d->HQ / d->HKV;
    if ((long long)d->n_layers * d->B * d->HKV > 65535 || ((long long)G * d->T + kRB - 1) / kRB > 65535)
        return fail(TSV_ECAPACITY, "tree_verify_attention: grid too large");
    for (int l = 0; l < d->n_layers; ++l) {
        if (!d->q[l] || !d->k[l] || !d->v[l] || !d->o[l])
            return fail(TSV_EINVAL, "tree_verify_attention: layer %d has a null Q/K/V/O", l);
        if (((uintptr_t)d->q[l] | (uintptr_t)d->k[l] | (uintptr_t)d->v[l] | (uintptr_t)d->o[l]) & 15)
            return fail(TSV_EINVAL, "tree_verify_attention: layer %d Q/K/V/O not 16-byte aligned", l);
        if (d->kv_dtype == TSV_I8_SCALED && (!d->k_scale[l] || !d->v_scale[l]))
            return fail(TSV_EINVAL, "tree_verify_attention: layer %d Int8 cache without scales", l);
    }
    return TSV_OK;
}

}  // namespace tsv

extern "C" size_t tsv_attention_workspace_size(const tsv_attn_desc* d) {
    using namespace tsv;
    if (!d || d->HKV < 1 || d->HQ % d->HKV) return 0;
    return ws_bytes_for(d, attn_geom(d));
}

extern "C" tsv_status tsv_tree_verify_attention(const tsv_attn_desc* d, void* workspace, size_t ws_bytes,
                                                int32_t* dev_status, cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    tsv_status st = check_desc(d);
    if (st != TSV_OK) return st;
    if (d->B == 0) return TSV_OK;
    const AttnGeom g = attn_geom(d);
    const size_t need = ws_bytes_for(d, g);
    if (need > 0 && (!workspace || ws_bytes < need))
        return fail(TSV_ECAPACITY, "tree_verify_attention: workspace %zu < %zu bytes", ws_bytes, need);
    float* ws_o = (float*)workspace;
    float* ws_ml = need ? (float*)((char*)workspace + ((((size_t)g.units * g.splits * g.rows_unit) * d->D * 4 + 255) & ~(size_t)255)) : nullptr;
    if (g.path == TSV_ATTN_TCGEN05) {
        st = launch_tc(d, g.splits, g.chunk, ws_o, ws_ml, dev_status, stream);
        if (st != TSV_OK || g.splits == 1) return st;
        dim3 cg((g.rows_unit + kCombRows - 1) / kCombRows, g.units);
        launch_pdl(attn_combine_kernel, cg, kCombRows * 32, 0, stream, *d, g.splits, ws_o, ws_ml);
        return check_launch("tree_verify_attention(combine)");
    }
    switch (d->D) {
        case 64: launch_simt<64>(d, g, ws_o, ws_ml, dev_status, stream); break;
        case 128: launch_simt<128>(d, g, ws_o, ws_ml, dev_status, stream); break;
        default: launch_simt<256>(d, g, ws_o, ws_ml, dev_status, stream); break;
    }
    st = check_launch("tree_verify_attention");
    if (st != TSV_OK || g.splits == 1) return st;
    dim3 cg((g.rows_unit + kCombRows - 1) / kCombRows, g.units);
    launch_pdl(attn_combine_kernel, cg, kCombRows * 32, 0, stream, *d, g.splits, ws_o, ws_ml);
    return check_launch("tree_verify_attention(combine)");
}
