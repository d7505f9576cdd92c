// tsv_tree_append: the verify block appended to every layer's cache, each
// node at its own position.
//
// mlxcel issue #1185, the closing comment's follow-up list: the tree path
// verifies the tree at its own positions.  Node i of the block is verified at position
// S + depth(i), while its K/V rows keep the topological slot S + i.  Q and
// the new K rows are rotated (rotary embedding of the first rot_dim
// features); V is not.  Int8 caches (PR #1212, gather_positions commit: one
// scale per token) quantise every row symmetrically by its absolute maximum.
//
// One CTA per (sequence, node, layer): the node's angles (inverse
// frequencies from the host in fp64, fp64 angle and range reduction, fp32
// sine/cosine) go to shared memory; each warp takes
// whole rows (Q heads, then K and V heads), one vector load and one vector
// store per lane and row, with the rotation done in a shared-memory copy of
// the row (pairs span lanes) and Int8 scales from a warp maximum.  The traffic
// is a few rows per node; the kernel is latency-bound.
#include <cmath>

#include "common.cuh"

namespace tsv {

constexpr int kApThreads = 256;
constexpr int kApWarps = kApThreads / 32;
constexpr int kApBatch = 4;  // rows per warp whose loads are in flight together

// E consecutive bf16 values (E = 2, 4, 8) from global memory as fp32.
template <int E>
__device__ __forceinline__ void load_bf16(const uint16_t* src, float* out) {
    uint32_t w[E / 2];
    if constexpr (E == 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (E == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(src);
        w[0] = v.x; w[1] = v.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t*>(src);
    }
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
        out[2 * k] = bf16_lo(w[k]);
        out[2 * k + 1] = bf16_hi(w[k]);
    }
}

template <int E>
__device__ __forceinline__ void store_words(void* dst, const uint32_t* w) {
    if constexpr (E == 8) *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    else if constexpr (E == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    else *reinterpret_cast<uint32_t*>(dst) = w[0];
}

// One row: this lane's E values x (features lane*E ..) -> stored form: bf16 (Q), fp16 / bf16 or Int8 codes
// + fp16 scale (cache rows).
template <int E>
__device__ __forceinline__ void store_row(const float* x, int lane, int dtype, void* dst, size_t e0,
                                          uint16_t* scale_dst) {
    if (dtype == TSV_I8_SCALED) {
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < E; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const __half sh = __float2half_rn(__fdiv_rn(amax, 127.f));
        const float s = __half2float(sh);
        uint32_t w[E / 4 > 0 ? E / 4 : 1] = {0};
#pragma unroll
        for (int k = 0; k < E; ++k) {
            const float q = s != 0.f ? fminf(127.f, fmaxf(-127.f, rintf(__fdiv_rn(x[k], s)))) : 0.f;
            w[k / 4] |= ((uint32_t)(uint8_t)(int8_t)(int)q) << (8 * (k % 4));
        }
        int8_t* out = reinterpret_cast<int8_t*>(dst) + e0 + (size_t)lane * E;
        if constexpr (E == 8) *reinterpret_cast<uint2*>(out) = make_uint2(w[0], w[1]);
        else if constexpr (E == 4) *reinterpret_cast<uint32_t*>(out) = w[0];
        else *reinterpret_cast<uint16_t*>(out) = (uint16_t)w[0];
        if (lane == 0) *scale_dst = __half_as_ushort(sh);
    } else {
        uint32_t w[E / 2];
#pragma unroll
        for (int k = 0; k < E / 2; ++k) {
            if (dtype == TSV_F16) {
                const __half2 h = __floats2half2_rn(x[2 * k], x[2 * k + 1]);
                w[k] = *reinterpret_cast<const uint32_t*>(&h);
            } else {
                const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
                w[k] = *reinterpret_cast<const uint32_t*>(&h);
            }
        }
        store_words<E>(reinterpret_cast<uint16_t*>(dst) + e0 + (size_t)lane * E, w);
    }
}

// Rotate this lane's E values of one row to the node's position (pairs may span lanes, so the row passes
// through the warp's shared-memory row once).
template <int E>
__device__ __forceinline__ void rotate_row(float* x, int rot_dim, bool interleaved, const float* cs, const float* sn,
                                           float* srow, int lane) {
#pragma unroll
    for (int k = 0; k < E; ++k) srow[lane * E + k] = x[k];
    __syncwarp();
    const int h = rot_dim / 2;
    for (int j = lane; j < h; j += 32) {
        const int ea = interleaved ? 2 * j : j, eb = interleaved ? 2 * j + 1 : j + h;
        const float a = srow[ea], b = srow[eb];
        srow[ea] = __fsub_rn(__fmul_rn(a, cs[j]), __fmul_rn(b, sn[j]));
        srow[eb] = __fadd_rn(__fmul_rn(b, cs[j]), __fmul_rn(a, sn[j]));
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < E; ++k) x[k] = srow[lane * E + k];
    __syncwarp();
}

// First bf16 element of row r of (sequence b, node i, layer l): Q heads, then new K heads, then new V heads.
__device__ __forceinline__ const uint16_t* row_src(const tsv_append_desc& d, int b, int i, int l, int r, int D) {
    if (r < d.HQ) return reinterpret_cast<const uint16_t*>(d.q_in[l]) + ((size_t)(b * d.T + i) * d.HQ + r) * D;
    const bool isK = r < d.HQ + d.HKV;
    const int kvh = r - d.HQ - (isK ? 0 : d.HKV);
    return reinterpret_cast<const uint16_t*>(isK ? d.k_new[l] : d.v_new[l]) + ((size_t)(b * d.T + i) * d.HKV + kvh) * D;
}

// Kernel parameters: the caller's descriptor plus the inverse frequencies base^(-2j / rot_dim), computed once
// on the host in fp64 (on the device fp64 transcendentals cost more than the rest of the kernel).
struct ApParams {
    tsv_append_desc d;
    double inv_freq[128];
};

// grid (B * T, n_layers): one CTA per (sequence, node, layer); each warp takes whole rows.
template <int D>
__global__ void __launch_bounds__(kApThreads) tree_append_kernel(const __grid_constant__ ApParams ap,
                                                                 const int32_t* __restrict__ kv_len, int32_t* status) {
    griddep_begin();
    const tsv_append_desc& d = ap.d;
    constexpr int E = D / 32;  // features per lane
    __shared__ float cs[128], sn[128];
    __shared__ float rows[kApWarps][D];
    const int T = d.T;
    const int b = blockIdx.x / T, i = blockIdx.x % T, l = blockIdx.y;
    if (d.depth[(size_t)b * T] != 0) return;  // this sequence's mask call failed: skip it
    const int S = kv_len[b];
    if (S < 0 || (int64_t)S + T > d.s_cap) {
        if (i == 0 && l == 0 && threadIdx.x == 0) dev_fail(status, TSV_DEV_BAD_KV_LEN, b, S);
        return;
    }
    const double pos = (double)S + (double)d.depth[(size_t)b * T + i];
    for (int j = threadIdx.x; j < d.rot_dim / 2; j += blockDim.x) {
        const double ang = pos * ap.inv_freq[j];
        const double r = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);  // into [-pi, pi]
        float s, c;
        sincosf((float)r, &s, &c);
        cs[j] = c;
        sn[j] = s;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool il = d.interleaved != 0;
    float* srow = rows[warp];
    const int nrows = d.HQ + 2 * d.HKV;
    // Rows in batches of kApBatch per warp: every load of a batch is issued before the first row is processed.
    for (int r0 = warp; r0 < nrows; r0 += kApWarps * kApBatch) {
        float x[kApBatch][E];
#pragma unroll
        for (int u = 0; u < kApBatch; ++u) {
            const int r = r0 + u * kApWarps;
            if (r < nrows) load_bf16<E>(row_src(d, b, i, l, r, D) + (size_t)lane * E, x[u]);
        }
#pragma unroll
        for (int u = 0; u < kApBatch; ++u) {
            const int r = r0 + u * kApWarps;
            if (r >= nrows) break;
            const bool isQ = r < d.HQ, isK = !isQ && r < d.HQ + d.HKV;
            if (isQ || isK) rotate_row<E>(x[u], d.rot_dim, il, cs, sn, srow, lane);
            if (isQ) {
                store_row<E>(x[u], lane, TSV_BF16, d.q_out[l], ((size_t)(b * T + i) * d.HQ + r) * D, nullptr);
            } else {
                const int kvh = r - d.HQ - (isK ? 0 : d.HKV);
                const size_t slot = ((size_t)b * d.HKV + kvh) * (size_t)d.s_cap + (size_t)(S + i);
                uint16_t* sc = d.kv_dtype == TSV_I8_SCALED
                                   ? reinterpret_cast<uint16_t*>(isK ? d.k_scale[l] : d.v_scale[l]) + slot
                                   : nullptr;
                store_row<E>(x[u], lane, d.kv_dtype, isK ? d.k[l] : d.v[l], slot * D, sc);
            }
        }
    }
}

// kv_len[b] += T for every sequence the append kernel wrote.
__global__ void append_kv_len_kernel(const int32_t* __restrict__ depth, int B, int T, int64_t s_cap,
                                     int32_t* __restrict__ kv_len) {
    griddep_begin();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B || depth[(size_t)b * T] != 0) return;
    const int S = kv_len[b];
    if (S >= 0 && (int64_t)S + T <= s_cap) kv_len[b] = S + T;
}

static tsv_status check_append(const tsv_append_desc* d, const int32_t* kv_len) {
    if (!d) return fail(TSV_EINVAL, "tree_append: null descriptor");
    if (d->n_layers < 1 || d->n_layers > TSV_MAX_LAYERS)
        return fail(TSV_ECAPACITY, "tree_append: n_layers=%d outside [1, %d]", d->n_layers, TSV_MAX_LAYERS);
    if (d->T < 1 || d->T > TSV_MAX_T) return fail(TSV_ECAPACITY, "tree_append: T=%d outside [1, %d]", d->T, TSV_MAX_T);
    if (d->B < 0 || d->HKV < 1 || d->HQ < 1 || d->HQ % d->HKV)
        return fail(TSV_EINVAL, "tree_append: B=%d HQ=%d HKV=%d", d->B, d->HQ, d->HKV);
    if (d->D != 64 && d->D != 128 && d->D != 256)
        return fail(TSV_EUNSUPPORTED, "tree_append: head dim %d is not 64, 128 or 256", d->D);
    if (d->kv_dtype != TSV_F16 && d->kv_dtype != TSV_BF16 && d->kv_dtype != TSV_I8_SCALED)
        return fail(TSV_EUNSUPPORTED, "tree_append: cache format %d", d->kv_dtype);
    if (d->rot_dim < 2 || d->rot_dim > d->D || d->rot_dim % 2)
        return fail(TSV_EINVAL, "tree_append: rot_dim=%d must be even and in [2, D=%d]", d->rot_dim, d->D);
    if (!(d->rope_base > 0.0) || d->rope_base > 1e30)
        return fail(TSV_EINVAL, "tree_append: rope_base=%g must be positive and finite", d->rope_base);
    if (d->s_cap < d->T) return fail(TSV_EINVAL, "tree_append: s_cap=%lld < T", (long long)d->s_cap);
    if ((long long)d->B * d->T > 0x7FFFFFFFLL) return fail(TSV_ECAPACITY, "tree_append: grid too large");
    if (d->B == 0) return TSV_OK;  // an empty batch: no pointer is read
    if (!d->depth || !kv_len) return fail(TSV_EINVAL, "tree_append: depth and kv_len must be non-null");
    for (int l = 0; l < d->n_layers; ++l) {
        if (!d->q_in[l] || !d->q_out[l] || !d->k_new[l] || !d->v_new[l] || !d->k[l] || !d->v[l])
            return fail(TSV_EINVAL, "tree_append: layer %d has a null pointer", l);
        if (d->kv_dtype == TSV_I8_SCALED && (!d->k_scale[l] || !d->v_scale[l]))
            return fail(TSV_EINVAL, "tree_append: layer %d Int8 cache without scales", l);
        if (((uintptr_t)d->q_in[l] | (uintptr_t)d->q_out[l] | (uintptr_t)d->k_new[l] | (uintptr_t)d->v_new[l] |
             (uintptr_t)d->k[l] | (uintptr_t)d->v[l]) & 15)
            return fail(TSV_EINVAL, "tree_append: layer %d buffers not 16-byte aligned", l);
    }
    return TSV_OK;
}

}  // namespace tsv

extern "C" tsv_status tsv_tree_append(const tsv_append_desc* d, int32_t* kv_len, int32_t* dev_status,
                                      cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    tsv_status st = check_append(d, kv_len);
    if (st != TSV_OK) return st;
    if (d->B == 0) return TSV_OK;
    if (d->n_layers > 65535) return fail(TSV_ECAPACITY, "tree_append: too many layers");
    static thread_local ApParams ap;
    ap.d = *d;
    for (int j = 0; j < d->rot_dim / 2; ++j) ap.inv_freq[j] = pow(d->rope_base, -2.0 * j / d->rot_dim);
    const dim3 grid((unsigned)(d->B * d->T), (unsigned)d->n_layers);
    if (d->D == 64) launch_pdl(tree_append_kernel<64>, grid, kApThreads, 0, stream, ap, kv_len, dev_status);
    else if (d->D == 128) launch_pdl(tree_append_kernel<128>, grid, kApThreads, 0, stream, ap, kv_len, dev_status);
    else launch_pdl(tree_append_kernel<256>, grid, kApThreads, 0, stream, ap, kv_len, dev_status);
    st = check_launch("tree_append");
    if (st != TSV_OK) return st;
    launch_pdl(append_kv_len_kernel, (d->B + 127) / 128, 128, 0, stream, d->depth, d->B, d->T, d->s_cap, kv_len);
    return check_launch("tree_append(kv_len)");
}
