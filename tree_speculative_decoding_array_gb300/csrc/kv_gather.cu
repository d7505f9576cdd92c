// tsv_kv_gather_positions: compact the verify block of every KV cache to the
// accepted path, in place.
//
// mlxcel issue #1204, "The rollback constraint, which decides feasibility": a
// chain rolls back by trimming the tail, which is only correct for a prefix;
// a tree's accepted path is scattered, so survivors must be selected and
// closed up.  PR #1212's gather_positions commit: Int8 scale sidecars move
// with their tokens, a prefix selection equals trim_to and the identity
// selection short-circuits (a full-accept round pays no rewrite).  Its
// gather_within_tail commit: rewrite only [tail_start, tail_start + kept_len)
// so the cost scales with the block, not with the context, and the
// allocation survives.
//
// One CTA per (layer, sequence, kv head, K-or-V).  path is strictly
// increasing, so path[j] >= j: a sequential ascending copy would be safe, but
// a parallel one is not (row S + j may be a source of a later row).  The CTA
// therefore stages every moved row in shared memory (at most 64 rows of
// D * element bytes) before writing any of them.  Rows before the first j
// with path[j] != j are already in place and are not touched; when there is
// no such j nothing moves.  A second, tiny kernel then advances kv_len.
#include "common.cuh"

namespace tsv {

struct GatherCheck {
    int ok, len, S, first;
};

// Validates sequence b's path and length; identical in both kernels.
__device__ __forceinline__ GatherCheck gather_check(const int32_t* __restrict__ kv_len,
                                                    const int32_t* __restrict__ path,
                                                    const int32_t* __restrict__ path_len, int b, int T,
                                                    int64_t s_cap, int* sp) {
    GatherCheck g;
    g.len = path_len[b];
    const int kvl = kv_len[b];
    g.S = kvl - T;
    g.ok = 1;
    if (kvl < T || (int64_t)kvl > s_cap) g.ok = -TSV_DEV_BAD_KV_LEN;
    else if (g.len < 1 || g.len > T) g.ok = -TSV_DEV_BAD_PATH;
    g.first = g.len;
    if (g.ok == 1) {
        int prev = -1;
        for (int j = 0; j < g.len; ++j) {
            const int p = path[(size_t)b * T + j];
            if ((j == 0 && p != 0) || p <= prev || p >= T) {
                g.ok = -TSV_DEV_BAD_PATH;
                break;
            }
            if (p != j && g.first == g.len) g.first = j;
            if (sp) sp[j] = p;
            prev = p;
        }
    }
    return g;
}

constexpr int kGatherThreads = 256;
constexpr int kMaxRowBytes = 512;  // D = 256 at 2 bytes

__global__ void __launch_bounds__(kGatherThreads) kv_gather_kernel(const __grid_constant__ tsv_kv_desc kv,
                                                                   const int32_t* __restrict__ kv_len,
                                                                   const int32_t* __restrict__ path,
                                                                   const int32_t* __restrict__ path_len, int T,
                                                                   int32_t* status) {
    griddep_begin();
    __shared__ uint4 buf[TSV_MAX_T * kMaxRowBytes / 16];
    __shared__ uint16_t sbuf[TSV_MAX_T];
    __shared__ int sp[TSV_MAX_T];
    __shared__ GatherCheck g;
    const int unit = blockIdx.x;
    const int h = unit % kv.HKV;
    const int b = (unit / kv.HKV) % kv.B;
    const int layer = unit / (kv.HKV * kv.B);
    const int which = blockIdx.y;  // 0 = K, 1 = V
    if (threadIdx.x == 0) {
        g = gather_check(kv_len, path, path_len, b, T, kv.s_cap, sp);
        if (g.ok < 0 && layer == 0 && h == 0 && which == 0) dev_fail(status, -g.ok, b, 0);
    }
    __syncthreads();
    if (g.ok < 0 || g.first == g.len) return;  // invalid, or identity selection: nothing moves

    const int elt = kv.kv_dtype == TSV_I8_SCALED ? 1 : 2;
    const int vpr = kv.D * elt / 16;  // 16-byte vectors per row
    const size_t seq_row0 = ((size_t)b * kv.HKV + h) * (size_t)kv.s_cap;
    uint4* base = reinterpret_cast<uint4*>(which ? kv.v[layer] : kv.k[layer]) + seq_row0 * vpr;
    const int first = g.first, n = g.len - g.first, S = g.S;
    for (int e = threadIdx.x; e < n * vpr; e += blockDim.x) {
        const int r = e / vpr, c = e % vpr;
        buf[e] = base[(size_t)(S + sp[first + r]) * vpr + c];
    }
    uint16_t* sc = nullptr;
    if (kv.kv_dtype == TSV_I8_SCALED) {
        sc = reinterpret_cast<uint16_t*>(which ? kv.v_scale[layer] : kv.k_scale[layer]) + seq_row0;
        for (int r = threadIdx.x; r < n; r += blockDim.x) sbuf[r] = sc[S + sp[first + r]];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * vpr; e += blockDim.x) {
        const int r = e / vpr, c = e % vpr;
        base[(size_t)(S + first + r) * vpr + c] = buf[e];
    }
    if (sc)
        for (int r = threadIdx.x; r < n; r += blockDim.x) sc[S + first + r] = sbuf[r];
}

__global__ void kv_len_update_kernel(int32_t* __restrict__ kv_len, const int32_t* __restrict__ path,
                                     const int32_t* __restrict__ path_len, int B, int T, int64_t s_cap) {
    griddep_begin();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const GatherCheck g = gather_check(kv_len, path, path_len, b, T, s_cap, nullptr);
    if (g.ok == 1) kv_len[b] = g.S + g.len;
}

}  // namespace tsv

extern "C" tsv_status tsv_kv_gather_positions(const tsv_kv_desc* kv, int32_t* kv_len, const int32_t* path,
                                              const int32_t* path_len, int32_t T, int32_t* dev_status,
                                              cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (!kv) return fail(TSV_EINVAL, "kv_gather_positions: null descriptor");
    if (kv->B == 0 && T >= 1 && T <= TSV_MAX_T) return TSV_OK;  // an empty batch: nothing to read or write
    if (!kv_len || !path || !path_len) return fail(TSV_EINVAL, "kv_gather_positions: null pointer argument");
    if (T < 1 || T > TSV_MAX_T) return fail(TSV_ECAPACITY, "kv_gather_positions: T=%d outside [1, %d]", T, TSV_MAX_T);
    if (kv->n_layers < 1 || kv->n_layers > TSV_MAX_LAYERS)
        return fail(TSV_ECAPACITY, "kv_gather_positions: n_layers=%d outside [1, %d]", kv->n_layers, TSV_MAX_LAYERS);
    if (kv->B < 0 || kv->HKV < 1) return fail(TSV_EINVAL, "kv_gather_positions: B=%d HKV=%d", kv->B, kv->HKV);
    if (kv->D != 64 && kv->D != 128 && kv->D != 256)
        return fail(TSV_EUNSUPPORTED, "kv_gather_positions: head dim %d is not 64, 128 or 256", kv->D);
    if (kv->kv_dtype != TSV_F16 && kv->kv_dtype != TSV_BF16 && kv->kv_dtype != TSV_I8_SCALED)
        return fail(TSV_EUNSUPPORTED, "kv_gather_positions: cache format %d has no gather (only fp16, bf16 and "
                                      "Int8 with per-token scales keep all per-token state on the sequence axis)",
                    kv->kv_dtype);
    if (kv->s_cap < T) return fail(TSV_EINVAL, "kv_gather_positions: s_cap=%lld < T", (long long)kv->s_cap);
    if (kv->B == 0) return TSV_OK;
    for (int l = 0; l < kv->n_layers; ++l) {
        if (!kv->k[l] || !kv->v[l]) return fail(TSV_EINVAL, "kv_gather_positions: layer %d has a null K or V", l);
        if (((uintptr_t)kv->k[l] | (uintptr_t)kv->v[l]) & 15)
            return fail(TSV_EINVAL, "kv_gather_positions: layer %d K/V not 16-byte aligned", l);
        if (kv->kv_dtype == TSV_I8_SCALED && (!kv->k_scale[l] || !kv->v_scale[l]))
            return fail(TSV_EINVAL, "kv_gather_positions: layer %d Int8 cache without scale sidecars", l);
    }
    const long long units = (long long)kv->n_layers * kv->B * kv->HKV;
    if (units > 0x7FFFFFFFLL) return fail(TSV_ECAPACITY, "kv_gather_positions: too many (layer, seq, head) units");
    dim3 grid((unsigned)units, 2);
    launch_pdl(kv_gather_kernel, grid, kGatherThreads, 0, stream, *kv, kv_len, path, path_len, T, dev_status);
    tsv_status st = check_launch("kv_gather_positions");
    if (st != TSV_OK) return st;
    launch_pdl(kv_len_update_kernel, (kv->B + 127) / 128, 128, 0, stream, kv_len, path, path_len, kv->B, T, kv->s_cap);
    return check_launch("kv_gather_positions(kv_len)");
}

// ---------------------------------------------------------------------------------------------------------------
// tsv_gather_positions: the absolute form.  PR #1212's gather_positions commit: the new sequence is the old
// positions kept[0] < kept[1] < ... in order; a prefix selection equals trim_to; the identity selection moves
// nothing; Int8 scale sidecars move with their tokens.  The kept list may be as long as the cache.
//
// In place with kept strictly increasing: kept[j] >= j, so a row is only ever read by a destination at or
// below it.  One CTA per (layer, sequence, kv head, K-or-V) walks the destinations upwards in chunks of
// kChunkBytes: it loads a chunk's source rows into shared memory, synchronises, then stores them.  The loads of
// chunk c + 1 read rows >= its first destination, above every row chunk c writes, so they need no ordering
// against chunk c's stores; a row that chunk c + 1 overwrites was read either by an earlier chunk (before an
// earlier barrier) or by chunk c + 1 itself (before its own barrier).  Two shared buffers alternate, so one
// barrier per chunk suffices.  Destinations below the first j with kept[j] != j are already in place.
namespace tsv {

constexpr int kAbsThreads = 512;
constexpr int kChunkBytes = 16384;

struct KeptCheck {
    int ok, n, first;
};

// The whole block validates sequence b's kept list; every thread returns the same result.
__device__ KeptCheck kept_check(const int32_t* __restrict__ kv_len, const int32_t* __restrict__ kept,
                                const int32_t* __restrict__ kept_len, int b, int max_kept, int64_t s_cap) {
    __shared__ int s_first, s_bad;
    const int kvl = kv_len[b];
    const int n = kept_len[b];
    KeptCheck k;
    k.n = n;
    k.ok = 1;
    if (kvl < 0 || (int64_t)kvl > s_cap) k.ok = -TSV_DEV_BAD_KV_LEN;
    else if (n < 0 || n > max_kept || n > kvl) k.ok = -TSV_DEV_BAD_PATH;
    if (threadIdx.x == 0) {
        s_first = n;
        s_bad = 0;
    }
    __syncthreads();
    if (k.ok == 1) {
        const int32_t* row = kept + (size_t)b * max_kept;
        int first = n, bad = 0;
        for (int j = threadIdx.x; j < n; j += blockDim.x) {
            const int p = row[j];
            if (p < 0 || p >= kvl || (j > 0 && row[j - 1] >= p)) bad = 1;
            if (p != j && j < first) first = j;
        }
        if (bad) atomicOr(&s_bad, 1);
        if (first < n) atomicMin(&s_first, first);
    }
    __syncthreads();
    if (k.ok == 1 && s_bad) k.ok = -TSV_DEV_BAD_PATH;
    k.first = s_first;
    __syncthreads();  // s_first / s_bad may be reused by a later call in the same thread block
    return k;
}

__global__ void __launch_bounds__(kAbsThreads) gather_abs_kernel(const __grid_constant__ tsv_kv_desc kv,
                                                                 const int32_t* __restrict__ kv_len,
                                                                 const int32_t* __restrict__ kept,
                                                                 const int32_t* __restrict__ kept_len, int max_kept,
                                                                 int32_t* status) {
    griddep_begin();
    __shared__ uint4 buf[2][kChunkBytes / 16];
    __shared__ uint16_t sbuf[2][kChunkBytes / 64];  // one scale per row; rows per chunk <= kChunkBytes / 64
    const int unit = blockIdx.x;
    const int h = unit % kv.HKV;
    const int b = (unit / kv.HKV) % kv.B;
    const int layer = unit / (kv.HKV * kv.B);
    const int which = blockIdx.y;  // 0 = K, 1 = V
    const KeptCheck g = kept_check(kv_len, kept, kept_len, b, max_kept, kv.s_cap);
    if (g.ok < 0) {
        if (threadIdx.x == 0 && layer == 0 && h == 0 && which == 0) dev_fail(status, -g.ok, b, 0);
        return;
    }
    if (g.first >= g.n) return;  // identity (or prefix) selection: a trim, nothing moves

    const int elt = kv.kv_dtype == TSV_I8_SCALED ? 1 : 2;
    const int vpr = kv.D * elt / 16;          // 16-byte vectors per row (4 .. 32)
    const int rows = kChunkBytes / (vpr * 16);  // rows per chunk (32 .. 256)
    const size_t seq_row0 = ((size_t)b * kv.HKV + h) * (size_t)kv.s_cap;
    uint4* base = reinterpret_cast<uint4*>(which ? kv.v[layer] : kv.k[layer]) + seq_row0 * vpr;
    uint16_t* sc = kv.kv_dtype == TSV_I8_SCALED
                       ? reinterpret_cast<uint16_t*>(which ? kv.v_scale[layer] : kv.k_scale[layer]) + seq_row0
                       : nullptr;
    const int32_t* row = kept + (size_t)b * max_kept;
    int s = 0;
    for (int j0 = g.first; j0 < g.n; j0 += rows, s ^= 1) {
        const int cnt = min(rows, g.n - j0);
        for (int e = threadIdx.x; e < cnt * vpr; e += blockDim.x) {
            const int r = e / vpr, c = e - r * vpr;
            buf[s][e] = base[(size_t)__ldg(row + j0 + r) * vpr + c];
        }
        if (sc)
            for (int r = threadIdx.x; r < cnt; r += blockDim.x) sbuf[s][r] = sc[__ldg(row + j0 + r)];
        __syncthreads();
        for (int e = threadIdx.x; e < cnt * vpr; e += blockDim.x) {
            const int r = e / vpr, c = e - r * vpr;
            base[(size_t)(j0 + r) * vpr + c] = buf[s][e];
        }
        if (sc)
            for (int r = threadIdx.x; r < cnt; r += blockDim.x) sc[j0 + r] = sbuf[s][r];
    }
}

__global__ void __launch_bounds__(256) gather_abs_len_kernel(int32_t* __restrict__ kv_len,
                                                             const int32_t* __restrict__ kept,
                                                             const int32_t* __restrict__ kept_len, int max_kept,
                                                             int64_t s_cap) {
    griddep_begin();
    const KeptCheck g = kept_check(kv_len, kept, kept_len, blockIdx.x, max_kept, s_cap);
    if (threadIdx.x == 0 && g.ok == 1) kv_len[blockIdx.x] = g.n;
}

}  // namespace tsv

extern "C" tsv_status tsv_gather_positions(const tsv_kv_desc* kv, int32_t* kv_len, const int32_t* kept,
                                           const int32_t* kept_len, int32_t max_kept, int32_t* dev_status,
                                           cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (!kv) return fail(TSV_EINVAL, "gather_positions: null descriptor");
    if (max_kept < 0) return fail(TSV_EINVAL, "gather_positions: max_kept=%d < 0", max_kept);
    if (kv->B < 0 || kv->HKV < 1) return fail(TSV_EINVAL, "gather_positions: B=%d HKV=%d", kv->B, kv->HKV);
    if (kv->B == 0) return TSV_OK;  // an empty batch: nothing to read or write
    if (!kv_len || !kept_len || (!kept && max_kept > 0))
        return fail(TSV_EINVAL, "gather_positions: null pointer argument");
    if (kv->n_layers < 1 || kv->n_layers > TSV_MAX_LAYERS)
        return fail(TSV_ECAPACITY, "gather_positions: n_layers=%d outside [1, %d]", kv->n_layers, TSV_MAX_LAYERS);
    if (kv->D != 64 && kv->D != 128 && kv->D != 256)
        return fail(TSV_EUNSUPPORTED, "gather_positions: head dim %d is not 64, 128 or 256", kv->D);
    if (kv->kv_dtype != TSV_F16 && kv->kv_dtype != TSV_BF16 && kv->kv_dtype != TSV_I8_SCALED)
        return fail(TSV_EUNSUPPORTED, "gather_positions: cache format %d has no gather (only fp16, bf16 and Int8 "
                                      "with per-token scales keep all per-token state on the sequence axis)",
                    kv->kv_dtype);
    if (kv->s_cap < 1 || kv->s_cap > 0x7FFFFFFFLL)
        return fail(TSV_EINVAL, "gather_positions: s_cap=%lld outside [1, 2^31)", (long long)kv->s_cap);
    for (int l = 0; l < kv->n_layers; ++l) {
        if (!kv->k[l] || !kv->v[l]) return fail(TSV_EINVAL, "gather_positions: layer %d has a null K or V", l);
        if (((uintptr_t)kv->k[l] | (uintptr_t)kv->v[l]) & 15)
            return fail(TSV_EINVAL, "gather_positions: layer %d K/V not 16-byte aligned", l);
        if (kv->kv_dtype == TSV_I8_SCALED && (!kv->k_scale[l] || !kv->v_scale[l]))
            return fail(TSV_EINVAL, "gather_positions: layer %d Int8 cache without scale sidecars", l);
    }
    const long long units = (long long)kv->n_layers * kv->B * kv->HKV;
    if (units > 0x7FFFFFFFLL) return fail(TSV_ECAPACITY, "gather_positions: too many (layer, seq, head) units");
    if (max_kept > 0) {
        launch_pdl(gather_abs_kernel, dim3((unsigned)units, 2), kAbsThreads, 0, stream, *kv, kv_len, kept, kept_len,
                   max_kept, dev_status);
        tsv_status st = check_launch("gather_positions");
        if (st != TSV_OK) return st;
    }
    launch_pdl(gather_abs_len_kernel, kv->B, 256, 0, stream, kv_len, kept, kept_len, max_kept, kv->s_cap);
    return check_launch("gather_positions(kv_len)");
}
