// tsv_sample_nucleus: every tree node's draw from the nucleus-filtered target
// distribution, for sampled (temperature > 0) verification.
//
// Splash issue #728, "What it does": for sampled requests each node draws from
// the nucleus-filtered distribution with its own uniform, so the committed
// tokens keep the chain verify's output distribution; the accept walk then
// follows the child whose draft token equals the draw.  Filter order (a
// reading; the page names temperature, top-p and top-k): logits / T, the top_k
// largest (ties to the lower index), softmax, the shortest descending prefix
// whose mass reaches top_p, renormalised, inverted at the node's uniform.
//
// Top-k selection is exact and two-level: CTAs take the top_k of 4096-entry
// chunks of a row's packed keys (orderable logit << 32 | ~index, so larger
// logit first and the lower index first among ties) by rounds of warp maxima
// over per-lane sorted keys; further passes reduce the survivors until one
// chunk remains.  One warp per row then draws: softmax weights with expf,
// warp prefix sums, the nucleus cut and the inverse-CDF pick by ballots.
#include "common.cuh"

namespace tsv {

constexpr int kSortN = 4096;
constexpr int kSortThreads = 512;
constexpr int kMaxTopK = 64;

// Largest 64-bit key of the warp (keys are unique: they carry their index).
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long k) {
    const uint32_t hi = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(k >> 32));
    const uint32_t lo = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(k >> 32) == hi ? (uint32_t)k : 0u);
    return ((unsigned long long)hi << 32) | lo;
}

// Compare-exchange keeping a >= b.
__device__ __forceinline__ void cx(unsigned long long& a, unsigned long long& b) {
    const unsigned long long x = a > b ? a : b, y = a > b ? b : a;
    a = x;
    b = y;
}

// grid (chunks, rows): the top K keys (largest first) of every kSortN-entry chunk of a row.  FROM_LOGITS: the
// input is the row's fp32 logits [n]; else packed keys [n] from an earlier pass.  Each warp sorts its lanes'
// 8 keys, takes its own top K by K rounds of a warp maximum (the winning lane pops its head), and warp 0 merges
// the 16 warps' sorted lists the same way.
// With lse_part != NULL (the first pass over logits) each CTA also writes its chunk's (max, sum of exp(x - max))
// to lse_part[row][chunk], for log-probabilities.
template <bool FROM_LOGITS>
__global__ void __launch_bounds__(kSortThreads) topk_chunk_kernel(const void* __restrict__ in, int n, int K,
                                                                  unsigned long long* __restrict__ out,
                                                                  float2* __restrict__ lse_part) {
    griddep_begin();
    __shared__ unsigned long long wtop[kSortThreads / 32][kMaxTopK];
    __shared__ float2 wlse[kSortThreads / 32];
    const int row = blockIdx.y, ch = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t base = (size_t)row * n;
    unsigned long long a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = ch * kSortN + warp * 256 + j * 32 + lane;
        unsigned long long key = 0ull;  // below every real key
        if (e < n) {
            if (FROM_LOGITS) key = pack_best(reinterpret_cast<const float*>(in)[base + e], (uint32_t)e);
            else key = reinterpret_cast<const unsigned long long*>(in)[base + e];
        }
        a[j] = key;
    }
    if (FROM_LOGITS && lse_part) {  // this chunk's (max, sum exp(x - max)); padding keys (0) are not logits
        float m = -INFINITY, sum = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (a[j] != 0ull) m = fmaxf(m, unorderable((uint32_t)(a[j] >> 32)));
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (a[j] != 0ull && m != -INFINITY) sum += expf(unorderable((uint32_t)(a[j] >> 32)) - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o), s2 = __shfl_xor_sync(0xFFFFFFFFu, sum, o);
            const float mm = fmaxf(m, m2);
            sum = (m == -INFINITY ? 0.f : sum * expf(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * expf(m2 - mm));
            m = mm;
        }
        if (lane == 0) wlse[warp] = make_float2(m, sum);
        __syncthreads();
        if (threadIdx.x == 0) {
            float M = -INFINITY, S = 0.f;
            for (int w = 0; w < kSortThreads / 32; ++w) {
                const float mm = fmaxf(M, wlse[w].x);
                S = (M == -INFINITY ? 0.f : S * expf(M - mm)) + (wlse[w].x == -INFINITY ? 0.f : wlse[w].y * expf(wlse[w].x - mm));
                M = mm;
            }
            lse_part[(size_t)row * gridDim.x + ch] = make_float2(M, S);
        }
    }
    // sorting network for 8 keys, descending
    cx(a[0], a[1]); cx(a[2], a[3]); cx(a[4], a[5]); cx(a[6], a[7]);
    cx(a[0], a[2]); cx(a[1], a[3]); cx(a[4], a[6]); cx(a[5], a[7]);
    cx(a[1], a[2]); cx(a[5], a[6]); cx(a[0], a[4]); cx(a[3], a[7]);
    cx(a[1], a[5]); cx(a[2], a[6]);
    cx(a[1], a[4]); cx(a[3], a[6]);
    cx(a[2], a[4]); cx(a[3], a[5]);
    cx(a[3], a[4]);
    for (int t = 0; t < K; ++t) {
        const unsigned long long m = warp_max_u64(a[0]);
        if (a[0] == m) {  // the winning lane pops its head
#pragma unroll
            for (int j = 0; j < 7; ++j) a[j] = a[j + 1];
            a[7] = 0ull;
        }
        if (lane == 0) wtop[warp][t] = m;
    }
    __syncthreads();
    if (warp == 0) {
        // lanes 0..15 own warp lists 0..15; the others hold nothing
        int pos = 0;
        const bool own = lane < kSortThreads / 32;
        for (int t = 0; t < K; ++t) {
            const unsigned long long h = own && pos < K ? wtop[lane][pos] : 0ull;
            const unsigned long long m = warp_max_u64(h);
            if (own && h == m && m != 0ull) ++pos;
            if (lane == 0) out[((size_t)row * gridDim.x + ch) * K + t] = m;
        }
    }
}

// One warp per row: the node's draw from its top K keys (sorted, largest first).
__global__ void nucleus_draw_kernel(const unsigned long long* __restrict__ top, int rows, int K, float inv_temp,
                                    float top_p, const float* __restrict__ uniforms, int32_t* __restrict__ tokens) {
    griddep_begin();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const unsigned long long* t = top + (size_t)row * K;
    const bool ha = lane < K, hb = 32 + lane < K;
    const unsigned long long ka = ha ? t[lane] : 0ull, kb = hb ? t[32 + lane] : 0ull;
    const float lmax = unorderable((uint32_t)(t[0] >> 32));
    const float pa = ha ? expf((unorderable((uint32_t)(ka >> 32)) - lmax) * inv_temp) : 0.f;
    const float pb = hb ? expf((unorderable((uint32_t)(kb >> 32)) - lmax) * inv_temp) : 0.f;
    // inclusive prefix sums over j = 0 .. K-1 (first half in lanes, then the second half)
    float ca = pa, cb = pb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float xa = __shfl_up_sync(0xFFFFFFFFu, ca, o), xb = __shfl_up_sync(0xFFFFFFFFu, cb, o);
        if (lane >= o) {
            ca += xa;
            cb += xb;
        }
    }
    cb += __shfl_sync(0xFFFFFFFFu, ca, 31);
    const float Z = K > 32 ? __shfl_sync(0xFFFFFFFFu, cb, (K - 33)) : __shfl_sync(0xFFFFFFFFu, ca, K - 1);
    // nucleus: m = 1 + the first j with c_j >= top_p * Z
    const float thr = top_p * Z;
    const unsigned ba = __ballot_sync(0xFFFFFFFFu, ha && ca >= thr), bb = __ballot_sync(0xFFFFFFFFu, hb && cb >= thr);
    const int m = ba ? __ffs(ba) : (bb ? 32 + __ffs(bb) : K);
    const float cm = m <= 32 ? __shfl_sync(0xFFFFFFFFu, ca, m - 1) : __shfl_sync(0xFFFFFFFFu, cb, m - 33);
    // inverse CDF: the first j < m with c_j > u * c_{m-1}
    const float target = uniforms[row] * cm;
    const unsigned da = __ballot_sync(0xFFFFFFFFu, lane < m && ha && ca > target);
    const unsigned db = __ballot_sync(0xFFFFFFFFu, 32 + lane < m && hb && cb > target);
    const int j = da ? __ffs(da) - 1 : (db ? 32 + __ffs(db) - 1 : m - 1);
    if (lane == 0) tokens[row] = (int32_t)(0xFFFFFFFFu - (uint32_t)(t[j] & 0xFFFFFFFFull));
}

static int chunks_of(long long n) { return (int)((n + kSortN - 1) / kSortN); }

}  // namespace tsv

extern "C" size_t tsv_sample_workspace_size(int32_t rows, int32_t V, int32_t top_k) {
    using namespace tsv;
    if (rows < 1 || V < 1 || top_k < 1) return 0;
    const int K = top_k < V ? (top_k < kMaxTopK ? top_k : kMaxTopK) : V;
    const size_t one = ((size_t)rows * chunks_of(V) * K * sizeof(unsigned long long) + 255) & ~(size_t)255;
    return 2 * one;
}

extern "C" tsv_status tsv_sample_nucleus(const float* logits, int32_t rows, int32_t V, float temperature,
                                         int32_t top_k, float top_p, const float* uniforms, int32_t* tokens,
                                         void* workspace, size_t ws_bytes, cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (rows < 1 || rows > 65535 || V < 1)
        return fail(TSV_EINVAL, "sample_nucleus: rows=%d (1..65535) V=%d", rows, V);
    if (top_k < 1 || top_k > kMaxTopK)
        return fail(TSV_EUNSUPPORTED, "sample_nucleus: top_k=%d outside [1, %d]", top_k, kMaxTopK);
    if (!(temperature > 0.f) || !(top_p > 0.f && top_p <= 1.f))
        return fail(TSV_EINVAL, "sample_nucleus: temperature=%g must be > 0 and top_p=%g in (0, 1]", temperature,
                    top_p);
    if (!logits || !uniforms || !tokens || !workspace) return fail(TSV_EINVAL, "sample_nucleus: null pointer argument");
    const size_t need = tsv_sample_workspace_size(rows, V, top_k);
    if (ws_bytes < need) return fail(TSV_ECAPACITY, "sample_nucleus: workspace %zu < %zu bytes", ws_bytes, need);
    const int K = top_k < V ? top_k : V;
    unsigned long long* buf[2] = {(unsigned long long*)workspace, (unsigned long long*)((char*)workspace + need / 2)};
    int cur = 0;
    int nch = chunks_of(V);
    launch_pdl(topk_chunk_kernel<true>, dim3(nch, rows), kSortThreads, 0, stream, logits, V, K, buf[cur], nullptr);
    tsv_status st = check_launch("sample_nucleus(top-k)");
    if (st != TSV_OK) return st;
    long long n = (long long)nch * K;  // survivors per row
    while (nch > 1) {
        nch = chunks_of(n);
        launch_pdl(topk_chunk_kernel<false>, dim3(nch, rows), kSortThreads, 0, stream, buf[cur], (int)n, K, buf[cur ^ 1],
                                                                              nullptr);
        st = check_launch("sample_nucleus(top-k merge)");
        if (st != TSV_OK) return st;
        cur ^= 1;
        n = (long long)nch * K;
    }
    launch_pdl(nucleus_draw_kernel, (rows + 7) / 8, 256, 0, stream, buf[cur], rows, K, 1.f / temperature, top_p, uniforms,
                                                            tokens);
    return check_launch("sample_nucleus(draw)");
}

// ---------------------------------------------------------------------------
// tsv_draft_children: the drafter's candidate children of every expanded
// node - its top_k tokens and their log-probabilities log_softmax(logits) -
// the confidence signal the draft tree branches on (mlxcel issue #1204, "What
// this needs", the fourth decision: EAGLE-2 branches by drafter confidence).
// ---------------------------------------------------------------------------
namespace tsv {

// One warp per row: log(sum exp(x)) from the chunks' (max, sum) partials, then the row's K children.
__global__ void draft_children_kernel(const unsigned long long* __restrict__ top, const float2* __restrict__ lse_part,
                                      int nch, int rows, int K, int32_t* __restrict__ tokens, float* __restrict__ logp) {
    griddep_begin();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    float m = -INFINITY, sum = 0.f;
    for (int c = lane; c < nch; c += 32) {
        const float2 p = lse_part[(size_t)row * nch + c];
        const float mm = fmaxf(m, p.x);
        sum = (m == -INFINITY ? 0.f : sum * expf(m - mm)) + (p.x == -INFINITY ? 0.f : p.y * expf(p.x - mm));
        m = mm;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o), s2 = __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        const float mm = fmaxf(m, m2);
        sum = (m == -INFINITY ? 0.f : sum * expf(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * expf(m2 - mm));
        m = mm;
    }
    const float lse = m + logf(sum);
    for (int j = lane; j < K; j += 32) {
        const unsigned long long key = top[(size_t)row * K + j];
        tokens[(size_t)row * K + j] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
        logp[(size_t)row * K + j] = unorderable((uint32_t)(key >> 32)) - lse;
    }
}

}  // namespace tsv

extern "C" size_t tsv_draft_children_workspace_size(int32_t rows, int32_t V, int32_t top_k) {
    const size_t base = tsv_sample_workspace_size(rows, V, top_k);
    return base ? base + (((size_t)rows * tsv::chunks_of(V) * sizeof(float2) + 255) & ~(size_t)255) : 0;
}

extern "C" tsv_status tsv_draft_children(const float* draft_logits, int32_t rows, int32_t V, int32_t top_k,
                                         int32_t* child_tokens, float* child_logp, void* workspace, size_t ws_bytes,
                                         cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (rows < 1 || rows > 65535 || V < 1) return fail(TSV_EINVAL, "draft_children: rows=%d (1..65535) V=%d", rows, V);
    if (top_k < 1 || top_k > kMaxTopK || top_k > V)
        return fail(TSV_EUNSUPPORTED, "draft_children: top_k=%d outside [1, min(%d, V)]", top_k, kMaxTopK);
    if (!draft_logits || !child_tokens || !child_logp || !workspace)
        return fail(TSV_EINVAL, "draft_children: null pointer argument");
    const size_t need = tsv_draft_children_workspace_size(rows, V, top_k);
    if (ws_bytes < need) return fail(TSV_ECAPACITY, "draft_children: workspace %zu < %zu bytes", ws_bytes, need);
    const size_t half = tsv_sample_workspace_size(rows, V, top_k) / 2;
    unsigned long long* buf[2] = {(unsigned long long*)workspace, (unsigned long long*)((char*)workspace + half)};
    float2* lse_part = (float2*)((char*)workspace + 2 * half);
    const int K = top_k;
    const int nch0 = chunks_of(V);
    int cur = 0, nch = nch0;
    launch_pdl(topk_chunk_kernel<true>, dim3(nch, rows), kSortThreads, 0, stream, draft_logits, V, K, buf[cur], lse_part);
    tsv_status st = check_launch("draft_children(top-k)");
    if (st != TSV_OK) return st;
    long long n = (long long)nch * K;
    while (nch > 1) {
        nch = chunks_of(n);
        launch_pdl(topk_chunk_kernel<false>, dim3(nch, rows), kSortThreads, 0, stream, buf[cur], (int)n, K, buf[cur ^ 1],
                                                                              nullptr);
        st = check_launch("draft_children(top-k merge)");
        if (st != TSV_OK) return st;
        cur ^= 1;
        n = (long long)nch * K;
    }
    launch_pdl(draft_children_kernel, (rows + 7) / 8, 256, 0, stream, buf[cur], lse_part, nch0, rows, K, child_tokens,
                                                              child_logp);
    return check_launch("draft_children");
}
