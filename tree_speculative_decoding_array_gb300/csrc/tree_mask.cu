// tsv_tree_mask: topology check, per-node ancestor bitmask and depth.
//
// mlxcel issue #1204, "What this needs" item 1: a node attends to its
// ancestors only, and the mask is rebuilt every round from the topology.
// "Increment 1": nodes are in topological order, parents[i] < i.  The mask is
// kept as one 64-bit word per node (bit j = node j is an ancestor or the node
// itself) instead of a dense T x T tensor; the attention kernels test bits.
// PR #1212's history-mask commit gives the dense [T, offset + T] additive form
// (history columns attended in full) and its verify commit the -1e9 blocking
// value; the dense form is written only on request, for parity checks.
#include "common.cuh"

namespace tsv {

// One CTA of 64 threads per sequence; thread i owns node i.
__global__ void __launch_bounds__(64) tree_mask_kernel(const int32_t* __restrict__ parents, int B, int T,
                                                       uint64_t* __restrict__ anc, int32_t* __restrict__ depth,
                                                       int32_t* status) {
    griddep_begin();
    __shared__ int par[TSV_MAX_T];
    __shared__ int bad;
    const int b = blockIdx.x;
    const int i = threadIdx.x;
    if (i == 0) bad = 0;
    __syncthreads();
    if (i < T) {
        const int p = parents[(size_t)b * T + i];
        par[i] = p;
        const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
        if (!ok) {
            atomicExch(&bad, 1);
            dev_fail(status, i == 0 ? TSV_DEV_BAD_ROOT : TSV_DEV_BAD_PARENT, b, i);
        }
    }
    __syncthreads();
    if (i >= T) return;
    uint64_t a = 0;
    int d = -1;
    if (!bad) {
        // parents strictly decrease along the chase, so it ends within i steps
        a = 1ull << i;
        d = 0;
        for (int u = par[i]; u >= 0; u = par[u]) {
            a |= 1ull << u;
            ++d;
        }
    }
    anc[(size_t)b * T + i] = a;
    depth[(size_t)b * T + i] = d;
}

// Dense additive mask [B, T, offset + T]: 0 for history columns and for
// ancestor-or-self block columns, -1e9 elsewhere.
__global__ void dense_mask_kernel(const uint64_t* __restrict__ anc, int B, int T, int offset,
                                  float* __restrict__ mask) {
    griddep_begin();
    const int W = offset + T;
    const size_t n = (size_t)B * T * W;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(e % W);
        const size_t row = e / W;  // b * T + q
        float v = 0.0f;
        if (c >= offset) v = ((anc[row] >> (c - offset)) & 1ull) ? 0.0f : -1e9f;
        mask[e] = v;
    }
}

}  // namespace tsv

extern "C" tsv_status tsv_tree_mask(const int32_t* parents, int32_t B, int32_t T, uint64_t* anc, int32_t* depth,
                                    float* dense_mask, int32_t mask_offset, int32_t* dev_status,
                                    cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (B < 0 || T < 0) return fail(TSV_EINVAL, "tree_mask: B=%d T=%d must be >= 0", B, T);
    if (T > TSV_MAX_T) return fail(TSV_ECAPACITY, "tree_mask: T=%d exceeds the maximum of %d nodes", T, TSV_MAX_T);
    if (B == 0 || T == 0) return TSV_OK;
    if (!parents || !anc || !depth) return fail(TSV_EINVAL, "tree_mask: parents, anc and depth must be non-null");
    if (dense_mask && mask_offset < 0) return fail(TSV_EINVAL, "tree_mask: mask_offset=%d < 0", mask_offset);
    launch_pdl(tree_mask_kernel, B, 64, 0, stream, parents, B, T, anc, depth, dev_status);
    tsv_status st = check_launch("tree_mask");
    if (st != TSV_OK || !dense_mask) return st;
    const size_t n = (size_t)B * T * (size_t)(mask_offset + T);
    const int grid = (int)((n + 255) / 256 < (size_t)sm_count() * 8 ? (n + 255) / 256 : (size_t)sm_count() * 8);
    launch_pdl(dense_mask_kernel, grid, 256, 0, stream, anc, B, T, mask_offset, dense_mask);
    return check_launch("tree_mask(dense)");
}

// ---------------------------------------------------------------------------
// tsv_sliding_band_mask: the dense mask of a sliding-window layer (PR #1212,
// the commit on caller masks and the sliding-window band): the caller's
// additive mask intersected, by element-wise minimum, with the band of query
// row q at position offset + q, which keeps columns offset + q - window < c
// <= offset + q.  Applied only where the two can disagree (offset + T >
// window), so shorter contexts keep exactly the caller's mask.
// ---------------------------------------------------------------------------
namespace tsv {

__global__ void sliding_band_kernel(float* __restrict__ mask, int B, int T, int offset, int window) {
    griddep_begin();
    const int W = offset + T;
    const size_t n = (size_t)B * T * W;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(e % W);
        const int q = (int)((e / W) % T);
        const int pos = offset + q;
        if (c > pos || c <= pos - window) mask[e] = fminf(mask[e], -1e9f);
    }
}

}  // namespace tsv

extern "C" tsv_status tsv_sliding_band_mask(float* dense_mask, int32_t B, int32_t T, int32_t mask_offset,
                                            int32_t window, cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (B < 0 || T < 0 || mask_offset < 0)
        return fail(TSV_EINVAL, "sliding_band_mask: B=%d T=%d mask_offset=%d must be >= 0", B, T, mask_offset);
    if (T > TSV_MAX_T) return fail(TSV_ECAPACITY, "sliding_band_mask: T=%d exceeds the maximum of %d nodes", T, TSV_MAX_T);
    if (window < 1) return fail(TSV_EINVAL, "sliding_band_mask: window=%d must be >= 1", window);
    if (B == 0 || T == 0 || (int64_t)mask_offset + T <= window) return TSV_OK;  // below the window: untouched
    if (!dense_mask) return fail(TSV_EINVAL, "sliding_band_mask: dense_mask is null");
    const size_t n = (size_t)B * T * (size_t)(mask_offset + T);
    const int grid = (int)((n + 255) / 256 < (size_t)sm_count() * 8 ? (n + 255) / 256 : (size_t)sm_count() * 8);
    launch_pdl(sliding_band_kernel, grid, 256, 0, stream, dense_mask, B, T, mask_offset, window);
    return check_launch("sliding_band_mask");
}
