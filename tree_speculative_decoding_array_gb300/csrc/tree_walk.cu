// tsv_tree_accept_walk: descend the draft tree along the target's argmaxes.
//
// mlxcel issue #1204, "What this needs" item 2: a tree walk descends the
// branch the target agreed with; "Increment 1": the accepted set is a path,
// never a subtree (the target emits one argmax per position, so one matching
// child is followed; with two matching siblings the lower index is taken).
// Splash issue #728, "What it does": every committed token is the target's
// selection at its path node, so emitted[j] = argmax[path[j]].
//
// One warp per sequence: lane l holds nodes l and l + 32.  Each step is one
// ballot over "my parent is u and my token is argmax[u]"; the lowest set bit
// is the next node.  The walk never leaves the device.
#include "common.cuh"

namespace tsv {

__global__ void __launch_bounds__(128) tree_walk_kernel(const int32_t* __restrict__ argmax,
                                                        const int32_t* __restrict__ tokens,
                                                        const int32_t* __restrict__ parents, int B, int T,
                                                        int32_t* __restrict__ path, int32_t* __restrict__ path_len,
                                                        int32_t* __restrict__ emitted, int32_t* status) {
    griddep_begin();
    const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const size_t base = (size_t)b * T;
    const int n0 = lane, n1 = lane + 32;
    const int p0 = n0 < T ? parents[base + n0] : -2;
    const int p1 = n1 < T ? parents[base + n1] : -2;
    const int t0 = n0 < T ? tokens[base + n0] : 0;
    const int t1 = n1 < T ? tokens[base + n1] : 0;
    const bool ok0 = n0 >= T || (n0 == 0 ? p0 == -1 : (p0 >= 0 && p0 < n0));
    const bool ok1 = n1 >= T || (p1 >= 0 && p1 < n1);
    const unsigned bad0 = __ballot_sync(0xFFFFFFFFu, !ok0), bad1 = __ballot_sync(0xFFFFFFFFu, !ok1);

    int len = 1;
    int u = 0;
    if (bad0 | bad1) {
        if (lane == 0) {
            const int where = bad0 ? __ffs(bad0) - 1 : 32 + __ffs(bad1) - 1;
            dev_fail(status, where == 0 ? TSV_DEV_BAD_ROOT : TSV_DEV_BAD_PARENT, b, where);
            path[base] = 0;
        }
    } else {
        if (lane == 0) path[base] = 0;
        for (;;) {
            const int target = argmax[base + u];
            const unsigned m0 = __ballot_sync(0xFFFFFFFFu, p0 == u && t0 == target);
            const unsigned m1 = __ballot_sync(0xFFFFFFFFu, p1 == u && t1 == target);
            int c;
            if (m0) c = __ffs(m0) - 1;
            else if (m1) c = 32 + __ffs(m1) - 1;
            else break;
            if (lane == 0) path[base + len] = c;
            ++len;
            u = c;  // children have larger indices, so at most T - 1 steps
        }
    }
    __syncwarp();
    // pad path, write emitted = argmax along the path
    for (int j = lane; j < T; j += 32) {
        if (j >= len) {
            path[base + j] = -1;
            emitted[base + j] = -1;
        }
    }
    __syncwarp();
    for (int j = lane; j < len; j += 32) emitted[base + j] = argmax[base + path[base + j]];
    if (lane == 0) path_len[b] = len;
}

}  // namespace tsv

extern "C" tsv_status tsv_tree_accept_walk(const int32_t* argmax, const int32_t* tokens, const int32_t* parents,
                                           int32_t B, int32_t T, int32_t* path, int32_t* path_len,
                                           int32_t* emitted, int32_t* dev_status, cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (B < 0) return fail(TSV_EINVAL, "tree_accept_walk: B=%d < 0", B);
    if (T < 1 || T > TSV_MAX_T) return fail(TSV_ECAPACITY, "tree_accept_walk: T=%d outside [1, %d]", T, TSV_MAX_T);
    if (B == 0) return TSV_OK;
    if (!argmax || !tokens || !parents || !path || !path_len || !emitted)
        return fail(TSV_EINVAL, "tree_accept_walk: null pointer argument");
    const int warps_per_block = 4;
    const int grid = (B + warps_per_block - 1) / warps_per_block;
    launch_pdl(tree_walk_kernel, grid, 32 * warps_per_block, 0, stream, argmax, tokens, parents, B, T, path, path_len,
                                                                  emitted, dev_status);
    return check_launch("tree_accept_walk");
}
