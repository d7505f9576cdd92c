// tsv_tree_select: the verified draft tree chosen from a candidate tree by
// the drafter's confidence, on the device.
//
// mlxcel issue #1204, "What this needs", the fourth decision: EAGLE-2 branches
// by the drafter's confidence; PR #1212, the draft_tree commit: the runner-up
// at an uncertain step is the alternative worth a verify position.  Reading:
// the tree is the root plus the T - 1 candidates with the highest cumulative
// log-probability (fp32, summed from the root down), within a depth cap, ties
// to the earlier candidate; listed in that order, which is topological.
//
// One CTA per sequence (up to 1024 candidates, one thread each): depths by
// pointer chasing, scores level by level, a bitonic sort of the packed keys
// (orderable score << 32 | ~index) in shared memory, then the relabelling.
#include "common.cuh"

namespace tsv {

constexpr int kSelThreads = TSV_MAX_CANDIDATES;

__global__ void __launch_bounds__(kSelThreads) tree_select_kernel(const int32_t* __restrict__ cparents,
                                                                  const int32_t* __restrict__ ctokens,
                                                                  const float* __restrict__ clogp, int N, int T,
                                                                  int depth_max, int32_t* __restrict__ parents,
                                                                  int32_t* __restrict__ tokens,
                                                                  int32_t* __restrict__ cand_index,
                                                                  int32_t* __restrict__ sizes, int32_t* status) {
    griddep_begin();
    __shared__ int par[kSelThreads], dep[kSelThreads], where[kSelThreads];
    __shared__ float score[kSelThreads];
    __shared__ unsigned long long key[kSelThreads];
    __shared__ int bad, maxdep;
    const int b = blockIdx.x, i = threadIdx.x;
    if (i == 0) {
        bad = 0;
        maxdep = 0;
    }
    __syncthreads();
    if (i < N) {
        const int p = cparents[(size_t)b * N + i];
        par[i] = p;
        if (i == 0 ? p != -1 : (p < 0 || p >= i)) {
            atomicExch(&bad, 1);
            dev_fail(status, i == 0 ? TSV_DEV_BAD_ROOT : TSV_DEV_BAD_PARENT, b, i);
        }
        where[i] = -1;
    }
    __syncthreads();
    if (bad) {
        if (i < T) {
            parents[(size_t)b * T + i] = -1;
            tokens[(size_t)b * T + i] = -1;
            cand_index[(size_t)b * T + i] = -1;
        }
        if (i == 0) sizes[b] = 0;
        return;
    }
    // depth (capped at depth_max + 1: deeper candidates are not eligible)
    int d = 0;
    if (i < N)
        for (int u = i; u > 0 && d <= depth_max; u = par[u]) ++d;
    if (i < N) {
        dep[i] = d;
        if (d <= depth_max) atomicMax(&maxdep, d);
        score[i] = 0.f;
    }
    __syncthreads();
    // scores level by level: score(i) = score(parent) + logp(i), in fp32 from the root down
    for (int lv = 1; lv <= maxdep; ++lv) {
        if (i < N && dep[i] == lv) score[i] = __fadd_rn(score[par[i]], clogp[(size_t)b * N + i]);
        __syncthreads();
    }
    key[i] = (i > 0 && i < N && dep[i] <= depth_max) ? pack_best(score[i], (uint32_t)i) : 0ull;
    __syncthreads();
    // bitonic sort of the keys, largest first
    for (int k = 2; k <= kSelThreads; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int ixj = i ^ j;
            if (ixj > i) {
                const unsigned long long x = key[i], y = key[ixj];
                if ((i & k) == 0 ? (x < y) : (x > y)) {
                    key[i] = y;
                    key[ixj] = x;
                }
            }
            __syncthreads();
        }
    // chosen: the root, then the first sorted keys; relabel parents through `where`
    const int chosen = i == 0 ? 0 : (i < T && key[i - 1] != 0ull ? (int)(0xFFFFFFFFu - (uint32_t)(key[i - 1] & 0xFFFFFFFFull)) : -1);
    if (chosen >= 0) where[chosen] = i;
    __syncthreads();
    if (chosen > 0 && where[par[chosen]] < 0) dev_fail(status, TSV_DEV_BAD_PARENT, b, chosen);  // a log-prob > 0
    if (i < T) {
        parents[(size_t)b * T + i] = chosen > 0 ? where[par[chosen]] : -1;
        tokens[(size_t)b * T + i] = chosen >= 0 ? ctokens[(size_t)b * N + chosen] : -1;
        cand_index[(size_t)b * T + i] = chosen;
    }
    if (i == 0) {
        int n = 1;
        while (n < T && key[n - 1] != 0ull) ++n;
        sizes[b] = n;
    }
}

}  // namespace tsv

extern "C" tsv_status tsv_tree_select(const int32_t* cand_parents, const int32_t* cand_tokens, const float* cand_logp,
                                      int32_t B, int32_t N, int32_t T, int32_t depth_max, int32_t* parents,
                                      int32_t* tokens, int32_t* cand_index, int32_t* sizes, int32_t* dev_status,
                                      cudaStream_t stream) {
    using namespace tsv;
    clear_error();
    if (B < 0 || N < 1 || T < 1) return fail(TSV_EINVAL, "tree_select: B=%d N=%d T=%d", B, N, T);
    if (N > TSV_MAX_CANDIDATES)
        return fail(TSV_ECAPACITY, "tree_select: N=%d candidates above the maximum of %d", N, TSV_MAX_CANDIDATES);
    if (T > TSV_MAX_T) return fail(TSV_ECAPACITY, "tree_select: T=%d exceeds the maximum of %d nodes", T, TSV_MAX_T);
    if (depth_max < 0) return fail(TSV_EINVAL, "tree_select: depth_max=%d < 0", depth_max);
    if (B == 0) return TSV_OK;
    if (!cand_parents || !cand_tokens || !cand_logp || !parents || !tokens || !cand_index || !sizes)
        return fail(TSV_EINVAL, "tree_select: null pointer argument");
    launch_pdl(tree_select_kernel, B, kSelThreads, 0, stream, cand_parents, cand_tokens, cand_logp, N, T, depth_max, parents,
                                                      tokens, cand_index, sizes, dev_status);
    return check_launch("tree_select");
}
