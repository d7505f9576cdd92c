/*
 * tsv.h - C ABI of the tree speculative-decoding verify step on GB300 (sm_103a).
 *
 * One verify round of tree speculative decoding, as five calls on one CUDA
 * stream (mask -> attention for every layer -> LM head + argmax -> accept walk
 * -> KV compaction).  The operations follow these pages:
 *
 *   [1204] mlxcel issue #1204, "perf(speculative): draft a tree instead of a
 *          chain, so an MTP round emits more than 2.33 tokens"
 *   [1212] mlxcel PR #1212, "feat(speculative): draft and verify a token tree,
 *          behind a flag, default off" (its commit messages)
 *   [1185] mlxcel issue #1185, "perf(speculative): cut the MTP drafter's
 *          per-step cost, now the binding constraint on M5-class hardware"
 *   [728]  Splash issue #728, "Experiment: qualify shared-prefix tree
 *          verification and conservative admission"
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership: every array argument is caller-owned memory.  Unless a parameter
 *   says "host", it is DEVICE memory of the current CUDA device.  The library
 *   keeps no pointer after a call returns and allocates no device memory;
 *   scratch comes from a caller-provided workspace whose size the matching
 *   *_workspace_size() call returns.
 * Streams: every call only enqueues work on `stream` (0 = legacy default
 *   stream) and returns without synchronising.  Results are ready when the
 *   stream reaches them.  Calls are capturable in CUDA graphs.  Every kernel
 *   is launched with programmatic stream serialization: it waits for the
 *   kernel before it on the stream to complete before it touches memory, and
 *   lets the kernel after it be scheduled early.  A kernel of the caller's
 *   launched after a call with that attribute set must therefore wait
 *   (griddepcontrol.wait / cudaGridDependencySynchronize) before it reads the
 *   call's outputs; ordinary launches, copies and events need nothing.
 * Host errors: a call returns TSV_OK when its work was enqueued.  Any other
 *   status means nothing was enqueued; tsv_last_error() then names the reason
 *   (a per-thread string, valid until the next call on the same thread).
 *   TSV_EUNSUPPORTED is a refusal ([1212], gather_positions commit: a layout
 *   the operation cannot serve refuses with a message, and the caller must
 *   decline tree drafting rather than proceed).
 * Device errors: topology or path errors that only the device can see are
 *   written to `dev_status` (int32[4], device memory) and never trap: word 0
 *   receives the first TSV_DEV_* code (atomic compare-and-swap from 0, so it
 *   is sticky), words 1..2 the sequence and node/position where it was found.
 *   The caller zeroes the words once and reads them whenever it chooses;
 *   outputs of a sequence with an error are unspecified (but in bounds).
 *   dev_status may be NULL, in which case device errors are dropped.
 * Sizes: 1 <= T <= 64 (one 64-bit ancestor word per node; tsv_tree_mask also
 *   accepts T == 0).  Layout shapes are row-major, innermost last.
 */
#ifndef TSV_H
#define TSV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TSV_OK = 0,
    TSV_EINVAL = 1,       /* bad argument: null pointer, size out of range, misaligned buffer */
    TSV_ETOPOLOGY = 2,    /* a host-visible topology error */
    TSV_EUNSUPPORTED = 3, /* a format or shape this build refuses (the caller must decline) */
    TSV_ECAPACITY = 4,    /* workspace too small, or a size above a compiled maximum */
    TSV_ECUDA = 5         /* the CUDA runtime reported an error while enqueueing */
} tsv_status;

typedef enum {
    TSV_F16 = 0,       /* IEEE binary16 */
    TSV_BF16 = 1,      /* bfloat16 */
    TSV_I8_SCALED = 2, /* int8 code x fp16 per-token scale (KV caches only) */
    TSV_Q4_G64 = 3     /* 4-bit affine, groups of 64 input features (LM head only) */
} tsv_dtype;

/* Device status codes (dev_status word 0). */
#define TSV_DEV_OK 0
#define TSV_DEV_BAD_ROOT 1    /* parents[b][0] != -1 */
#define TSV_DEV_BAD_PARENT 2  /* parents[b][i] outside [0, i) for i >= 1 */
#define TSV_DEV_BAD_PATH 3    /* path not strictly increasing from 0, or path_len outside [1, T]; or a
                                 kept list / kept_len of tsv_gather_positions out of order or range */
#define TSV_DEV_BAD_KV_LEN 4  /* kv_len[b] < T (< 0 for tsv_gather_positions), or kv_len[b] > capacity */
#define TSV_DEV_TIMEOUT 5     /* a bounded wait inside a kernel expired (a library bug; outputs unspecified) */

#define TSV_MAX_T 64
#define TSV_MAX_CANDIDATES 1024 /* candidate-tree nodes per sequence for tsv_tree_select */
#define TSV_MAX_LAYERS 64

/* Reason for the last non-TSV_OK status returned on this thread ("" if none). */
const char* tsv_last_error(void);

/*
 * tsv_selftest_bounded_wait - checks the failure path every tensor-core
 * kernel relies on (no page counterpart: a property of this implementation).
 * One CTA waits on a barrier that nothing completes; the library's bounded
 * wait gives up after 1 s, raises the CTA's abort flag (which ends the other
 * warps' waits) and records TSV_DEV_TIMEOUT in dev_status (words 1..2: the
 * flag, the warp).  The device stays usable.  dev_status: int32[4], device
 * memory, zeroed by the caller.
 */
tsv_status tsv_selftest_bounded_wait(int32_t* dev_status, cudaStream_t stream);

/* ABI version of this library (major * 100 + minor). */
int tsv_version(void);

/*
 * tsv_tree_mask - topology check, ancestor bitmask and depth of every node.
 *   [1204] "What this needs" item 1: each node attends to its ancestors only,
 *   rebuilt every round from the topology; [1204] "Increment 1": nodes in
 *   topological order with parents[i] < i; [1212] history-mask commit: the
 *   [n, offset + n] additive form, history columns attended in full; [1212]
 *   verify commit: blocked entries are -1e9, never -inf.
 *
 *   parents    int32 [B, T]   parents[b][0] == -1, 0 <= parents[b][i] < i.
 *   anc        uint64 [B, T]  out: bit j of anc[b][i] set iff node j is an
 *                             ancestor of node i or i itself.
 *   depth      int32 [B, T]   out: edges from the root (root = 0).
 *   dense_mask float [B, T, mask_offset + T] or NULL; out: the additive mask
 *                             (0 = attend, -1e9 = blocked) for a history of
 *                             mask_offset positions.  Provided for parity
 *                             checks; the attention call never reads it.
 *   Device errors: TSV_DEV_BAD_ROOT / TSV_DEV_BAD_PARENT; that sequence's anc
 *   and depth are then 0 / -1.
 */
tsv_status tsv_tree_mask(const int32_t* parents, int32_t B, int32_t T, uint64_t* anc, int32_t* depth,
                         float* dense_mask, int32_t mask_offset, int32_t* dev_status, cudaStream_t stream);

/*
 * tsv_sliding_band_mask - the mask a sliding-window layer attends with, in place.
 *   [1212], the commit on caller masks and the sliding-window band: a
 *   sliding-window layer takes the intersection of the caller's mask (here the
 *   dense tree mask of tsv_tree_mask) with its band, by element-wise minimum
 *   of the additive masks, and only where the two can disagree.  Query row q
 *   sits at position mask_offset + q; its band keeps columns c with
 *   mask_offset + q - window < c <= mask_offset + q, all else becomes
 *   min(mask, -1e9).  Every row keeps its own position.
 *   dense_mask float [B, T, mask_offset + T], in/out.  window >= 1; when
 *   mask_offset + T <= window the mask is left untouched (nothing is launched).
 *   The attention call applies the same band itself from tsv_attn_desc.window;
 *   this call is provided for parity checks.
 */
tsv_status tsv_sliding_band_mask(float* dense_mask, int32_t B, int32_t T, int32_t mask_offset, int32_t window,
                                 cudaStream_t stream);

/*
 * Building the draft tree from the drafter's confidence (two calls).
 *   [1204] "What this needs", the fourth decision: EAGLE-2 branches by the
 *   drafter's confidence, which needs the drafter's logits; [1212], the
 *   draft_tree commit: the runner-up at an uncertain step is the alternative
 *   worth a verify position; [728] "What it does": the chain plus likely
 *   alternatives from the draft's top-k selector.
 *
 * tsv_draft_children - for every expanded node (row of drafter logits
 *   [rows, V] fp32), its top_k tokens (ties to the lower index) and their
 *   log-probabilities log_softmax(logits)[token]: child_tokens int32 and
 *   child_logp float, [rows, top_k], largest first.  1 <= top_k <= min(64, V).
 * tsv_tree_select - the verified tree from a candidate tree (reading: the
 *   root plus the T - 1 candidates of highest cumulative log-probability,
 *   summed in fp32 from the root down, depth <= depth_max, ties to the earlier
 *   candidate - what best-first expansion by path probability selects).
 *   cand_parents int32 [B, N] (topological: [b][0] = -1, 0 <= [b][i] < i),
 *   cand_tokens int32 [B, N], cand_logp float [B, N] (log-probability of the
 *   candidate given its parent, <= 0; the root's is ignored).  N <= 1024.
 *   Out: parents, tokens, cand_index int32 [B, T] in selection order (descending
 *   score, so topological; the root first), sizes int32 [B] = nodes chosen
 *   (< T when fewer candidates qualify; the rest of the row is -1).
 *   Device errors: TSV_DEV_BAD_ROOT / TSV_DEV_BAD_PARENT for a candidate tree
 *   that is not topological (that sequence's outputs are -1, size 0) or whose
 *   chosen node's parent was not chosen (a log-probability above 0).
 */
size_t tsv_draft_children_workspace_size(int32_t rows, int32_t V, int32_t top_k);

tsv_status tsv_draft_children(const float* draft_logits, int32_t rows, int32_t V, int32_t top_k, int32_t* child_tokens,
                              float* child_logp, void* workspace, size_t ws_bytes, cudaStream_t stream);

tsv_status tsv_tree_select(const int32_t* cand_parents, const int32_t* cand_tokens, const float* cand_logp, int32_t B,
                           int32_t N, int32_t T, int32_t depth_max, int32_t* parents, int32_t* tokens,
                           int32_t* cand_index, int32_t* sizes, int32_t* dev_status, cudaStream_t stream);

/*
 * Tree-masked GQA attention of the verify block, for n_layers layers at once.
 *   [1204] "What this needs" item 1 and "Increment 3"; [1212] history-mask and
 *   verify_forward_with_mask commits; [728] "Earlier shader evidence" (split-KV
 *   attention with fp32 partials and statistics, 16 nodes x 24 heads x D256).
 *   For every layer l, sequence b, query head h and node i:
 *     O[b,i,h,:] = sum_c p_c V[b, h/G, c, :],  p = softmax_c( Q[b,i,h,:] . K[b,h/G,c,:] / sqrt(D) )
 *   over c in [0, S_b) and c = S_b + j for every j set in anc[b][i], where
 *   S_b = kv_len[b] - T (the block was appended in topological order at
 *   [S_b, S_b + T)).  G = HQ / HKV.  Int8: K = code * k_scale[c], V = code * v_scale[c].
 *   Sliding-window layers ([1212], the commit on caller masks and the
 *   sliding-window band): with window[l] > 0, node i (at cache position
 *   S_b + i) keeps only those of the keys above whose position c satisfies
 *   c > S_b + i - window[l]: the intersection of the tree mask with the
 *   layer's band.  Every node keeps itself.  window[l] == 0 is a full-attention layer.
 *   Accumulation is fp32; O is rounded to bf16 once.
 */
typedef struct {
    int32_t n_layers;   /* 1 .. TSV_MAX_LAYERS */
    int32_t B, T, HQ, HKV, D; /* HQ % HKV == 0; D in {64, 128, 256} */
    int64_t s_cap;      /* capacity of every cache buffer's sequence axis, in positions */
    int32_t max_kv_len; /* host-known upper bound of every kv_len[b] (<= s_cap); sizes the grid */
    int32_t kv_dtype;   /* TSV_F16, TSV_BF16 or TSV_I8_SCALED */
    int32_t splits;     /* key-range splits per (layer, sequence, kv head); 0 = automatic; at most 64 */
    int32_t path;       /* TSV_ATTN_AUTO, TSV_ATTN_SIMT or TSV_ATTN_TCGEN05 */
    const void* q[TSV_MAX_LAYERS];       /* per layer: bf16 [B, T, HQ, D] */
    const void* k[TSV_MAX_LAYERS];       /* per layer: [B, HKV, s_cap, D] in kv_dtype (int8 codes) */
    const void* v[TSV_MAX_LAYERS];       /* per layer: as k */
    const void* k_scale[TSV_MAX_LAYERS]; /* per layer: fp16 [B, HKV, s_cap] (Int8 only, else NULL) */
    const void* v_scale[TSV_MAX_LAYERS]; /* per layer: as k_scale */
    void* o[TSV_MAX_LAYERS];             /* per layer: bf16 [B, T, HQ, D], out */
    const int32_t* kv_len;               /* int32 [B]: S_b + T */
    const uint64_t* anc;                 /* uint64 [B, T] from tsv_tree_mask */
    int32_t window[TSV_MAX_LAYERS];      /* per layer: sliding window in positions, 0 = full attention */
} tsv_attn_desc;

/* Kernel choice.  AUTO takes the tensor-core (tcgen05) kernel where it applies
 * (D == 256 with an fp16, bf16 or Int8 cache) and the CUDA-core kernel elsewhere.
 * TCGEN05 lets the library pick the tensor-core kernel's score-tile width (128
 * keys for Int8 caches and for units of more than 128 query rows, else 64);
 * TCGEN05_64 and TCGEN05_128 force one (both compute the same result).
 * On the tensor-core path Q is rounded to the cache's 16-bit type for the
 * Q K^T product (exact for bf16; for fp16 caches |q| must lie in fp16 range)
 * and the softmax weights P enter P V as 16-bit values. */
#define TSV_ATTN_AUTO 0
#define TSV_ATTN_SIMT 1
#define TSV_ATTN_TCGEN05 2
#define TSV_ATTN_TCGEN05_64 3
#define TSV_ATTN_TCGEN05_128 4

size_t tsv_attention_workspace_size(const tsv_attn_desc* d);

/* Device errors: TSV_DEV_BAD_KV_LEN (that sequence's outputs are left unwritten). */
tsv_status tsv_tree_verify_attention(const tsv_attn_desc* d, void* workspace, size_t ws_bytes,
                                     int32_t* dev_status, cudaStream_t stream);

/*
 * tsv_lm_head_argmax - LM-head projection fused with a greedy argmax; the
 * logits are never written.  [1185] "Phase 2" item 2a (fused projection and
 * argmax at temperature 0) and "Phase 3" (affine group-64 4-bit weights with
 * scales and biases); [1204] "What this needs" item 2 (one target argmax per
 * verified position).
 *   hidden  bf16 [rows, H]
 *   W       TSV_F16 / TSV_BF16: [V, H].  TSV_Q4_G64: uint8 [V, H/2], byte j of a
 *           row holds element 2j in its low nibble and 2j+1 in its high nibble;
 *           scales, biases: bf16 [V, H/64]; w = scale * q + bias, q in [0, 15].
 *   argmax  int32 [rows], out: index of the largest logit, ties -> lowest index.
 *   maxlogit float [rows] or NULL, out: that logit (fp32 accumulation).
 *   H % 64 == 0 (H % 256 == 0 for TSV_F16/TSV_BF16), 1 <= V < 2^31, rows >= 1.
 *   fp16 and bf16 heads with up to 4 rows stream the head once through CUDA
 *   cores; more rows, and 4-bit heads at any row count (H % 512 == 0, scales
 *   and biases 16-byte aligned), use the tcgen05 kernels (fp16 or bf16
 *   operands, fp32 accumulation; 4-bit weights are dequantised to fp16 with
 *   one rounding, and hidden is rounded to fp16 for fp16 and 4-bit heads).
 */
/* Workspace bytes for tsv_lm_head_argmax: 8 per hidden row (running bests), plus, when the tensor-core
 * kernel applies to an fp16 or 4-bit head, an fp16 copy of hidden (rows * H * 2, rounded up to 256).  A
 * smaller workspace (at least 8 bytes per row) is accepted and selects the CUDA-core kernel. */
size_t tsv_lm_head_workspace_size(int32_t rows, int32_t H, int32_t V, int32_t w_dtype);

tsv_status tsv_lm_head_argmax(const void* hidden, int32_t rows, int32_t H, int32_t V, int32_t w_dtype,
                              const void* W, const void* scales, const void* biases, int32_t* argmax,
                              float* maxlogit, void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * tsv_lm_head_logits - the same projection, writing every logit instead of the
 * argmax: logits float [rows, V] (fp32 accumulation, same kernels and
 * workspace as tsv_lm_head_argmax).  The input of sampled verification
 * (tsv_sample_nucleus): Splash issue #728, "What it does" - sampled requests
 * draw from the target's nucleus-filtered distribution at every node.
 */
tsv_status tsv_lm_head_logits(const void* hidden, int32_t rows, int32_t H, int32_t V, int32_t w_dtype,
                              const void* W, const void* scales, const void* biases, float* logits,
                              void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * tsv_sample_nucleus - each node's draw for sampled (temperature > 0)
 * verification.  Splash issue #728, "What it does": every node draws from
 * the nucleus-filtered distribution with its own uniform, which keeps the
 * chain verify's output distribution; the walk (tsv_tree_accept_walk, with
 * these tokens in place of the argmax) then follows the child whose draft
 * token equals the draw.  Filter order (reading; the page names the three
 * knobs): logits / temperature, the top_k largest (ties to the lower index),
 * softmax over them, the shortest descending prefix whose mass reaches top_p,
 * renormalised; the token is the first whose cumulative mass exceeds
 * uniforms[row] * (kept mass).
 *   logits   float [rows, V] (tsv_lm_head_logits); uniforms float [rows] in
 *            [0, 1), one per node, drawn by the caller; tokens int32 [rows], out.
 *   1 <= top_k <= 64 (TSV_EUNSUPPORTED above: the top-k selection is exact
 *   and bounded), temperature > 0, 0 < top_p <= 1, rows <= 65535.
 *   Arithmetic: softmax weights and prefix sums in fp32.
 */
size_t tsv_sample_workspace_size(int32_t rows, int32_t V, int32_t top_k);

tsv_status tsv_sample_nucleus(const float* logits, int32_t rows, int32_t V, float temperature, int32_t top_k,
                              float top_p, const float* uniforms, int32_t* tokens, void* workspace, size_t ws_bytes,
                              cudaStream_t stream);

/*
 * tsv_lm_head_argmax_noalloc - tsv_lm_head_argmax without a workspace argument.
 *   The pages have no counterpart: this entry point exists only in this
 *   library, for callers that cannot allocate device memory themselves -
 *   for example a plugin whose host framework owns every device buffer
 *   through its own pool, or a latency-critical caller that may not pay for
 *   cudaMalloc's implicit synchronisation.  Its scratch is a fixed array of
 *   TSV_NOALLOC_MAX_ROWS 64-bit entries (32 KiB) inside this library's device
 *   image, held by every GPU that loads the library until the process exits.
 *   Arguments, results and errors are those of tsv_lm_head_argmax, plus
 *   TSV_ECAPACITY when rows > TSV_NOALLOC_MAX_ROWS.  The library allocates
 *   nothing for it: the first call on each device looks up the array's
 *   device address (with that device current), and every call clears the
 *   entries it uses on `stream` before the projection.  All calls share the
 *   one array, so calls whose work overlaps on the GPU (on different streams,
 *   or from different host threads) race and give wrong results; serialise
 *   them on one stream.
 *   Speed: the array is also the call's workspace, and for fp16 and 4-bit
 *   heads the tensor-core kernel needs an fp16 copy of hidden beside the
 *   bests (rows * H * 2 bytes, rounded up to 256, after 8 bytes per row
 *   rounded up to 256).  When that does not fit the 32 KiB (H = 5120: more
 *   than 3 rows), the call takes the CUDA-core kernel instead, which streams
 *   the whole head once per 8 hidden rows and, for a 4-bit head, dequantises
 *   every weight again for each row (248,320 x 5120 4-bit head: about 2.1 ms
 *   per 8-row pass, so 4096 rows take about a second instead of a few ms).
 *   bf16 heads need no copy and keep the tensor-core kernel.  Callers with
 *   many rows and an fp16 or 4-bit head should use tsv_lm_head_argmax with a
 *   workspace.
 */
#define TSV_NOALLOC_MAX_ROWS 4096

tsv_status tsv_lm_head_argmax_noalloc(const void* hidden, int32_t rows, int32_t H, int32_t V, int32_t w_dtype,
                                      const void* W, const void* scales, const void* biases, int32_t* argmax,
                                      float* maxlogit, cudaStream_t stream);

/*
 * tsv_tree_accept_walk - descend the tree along the target's argmaxes.
 *   [1204] "What this needs" item 2 and "Increment 1" (the accepted set is a
 *   path, never a subtree); [1212] first commit; [728] "What it does" (every
 *   committed token is the target's selection at its path node).
 *   From u = 0: take the lowest-index child c of u with tokens[c] == argmax[u],
 *   append it, repeat; stop when no child matches.
 *   argmax, tokens, parents  int32 [B, T]
 *   path      int32 [B, T] out: accepted nodes from the root, -1 padded.
 *   path_len  int32 [B]    out: accepted + 1.
 *   emitted   int32 [B, T] out: argmax[path[j]] for j < path_len, -1 padded.
 *   Device errors: TSV_DEV_BAD_ROOT / TSV_DEV_BAD_PARENT (that sequence gets
 *   path = [0], path_len = 1).
 */
tsv_status tsv_tree_accept_walk(const int32_t* argmax, const int32_t* tokens, const int32_t* parents, int32_t B,
                                int32_t T, int32_t* path, int32_t* path_len, int32_t* emitted, int32_t* dev_status,
                                cudaStream_t stream);

/*
 * tsv_kv_gather_positions - compact the verify block of every cache to the
 * accepted path, in place.  [1204] "The rollback constraint, which decides
 * feasibility"; [1212] gather_positions commit (Int8 scale sidecars move with
 * their tokens; a prefix selection equals trim_to; the identity selection
 * short-circuits) and gather_within_tail commit (only [tail_start, tail_start
 * + kept_len) is rewritten; cost scales with the block, not the context).
 *   For every layer, sequence b and kv head, with S = kv_len[b] - T:
 *     rows S + j <- rows S + path[b][j] for j < path_len[b] (K, V and, for
 *     Int8, k_scale and v_scale); then kv_len[b] = S + path_len[b].
 *   Rows below S and at or beyond the new kv_len are not written.  When
 *   path[b][j] == j for every j, no cache byte is moved.
 *   path: strictly increasing with path[b][0] == 0 (every root path of a
 *   topological tree is), 1 <= path_len[b] <= T.
 *   Device errors: TSV_DEV_BAD_PATH, TSV_DEV_BAD_KV_LEN (that sequence is left
 *   untouched, kv_len included).
 */
typedef struct {
    int32_t n_layers, B, HKV, D;
    int64_t s_cap;
    int32_t kv_dtype; /* TSV_F16, TSV_BF16 or TSV_I8_SCALED */
    int32_t reserved;
    void* k[TSV_MAX_LAYERS];       /* per layer: [B, HKV, s_cap, D] */
    void* v[TSV_MAX_LAYERS];
    void* k_scale[TSV_MAX_LAYERS]; /* per layer: fp16 [B, HKV, s_cap] (Int8 only) */
    void* v_scale[TSV_MAX_LAYERS];
} tsv_kv_desc;

tsv_status tsv_kv_gather_positions(const tsv_kv_desc* kv, int32_t* kv_len, const int32_t* path,
                                   const int32_t* path_len, int32_t T, int32_t* dev_status, cudaStream_t stream);

/*
 * tsv_gather_positions - the absolute form of the compaction: keep the cache
 * positions listed in kept, in order, and close them up from position 0.
 *   [1212] gather_positions commit: select and compact positions on the
 *   sequence axis (kept strictly increasing); Int8 scale sidecars move with
 *   their tokens; a prefix selection [0, 1, ..., n-1] equals trim_to(n) and
 *   the identity selection moves nothing.  tsv_kv_gather_positions is the
 *   tail form of the same selection ([1212] gather_within_tail commit) for
 *   kept = [0, S_b) followed by S_b + path[b][j].
 *   For every layer, sequence b and kv head:
 *     rows j <- rows kept[b][j] for j < kept_len[b] (K, V and, for Int8,
 *     k_scale and v_scale); then kv_len[b] = kept_len[b].
 *   Rows at or beyond the new kv_len are not written.  Rows below the first j
 *   with kept[b][j] != j are not written either, so a prefix or identity
 *   selection moves no cache byte.
 *   kept      int32 [B, max_kept] (row stride max_kept): kept[b][0..kept_len[b])
 *             strictly increasing within [0, kv_len[b]).  May be NULL when
 *             max_kept == 0.
 *   kept_len  int32 [B]: 0 <= kept_len[b] <= min(max_kept, kv_len[b]).
 *   kv_len    int32 [B], in/out: in, the current length (<= s_cap); out,
 *             kept_len[b].
 *   The list may be as long as the cache; every (layer, sequence, kv head)
 *   moves its rows in ascending chunks, so the cost is the rows moved.
 *   Device errors: TSV_DEV_BAD_PATH (a kept list that is not strictly
 *   increasing, leaves [0, kv_len[b]), or a kept_len out of range),
 *   TSV_DEV_BAD_KV_LEN (kv_len[b] outside [0, s_cap]); that sequence is left
 *   untouched, kv_len included.
 */
tsv_status tsv_gather_positions(const tsv_kv_desc* kv, int32_t* kv_len, const int32_t* kept, const int32_t* kept_len,
                                int32_t max_kept, int32_t* dev_status, cudaStream_t stream);

/*
 * tsv_tree_append - append the verify block to every layer's cache, each node
 * at its own position, ahead of the attention call.
 *   [1185], the closing comment's list of follow-ups: the tree path verifies
 *   the tree at its own positions (the title of the PR that added tree
 *   drafting there).  Node i is verified at position S_b + depth(i)
 *   (the root, the last committed token, at S_b; a chain gets S_b + i); its K
 *   and V rows still go to cache slot S_b + i, the topological block layout
 *   tsv_tree_verify_attention and tsv_kv_gather_positions use.  Rotary
 *   embedding (reading; the pages name only positions): the first rot_dim
 *   features are rotated in pairs (j, j + rot_dim/2) - or (2j, 2j + 1) when
 *   interleaved - by the angle pos * rope_base^(-2j / rot_dim); Q and K are
 *   rotated, V is not.  Int8 caches ([1212] gather_positions commit: one scale
 *   per token; a per-token scale maps every single-valued token to the same
 *   code): scale = fp16(absmax / 127) with the division in fp32, code =
 *   round-half-to-even(x / scale) in fp32, clamped to [-127, 127]; a token whose
 *   scale is 0 stores zero codes.  fp16 / bf16 caches store the rotated fp32
 *   values rounded to nearest even.  Angles are reduced in fp64, so positions
 *   up to 2^31 keep fp32 accuracy.
 *   kv_len: in, S_b per sequence; out, S_b + T.  depth: from tsv_tree_mask.
 *   Device errors: TSV_DEV_BAD_KV_LEN when S_b + T > s_cap; a sequence whose
 *   depth[b][0] != 0 (its mask call failed) is skipped.  Skipped sequences
 *   keep their caches and kv_len.
 */
typedef struct {
    int32_t n_layers;   /* 1 .. TSV_MAX_LAYERS */
    int32_t B, T, HQ, HKV, D; /* HQ % HKV == 0; D in {64, 128, 256} */
    int64_t s_cap;
    int32_t kv_dtype;   /* TSV_F16, TSV_BF16 or TSV_I8_SCALED */
    int32_t rot_dim;    /* even, 2 <= rot_dim <= D; features >= rot_dim are copied */
    int32_t interleaved; /* 0: pairs (j, j + rot_dim/2); 1: pairs (2j, 2j + 1) */
    int32_t reserved;
    double rope_base;   /* > 0, e.g. 1e4 or 1e6 */
    const void* q_in[TSV_MAX_LAYERS];  /* per layer: bf16 [B, T, HQ, D], not yet rotated */
    void* q_out[TSV_MAX_LAYERS];       /* per layer: bf16 [B, T, HQ, D], out (may equal q_in) */
    const void* k_new[TSV_MAX_LAYERS]; /* per layer: bf16 [B, T, HKV, D], not yet rotated */
    const void* v_new[TSV_MAX_LAYERS]; /* per layer: bf16 [B, T, HKV, D] */
    void* k[TSV_MAX_LAYERS];           /* per layer caches as in tsv_kv_desc */
    void* v[TSV_MAX_LAYERS];
    void* k_scale[TSV_MAX_LAYERS];
    void* v_scale[TSV_MAX_LAYERS];
    const int32_t* depth;              /* int32 [B, T] */
} tsv_append_desc;

tsv_status tsv_tree_append(const tsv_append_desc* d, int32_t* kv_len, int32_t* dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TSV_H */
