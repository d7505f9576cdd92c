"""Torch-facing wrappers of the tsv C ABI (argument marshalling only).

Every function checks shapes/dtypes/devices of its torch tensors, passes raw
device pointers and the current CUDA stream to the library, and raises
``TsvError`` on any status other than TSV_OK.  All computation happens in the
library's CUDA kernels.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass, field

import torch

from . import _abi
from ._abi import BF16, F16, I8_SCALED, MAX_LAYERS, Q4_G64, AppendDesc, AttnDesc, KvDesc, check, load

KV_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, I8_SCALED: torch.int8}


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _cuda(t, name, dtype=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# ----------------------------------------------------------------------------- a1 tree mask
def tree_mask(parents, anc, depth, dense_mask=None, mask_offset=0, dev_status=None, stream=None):
    """parents int32 [B,T] -> anc int64 [B,T] (uint64 bits), depth int32 [B,T], optional dense mask."""
    lib = load()
    B, T = parents.shape
    _cuda(parents, "parents", torch.int32)
    _cuda(anc, "anc", torch.int64, (B, T))
    _cuda(depth, "depth", torch.int32, (B, T))
    if dense_mask is not None:
        _cuda(dense_mask, "dense_mask", torch.float32, (B, T, mask_offset + T))
    check(lib.tsv_tree_mask(_p(parents), B, T, _p(anc), _p(depth), _p(dense_mask), int(mask_offset),
                            _p(dev_status), _stream(stream)), "tree_mask")


def sliding_band_mask(dense_mask, mask_offset, window, stream=None):
    """In place: intersect a dense [B, T, mask_offset + T] fp32 mask with a sliding-window band."""
    B, T = dense_mask.shape[0], dense_mask.shape[1]
    _cuda(dense_mask, "dense_mask", torch.float32, (B, T, mask_offset + T))
    check(load().tsv_sliding_band_mask(_p(dense_mask), B, T, int(mask_offset), int(window), _stream(stream)),
          "sliding_band_mask")


def draft_children(draft_logits, child_tokens, child_logp, *, top_k, workspace=None, stream=None):
    """Top-k children of every expanded node: draft_logits fp32 [rows, V] -> tokens int32, logp fp32 [rows, k]."""
    lib = load()
    rows, V = draft_logits.shape
    _cuda(draft_logits, "draft_logits", torch.float32, (rows, V))
    _cuda(child_tokens, "child_tokens", torch.int32, (rows, top_k))
    _cuda(child_logp, "child_logp", torch.float32, (rows, top_k))
    if workspace is None:
        workspace = torch.empty(max(int(lib.tsv_draft_children_workspace_size(rows, V, top_k)), 256),
                                dtype=torch.uint8, device=draft_logits.device)
    check(lib.tsv_draft_children(_p(draft_logits), rows, V, int(top_k), _p(child_tokens), _p(child_logp),
                                 _p(workspace), workspace.numel(), _stream(stream)), "draft_children")


def tree_select(cand_parents, cand_tokens, cand_logp, parents, tokens, cand_index, sizes, *, depth_max,
                dev_status=None, stream=None):
    """Verified tree [B, T] from a candidate tree [B, N] by cumulative drafter log-probability."""
    B, N = cand_parents.shape
    T = parents.shape[1]
    for t, name, dt, shape in ((cand_parents, "cand_parents", torch.int32, (B, N)),
                               (cand_tokens, "cand_tokens", torch.int32, (B, N)),
                               (cand_logp, "cand_logp", torch.float32, (B, N)), (parents, "parents", torch.int32, (B, T)),
                               (tokens, "tokens", torch.int32, (B, T)), (cand_index, "cand_index", torch.int32, (B, T)),
                               (sizes, "sizes", torch.int32, (B,))):
        _cuda(t, name, dt, shape)
    check(load().tsv_tree_select(_p(cand_parents), _p(cand_tokens), _p(cand_logp), B, N, T, int(depth_max),
                                 _p(parents), _p(tokens), _p(cand_index), _p(sizes), _p(dev_status), _stream(stream)),
          "tree_select")


# ----------------------------------------------------------------------------- a2 attention
def attn_desc(q, k, v, o, kv_len, anc, *, T, HQ, HKV, D, kv_dtype, max_kv_len, k_scale=None, v_scale=None,
              splits=0, path=0, window=None) -> AttnDesc:
    """Descriptor over per-layer lists: q/o bf16 [B,T,HQ,D]; k/v [B,HKV,s_cap,D]; scales fp16 [B,HKV,s_cap].

    window: per-layer sliding windows (0 = full attention), or None for all full-attention layers.
    """
    n = len(q)
    if not (1 <= n <= MAX_LAYERS) or not (len(k) == len(v) == len(o) == n):
        raise ValueError("per-layer lists must have the same length in [1, 64]")
    if window is not None and len(window) != n:
        raise ValueError("window needs one entry per layer")
    B = q[0].shape[0]
    s_cap = k[0].shape[2]
    d = AttnDesc()
    d.n_layers, d.B, d.T, d.HQ, d.HKV, d.D = n, B, T, HQ, HKV, D
    d.s_cap, d.max_kv_len, d.kv_dtype, d.splits, d.path = s_cap, int(max_kv_len), kv_dtype, int(splits), int(path)
    kvt = KV_TORCH_DTYPE[kv_dtype]
    for l in range(n):
        _cuda(q[l], "q", torch.bfloat16, (B, T, HQ, D))
        _cuda(o[l], "o", torch.bfloat16, (B, T, HQ, D))
        _cuda(k[l], "k", kvt, (B, HKV, s_cap, D))
        _cuda(v[l], "v", kvt, (B, HKV, s_cap, D))
        d.q[l], d.k[l], d.v[l], d.o[l] = q[l].data_ptr(), k[l].data_ptr(), v[l].data_ptr(), o[l].data_ptr()
        if kv_dtype == I8_SCALED:
            _cuda(k_scale[l], "k_scale", torch.float16, (B, HKV, s_cap))
            _cuda(v_scale[l], "v_scale", torch.float16, (B, HKV, s_cap))
            d.k_scale[l], d.v_scale[l] = k_scale[l].data_ptr(), v_scale[l].data_ptr()
    _cuda(kv_len, "kv_len", torch.int32, (B,))
    _cuda(anc, "anc", torch.int64, (B, T))
    d.kv_len, d.anc = kv_len.data_ptr(), anc.data_ptr()
    for l in range(n):
        d.window[l] = 0 if window is None else int(window[l])
    return d


def attention_workspace_size(desc: AttnDesc) -> int:
    return int(load().tsv_attention_workspace_size(C.byref(desc)))


def tree_verify_attention(desc: AttnDesc, workspace=None, dev_status=None, stream=None):
    lib = load()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(lib.tsv_tree_verify_attention(C.byref(desc), _p(workspace), ws_bytes, _p(dev_status), _stream(stream)),
          "tree_verify_attention")


# ----------------------------------------------------------------------------- block append (rotary + Int8)
def append_desc(q_in, q_out, k_new, v_new, k, v, depth, *, T, HQ, HKV, D, kv_dtype, rot_dim, rope_base,
                interleaved=False, k_scale=None, v_scale=None) -> AppendDesc:
    """Descriptor over per-layer lists: q_in/q_out bf16 [B,T,HQ,D]; k_new/v_new bf16 [B,T,HKV,D]; caches as
    for attn_desc."""
    n = len(q_in)
    if not (1 <= n <= MAX_LAYERS) or not (len(q_out) == len(k_new) == len(v_new) == len(k) == len(v) == n):
        raise ValueError("per-layer lists must have the same length in [1, 64]")
    B = q_in[0].shape[0]
    s_cap = k[0].shape[2]
    d = AppendDesc()
    d.n_layers, d.B, d.T, d.HQ, d.HKV, d.D, d.s_cap = n, B, T, HQ, HKV, D, s_cap
    d.kv_dtype, d.rot_dim, d.interleaved, d.rope_base = kv_dtype, int(rot_dim), int(bool(interleaved)), float(rope_base)
    kvt = KV_TORCH_DTYPE[kv_dtype]
    for l in range(n):
        _cuda(q_in[l], "q_in", torch.bfloat16, (B, T, HQ, D))
        _cuda(q_out[l], "q_out", torch.bfloat16, (B, T, HQ, D))
        _cuda(k_new[l], "k_new", torch.bfloat16, (B, T, HKV, D))
        _cuda(v_new[l], "v_new", torch.bfloat16, (B, T, HKV, D))
        _cuda(k[l], "k", kvt, (B, HKV, s_cap, D))
        _cuda(v[l], "v", kvt, (B, HKV, s_cap, D))
        d.q_in[l], d.q_out[l] = q_in[l].data_ptr(), q_out[l].data_ptr()
        d.k_new[l], d.v_new[l], d.k[l], d.v[l] = k_new[l].data_ptr(), v_new[l].data_ptr(), k[l].data_ptr(), v[l].data_ptr()
        if kv_dtype == I8_SCALED:
            _cuda(k_scale[l], "k_scale", torch.float16, (B, HKV, s_cap))
            _cuda(v_scale[l], "v_scale", torch.float16, (B, HKV, s_cap))
            d.k_scale[l], d.v_scale[l] = k_scale[l].data_ptr(), v_scale[l].data_ptr()
    _cuda(depth, "depth", torch.int32, (B, T))
    d.depth = depth.data_ptr()
    return d


def tree_append(desc: AppendDesc, kv_len, dev_status=None, stream=None):
    """Append the block at the nodes' positions; kv_len int32 [B]: S_b in, S_b + T out."""
    _cuda(kv_len, "kv_len", torch.int32, (desc.B,))
    check(load().tsv_tree_append(C.byref(desc), _p(kv_len), _p(dev_status), _stream(stream)), "tree_append")


# ----------------------------------------------------------------------------- a3 LM head
def lm_head_workspace_size(rows: int, H: int, V: int, w_dtype: int) -> int:
    return int(load().tsv_lm_head_workspace_size(rows, H, V, w_dtype))


def lm_head_argmax(hidden, W, argmax, *, w_dtype, V, scales=None, biases=None, maxlogit=None, workspace=None,
                   stream=None):
    """hidden bf16 [rows,H]; W fp16/bf16 [V,H] or uint8 [V,H/2] (+ bf16 scales/biases [V,H/64])."""
    lib = load()
    rows, H = hidden.shape
    _cuda(hidden, "hidden", torch.bfloat16)
    if w_dtype == Q4_G64:
        _cuda(W, "W", torch.uint8, (V, H // 2))
        _cuda(scales, "scales", torch.bfloat16, (V, H // 64))
        _cuda(biases, "biases", torch.bfloat16, (V, H // 64))
    else:
        _cuda(W, "W", torch.bfloat16 if w_dtype == BF16 else torch.float16, (V, H))
    _cuda(argmax, "argmax", torch.int32, (rows,))
    if maxlogit is not None:
        _cuda(maxlogit, "maxlogit", torch.float32, (rows,))
    if workspace is None:
        workspace = torch.empty(lm_head_workspace_size(rows, H, V, w_dtype), dtype=torch.uint8, device=hidden.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    check(lib.tsv_lm_head_argmax(_p(hidden), rows, H, V, w_dtype, _p(W), _p(scales), _p(biases), _p(argmax),
                                 _p(maxlogit), _p(workspace), ws_bytes, _stream(stream)), "lm_head_argmax")


def lm_head_logits(hidden, W, logits, *, w_dtype, V, scales=None, biases=None, workspace=None, stream=None):
    """Every logit: hidden bf16 [rows, H] -> logits fp32 [rows, V]."""
    lib = load()
    rows, H = hidden.shape
    _cuda(logits, "logits", torch.float32, (rows, V))
    if workspace is None:
        workspace = torch.empty(max(lm_head_workspace_size(rows, H, V, w_dtype), 256), dtype=torch.uint8,
                                device=hidden.device)
    check(lib.tsv_lm_head_logits(_p(hidden), rows, H, V, w_dtype, _p(W), _p(scales), _p(biases), _p(logits),
                                 _p(workspace), workspace.numel(), _stream(stream)), "lm_head_logits")


def sample_workspace_size(rows: int, V: int, top_k: int) -> int:
    return int(load().tsv_sample_workspace_size(rows, V, top_k))


def sample_nucleus(logits, uniforms, tokens, *, temperature, top_k, top_p, workspace=None, stream=None):
    """Each row's draw from its nucleus-filtered distribution: logits fp32 [rows, V], uniforms fp32 [rows]."""
    lib = load()
    rows, V = logits.shape
    _cuda(uniforms, "uniforms", torch.float32, (rows,))
    _cuda(tokens, "tokens", torch.int32, (rows,))
    if workspace is None:
        workspace = torch.empty(max(sample_workspace_size(rows, V, top_k), 256), dtype=torch.uint8,
                                device=logits.device)
    check(lib.tsv_sample_nucleus(_p(logits), rows, V, float(temperature), int(top_k), float(top_p), _p(uniforms),
                                 _p(tokens), _p(workspace), workspace.numel(), _stream(stream)), "sample_nucleus")


# ----------------------------------------------------------------------------- a4 walk
def tree_accept_walk(argmax, tokens, parents, path, path_len, emitted, dev_status=None, stream=None):
    lib = load()
    B, T = parents.shape
    for t, n in ((argmax, "argmax"), (tokens, "tokens"), (parents, "parents"), (path, "path"), (emitted, "emitted")):
        _cuda(t, n, torch.int32, (B, T))
    _cuda(path_len, "path_len", torch.int32, (B,))
    check(lib.tsv_tree_accept_walk(_p(argmax), _p(tokens), _p(parents), B, T, _p(path), _p(path_len), _p(emitted),
                                   _p(dev_status), _stream(stream)), "tree_accept_walk")


# ----------------------------------------------------------------------------- a5 gather
def kv_desc(k, v, *, HKV, D, kv_dtype, k_scale=None, v_scale=None) -> KvDesc:
    n = len(k)
    B, _, s_cap, _ = k[0].shape
    d = KvDesc()
    d.n_layers, d.B, d.HKV, d.D, d.s_cap, d.kv_dtype = n, B, HKV, D, s_cap, kv_dtype
    kvt = KV_TORCH_DTYPE[kv_dtype]
    for l in range(n):
        _cuda(k[l], "k", kvt, (B, HKV, s_cap, D))
        _cuda(v[l], "v", kvt, (B, HKV, s_cap, D))
        d.k[l], d.v[l] = k[l].data_ptr(), v[l].data_ptr()
        if kv_dtype == I8_SCALED:
            _cuda(k_scale[l], "k_scale", torch.float16, (B, HKV, s_cap))
            _cuda(v_scale[l], "v_scale", torch.float16, (B, HKV, s_cap))
            d.k_scale[l], d.v_scale[l] = k_scale[l].data_ptr(), v_scale[l].data_ptr()
    return d


def kv_gather_positions(desc: KvDesc, kv_len, path, path_len, T: int, dev_status=None, stream=None):
    lib = load()
    _cuda(kv_len, "kv_len", torch.int32, (desc.B,))
    _cuda(path, "path", torch.int32, (desc.B, T))
    _cuda(path_len, "path_len", torch.int32, (desc.B,))
    check(lib.tsv_kv_gather_positions(C.byref(desc), _p(kv_len), _p(path), _p(path_len), T, _p(dev_status),
                                      _stream(stream)), "kv_gather_positions")


def gather_positions(desc: KvDesc, kv_len, kept, kept_len, dev_status=None, stream=None):
    """Absolute form: every cache keeps positions kept[b, :kept_len[b]] (strictly increasing), closed up from 0;
    kv_len[b] becomes kept_len[b].  kept int32 [B, max_kept], kept_len int32 [B]."""
    _cuda(kv_len, "kv_len", torch.int32, (desc.B,))
    _cuda(kept_len, "kept_len", torch.int32, (desc.B,))
    if kept is None or kept.numel() == 0:
        kept, max_kept = None, 0
    else:
        _cuda(kept, "kept", torch.int32)
        if kept.dim() != 2 or kept.shape[0] != desc.B:
            raise ValueError(f"kept must have shape [B={desc.B}, max_kept], got {tuple(kept.shape)}")
        max_kept = kept.shape[1]
    check(load().tsv_gather_positions(C.byref(desc), _p(kv_len), _p(kept), _p(kept_len), int(max_kept), _p(dev_status),
                                      _stream(stream)), "gather_positions")


# ----------------------------------------------------------------------------- one verify round
@dataclass
class VerifyRound:
    """Device buffers of one verify round and the five calls in order on one stream.

    Caches (k, v[, k_scale, v_scale]) and the LM head are resident state; the
    per-round inputs are parents, tokens, q (per layer), hidden and kv_len.
    The int32 results (path, path_len, emitted, argmax) are views into one
    block, ``outs["result"]``.
    """
    T: int
    HQ: int
    HKV: int
    D: int
    V: int
    kv_dtype: int
    w_dtype: int
    max_kv_len: int
    parents: torch.Tensor
    tokens: torch.Tensor
    q: list
    k: list
    v: list
    hidden: torch.Tensor
    W: torch.Tensor
    kv_len: torch.Tensor
    k_scale: list = None
    v_scale: list = None
    w_scales: torch.Tensor = None
    w_biases: torch.Tensor = None
    splits: int = 0
    attn_path: int = 0
    window: tuple = None
    q_in: list = None      # block append (optional): pre-rotation Q, new K and V rows per layer
    k_new: list = None
    v_new: list = None
    rot_dim: int = 0
    rope_base: float = 1e6
    sample: tuple = None   # sampled verification (optional): (temperature, top_k, top_p)
    uniforms: torch.Tensor = None  # fp32 [B * T], one per node
    outs: dict = field(default_factory=dict)

    def __post_init__(self):
        dev = self.parents.device
        B, T = self.parents.shape
        z = lambda *s, dt=torch.int32: torch.zeros(*s, dtype=dt, device=dev)
        n = len(self.q)
        # the round's int32 results share one block (outs["result"]: path, path_len, emitted, argmax, each at a
        # 64-byte offset), so that a caller reads them back with one copy
        a16 = lambda m: (m + 15) // 16 * 16
        BT = B * T
        res = z(3 * a16(BT) + a16(B))
        o_len, o_emit, o_arg = a16(BT), a16(BT) + a16(B), 2 * a16(BT) + a16(B)
        self.outs = dict(anc=z(B, T, dt=torch.int64), depth=z(B, T), argmax=res[o_arg:o_arg + BT],
                         maxlogit=z(B * T, dt=torch.float32), path=res[:BT].view(B, T), path_len=res[o_len:o_len + B],
                         emitted=res[o_emit:o_emit + BT].view(B, T), result=res, status=z(4),
                         o=[torch.empty(B, T, self.HQ, self.D, dtype=torch.bfloat16, device=dev) for _ in range(n)])
        self.adesc = attn_desc(self.q, self.k, self.v, self.outs["o"], self.kv_len, self.outs["anc"], T=T, HQ=self.HQ,
                               HKV=self.HKV, D=self.D, kv_dtype=self.kv_dtype, max_kv_len=self.max_kv_len,
                               k_scale=self.k_scale, v_scale=self.v_scale, splits=self.splits, path=self.attn_path,
                               window=self.window)
        self.kdesc = kv_desc(self.k, self.v, HKV=self.HKV, D=self.D, kv_dtype=self.kv_dtype, k_scale=self.k_scale,
                             v_scale=self.v_scale)
        self.apdesc = None
        if self.q_in is not None:  # the round appends its block: Q rotated from q_in into q, K/V rows into the caches
            self.apdesc = append_desc(self.q_in, self.q, self.k_new, self.v_new, self.k, self.v, self.outs["depth"], T=T,
                                      HQ=self.HQ, HKV=self.HKV, D=self.D, kv_dtype=self.kv_dtype, rot_dim=self.rot_dim,
                                      rope_base=self.rope_base, k_scale=self.k_scale, v_scale=self.v_scale)
        self.attn_ws = torch.empty(max(attention_workspace_size(self.adesc), 256), dtype=torch.uint8, device=dev)
        self.lm_ws = torch.empty(max(lm_head_workspace_size(B * T, self.hidden.shape[1], self.V, self.w_dtype), 256),
                                 dtype=torch.uint8, device=dev)
        if self.sample is not None:  # the LM stage writes every logit and draws each node's token
            self.outs["logits"] = torch.empty(B * T, self.V, dtype=torch.float32, device=dev)
            self.sample_ws = torch.empty(max(sample_workspace_size(B * T, self.V, int(self.sample[1])), 256),
                                         dtype=torch.uint8, device=dev)

    def run(self, stream=None, stages=("mask", "append", "attn", "lm", "walk", "gather")):
        """Issue the round's calls in order; "append" runs only when the round was built with append inputs."""
        o = self.outs
        B, T = self.parents.shape
        if "mask" in stages:
            tree_mask(self.parents, o["anc"], o["depth"], dev_status=o["status"], stream=stream)
        if "append" in stages and self.apdesc is not None:
            tree_append(self.apdesc, self.kv_len, dev_status=o["status"], stream=stream)
        if "attn" in stages:
            tree_verify_attention(self.adesc, self.attn_ws, dev_status=o["status"], stream=stream)
        if "lm" in stages and self.sample is None:
            lm_head_argmax(self.hidden, self.W, o["argmax"], w_dtype=self.w_dtype, V=self.V, scales=self.w_scales,
                           biases=self.w_biases, maxlogit=o["maxlogit"], workspace=self.lm_ws, stream=stream)
        elif "lm" in stages:  # sampled verification: o["argmax"] receives each node's draw, the walk's input
            t, k, p = self.sample
            lm_head_logits(self.hidden, self.W, o["logits"], w_dtype=self.w_dtype, V=self.V, scales=self.w_scales,
                           biases=self.w_biases, workspace=self.lm_ws, stream=stream)
            sample_nucleus(o["logits"], self.uniforms, o["argmax"], temperature=t, top_k=k, top_p=p,
                           workspace=self.sample_ws, stream=stream)
        if "walk" in stages:
            tree_accept_walk(o["argmax"].view(B, T), self.tokens, self.parents, o["path"], o["path_len"], o["emitted"],
                             dev_status=o["status"], stream=stream)
        if "gather" in stages:
            kv_gather_positions(self.kdesc, self.kv_len, o["path"], o["path_len"], T, dev_status=o["status"],
                                stream=stream)
        return o

    def capture(self, stages=("mask", "append", "attn", "lm", "walk", "gather")):
        """Record ``run(stages)`` once as a CUDA graph over this round's buffers.

        Every call reads its per-round inputs (parents, tokens, q, hidden, kv_len, ...) from device memory and
        takes its launch shapes from sizes fixed at construction, so one graph serves every later round: copy the
        round's inputs into the buffers, then ``replay()``.  The calls are validated on the host once, here.
        """
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(stages=stages)
        self._graph = g
        return g

    def replay(self):
        """Issue the captured round on the current stream (``capture()`` first)."""
        g = getattr(self, "_graph", None)
        if g is None:
            raise RuntimeError("VerifyRound.replay: capture() has not been called")
        g.replay()
        return self.outs
