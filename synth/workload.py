"""Device buffers of one synthetic verify round, ready for the tsv calls.

Caches, Q and the LM head are filled on the device by ``synth.device``; the
round's tree, tokens and planted hidden states come from ``synth.trees`` on the
host and are uploaded.  ``kv_len`` starts at S + T (the block was appended).
"""
from __future__ import annotations

import numpy as np
import torch

from . import device as sd
from . import trees
from .configs import I8, Config


def bits_to_bf16(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def _arena(specs, device, align: int = 256):
    """One uint8 device buffer holding every (name, shape, dtype) of ``specs`` at ``align``-byte offsets; returns
    the buffer and a dict of typed views into it."""
    offs, n = [], 0
    for _, shape, dt in specs:
        n = (n + align - 1) // align * align
        offs.append(n)
        n += int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
    buf = torch.zeros(max(n, 1), dtype=torch.uint8, device=device)
    views = {}
    for (name, shape, dt), o in zip(specs, offs):
        nb = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        views[name] = buf[o:o + nb].view(dt).view(shape)
    return buf, views


class Workload:
    """All device tensors of ``cfg`` (optionally a subset of layers, extra capacity)."""

    def __init__(self, cfg: Config, device="cuda", round_id: int = 0, n_layers: int | None = None,
                 s_cap: int | None = None, splits: int = 0, attn_path: int = 0):
        self.cfg = cfg
        self.device = device
        L = n_layers or cfg.n_layers
        self.s_cap = s_cap or cfg.NKV
        self.caches = [sd.alloc_cache(cfg, l, self.s_cap, device) for l in range(L)]
        # cfg.rot_dim > 0: every round appends its block first (Q rotated from q_in into q, K/V rows into [S, S+T))
        self.append = cfg.rot_dim > 0
        # Every per-round input lives in one device buffer (``inputs``), so that a round's inputs arrive with one
        # host-to-device copy: parents, tokens, hidden, Q (q_in when appending) and new K/V rows per layer, uniforms.
        B, T = cfg.B, cfg.T
        specs = [("parents", (B, T), torch.int32), ("tokens", (B, T), torch.int32),
                 ("hidden", (cfg.rows, cfg.H), torch.bfloat16)]
        specs += [(f"q{l}", (B, T, cfg.HQ, cfg.D), torch.bfloat16) for l in range(L)]
        if self.append:
            specs += [(f"{w}{l}", (B, T, cfg.HKV, cfg.D), torch.bfloat16) for l in range(L) for w in ("k_new", "v_new")]
        if cfg.sample:
            specs.append(("uniforms", (cfg.rows,), torch.float32))
        self._specs = specs
        self._splits, self._attn_path = splits, attn_path
        self.inputs, views = _arena(specs, device)
        q_fed = [sd.alloc_q(cfg, l, device, out=views[f"q{l}"]) for l in range(L)]
        self.q_in = self.new_kv = None
        if self.append:
            self.q_in = q_fed
            self.q = [torch.empty_like(t) for t in self.q_in]
            self.new_kv = [sd.alloc_new_kv(cfg, l, device, out={w: views[f"{w}{l}"] for w in ("k_new", "v_new")})
                           for l in range(L)]
        else:
            self.q = q_fed
        self.head = sd.alloc_head(cfg, device)
        self.round = trees.make_round(cfg, round_id)
        r = self.round
        self.parents, self.tokens, self.hidden = views["parents"], views["tokens"], views["hidden"]
        self.parents.copy_(torch.from_numpy(r["parents"]))
        self.tokens.copy_(torch.from_numpy(r["tokens"]))
        self.hidden.copy_(bits_to_bf16(r["hidden"], "cpu"))
        self.kv_len = torch.full((cfg.B,), cfg.S if self.append else cfg.NKV, dtype=torch.int32, device=device)
        self.uniforms = None
        if cfg.sample:  # sampled verification: one uniform per node and round
            from . import tensors as st
            self.uniforms = views["uniforms"]
            self.uniforms.copy_(torch.from_numpy(st.node_uniforms(cfg, round_id)))
        self.vr = self._verify_round(self.parents, self.tokens, self.q, self.hidden, self.q_in, self.new_kv,
                                     self.uniforms)
        self._tail = None

    def _verify_round(self, parents, tokens, q, hidden, q_in, new_kv, uniforms):
        """A VerifyRound over these per-round inputs and this workload's caches, head and kv_len."""
        from tree_speculative_decoding_array_gb300 import VerifyRound

        cfg = self.cfg
        i8 = cfg.kv_dtype == I8
        return VerifyRound(
            T=cfg.T, HQ=cfg.HQ, HKV=cfg.HKV, D=cfg.D, V=cfg.V, kv_dtype=cfg.kv_dtype, w_dtype=cfg.w_dtype,
            max_kv_len=self.s_cap, parents=parents, tokens=tokens, q=q,
            k=[c["k"] for c in self.caches], v=[c["v"] for c in self.caches], hidden=hidden,
            W=self.head["W"], kv_len=self.kv_len,
            k_scale=[c["ks"] for c in self.caches] if i8 else None,
            v_scale=[c["vs"] for c in self.caches] if i8 else None,
            w_scales=self.head["scales"], w_biases=self.head["biases"], splits=self._splits,
            attn_path=self._attn_path,
            window=tuple(cfg.layer_window(l) for l in range(len(self.caches))) if cfg.window else None,
            q_in=q_in, k_new=[x["k_new"] for x in new_kv] if self.append else None,
            v_new=[x["v_new"] for x in new_kv] if self.append else None, rot_dim=cfg.rot_dim,
            rope_base=cfg.rope_base, sample=tuple(cfg.sample) if cfg.sample else None, uniforms=uniforms)

    def twin(self):
        """A second input buffer of the same layout as ``inputs`` and a VerifyRound over it that shares this
        workload's caches, head and kv_len: a caller copies one round's inputs into one buffer while the round
        over the other buffer runs.  Returns (buffer, VerifyRound)."""
        L = len(self.caches)
        buf, views = _arena(self._specs, self.device)
        q_fed = [views[f"q{l}"] for l in range(L)]
        if self.append:
            q_in, q = q_fed, [torch.empty_like(t) for t in q_fed]
            new_kv = [{w: views[f"{w}{l}"] for w in ("k_new", "v_new")} for l in range(L)]
        else:
            q_in, q, new_kv = None, q_fed, None
        uniforms = views["uniforms"] if self.cfg.sample else None
        vr = self._verify_round(views["parents"], views["tokens"], q, views["hidden"], q_in, new_kv, uniforms)
        return buf, vr

    def set_round(self, round_id: int):
        """Load another round's tree, tokens and hidden states (same caches and head)."""
        self.round = trees.make_round(self.cfg, round_id)
        r = self.round
        self.parents.copy_(torch.from_numpy(r["parents"]))
        self.tokens.copy_(torch.from_numpy(r["tokens"]))
        self.hidden.copy_(bits_to_bf16(r["hidden"], "cpu"))
        if self.uniforms is not None:
            from . import tensors as st
            self.uniforms.copy_(torch.from_numpy(st.node_uniforms(self.cfg, round_id)))

    def save_tail(self):
        """Keep a pristine copy of the verify block [S, S+T) of every cache and of kv_len (the gather rewrites both).

        ``restore_tail`` then puts them back with one batched copy launch.  A round that appends its block keeps
        only kv_len (= S): the append rewrites the block rows every round.
        """
        S, T = self.cfg.S, self.cfg.T
        rows = []
        self._saved = []
        for c in ([] if self.append else self.caches):  # an appending round rewrites the block itself
            for name, t in c.items():
                tail = t[:, :, S:S + T]
                saved = tail.contiguous().clone()
                self._saved.append(saved)
                per = T * (t.shape[3] if t.dim() == 4 else 1) * t.element_size()  # bytes of one (b, kvh) tail
                for b in range(t.shape[0]):
                    for h in range(t.shape[1]):
                        rows.append((saved[b, h].data_ptr(), tail[b, h].data_ptr(), per))
        self._kv_len0 = self.kv_len.clone()
        rows.append((self._kv_len0.data_ptr(), self.kv_len.data_ptr(), self.kv_len.numel() * 4))
        self._table = torch.tensor(rows, dtype=torch.int64, device=self.device)
        self._tail = True

    def restore_tail(self):
        sd.copy_table(self._table)
