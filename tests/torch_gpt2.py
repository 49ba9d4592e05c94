"""Independent float64 restatement of the GPT-2 forward pass for pinning the
oracle.  Test-only.

It is written as a full-prefix, batched computation from torch library
primitives (``layer_norm``, ``scaled_dot_product_attention`` with a causal
mask, ``gelu(approximate='tanh')``, matrix products) rather than the oracle's
per-token cached loops, so a mistake in the oracle's loops, indexing or cache
handling shows up as a disagreement.  It parses the packed checkpoint itself
(LeanExe GPT-2 README, packed checkpoint paragraph; Hugging Face state-dict
block order, gpt2.s weight-layout paragraph).
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


class _Reader:
    def __init__(self, w):
        self.w = w
        self.pos = 0

    def take(self, *shape):
        n = int(np.prod(shape))
        t = self.w[self.pos:self.pos + n].view(*shape)
        self.pos += n
        return t


def parse(shape, weights: np.ndarray):
    w = torch.from_numpy(np.asarray(weights, dtype=np.float32).astype(np.float64))
    d, Fd, V, L = shape.d_model, shape.d_ff, shape.vocab, shape.n_layer
    r = _Reader(w)
    p = {"wte": r.take(V, d), "wpe": r.take(shape.n_pos, d), "blocks": []}
    for _ in range(L):
        b = {}
        b["ln1_g"], b["ln1_b"] = r.take(d), r.take(d)
        b["w_qkv"], b["b_qkv"] = r.take(d, 3 * d), r.take(3 * d)
        b["w_o"], b["b_o"] = r.take(d, d), r.take(d)
        b["ln2_g"], b["ln2_b"] = r.take(d), r.take(d)
        b["w_fc"], b["b_fc"] = r.take(d, Fd), r.take(Fd)
        b["w_p"], b["b_p"] = r.take(Fd, d), r.take(d)
        p["blocks"].append(b)
    p["lnf_g"], p["lnf_b"] = r.take(d), r.take(d)
    assert r.pos == w.numel()
    return p


def forward(shape, weights, tokens, params=None):
    """Returns (logits[n][V], keys[L][n][d], values[L][n][d]) in float64."""
    p = params if params is not None else parse(shape, weights)
    d, H = shape.d_model, shape.n_head
    dh = d // H
    toks = torch.as_tensor(np.asarray(tokens, dtype=np.int64))
    n = toks.numel()
    x = p["wte"][toks] + p["wpe"][torch.arange(n)]
    keys, values = [], []
    for b in p["blocks"]:
        a = F.layer_norm(x, (d,), b["ln1_g"], b["ln1_b"], eps=1e-5)
        qkv = a @ b["w_qkv"] + b["b_qkv"]
        q, k, v = qkv.split(d, dim=-1)
        keys.append(k)
        values.append(v)
        heads = lambda t: t.reshape(n, H, dh).transpose(0, 1)
        o = F.scaled_dot_product_attention(heads(q), heads(k), heads(v), is_causal=True)
        x = x + o.transpose(0, 1).reshape(n, d) @ b["w_o"] + b["b_o"]
        a = F.layer_norm(x, (d,), b["ln2_g"], b["ln2_b"], eps=1e-5)
        u = F.gelu(a @ b["w_fc"] + b["b_fc"], approximate="tanh")
        x = x + u @ b["w_p"] + b["b_p"]
    xf = F.layer_norm(x, (d,), p["lnf_g"], p["lnf_b"], eps=1e-5)
    logits = xf @ p["wte"].T
    return logits.numpy(), torch.stack(keys).numpy(), torch.stack(values).numpy()
