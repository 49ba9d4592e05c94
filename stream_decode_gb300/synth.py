"""Seeded synthetic inputs: packed GPT-2 checkpoints and token ids.

This module only draws numbers and places them in the packed binary32
checkpoint format; it holds none of the model's arithmetic.  Both the CUDA
path and the CPU oracle are fed the bytes it produces.

Random source: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used counter-style: draw i of a stream seeded
with ``seed`` is ``mix64(seed + (i + 1) * 0x9E3779B97F4A7C15)``.  Normal
deviates come from the Box-Muller transform in float64 on pairs of draws,
then are scaled and rounded once to binary32.

Checkpoint format (LeanExe GPT-2 README, packed checkpoint paragraph): little-
endian binary32 words in the order token embeddings ``wte[vocab][d]``, all
stored position rows ``wpe[n_pos][d]``, the blocks, then the final
normalization ``lnf_g[d], lnf_b[d]``.  Inside a block the order is the
Hugging Face GPT-2 state-dict order with Conv1D ``[in][out]`` matrices
(gpt2.s page, weight-layout paragraph): ``ln1_g, ln1_b, W_qkv[d][3d],
b_qkv[3d], W_o[d][d], b_o[d], ln2_g, ln2_b, W_fc[d][F], b_fc[F], W_p[F][d],
b_p[d]``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
SEED_124M = 0x5EED0124
SEED_TINY = 0x5EED0001
SEED_TOKENS = 42


@dataclass(frozen=True)
class Shape:
    """Model dimensions; ``max_pos`` is the largest accepted position + 1."""

    n_layer: int
    d_model: int
    n_head: int
    d_ff: int
    vocab: int
    n_pos: int
    max_pos: int

    def as_tuple(self):
        return (self.n_layer, self.d_model, self.n_head, self.d_ff,
                self.vocab, self.n_pos, self.max_pos)


# GPT-2 124M (LeanExe GPT-2 README, first paragraph); positions 0..127 accepted.
GPT2_124M = Shape(12, 768, 12, 3072, 50257, 1024, 128)
# Same weights, with every one of the 1024 stored position rows accepted.
GPT2_124M_LONG = Shape(12, 768, 12, 3072, 50257, 1024, 1024)
# Tiny pre-LN GPT-2 used for parity at oracle speed.
GPT2_TINY = Shape(2, 64, 4, 256, 512, 16, 16)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= np.uint64(0xBF58476D1CE4E5B9)
    z ^= z >> np.uint64(27)
    z *= np.uint64(0x94D049BB133111EB)
    z ^= z >> np.uint64(31)
    return z


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the SplitMix64 stream for ``seed``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN
    return _mix64(z)


def normals(seed: int, start: int, count: int) -> np.ndarray:
    """Standard normal deviates ``start .. start+count-1`` (float64).

    Deviate ``2k`` is the cosine branch and ``2k+1`` the sine branch of the
    Box-Muller transform of draws ``2k`` and ``2k+1``.
    """
    k0 = start // 2
    k1 = (start + count + 1) // 2
    r = splitmix64(seed, 2 * k0, 2 * (k1 - k0))
    u = ((r >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * np.pi * u2
    z = np.empty(2 * (k1 - k0), dtype=np.float64)
    z[0::2] = rad * np.cos(ang)
    z[1::2] = rad * np.sin(ang)
    off = start - 2 * k0
    return z[off:off + count]


def layout(s: Shape) -> dict:
    """Word offsets of every tensor in the packed checkpoint, and its size."""
    d, F = s.d_model, s.d_ff
    off = {}
    pos = 0

    def put(name, n):
        nonlocal pos
        off[name] = (pos, n)
        pos += n

    put("wte", s.vocab * d)
    put("wpe", s.n_pos * d)
    for l in range(s.n_layer):
        put(f"h{l}.ln1_g", d)
        put(f"h{l}.ln1_b", d)
        put(f"h{l}.w_qkv", d * 3 * d)
        put(f"h{l}.b_qkv", 3 * d)
        put(f"h{l}.w_o", d * d)
        put(f"h{l}.b_o", d)
        put(f"h{l}.ln2_g", d)
        put(f"h{l}.ln2_b", d)
        put(f"h{l}.w_fc", d * F)
        put(f"h{l}.b_fc", F)
        put(f"h{l}.w_p", F * d)
        put(f"h{l}.b_p", d)
    put("lnf_g", d)
    put("lnf_b", d)
    off["_words"] = pos
    return off


def weight_words(s: Shape) -> int:
    return layout(s)["_words"]


def checkpoint(s: Shape, seed: int, variant: str = "plain", block: int = 1 << 23) -> np.ndarray:
    """Packed checkpoint as a float32 array (little-endian on every host here).

    ``plain``: every matrix, wte and wpe ~ N(0, 0.02); LayerNorm gains 1,
    LayerNorm shifts and all biases 0.
    ``rich``: as plain, but biases and LayerNorm shifts ~ N(0, 0.02) and
    LayerNorm gains 1 + N(0, 0.1), so a dropped bias or gain shows up.
    ``zero_blocks``: as plain, but every block matrix and bias is zero, so
    each block is the identity map on the residual stream.
    ``outlier_channels``: as plain, but in every LayerNorm 4 fixed channels
    (0, d/4 + 1, d/2 + 2, 3d/4 + 3) have gain 20, so every normalised
    projection input carries a few coordinates about 20 times larger than
    the rest (the shape of the large-magnitude activation channels of
    trained GPT-2 models; used by the int8 scale-granularity ablation).
    ``offset_residual``: as rich, plus a residual stream that is hard on
    LayerNorm arithmetic: three fixed channels (5, d/3 + 7, 2d/3 + 11) of
    every wpe row are raised by 100 and every other wpe word by 3 (a nonzero
    residual mean), every block's b_o by 0.25 (the mean drifts from layer to
    layer) and channel d/2 of block 0's b_p by 100.  A variance formed as
    E[x^2] - mean^2, or a LayerNorm folded without removing the common
    offset first, loses most of its bits on such a stream.  wte (the tied
    vocabulary matrix) is left as in rich, so the logits keep the magnitude
    at which a binary32 tolerance of 2e-3 is meaningful.
    """
    if variant not in ("plain", "rich", "zero_blocks", "outlier_channels", "offset_residual"):
        raise ValueError(variant)
    if variant == "offset_residual":
        out = checkpoint(s, seed, "rich", block)
        lay = layout(s)
        d = s.d_model
        o, n = lay["wpe"]
        wpe = out[o:o + n].reshape(s.n_pos, d)
        wpe += np.float32(3.0)
        for ch in (5, d // 3 + 7, 2 * d // 3 + 11):
            wpe[:, ch] += np.float32(97.0)
        for l in range(s.n_layer):
            o, n = lay[f"h{l}.b_o"]
            out[o:o + n] += np.float32(0.25)
        o, n = lay["h0.b_p"]
        out[o + d // 2] += np.float32(100.0)
        return out
    lay = layout(s)
    n = lay["_words"]
    out = np.empty(n, dtype=np.float32)
    for b0 in range(0, n, block):
        cnt = min(block, n - b0)
        out[b0:b0 + cnt] = (0.02 * normals(seed, b0, cnt)).astype(np.float32)
    for name, val in lay.items():
        if name == "_words":
            continue
        o, cnt = val
        base = name.split(".")[-1]
        if base.endswith("_g"):  # LayerNorm gains
            if variant == "rich":
                out[o:o + cnt] = (1.0 + 0.1 * normals(seed ^ 0xA5A5, o, cnt)).astype(np.float32)
            else:
                out[o:o + cnt] = 1.0
                if variant == "outlier_channels":
                    for c in (0, cnt // 4 + 1, cnt // 2 + 2, 3 * cnt // 4 + 3):
                        out[o + c] = 20.0
        elif base.endswith("_b") and base.startswith("ln") or base.startswith("b_"):
            if variant != "rich":
                out[o:o + cnt] = 0.0
        elif base.startswith("w_") and variant == "zero_blocks":
            out[o:o + cnt] = 0.0
    return out


def tokens(vocab: int, count: int, seed: int = SEED_TOKENS, start: int = 0) -> np.ndarray:
    """Uniform token ids in [0, vocab): ``((draw >> 32) * vocab) >> 32``."""
    r = splitmix64(seed, start, count)
    t = ((r >> np.uint64(32)) * np.uint64(vocab)) >> np.uint64(32)
    return t.astype(np.uint32)


def uniform_f32(seed: int, count: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """Uniform float32 values in [lo, hi) for kernel-level parity inputs."""
    r = splitmix64(seed, 0, count)
    u = (r >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return (lo + (hi - lo) * u).astype(np.float32)


def cache(s: Shape, positions: int, seed: int, scale: float = 0.5) -> np.ndarray:
    """A KV cache of `positions` positions in the boundary layout (word
    (source*n_layer + layer)*2*d + offset), every word ~ N(0, scale^2): the
    magnitude of keys and values that N(0, 0.02) weights produce from a
    LayerNorm output (sqrt(768) * 0.02 ~ 0.55)."""
    n = positions * s.n_layer * 2 * s.d_model
    return (scale * normals(seed, 0, n)).astype(np.float32)
