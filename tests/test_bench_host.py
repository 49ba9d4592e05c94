"""Host-side pieces of bench.py (CPU only): the algorithmic byte counts
behind the roofline, checked against the packed-checkpoint layout tensor
by tensor, and the lookup of the recorded DRAM traffic."""
import json
import os

import bench
from stream_decode_gb300 import synth

S = synth.GPT2_124M
KV_ROW = 12 * 1536 * 4  # one cached position (README cachedStep paragraph)


def _layout_bytes(per_word_matrix, row_bytes_q8=None):
    """Bytes of one step's weights from the checkpoint layout: matrices at
    per_word_matrix bytes a weight (or int8 rows), wpe one row, the rest
    binary32."""
    lay = synth.layout(S)
    total = 0
    for name, v in lay.items():
        if name == "_words":
            continue
        _, n = v
        base = name.split(".")[-1]
        if name == "wpe":
            total += 4 * S.d_model
        elif name == "wte" or base.startswith("w_"):
            if row_bytes_q8 is None:
                total += per_word_matrix * n
            else:
                k = S.d_ff if base == "w_p" else S.d_model
                total += (n // k) * row_bytes_q8(k)
        else:
            total += 4 * n
    return total


def test_f32_step_bytes_are_every_used_checkpoint_word():
    # every packed word except the 1023 wpe rows a step does not read
    words = synth.weight_words(S) - (S.n_pos - 1) * S.d_model
    assert words * 4 == 494_616_576
    assert bench.step_bytes(S, "f32", 0) == words * 4 + KV_ROW + 4 * S.vocab
    assert _layout_bytes(4) == words * 4


def test_step_bytes_grow_by_one_cached_position():
    for q in ("f32", "f16", "int8", "int8_row"):
        assert bench.step_bytes(S, q, 101) - bench.step_bytes(S, q, 100) == KV_ROW


def test_reduced_formats_from_the_layout():
    tail = KV_ROW + 4 * S.vocab
    assert bench.step_bytes(S, "f16", 0) == _layout_bytes(2) + tail
    assert bench.step_bytes(S, "int8", 0) == _layout_bytes(None, lambda k: k + (k // 64) * 4) + tail
    assert bench.step_bytes(S, "int8_row", 0) == _layout_bytes(None, lambda k: k + 4) + tail


def test_traffic_record_lookup():
    path = os.path.join(bench.ROOT, "profiles", "step_kernel_traffic.json")
    with open(path) as f:
        rec = json.load(f)
    for q, e in rec.items():
        assert e["dram_bytes_per_launch_112_steps"] == e["dram_bytes_read"] + e["dram_bytes_write"]
        assert bench.traffic_from_profiles(e["kernel_sha256"], q) == e["dram_bytes_per_launch_112_steps"]
        assert bench.traffic_from_profiles("0" * 64, q) is None


def test_byte_components_match_the_printed_sizes():
    """The parts of the bench's byte count against the sizes the gpt2.s page
    prints for the same tensors (MB = 10^6 bytes, matched to the printed digits)."""
    with open(os.path.join(bench.ROOT, "tests", "golden", "page_identities.json")) as f:
        g = json.load(f)
    d, F, L, V = S.d_model, S.d_ff, S.n_layer, S.vocab
    blocks = 4 * L * (d * 3 * d + d * d + d * F + F * d)
    assert round(blocks / 1e6) == g["block_matrices_mb"]["value"]
    padded = (V + 63) // 64 * 64  # the vocabulary padded to whole 64-row tiles
    assert padded == g["wte_padded_rows"]["value"]
    assert int(4 * padded * d / 1e6) == g["wte_tiled_mb"]["value"]
    assert int(S.n_pos * KV_ROW / 1e6) == g["kv_cache_mb_1024"]["value"]
    # the f32 step reads exactly these blocks plus the unpadded wte and the small tensors
    small = bench.step_bytes(S, "f32", 0) - blocks - 4 * V * d - KV_ROW - 4 * V
    assert small == 4 * (L * (9 * d + F) + 2 * d + d)  # LN, biases, final LN, one wpe row
