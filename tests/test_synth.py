"""The seeded input generators (CPU only).  Both the oracle and the CUDA path
take their inputs from these, so they are pinned to their published
definitions and to the checkpoint layout."""
import numpy as np

from stream_decode_gb300 import synth

S = synth.GPT2_TINY


def test_splitmix64_reference_outputs():
    # the first outputs of SplitMix64 for seed 1234567 (Steele, Lea and
    # Flood's generator as published with its reference implementation)
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
            16408922859458223821]
    assert [int(x) for x in synth.splitmix64(1234567, 0, 5)] == want
    # counter-based: any window of the stream is the same draws
    assert np.array_equal(synth.splitmix64(99, 3, 4), synth.splitmix64(99, 0, 7)[3:])


def test_normals_windows_and_moments():
    a = synth.normals(7, 0, 11)
    for start, count in ((0, 11), (1, 5), (4, 7), (3, 1)):
        assert np.array_equal(synth.normals(7, start, count), a[start:start + count])
    z = synth.normals(11, 0, 400_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert abs(((z ** 4).mean()) - 3.0) < 0.05  # Gaussian fourth moment


def test_tokens_uniform_in_range():
    t = synth.tokens(50257, 200_000, seed=3)
    assert t.min() >= 0 and t.max() < 50257
    edges = np.arange(0, 50257 + 5026, 5026)  # ten bins of 5,026 ids (the last 5,023)
    counts, _ = np.histogram(t, bins=np.minimum(edges, 50257))
    expect = 200_000 * np.diff(np.minimum(edges, 50257)) / 50257
    assert (np.abs(counts - expect) < 0.05 * expect).all()


def test_checkpoint_variants_follow_the_layout():
    lay = synth.layout(S)
    assert lay["_words"] == synth.weight_words(S)
    plain = synth.checkpoint(S, synth.SEED_TINY)
    assert np.array_equal(plain, synth.checkpoint(S, synth.SEED_TINY, block=1000))  # block-size independent
    variants = {v: synth.checkpoint(S, synth.SEED_TINY, v) for v in ("rich", "zero_blocks", "outlier_channels")}
    big = {0, S.d_model // 4 + 1, S.d_model // 2 + 2, 3 * S.d_model // 4 + 3}
    for name, (o, n) in ((k, v) for k, v in lay.items() if k != "_words"):
        base = name.split(".")[-1]
        p = plain[o:o + n]
        if base.endswith("_g"):
            assert (p == 1.0).all()
            og = variants["outlier_channels"][o:o + n]
            assert set(np.nonzero(og != 1.0)[0].tolist()) == big and (og[list(big)] == 20.0).all()
            assert abs(variants["rich"][o:o + n].std() - 0.1) < 0.05
        elif base.startswith("b_") or base.endswith("_b"):
            assert (p == 0.0).all() and (variants["zero_blocks"][o:o + n] == 0.0).all()
            assert (variants["rich"][o:o + n] != 0.0).all()
        else:  # wte, wpe and the block matrices ~ N(0, 0.02)
            assert abs(p.std() - 0.02) < 0.002
            assert np.array_equal(variants["outlier_channels"][o:o + n], p)
            zb = variants["zero_blocks"][o:o + n]
            assert (zb == 0.0).all() if base.startswith("w_") else np.array_equal(zb, p)


def test_cache_shape_and_scale():
    c = synth.cache(S, 5, seed=1)
    assert c.dtype == np.float32 and c.size == 5 * S.n_layer * 2 * S.d_model
    assert abs(c.std() - 0.5) < 0.05


def test_offset_residual_variant_is_rich_plus_the_stated_offsets():
    lay = synth.layout(S)
    rich = synth.checkpoint(S, synth.SEED_TINY, "rich")
    off = synth.checkpoint(S, synth.SEED_TINY, "offset_residual")
    d = S.d_model
    diff = (off.astype(np.float64) - rich.astype(np.float64))
    o, n = lay["wpe"]
    wd = diff[o:o + n].reshape(S.n_pos, d)
    big = [5, d // 3 + 7, 2 * d // 3 + 11]
    assert np.allclose(wd[:, big], 100.0, atol=1e-3)
    assert np.allclose(np.delete(wd, big, axis=1), 3.0, atol=1e-5)
    for l in range(S.n_layer):
        o, n = lay[f"h{l}.b_o"]
        assert np.allclose(diff[o:o + n], 0.25, atol=1e-6)
    o, n = lay["h0.b_p"]
    bp = diff[o:o + n]
    assert abs(bp[d // 2] - 100.0) < 1e-3 and (np.delete(bp, d // 2) == 0.0).all()
    touched = np.zeros(off.size, bool)
    for name in ["wpe", "h0.b_p"] + [f"h{l}.b_o" for l in range(S.n_layer)]:
        o, n = lay[name]
        touched[o:o + n] = True
    assert (diff[~touched] == 0.0).all()
