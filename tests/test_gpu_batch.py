"""GPU parity of batched independent sessions (gpt2_batch_*): every session
of a batch against the oracle's own cached steps for that session alone.

Each session b starts from a seeded synthetic cache of p0_b positions (its
own length), takes a seeded first token and then the oracle's greedy
choices; the batch is fed the oracle's token sequences (teacher forcing:
every logit, choice and cache row is compared), and separately runs
greedily on the device from the same first tokens."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import AGREE_MIN, LOGIT_TOL, disagreements_are_near_ties, greedy_agreement  # noqa: E402
from stream_decode_gb300 import synth  # noqa: E402

import oracle_pins as P  # noqa: E402

GREEDY = 0xFFFFFFFF
# vocabulary not a multiple of the GEMM's 64-column tiles
RAGGED = synth.Shape(n_layer=2, d_model=64, n_head=4, d_ff=256, vocab=600, n_pos=16, max_pos=16)


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from stream_decode_gb300 import gpt2
    return gpt2


def _oracle_sessions(oracle, shape, w, B, n_steps, p0s, seed):
    """Per session: (cache_in, tokens fed, oracle logits [n][V], choices, cache_out)."""
    om = oracle.model(shape, w)
    out = []
    first = synth.tokens(shape.vocab, B, seed=seed)
    for b in range(B):
        c0 = synth.cache(shape, p0s[b], seed=seed + 17 * b)
        lg, ch, cache = om.session([int(first[b])] + [-1] * (n_steps - 1), n_steps, p0=p0s[b], cache=c0)
        fed = np.concatenate([[first[b]], ch[:-1]]).astype(np.int64)
        out.append((c0, fed, lg, ch, cache))
    om.close()
    return out


def _check_batch(g, oracle, shape, w, B, n_steps, p0s, seed=900):
    ref = _oracle_sessions(oracle, shape, w, B, n_steps, p0s, seed)
    model = g.Model(shape, w)
    bt = g.Batch(model, B)
    assert bt.size == B
    for b in range(B):
        assert bt.load_cache(b, ref[b][0]) == "ok" and bt.position(b) == p0s[b]
    V = shape.vocab
    toks = np.stack([r[1] for r in ref], axis=1).astype(np.uint32)  # [n_steps][B]
    d_in = torch.tensor(toks.view(np.int32), device="cuda")
    d_lg = torch.full((n_steps, B, V), float("nan"), device="cuda")
    d_out = torch.zeros((n_steps, B), dtype=torch.int32, device="cuda")
    assert bt.run(d_in, n_steps, d_lg, B * V, d_out) == "ok"
    assert bt.sync() == "ok"
    lg = d_lg.cpu().numpy()
    ch = d_out.cpu().numpy().view(np.uint32)
    for b in range(B):
        _, _, rl, rc, rcache = ref[b]
        assert np.abs(lg[:, b] - rl).max() <= LOGIT_TOL, b
        assert greedy_agreement(rl, ch[:, b]) >= AGREE_MIN
        assert disagreements_are_near_ties(rl, ch[:, b], LOGIT_TOL)
        assert bt.position(b) == p0s[b] + n_steps
        cache = bt.read_cache(b)
        assert cache.size == rcache.size and np.abs(cache - rcache).max() <= LOGIT_TOL, b
    # greedy on the device from the same first tokens follows each session's
    # oracle path up to its first near tie
    bt2 = g.Batch(model, B)
    for b in range(B):
        assert bt2.load_cache(b, ref[b][0]) == "ok"
    gt = np.full((n_steps, B), GREEDY, np.uint32)
    gt[0] = toks[0]
    d_gout = torch.zeros((n_steps, B), dtype=torch.int32, device="cuda")
    assert bt2.run(torch.tensor(gt.view(np.int32), device="cuda"), n_steps, None, 0, d_gout) == "ok"
    assert bt2.sync() == "ok"
    gch = d_gout.cpu().numpy().view(np.uint32)
    for b in range(B):
        rl, rc = ref[b][2], ref[b][3]
        d = np.nonzero(gch[:, b] != rc)[0]
        if d.size:
            top2 = np.sort(rl[d[0]])[-2:]
            assert top2[1] - top2[0] <= LOGIT_TOL, f"session {b} left the oracle's path at step {d[0]}"
    bt.close()
    bt2.close()
    model.close()


@pytest.mark.parametrize("B", [1, 3, 37, 130])
def test_tiny_batch(g, oracle, B):
    p0s = [(5 * b) % 9 for b in range(B)]
    _check_batch(g, oracle, synth.GPT2_TINY, synth.checkpoint(synth.GPT2_TINY, synth.SEED_TINY, "rich"), B, 7, p0s)


def test_ragged_vocab_batch(g, oracle):
    _check_batch(g, oracle, RAGGED, synth.checkpoint(RAGGED, 0x5EED0600, "rich"), 5, 8, [0, 1, 4, 7, 8])


def test_small_shape_batch(g, oracle):
    _check_batch(g, oracle, P.SMALL, synth.checkpoint(P.SMALL, P.SEED_SMALL, "rich"), 6, 8, [0, 2, 3, 5, 7, 8])


def test_124m_batch(g, oracle, w124m):
    """GPT-2 124M, 8 sessions at cached lengths 0..112, 16 steps each."""
    p0s = [0, 5, 16, 31, 64, 100, 111, 112]
    _check_batch(g, oracle, synth.GPT2_124M, w124m, len(p0s), 16, p0s)


def test_batch_validation(g):
    s = synth.GPT2_TINY
    w = synth.checkpoint(s, synth.SEED_TINY)
    model = g.Model(s, w)
    with pytest.raises(g.GPT2Error):
        g.Batch(model, 0)
    with pytest.raises(g.GPT2Error):
        g.Batch(model, 257)
    bt = g.Batch(model, 2)
    row = g.cache_words_per_position(s)
    assert bt.load_cache(0, np.zeros(s.max_pos * row, np.float32)) == "cache_len"
    assert bt.load_cache(0, np.zeros(row + 1, np.float32)) == "cache_len"
    assert bt.load_cache(2, np.zeros(row, np.float32)) == "arg"
    assert bt.load_cache(1, np.zeros(10 * row, np.float32)) == "ok"
    d_in = torch.zeros((8, 2), dtype=torch.int32, device="cuda")
    assert bt.run(d_in, 7, None, 0, None) == "position"  # session 1 would pass max_pos
    assert bt.run(d_in, 0, None, 0, None) == "tokens_len"
    d_lg = torch.empty((2, s.vocab), device="cuda")
    assert bt.run(d_in, 1, d_lg, s.vocab, None) == "arg"  # stride below B * vocab
    # a greedy token without a previous choice is reported at sync
    bad = torch.tensor(np.array([[1, GREEDY]], np.uint32).view(np.int32), device="cuda")
    assert bt.run(bad, 1, None, 0, None) == "ok"
    assert bt.sync() == "token"
    # rewind: every session must be at or past the target
    assert bt.rewind(11) == "position"
    assert bt.rewind(0) == "ok" and bt.position(0) == 0 and bt.position(1) == 0
    # an int8 model has no batched path
    mq = g.Model(s, w, quant=g.INT8_G64)
    with pytest.raises(g.GPT2Error):
        g.Batch(mq, 2)
    bt.close()
    mq.close()
    model.close()


def test_124m_long_context_batch(g, oracle, w124m):
    """The long-context configuration (max_pos 1024): three sessions at
    cached lengths 600, 900 and 1020 (seeded synthetic caches), two steps
    each, so the decode attention runs up to 64 passes of 16 keys."""
    _check_batch(g, oracle, synth.GPT2_124M_LONG, w124m, 3, 2, [600, 900, 1020])


@pytest.mark.parametrize("B", [64, 256])
def test_124m_batch_sizes_benched(g, oracle, w124m, B):
    """GPT-2 124M at the batch sizes the benchmark times (64 and 256
    sessions; two 128-row M tiles and four at 256), cached lengths 0..12, 3
    steps each."""
    p0s = [(7 * b) % 13 for b in range(B)]
    _check_batch(g, oracle, synth.GPT2_124M, w124m, B, 3, p0s, seed=1700 + B)
