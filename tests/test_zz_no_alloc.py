"""gpt2_cached_step_noalloc: the cached step for callers that may not
allocate device memory while stepping (their host framework owns every
device allocation, or the loop cannot afford cudaMalloc's device-wide
synchronisation).  Its scratch lives in a static device array inside the
library; the caller passes the model, its own KV cache and output buffers.

The check: several calls in a row through the C ABI give the same logits,
greedy choices and cache as the session entry point (gpt2_session_step): bit
for bit, since both run the same kernel on the same grid in the same order.
After the first call, further calls leave the device's free memory
unchanged: stepping allocates nothing.  This file is collected last so that
a failure here comes after every other test has run; it also passes alone in
a fresh process.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from stream_decode_gb300 import synth  # noqa: E402


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from stream_decode_gb300 import gpt2
    return gpt2


@pytest.fixture(params=["phase", "cluster"])
def kernel(request, monkeypatch):
    """Runs a binary32 / binary16 test on each step kernel (the variable is
    read when a model is created)."""
    monkeypatch.setenv("GPT2_STEP_KERNEL", request.param)
    return request.param


def _compare(g, shape, w, quant, n_calls=4):
    model = g.Model(shape, w, quant=quant)
    V, row = shape.vocab, g.cache_words_per_position(shape)
    toks = [int(t) for t in synth.tokens(V, n_calls, seed=77)]

    # existing entry point: a session, one gpt2_session_step per position
    sess = g.Session(model)
    ref_logits, ref_next = [], []
    d_logits = torch.empty(V, dtype=torch.float32, device="cuda")
    d_next = torch.empty(1, dtype=torch.int32, device="cuda")
    for t in toks:
        assert sess.step(t, d_logits, d_next) == "ok"
        assert sess.sync() == "ok"
        ref_logits.append(d_logits.cpu().numpy().copy())
        ref_next.append(int(d_next.item()) & 0xFFFFFFFF)
    ref_cache = sess.read_cache()

    # the no-allocation entry point, caller-owned buffers, calls in a row
    cache = torch.zeros(shape.max_pos * row, dtype=torch.float32, device="cuda")
    out = torch.empty(V, dtype=torch.float32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    got_all = torch.empty(n_calls, V, dtype=torch.float32, device="cuda")
    nxt_all = torch.empty(n_calls, dtype=torch.int32, device="cuda")
    free_after_first = None
    for p, t in enumerate(toks):
        out.fill_(float("nan"))
        assert model.cached_step_noalloc(cache, p, t, out, nxt) == "ok"
        got_all[p].copy_(out)
        nxt_all[p].copy_(nxt[0])
        if p == 0:
            torch.cuda.synchronize()
            free_after_first = torch.cuda.mem_get_info()[0]
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_after_first, "steady-state calls allocated device memory"
    got = got_all.cpu().numpy()
    for p in range(n_calls):
        assert np.array_equal(got[p].view(np.uint32), ref_logits[p].view(np.uint32)), f"call {p}"
        assert (int(nxt_all[p].item()) & 0xFFFFFFFF) == ref_next[p], f"call {p}"
    got_cache = cache[:n_calls * row].cpu().numpy()
    assert np.array_equal(got_cache.view(np.uint32), ref_cache.view(np.uint32))
    sess.close()
    model.close()


def test_noalloc_matches_session_step_tiny(g, kernel):
    shape = synth.GPT2_TINY
    _compare(g, shape, synth.checkpoint(shape, synth.SEED_TINY, "rich"), g.F32)


def test_noalloc_matches_session_step_124m(g, w124m, kernel):
    _compare(g, synth.GPT2_124M, w124m, g.F32, n_calls=3)


@pytest.mark.parametrize("fmt", ["INT8_G64", "F16", "INT8_ROW", "INT8_ROW_ACT"])
def test_noalloc_matches_session_step_other_formats(g, fmt):
    shape = synth.GPT2_TINY
    _compare(g, shape, synth.checkpoint(shape, synth.SEED_TINY, "rich"), getattr(g, fmt))


def test_noalloc_rejects_bad_arguments(g):
    shape = synth.GPT2_TINY
    model = g.Model(shape, synth.checkpoint(shape, synth.SEED_TINY))
    row = g.cache_words_per_position(shape)
    cache = torch.zeros(shape.max_pos * row, dtype=torch.float32, device="cuda")
    assert model.cached_step_noalloc(cache, 0, g.GREEDY) == "token"
    assert model.cached_step_noalloc(cache, 0, shape.vocab) == "token"
    assert model.cached_step_noalloc(cache, shape.max_pos, 1) == "position"
    assert g.STATUS[g.lib.gpt2_cached_step_noalloc(model.h, None, 0, 1, None, None, None)] == "arg"
    model.close()
