import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on CPU")


@pytest.fixture(scope="session")
def oracle():
    from oracle import Oracle
    return Oracle()


@pytest.fixture(scope="session")
def tiny():
    from stream_decode_gb300 import synth
    return synth.GPT2_TINY


@pytest.fixture(scope="session")
def tiny_plain():
    from stream_decode_gb300 import synth
    return synth.checkpoint(synth.GPT2_TINY, synth.SEED_TINY, "plain")


@pytest.fixture(scope="session")
def tiny_rich():
    from stream_decode_gb300 import synth
    return synth.checkpoint(synth.GPT2_TINY, synth.SEED_TINY, "rich")


@pytest.fixture(scope="session")
def w124m():
    from stream_decode_gb300 import synth
    return synth.checkpoint(synth.GPT2_124M, synth.SEED_124M, "plain")


@pytest.fixture(scope="session")
def w124m_rich():
    from stream_decode_gb300 import synth
    return synth.checkpoint(synth.GPT2_124M, synth.SEED_124M, "rich")
