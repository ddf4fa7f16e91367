import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def published_decode_ref(oracle_mod):
    """Oracle output of a whole published decode batch ("70b", "shared"), computed once
    per session: the batch is drawn on the GPU (its generator fixes the values), the
    oracle runs on host copies after the step's append."""
    import torch

    import synth
    from tests.helpers import oracle_decode_case
    cache = {}

    def get(name):
        if name not in cache:
            case = synth.build_case(name, "cuda")
            cache[name], _, _ = oracle_decode_case(oracle_mod, case)
            del case
            torch.cuda.empty_cache()
        return cache[name]
    return get
