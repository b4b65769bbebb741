"""Failure detection without a GPU fault: every on-chip wait in the kernels
is bounded, and a wait that runs out records ENGRAM_ST_TIMEOUT and returns.
engram_selftest_wait makes the two kinds of wait run out on purpose (an
mbarrier phase nothing completes, a global counter nothing increments); the
status word reports it and the context stays usable."""
import time

import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import DEV, require_gpu, setup, status

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_runs_out_sets_timeout_and_returns(which):
    st = status()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    eg.engram_selftest_wait(which, st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == eg.ST_TIMEOUT
    assert 0.2 < dt < 30.0, dt          # the budget is 2^31 SM cycles
    # the context is still usable: a library kernel runs and is right
    w, tm, lay_o, lay = setup("tiny")
    x = np.array([0, 1, 2 ** 40 + 7, 2 ** 63 - 1], dtype=np.uint64)
    got = eg.engram_selftest_mod(lay, 0, torch.from_numpy(x.view(np.int64)).to(DEV)).cpu().numpy()
    p = np.array(lay_o.layers[0].primes, dtype=object)
    off = np.array(lay_o.layers[0].offsets, dtype=object)
    want = np.array([[int(v) % int(p[j]) + int(off[j]) for j in range(len(p))] for v in x], dtype=np.int64)
    assert (got == want).all()


def test_invalid_selftest_argument_is_rejected_on_the_host():
    with pytest.raises(eg.EngramError):
        eg.engram_selftest_wait(2, status())
