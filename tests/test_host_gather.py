"""The host-side row gather (native, OpenMP) on CPU: bytes and bad-row handling."""
import numpy as np
import pytest

import hashed_gram_conditional_gb300 as eg
from workloads import ROW_BYTES, table_rows


@pytest.fixture(scope="module")
def lib():
    import os
    if not os.path.exists(eg.library_path()):
        from hashed_gram_conditional_gb300 import build
        build.build()
    return eg.lib()


@pytest.mark.parametrize("threads", [0, 1, 5])
def test_host_gather_copies_rows(lib, threads):
    n = 20_000
    table = table_rows(11, np.arange(n)).reshape(-1)
    rng = np.random.default_rng(threads)
    ids = rng.integers(0, n, size=24 * 333).astype(np.int32)
    ids[[5, 77, 1000]] = [n, -1, 2 ** 30]
    staging = np.empty(len(ids) * ROW_BYTES, dtype=np.uint8)
    bad = eg.engram_host_gather(table, n, ids, staging, threads)
    assert bad == 3
    got = staging.reshape(len(ids), ROW_BYTES)
    good = (ids >= 0) & (ids < n)
    assert (got[good] == table.reshape(n, ROW_BYTES)[ids[good]]).all()
    assert (got[~good] == 0).all()


def test_host_gather_empty_and_errors(lib):
    assert eg.engram_host_gather(np.zeros(ROW_BYTES, np.uint8), 1, np.zeros(0, np.int32),
                                 np.zeros(0, np.uint8)) == 0
    assert lib.engram_host_gather(None, 1, None, 5, None, 0, None) == -1
