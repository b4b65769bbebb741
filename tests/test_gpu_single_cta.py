"""The alternative projection kernels pass the same parity tests as the
defaults: the single-CTA bf16 kernels at every size (ENGRAM_SINGLE_CTA_MMA=1),
the CTA-pair bf16 kernels at every size (=0; by default batches of at most
128 tokens take the single-CTA kernel), the CTA-pair block-FP8 kernels
(ENGRAM_FP8_PAIR=1), the fused block-FP8 kernels (ENGRAM_FP8_FUSED=1; by
default the FP8 gate runs as a separate kernel), the TMA bulk-copy gather
(ENGRAM_GATHER=bulk) and the fused projection launched without the
cooperative attribute (ENGRAM_COOPERATIVE=0, the mode profilers need).

The selection is read once per process, so the tests run in a child process.
"""
import os
import subprocess
import sys

import pytest

from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


def test_single_cta_kernels_pass_projection_parity():
    require_gpu()
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, ENGRAM_SINGLE_CTA_MMA="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(here, "test_gpu_project.py"), "-m", "gpu", "-q",
                        "-p", "no:cacheprovider"], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


def test_fp8_pair_kernels_pass_fp8_parity():
    require_gpu()
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, ENGRAM_FP8_PAIR="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(here, "test_gpu_fp8.py"), "-m", "gpu", "-q",
                        "-p", "no:cacheprovider"], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]



def test_pair_kernels_at_every_size_pass_projection_parity():
    require_gpu()
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, ENGRAM_SINGLE_CTA_MMA="0")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(here, "test_gpu_project.py"), "-m", "gpu", "-q",
                        "-p", "no:cacheprovider"], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


@pytest.mark.parametrize("pair", ["0", "1"])
def test_fused_fp8_kernels_pass_fp8_parity(pair):
    require_gpu()
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, ENGRAM_FP8_FUSED="1", ENGRAM_FP8_PAIR=pair)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(here, "test_gpu_fp8.py"), "-m", "gpu", "-q",
                        "-p", "no:cacheprovider"], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


@pytest.mark.parametrize("env_var,value,test_file", [("ENGRAM_GATHER", "bulk", "test_gpu_gather.py"),
                                                     ("ENGRAM_COOPERATIVE", "0", "test_gpu_project.py")])
def test_alternative_launch_modes_pass_parity(env_var, value, test_file):
    require_gpu()
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, **{env_var: value})
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(here, test_file), "-m", "gpu", "-q",
                        "-p", "no:cacheprovider"], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
