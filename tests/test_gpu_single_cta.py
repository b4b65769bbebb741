"""The alternative kernels pass the same parity tests as the defaults.

engram_kernel_options selects them: the single-CTA bf16 kernels at every
size (projection_cta = 1), the CTA-pair bf16 kernels at every size (= 2; by
default batches of at most 128 tokens take the single-CTA kernel), the
CTA-pair block-FP8 kernels (fp8_pair), the fused block-FP8 kernels
(fp8_fused; by default the FP8 gate runs as a separate kernel), the TMA
bulk-copy gather (gather_copy = 1) and the fused projection launched without
the cooperative attribute (plain_launch, the mode profilers need).

Each case reruns a parity test file in a child process with the options set
for the whole run (--kernel-options), so the defaults stay in force here.
"""
import os
import subprocess
import sys

import pytest

from gpu_util import require_gpu

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("options,test_file", [
    ("projection_cta=1", "test_gpu_project.py"),
    ("projection_cta=2", "test_gpu_project.py"),
    ("fp8_pair=1", "test_gpu_fp8.py"),
    ("fp8_fused=1,fp8_pair=0", "test_gpu_fp8.py"),
    ("fp8_fused=1,fp8_pair=1", "test_gpu_fp8.py"),
    ("gather_copy=1", "test_gpu_gather.py"),
    ("plain_launch=1", "test_gpu_project.py"),
])
def test_alternative_kernels_pass_parity(options, test_file):
    require_gpu()
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, test_file), "-m", "gpu", "-q",
                        "-p", "no:cacheprovider", f"--kernel-options={options}"],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
