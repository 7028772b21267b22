"""The debug-checks build over the tiny shape sweeps.

The same sources compiled with -DALIBI_CHECKS test every TMA coordinate, TMEM
address and shared-memory operand of the tensor-core kernels before use and
record any bad one in the device status word (alibi_check_error then returns
ALIBI_ERR_CHECK). This stands in for the memory checker, which is not available
here: the parity tests of the shape sweeps (ragged sizes, every head size, both
masks, the mitigations, skipping, the backward) run in a child process with that
library loaded, and every call must come back with a clean status word and the
same results as the oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

SWEEPS = [
    "test_gpu_prefill.py::test_prefill_shape_sweep",
    "test_gpu_prefill.py::test_prefill_small_head_sizes",
    "test_gpu_prefill.py::test_prefill_small_head_skip_is_bit_identical",
    "test_gpu_prefill.py::test_lazy_rescale_with_divergent_rows",
    "test_gpu_noncausal.py::test_noncausal_shape_sweep",
    "test_gpu_noncausal.py::test_noncausal_mitigations",
    "test_gpu_variants.py::test_mitigation_variants",
    "test_gpu_skip.py::test_skip_is_bit_identical",
    "test_gpu_bwd.py::test_bwd_bf16_vs_oracle",
    "test_gpu_bwd.py::test_bwd_mitigations",
    "test_gpu_bwd.py::test_bwd_deterministic",
]


def test_checks_build_passes_the_shape_sweeps():
    from alibi_positional_bias_gb300 import _build
    lib = _build.build(checks=True)
    env = dict(os.environ, ALIBI_CHECKS="1")
    # the child loads the checks library, not the default one
    probe = subprocess.run(
        [sys.executable, "-c",
         "import alibi_positional_bias_gb300 as ab; ab.load(); print(ab.lib_path())"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr
    assert probe.stdout.strip() == lib
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        *[os.path.join(HERE, s) for s in SWEEPS]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    summary = [ln for ln in r.stdout.splitlines() if " passed" in ln][-1]
    assert int(summary.split(" passed")[0].split()[-1]) >= 88, summary  # every case of the selection ran
