"""The small GPU cases under the checking build of the library (FLARE_DEBUG).

That build checks, on the device, the place of every TMA tile (token row,
head, batch and a 16-byte-aligned innermost coordinate inside the tensor),
the tile cursors against their shards and every workspace index before the
access; a failed check is reported as FLARE_ERR_DEVICE_CHECK. The canary and
small parity tests run in a child process that loads that build
(FLARE_LIBRARY_VARIANT=debug), so they fail if any check fires. This file
sorts after the other GPU tests (the build takes a minute or two).
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

pytestmark = pytest.mark.gpu


def test_small_cases_pass_under_the_checking_build(cuda_device):
    sys.path.insert(0, ROOT)
    from latent_query_split_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, FLARE_LIBRARY_VARIANT="debug")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_gpu_guards.py"), os.path.join(HERE, "test_gpu_failure.py"),
           os.path.join(HERE, "test_gpu_parity.py"), "-k",
           "not full_size and (guards or tiny or empty or shard or bounded or B1H3M128 or B2H2M64 "
           "or encoder_bwd or decode_bwd)"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
