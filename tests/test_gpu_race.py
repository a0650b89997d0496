"""Race check of the decode kernel's copy/compute overlap.

The decode kernel computes on a warp's ring stages while TMA copies into the
other stages are in flight, and reuses a stage as soon as a step has read
it.  A missing wait or a stage reused too early would let a copy overwrite
data still being read, or a step read data not yet landed.  A verification
build (OSCAR_SERIAL_COPIES=1) waits for every copy right after issuing it, so
nothing overlaps; with every sum in a fixed order, both builds must give the
same output bit for bit on a workload that refills every ring many times.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import harness as H

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

SCRIPT = r'''
import sys, numpy as np
sys.path.insert(0, %r)
sys.path.insert(0, %r)
import harness as H
sc = H.Scenario(1002, [100_000], n_kv=8, g=4, cal=(1024, 512))
cache, q = H.to_device(sc)
out, status = H.run_decode(cache, q)
assert status == 0, status
np.save(%r, out)
'''


@pytest.fixture(scope="module", autouse=True)
def _cuda(built_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_serial_copy_build_gives_bit_identical_output(tmp_path):
    from bit_rotated_kv_split_gb300 import build as _b
    lib = _b.build_variant(str(tmp_path / "liboscar_serial.so"), ["OSCAR_SERIAL_COPIES=1"], str(tmp_path / "obj"))
    path = str(tmp_path / "serial.npy")
    env = dict(os.environ, OSCAR_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", SCRIPT % (HERE, ROOT, path)], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    serial = np.load(path)
    sc = H.Scenario(1002, [100_000], n_kv=8, g=4, cal=(1024, 512))
    cache, q = H.to_device(sc)
    out, status = H.run_decode(cache, q)
    assert status == 0
    np.testing.assert_array_equal(out, serial)
