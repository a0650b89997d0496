"""The OScaR variant on the GPU path: demotion and decode with the
block-diagonal (canalized) rotation, against the float64 oracle.

[CSDN] section 四.2: channels split into groups and rotated within each
group.  The kernels take R as data, so the same calls serve the variant;
these cases check that nothing in them assumes the OSCAR eigenbasis (a dense
R).  Bars as in the other parity tests: the code rule of harness.code_parity
and max|o - o_ref| / max|o_ref| <= 2e-3 per (request, query head).
"""
import numpy as np
import pytest

import harness as H
import oracle as O
import synth
from test_gpu_demote import _run

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda(built_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("block", [32, 128])
def test_demote_with_canalized_rotation_per_step_path(block):
    g = synth.generator(5, 1)
    pos = g.permutation(600)[:257]
    _run(2101, 257, 4, positions=pos, canalized_block=block)


def test_demote_with_canalized_rotation_bulk_path():
    _run(2102, 1500, 2, canalized_block=16)


@pytest.mark.parametrize("g", [4, 8])
def test_decode_with_canalized_rotation(g):
    outl = synth.outlier_channels(2103, 0, 2)
    rot = H.canalized_rotations(2103, 0, 2, outl, 32)
    sc = H.Scenario(2103, [4000, 1337, 333], n_kv=2, g=g, rot=rot)
    cache, q = H.to_device(sc)
    out, status = H.run_decode(cache, q)
    assert status == 0
    err = H.relative_error(out, sc.expected())
    assert np.all(np.isfinite(out))
    assert err.max() <= TOL, err.max()
