"""Calibration covariance on the GPU (oscar_covariance) against the float64
oracle, and the rotation built from it.

[GIST] 2.1 and 2.2 A: C_Q = Q^T Q / N over calibration queries, C_S =
(S V)^T (S V) / N.  The device computes fp32 sums of exact bf16 products
(partials of at most 2048 rows, then the partials in chunk order), so each
entry must lie within the summation bound gamma_m * sum_r |x_ri x_rj| / N of
the oracle's value, m = 2048 + (number of partials) + 2.
"""
import numpy as np
import pytest

import harness as H
import oracle as O
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(built_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _device_cov(x64, pitch=128):
    """oscar_covariance of the bf16-valued rows x64 [n][128], stored with row pitch `pitch`."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    n = x64.shape[0]
    buf = torch.zeros((n, pitch), dtype=torch.bfloat16)
    buf[:, :128] = torch.from_numpy(x64.astype(np.float32)).to(torch.bfloat16)
    xd = buf.cuda()[:, :128]
    c = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.oscar_covariance_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    B.oscar_covariance(xd, c, ws)
    torch.cuda.synchronize()
    return c.cpu().numpy().astype(np.float64)


def _check(x64, c_gpu):
    n = x64.shape[0]
    ref = x64.T @ x64 / n
    chunks = -(-n // 2048)
    m = 2048 + chunks + 2
    gamma = m * 2.0 ** -24 / (1 - m * 2.0 ** -24)
    bound = gamma * (np.abs(x64).T @ np.abs(x64)) / n + 2.0 ** -24 * np.abs(ref)
    err = np.abs(c_gpu - ref)
    assert np.all(err <= bound), "max err/bound %.3g" % (err / bound).max()
    return ref


def test_query_covariance_matches_oracle():
    outl = synth.outlier_channels(3001, 0, 1)
    cal = synth.calibration_set(3001, 0, 0, outl[0], n_q=4096, n_k=512)
    ref = _check(cal["q"], _device_cov(cal["q"]))
    np.testing.assert_allclose(ref, O.query_covariance(cal["q"]), rtol=1e-12, atol=1e-12)


def test_value_covariance_rows_ragged_and_strided():
    # S.V rows (bf16-rounded, as a device would hold them), 3000 of them: a
    # partial 2048-row chunk and a partial 64-row stage; rows 256 values apart
    outl = synth.outlier_channels(3002, 0, 1)
    cal = synth.calibration_set(3002, 0, 0, outl[0], n_q=3000, n_k=700)
    sv = O.score_weighted_values(cal["q"], cal["k"], cal["v"])
    sv_b = synth.to_bf16(sv.astype(np.float32)).astype(np.float64)
    _check(sv_b, _device_cov(sv_b, pitch=256))


def test_rotation_from_device_covariance():
    from bit_rotated_kv_split_gb300 import binding as B
    outl = synth.outlier_channels(3003, 0, 1)
    cal = synth.calibration_set(3003, 0, 0, outl[0], n_q=4096, n_k=512)
    c_gpu = _device_cov(cal["q"])
    r, w = B.oscar_build_rotation_from_covariance(c_gpu)
    np.testing.assert_allclose(r @ r.T, np.eye(128), atol=1e-12)
    w_ref = np.sort(np.linalg.eigvalsh(O.query_covariance(cal["q"])))[::-1]
    np.testing.assert_allclose(w, w_ref, rtol=1e-5, atol=1e-5 * w_ref[0])
