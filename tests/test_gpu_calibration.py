"""Calibration covariance on the GPU (oscar_covariance) against the float64
oracle, and the rotation built from it.

[GIST] 2.1 and 2.2 A: C_Q = Q^T Q / N over calibration queries, C_S =
(S V)^T (S V) / N.  The device computes fp32 sums of exact bf16 products
(partials of at most 2048 rows, then the partials in a fixed order of at
most as many additions per path), so each entry must lie within the
summation bound gamma_m * sum_r |x_ri x_rj| / N of the oracle's value,
m = 2048 + (number of partials) + 2.
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


def _device_value_cov(q64, k64, v64, pitch=128):
    import torch
    from bit_rotated_kv_split_gb300 import binding as B

    def up(x):
        buf = torch.zeros((x.shape[0], pitch), dtype=torch.bfloat16)
        buf[:, :128] = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
        return buf.cuda()[:, :128]
    q, k, v = up(q64), up(k64), up(v64)
    c = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.oscar_value_covariance_workspace_bytes(q.shape[0]), dtype=torch.uint8, device="cuda")
    B.oscar_value_covariance(q, k, v, c, ws)
    torch.cuda.synchronize()
    return c.cpu().numpy().astype(np.float64)


def _value_cov_bound(q, k, v):
    """Entrywise bound on |C_S(device) - C_S(oracle)| from the device's
    arithmetic, worst case.  Each weight p = 2^(s log2e - m) carries the fp32
    score sum of 128 exact bf16 products (gamma_128 sum|q_i k_i| / sqrt(128)),
    the rounding of the scaling and of s - m (2 u |s| each), exp2f (2 ulp),
    and the rounding of its bf16 lo part (2^-18 p); the tile rescalings are
    applied to numerator and denominator alike (only their 2 u per tile
    remain); the fp32 sums over the n_k keys add gamma_nk to each of the
    numerator and the denominator.  With eps the sum of those relative terms,
    |d sv_n| <= 3 eps (P |V|)_n, and C's own fp32 sums (256 rows, then the
    partials) add gamma_m (|sv|^T |sv|) / N."""
    u = 2.0 ** -24
    gam = lambda n: n * u / (1 - n * u)
    n_q, n_k = q.shape[0], k.shape[0]
    s = q @ k.T / np.sqrt(128.0)
    eps = (gam(128) * (np.abs(q) @ np.abs(k).T).max() / np.sqrt(128.0) + 4 * u * np.abs(s).max()
           + 2.0 ** -21 + 2.0 ** -18 + 2 * u * (-(-n_k // 64)) + 2 * gam(n_k))
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    sv = p @ v
    w = 3 * eps * (p @ np.abs(v))
    a = np.abs(sv)
    m = 256 + (-(-n_q // 256)) + 2
    return ((w.T @ a + a.T @ w + w.T @ w) + gam(m) * (a.T @ a)) / n_q + u * np.abs(sv.T @ sv) / n_q


@pytest.mark.parametrize("n_q,n_k,pitch", [(4096, 2048, 128), (1000, 777, 256)])
def test_value_covariance_on_device_matches_oracle(n_q, n_k, pitch):
    """C_S = (S V)^T (S V) / N formed on the device from bf16 calibration
    rows (row and key counts off the tile sizes, strided rows) against the
    float64 oracle, within the worst-case bound of the device's arithmetic;
    and the rotation built from it."""
    from bit_rotated_kv_split_gb300 import binding as B
    outl = synth.outlier_channels(3004, 0, 1)
    cal = synth.calibration_set(3004, 0, 0, outl[0], n_q=n_q, n_k=n_k)
    c_gpu = _device_value_cov(cal["q"], cal["k"], cal["v"], pitch)
    ref = O.value_covariance(cal["q"], cal["k"], cal["v"])
    bound = _value_cov_bound(cal["q"], cal["k"], cal["v"])
    err = np.abs(c_gpu - ref)
    print("max err/bound %.3g, max rel err %.3g" % ((err / bound).max(), (err / np.abs(ref).max()).max()))
    assert np.all(err <= bound), "max err/bound %.3g" % (err / bound).max()
    r, w = B.oscar_build_rotation_from_covariance(c_gpu)
    np.testing.assert_allclose(r @ r.T, np.eye(128), atol=1e-12)


def test_value_covariance_uniform_scores():
    """Special case with a closed form: every key equal, so S is uniform
    (every score equal, each weight exactly 1) and every S V row is the mean
    value row v_bar; C_S = v_bar^T v_bar whatever the queries."""
    outl = synth.outlier_channels(3005, 0, 1)
    cal = synth.calibration_set(3005, 0, 0, outl[0], n_q=333, n_k=300)
    k = np.repeat(cal["k"][:1], 300, axis=0)
    c_gpu = _device_value_cov(cal["q"], k, cal["v"])
    vbar = cal["v"].mean(axis=0)
    ref = np.outer(vbar, vbar)
    # fp32 sums of 300 values (gamma_300 sum|v| / 300 per mean) and the
    # covariance's own fp32 sums
    u = 2.0 ** -24
    dv = 305 * u * np.abs(cal["v"]).mean(axis=0)
    bound = np.outer(dv, np.abs(vbar)) + np.outer(np.abs(vbar), dv) + np.outer(dv, dv) + 300 * u * np.abs(ref)
    assert np.all(np.abs(c_gpu - ref) <= bound + 1e-30)
