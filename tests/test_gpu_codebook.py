"""GPU parity for the Lloyd-Max codebook (four fp16 levels per layer, K and V).

The levels are the oracle's fit on seeded calibration rows (the library's
own fit is checked against it on the CPU).  Demotion: both kernels
write nearest-level codes with the uniform codec's (scale, zero); codes are
compared with the oracle's by `harness.code_parity` with the codebook's
thresholds as rounding boundaries.  Decode: the oracle quantises and packs
the history with the same levels; bar max|o_gpu - o_ref| / max|o_ref| <= 2e-3
per (request, query head).
"""
import numpy as np
import pytest

import harness as H
import oracle as O
import synth
from test_gpu_decode import _check
from test_gpu_demote import _run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(built_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _levels(seed, n_kv=2):
    """(levels_k, levels_v): the oracle's fit on seeded calibration rows (the
    library's fit is checked against it on the CPU)."""
    outl = synth.outlier_channels(seed, 0, n_kv)
    rk32, rv32, tau_k, tau_v = H.rotations(seed, 0, n_kv, outl, n_q=1024, n_k=512)
    xk = np.concatenate([synth.calibration_set(seed, 0, h, outl[h], n_q=64, n_k=512)["k"] @ rk32[h].astype(np.float64)
                         for h in range(n_kv)])
    xv = np.concatenate([synth.calibration_set(seed, 0, h, outl[h], n_q=64, n_k=512)["v"] @ rv32[h].astype(np.float64)
                         for h in range(n_kv)])
    eye = np.eye(128)
    lk = O.fit_codebook(xk, eye, tau_k)
    lv = O.fit_codebook(xv, eye, tau_v)
    assert not np.array_equal(lk.astype(np.float32), [0, 1, 2, 3])
    return lk, lv


def test_demote_per_token_kernel_codebook():
    g = synth.generator(41, 1)
    pos = g.permutation(700)[:333]
    print(_run(4001, 333, 8, positions=pos, levels=_levels(4001)))


def test_demote_per_token_kernel_codebook_with_new_tokens():
    _run(4002, 512, 4, with_new=True, levels=_levels(4002, 4))


def test_demote_bulk_gathered_rows_codebook():
    g = synth.generator(42, 1)
    pos = g.permutation(4000)[:3000]
    print(_run(4003, 3000, 4, positions=pos, levels=_levels(4003)))


def test_demote_bulk_contiguous_rows_codebook():
    g = synth.generator(43, 1)
    pos = g.permutation(3000)[:2100]
    print(_run(4004, 2100, 8, positions=pos, first_row=77, levels=_levels(4004)))


@pytest.mark.parametrize("g", [4, 8])
def test_decode_codebook_ragged_batch(g):
    sc = H.Scenario(4100 + g, [2048, 777, 5000, 321], n_kv=2, g=g, levels=_levels(4100 + g))
    _check(sc)


def test_decode_codebook_edge_lengths():
    sc = H.Scenario(4200, [1, 64, 65, 320, 321, 336, 337, 16 * 7 + 320 + 5], n_kv=1, g=4,
                    levels=_levels(4200, 1))
    _check(sc)


@pytest.mark.parametrize("levels", [(0.25, 1.0, 2.0, 2.75), (0.0, 1.0, 2.0, 3.0), (0.5, 0.75, 1.25, 3.0)])
def test_decode_codebook_fixed_levels(levels):
    # hand-set levels, the uniform ones among them (the level coefficients
    # of the second- and third-order planes vanish) and a lopsided set
    lv = np.array(levels, np.float16)
    sc = H.Scenario(4300, [3000, 1500], n_kv=2, g=4, levels=(lv, lv.copy()))
    _check(sc)


@pytest.mark.parametrize("with_levels", [False, True])
def test_masked_tail_slots_with_nan_bytes_do_not_leak(with_levels):
    # token slots past the history length of a partial last page are masked;
    # their (scale, zero) bytes are set to fp16 NaN and their codes to 0xFF,
    # and the output must still match the oracle (selects, not p = 0 products)
    import torch
    levels = _levels(4400, 2) if with_levels else None
    sc = H.Scenario(4400, [64 + 1000 + 256, 64 + 777 + 256], n_kv=2, g=4, levels=levels)
    assert all(int(h) % 16 for h in sc.hist_len)
    cache, q = H.to_device(sc)
    pool = cache.pages.cpu().numpy().copy()
    nan = np.array([0x7E00, 0x7E00], np.uint16).view(np.uint8)
    for b in range(sc.B):
        h = int(sc.hist_len[b])
        page = int(sc.table[b, (h - 1) // 16])
        for head in range(sc.n_kv):
            base = (page * sc.n_kv + head) * O.BLOCK_BYTES
            for which in (0, 1):
                for slot in range(h % 16, 16):
                    pool[base + O.code_byte_offset(which, slot, np.arange(32))] = 0xFF
                    so = base + int(O.pair_offset(which, slot, 0))
                    pool[so:so + 4] = nan
    cache.pages.copy_(torch.from_numpy(pool))
    _check(sc)
