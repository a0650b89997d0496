"""GPU parity for quantisation groups of 32 / 64 channels (K and V chosen apart).

Demotion: both kernels (the per-token kernel, and the tensor-core bulk
kernel with gathered and with contiguous rows) write the grouped page format;
codes and each group's (scale, zero) are read back with the oracle's reader
and compared with the oracle's grouped quantiser by the rule in
`harness.code_parity`, group by group.  Decode: the oracle quantises and packs
the history in the grouped format, the CUDA path attends over it; bar
max|o_gpu - o_ref| / max|o_ref| <= 2e-3 per (request, query head).
"""
import numpy as np
import pytest

import harness as H
import synth
from test_gpu_decode import _check
from test_gpu_demote import _run

pytestmark = pytest.mark.gpu

GROUPS = [(32, 32), (64, 64), (32, 128), (128, 32), (64, 32)]


@pytest.fixture(scope="module", autouse=True)
def _cuda(built_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("groups", GROUPS)
def test_demote_per_token_kernel_groups(groups):
    g = synth.generator(21, 1)
    pos = g.permutation(700)[:333]
    print(_run(3001, 333, 8, positions=pos, groups=groups))


@pytest.mark.parametrize("groups", [(32, 32), (64, 128), (128, 64)])
def test_demote_per_token_kernel_groups_with_new_tokens(groups):
    _run(3002, 512, 4, with_new=True, groups=groups)


@pytest.mark.parametrize("groups", GROUPS)
def test_demote_bulk_gathered_rows_groups(groups):
    g = synth.generator(22, 1)
    pos = g.permutation(4000)[:3000]
    print(_run(3003, 3000, 4, positions=pos, groups=groups))


@pytest.mark.parametrize("groups", [(32, 32), (64, 64), (32, 64)])
def test_demote_bulk_contiguous_rows_groups(groups):
    g = synth.generator(23, 1)
    pos = g.permutation(3000)[:2100]
    print(_run(3004, 2100, 8, positions=pos, first_row=77, groups=groups))


@pytest.mark.parametrize("g", [4, 8])
@pytest.mark.parametrize("groups", GROUPS + [(64, 128), (128, 64)])
def test_decode_groups_ragged_batch(g, groups):
    sc = H.Scenario(3100 + g, [2048, 777, 5000, 321], n_kv=2, g=g, groups=groups)
    _check(sc)


@pytest.mark.parametrize("groups", [(32, 32), (64, 32)])
def test_decode_groups_edge_lengths(groups):
    sc = H.Scenario(3200, [1, 64, 65, 320, 321, 336, 337, 16 * 7 + 320 + 5], n_kv=1, g=4, groups=groups)
    _check(sc)


def test_decode_groups_with_equal_pairs_match_one_group():
    # The grouped pool holding a single (scale, zero) in every group decodes
    # exactly like the one-group pool: the grouped kernel's QK and PV sums per
    # group add up to the one-group sums (up to fp32 reassociation).
    import oracle as O
    import torch
    from bit_rotated_kv_split_gb300.cache import LayerCache
    sc = H.Scenario(3300, [3000, 1200], n_kv=2, g=4)
    cache1, q = H.to_device(sc)
    out1, st1 = H.run_decode(cache1, q)
    pool4 = np.zeros(sc.n_pages * sc.n_kv * O.block_bytes(4, 4), np.uint8)
    for b in range(sc.B):
        h = sc.hist[b]
        if not len(h["codes_k"]):
            continue
        for which, c, s, z in ((0, h["codes_k"], h["scale_k"], h["zero_k"]),
                               (1, h["codes_v"], h["scale_v"], h["zero_v"])):
            O.store_history_groups(pool4, sc.table, sc.n_kv, b, 0, c, np.repeat(s[..., None], 4, -1),
                                   np.repeat(z[..., None], 4, -1), which, 4, 4)
    cache4 = LayerCache(sc.B, sc.h_q, sc.n_kv, sc.table.shape[1], sc.n_pages, cache1.r_k, cache1.r_v,
                        sc.tau_k, sc.tau_v, device=q.device, quant_group_k=32, quant_group_v=32)
    for name in ("page_table", "hist_len", "sink_len", "recent_len", "recent_start", "sink_k", "sink_v",
                 "recent_k", "recent_v"):
        getattr(cache4, name).copy_(getattr(cache1, name))
    cache4.pages.copy_(torch.from_numpy(pool4))
    cache4.max_hist = cache1.max_hist
    out4, st4 = H.run_decode(cache4, q)
    assert st1 == 0 and st4 == 0
    np.testing.assert_allclose(out4, out1, rtol=0, atol=2e-5 * np.abs(out1).max())
