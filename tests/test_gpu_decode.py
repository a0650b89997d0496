"""GPU parity of oscar_decode_attention against the float64 oracle.

The INT2 history is quantised and packed by the oracle, uploaded, and read by
the CUDA path, so both sides attend over identical codes.  Bar (per request
and query head): max|o_gpu - o_ref| / max|o_ref| <= 2e-3 (BF16 inputs, fp32
accumulate, fp32 output).
"""
import numpy as np
import pytest

import harness as H

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda(built_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(sc, **kw):
    cache, q = H.to_device(sc)
    out, status = H.run_decode(cache, q, **kw)
    ref = sc.expected()
    err = H.relative_error(out, ref)
    assert status == 0, "device status %#x" % status
    assert np.all(np.isfinite(out))
    assert err.max() <= TOL, "max relative error %.3g at %s" % (err.max(), np.unravel_index(err.argmax(), err.shape))
    return out, err


def test_tiny_single_layer_config():
    # batch 1, 1 KV head, GQA 4, context 2048 = 64 + 1728 INT2 + 256, rotations
    # from 4096 calibration queries (the tiny workload of the benchmark list)
    sc = H.Scenario(1001, [2048], n_kv=1, g=4, cal=(4096, 2048))
    assert (sc.sink_len[0], sc.hist_len[0], sc.recent_len[0]) == (64, 1728, 256)
    _check(sc)


def test_ragged_batch_many_splits():
    sc = H.Scenario(11, [2048, 777, 5000, 321, 4113], n_kv=2, g=4)
    _check(sc)


def test_gqa8():
    sc = H.Scenario(12, [3000, 1500, 337], n_kv=2, g=8)
    _check(sc)


@pytest.mark.parametrize("g", [4, 8])
def test_edge_lengths(g):
    # sink only, full sink, one recent token, no history, one history token,
    # exactly one full page, one page plus one token
    sc = H.Scenario(13 + g, [1, 64, 65, 320, 321, 336, 337, 16 * 7 + 320 + 5], n_kv=1, g=g)
    _check(sc)


def test_ring_start_wraps():
    for start in (0, 255, 100):
        sc = H.Scenario(14, [300, 2000], n_kv=1, g=4, ring_start=start)
        _check(sc)


def test_page_permutation_is_invisible():
    a = H.Scenario(15, [3000, 1800], n_kv=2, g=4)
    b = H.Scenario(15, [3000, 1800], n_kv=2, g=4, identity_pages=True)
    out_a, _ = _check(a)
    out_b, _ = _check(b)
    np.testing.assert_array_equal(out_a, out_b)


def test_shared_prefix_pages_equal_private_copies():
    import torch
    sc = H.Scenario(16, [2000, 1200, 900, 3000], n_kv=2, g=4, shared_prefix_hist=512)
    shared_ids = set(int(x) for x in sc.table[0, :512 // 16])
    assert all(int(x) in shared_ids for x in sc.table[1, :512 // 16])
    out_shared, _ = _check(sc)
    # private copy of every page reference
    import oracle as O
    blocks = sc.pool.reshape(sc.n_pages, sc.n_kv, O.BLOCK_BYTES)
    refs = [(b, p) for b in range(sc.B) for p in range(sc.table.shape[1]) if sc.table[b, p] >= 0]
    private = np.zeros((len(refs), sc.n_kv, O.BLOCK_BYTES), np.uint8)
    table = np.full_like(sc.table, -1)
    for i, (b, p) in enumerate(refs):
        private[i] = blocks[sc.table[b, p]]
        table[b, p] = i
    cache, q = H.to_device(sc)
    cache.pages = torch.from_numpy(private.reshape(-1)).cuda()
    cache.n_pages = len(refs)
    cache.page_table.copy_(torch.from_numpy(table))
    out_private, status = H.run_decode(cache, q)
    assert status == 0
    np.testing.assert_array_equal(out_shared, out_private)


def test_out_of_range_page_is_flagged_not_faulted():
    import torch
    sc = H.Scenario(17, [2000], n_kv=1, g=4)
    cache, q = H.to_device(sc)
    bad = cache.page_table.clone()
    bad[0, 3] = sc.n_pages + 1000
    cache.page_table.copy_(bad)
    out, status = H.run_decode(cache, q)
    assert status & 0x1
    assert np.all(np.isfinite(out))


def test_history_longer_than_bound_is_flagged():
    sc = H.Scenario(18, [2000], n_kv=1, g=4)
    cache, q = H.to_device(sc)
    _, status = H.run_decode(cache, q, max_hist=100)
    assert status & 0x2


@pytest.mark.slow
def test_full_size_qwen3_8b_layer_100k():
    # Qwen3-8B-shaped single layer: 32 query heads, 8 KV heads, context
    # 100,000 = 64 + 99,680 INT2 + 256; every output compared, same launch
    # configuration as the benchmark (plan depends only on dims and device)
    sc = H.Scenario(1002, [100_000], n_kv=8, g=4, cal=(4096, 2048))
    _check(sc)


def test_workspace_is_reusable_across_calls():
    # the merge tickets reset themselves: back-to-back calls on one workspace
    # give identical outputs
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    sc = H.Scenario(19, [4000, 900], n_kv=2, g=4)
    cache, q = H.to_device(sc)
    desc = cache.desc()
    ws = torch.zeros(B.oscar_decode_workspace_bytes(desc), dtype=torch.uint8, device=q.device)
    outs = []
    for _ in range(3):
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        B.oscar_decode_attention(desc, q, out, ws)
        outs.append(out)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    err = H.relative_error(outs[0].cpu().numpy().astype(np.float64), sc.expected())
    assert err.max() <= TOL


@pytest.mark.parametrize("scales", [(2.0 ** -8, 2.0 ** -8, 1.0), (2.0 ** 8, 2.0 ** 8, 1.0),
                                    (1.0, 2.0 ** 8, 2.0 ** -8), (2.0 ** 8, 2.0 ** -8, 2.0 ** 8)])
def test_scaled_caches(scales):
    """Keys, values and queries scaled by 2^-8 .. 2^8: the fp16 hi/lo splits of
    q~ (per-head power-of-two scale) and of p s_V (scale from tau_v) and the
    subnormal code operands keep the output within the bar."""
    sc = H.Scenario(1013, [3000, 1500], n_kv=2, g=4, scales=scales)
    _check(sc)


def test_expired_page_waits_are_flagged_and_the_workspace_recovers():
    """With the page-scan budget at 20 ns every warp gives up its pages at
    its first step: the call returns, the timeout bit is set, and the copies
    already issued land before the kernel exits.  With the default limit
    restored, the next call on the same workspace gives the oracle's output."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    sc = H.Scenario(1002, [100_000], n_kv=8, g=4, cal=(1024, 512))
    cache, q = H.to_device(sc)
    desc = cache.desc()
    nbytes = B.oscar_decode_workspace_bytes(desc)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    prev = B.oscar_set_page_wait_limit(20)
    try:
        for _ in range(2):
            cache.dev_status.zero_()
            B.oscar_decode_attention(desc, q, out, ws, nbytes)
            torch.cuda.synchronize()
            assert int(cache.dev_status.item()) == B.DEV_TIMEOUT
    finally:
        assert B.oscar_set_page_wait_limit(prev) == 20
    cache.dev_status.zero_()
    B.oscar_decode_attention(desc, q, out, ws, nbytes)
    torch.cuda.synchronize()
    assert int(cache.dev_status.item()) == 0
    err = H.relative_error(out.cpu().numpy().astype(np.float64), sc.expected())
    assert err.max() <= TOL
