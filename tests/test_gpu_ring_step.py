"""GPU checks of the one-kernel decode step (oscar_decode_step_ring).

[ZAKER] "从离线校准到在线推理的 pipeline": per decode step the oldest recent
token is demoted into INT2 history and the new token takes its ring slot,
then attention runs over sink | history | recent.  The one-kernel step must
equal the separate calls - oscar_quantize_append (the displaced token into
history position hist_len - 1, the new rows into its slot) and
oscar_decode_attention - bit for bit: pool bytes, ring rows and output.
The separate calls are themselves checked against the oracle elsewhere; the
output is also held to the oracle's bar here through the pool both paths
leave.
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


def _separate(sc, cache, q, new_k, new_v):
    """Reference: quantize_append for the requests that demote, a plain write
    of the new rows for those that do not, then the decode."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    dev = q.device
    cap = sc.recent_cap
    dem, src, pos = [], [], []
    for b in range(sc.B):
        rl, st, h = int(sc.recent_len[b]), int(sc.recent_start[b]), int(sc.hist_len[b])
        if rl < 1:
            continue
        t = (st + rl - 1) % cap
        if rl == cap and h >= 1:
            dem.append(b)
            src.append(b * cap + t)
            pos.append(h - 1)
        else:
            cache.recent_k[b, t] = new_k[b]
            cache.recent_v[b, t] = new_v[b]
    desc = cache.desc()
    if dem:
        idx = torch.tensor(dem, dtype=torch.int64, device=dev)
        B.oscar_quantize_append(desc, cache.recent_k.view(torch.uint16), cache.recent_v.view(torch.uint16),
                                sc.B * cap, sc.n_kv * 128, torch.tensor(src, dtype=torch.int32, device=dev),
                                torch.tensor(dem, dtype=torch.int32, device=dev),
                                torch.tensor(pos, dtype=torch.int32, device=dev), len(dem),
                                new_k[idx].contiguous().view(torch.uint16),
                                new_v[idx].contiguous().view(torch.uint16))
    ws = torch.zeros(B.oscar_decode_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    B.oscar_decode_attention(desc, q, out, ws)
    torch.cuda.synchronize()
    return out


def _ring(sc, cache, q, new_k, new_v):
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    desc = cache.desc()
    ws = torch.zeros(B.oscar_decode_workspace_bytes(desc), dtype=torch.uint8, device=q.device)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    B.oscar_decode_step_ring(desc, new_k.view(torch.uint16), new_v.view(torch.uint16), q, out, ws)
    torch.cuda.synchronize()
    return out


def _compare(sc):
    import torch
    cache_a, q = H.to_device(sc)
    cache_b, _ = H.to_device(sc)
    dev = q.device
    nk = synth.activations(sc.seed, (9, 0), sc.B, sc.outl)
    nv = synth.activations(sc.seed, (9, 1), sc.B, sc.outl)
    new_k = torch.from_numpy(nk).to(torch.bfloat16).to(dev).contiguous()
    new_v = torch.from_numpy(nv).to(torch.bfloat16).to(dev).contiguous()
    out_a = _separate(sc, cache_a, q, new_k, new_v)
    out_b = _ring(sc, cache_b, q, new_k, new_v)
    assert int(cache_a.dev_status.item()) == 0 and int(cache_b.dev_status.item()) == 0
    assert torch.equal(cache_a.pages, cache_b.pages)
    assert torch.equal(cache_a.recent_k.view(torch.int16), cache_b.recent_k.view(torch.int16))
    assert torch.equal(cache_a.recent_v.view(torch.int16), cache_b.recent_v.view(torch.int16))
    oa, ob = out_a.cpu().numpy(), out_b.cpu().numpy()
    np.testing.assert_array_equal(oa, ob)
    # the output against the oracle over the pool the step left (history
    # read back with the oracle's layout functions; sink and ring from the
    # device rows)
    pool = cache_b.pages.cpu().numpy()
    rk = cache_b.recent_k.float().cpu().numpy()
    rv = cache_b.recent_v.float().cpu().numpy()
    sk = cache_b.sink_k.float().cpu().numpy()
    sv = cache_b.sink_v.float().cpu().numpy()
    for b in range(sc.B):
        h, s, rl, st = int(sc.hist_len[b]), int(sc.sink_len[b]), int(sc.recent_len[b]), int(sc.recent_start[b])
        slots = [(st + i) % sc.recent_cap for i in range(rl)]
        hist = {}
        for which, nm in ((0, "k"), (1, "v")):
            c, sz, z = O.load_history_bulk(pool, sc.table, sc.n_kv, b, h, which)
            hist["codes_" + nm], hist["scale_" + nm], hist["zero_" + nm] = c, sz, z
        ref = O.decode_attention(sc.q[b].astype(np.float64), sk[b, :s].astype(np.float64),
                                 sv[b, :s].astype(np.float64), hist, rk[b, slots].astype(np.float64),
                                 rv[b, slots].astype(np.float64), sc.rk32.astype(np.float64),
                                 sc.rv32.astype(np.float64))
        err = H.relative_error(ob[b:b + 1].astype(np.float64), ref[None])
        assert err.max() <= 2e-3, (b, err.max())
    return oa


@pytest.mark.parametrize("g", [4, 8])
def test_ring_step_equals_separate_calls(g):
    # history lengths 1 (the first demotion), 17, 457, 4680 and 1 page + 1;
    # a context inside the ring (no demotion) and one inside the sink (no
    # write); random ring starts
    ctxs = [64 + 256 + 1, 64 + 256 + 17, 777, 5000, 64 + 100, 1, 64 + 256 + 16 + 1]
    _compare(H.Scenario(5100 + g, ctxs, n_kv=2, g=g))


@pytest.mark.parametrize("start", [0, 255])
def test_ring_step_at_ring_edges(start):
    # the newest slot at the ring's last and first rows
    _compare(H.Scenario(5200 + start, [3000, 64 + 256 + 33, 64 + 256], n_kv=1, g=4, ring_start=start))


def test_ring_step_many_splits_batch():
    # a ragged batch whose longest request takes many splits, so the
    # demoted token's page sits in a later split than the new token's reader
    _compare(H.Scenario(5300, [20000, 64 + 256 + 5, 9000, 1500], n_kv=2, g=4))
