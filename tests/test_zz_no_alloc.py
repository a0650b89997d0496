"""The no-allocation decode entry point against the regular one.

oscar_decode_attention_static serves callers that cannot allocate device
memory (a host framework that owns all allocations, or a serving loop that
forbids allocating after start-up): it runs the same decode with a fixed
workspace inside the library.  Two calls in a row must each give the
regular entry point's output on the same inputs, bit for bit.  This file is collected
last on purpose.
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


def test_static_workspace_matches_regular_entry_point_twice():
    """Decode is deterministic (fixed-order reductions), so the fixed
    workspace must give the regular entry point's output bit for bit, on
    two calls in a row; both are also within the attention tolerance of the
    float64 oracle."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    sc = H.Scenario(31, [3000, 800, 2049], n_kv=2, g=4)
    cache, q = H.to_device(sc)
    ref, status = H.run_decode(cache, q)
    assert status == 0
    assert H.relative_error(ref, sc.expected()).max() <= TOL
    desc = cache.desc()
    for _ in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=q.device)
        B.oscar_decode_attention_static(desc, q, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        np.testing.assert_array_equal(got, ref)
    assert int(cache.dev_status.item()) == 0


def test_static_workspace_rejects_oversized_problems():
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    from bit_rotated_kv_split_gb300.cache import LayerCache
    # 1024 requests x 8 KV heads x GQA 8 at 128k tokens: at least one split
    # partial per (request, query head) is far more than the fixed array; the
    # call must refuse before launching anything
    r = torch.eye(128).repeat(8, 1, 1)
    cache = LayerCache(1024, 64, 8, 8192, 16, r, r, 4.0, 4.0, sink_cap=0, recent_cap=0)
    desc = cache.desc(131_072 - 320)
    assert B.oscar_decode_workspace_bytes(desc) > (8 << 20)
    out = torch.empty((1024, 64, 128), dtype=torch.float32, device="cuda")
    q = torch.zeros((1024, 64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.OscarError) as err:
        B.oscar_decode_attention_static(desc, q.view(torch.uint16), out)
    assert err.value.status == 3
