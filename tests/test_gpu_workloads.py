"""Full-size GPU parity at the stated workloads, on sampled outputs.

* Qwen3-32B-shaped layer: 64 query heads, 8 KV heads (GQA 8), batch 64,
  contexts ragged uniform in [8k, 128k], the first 32k tokens a shared
  prefix whose INT2 pages every request's page table references.
* Qwen3-4B-shaped layer: 32 query heads, 8 KV heads, batch 28 x 100k
  tokens, plus one demotion per request (the per-layer part of the 36-layer
  decode step).
* Bulk demotion of a 128k-token prefill for 8 KV heads (every code, scale
  and zero point checked), then batch-1 decode (GQA 4) over that history
  with the oracle's codes in the pool, so both sides decode identical codes.

For the decode-only cases the INT2 history is seeded random code bytes with
plausible fp16 (scale, zero): decode parity does not depend on how the codes
were produced, and the oracle reads the very bytes the GPU reads (no value
from the CUDA path enters the expectation).  Every output of the sampled
requests is compared with the oracle at the decode tolerance.
"""
import numpy as np
import pytest

import harness as H
import oracle as O
import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda(built_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class RandomHistory:
    """Batch of three-segment caches whose INT2 history is random code bytes.

    Provides what `harness.to_device` reads, and oracle outputs for chosen
    requests.  Sink/recent tokens and queries follow the synthetic recipe
    (N(0,1), 4 outlier channels x20, bf16).
    """

    def __init__(self, seed, ctxs, n_kv, g, shared_prefix_hist=0, n_extra_pages=1):
        self.seed, self.n_kv, self.g = seed, n_kv, g
        self.ctxs = [int(c) for c in ctxs]
        self.B = len(self.ctxs)
        self.h_q = n_kv * g
        self.sink_cap, self.recent_cap = 64, 256
        self.outl = synth.outlier_channels(seed, 0, n_kv)
        self.rk32, self.rv32, self.tau_k, self.tau_v = H.rotations(seed, 0, n_kv, self.outl, n_q=1024, n_k=512)
        splits = [synth.history_split(c) for c in self.ctxs]
        self.sink_len = np.array([s[0] for s in splits], np.int32)
        self.hist_len = np.array([s[1] for s in splits], np.int32)
        self.recent_len = np.array([s[2] for s in splits], np.int32)
        self.recent_start = synth.generator(seed, 77).integers(0, 256, size=self.B).astype(np.int32)
        self.table, self.n_pages = synth.page_table(seed, self.hist_len, n_extra_pages=n_extra_pages,
                                                    shared_prefix_tokens=shared_prefix_hist)
        n_blocks = self.n_pages * n_kv
        self.pool = synth.random_bytes(seed, (1,), n_blocks * O.BLOCK_BYTES)
        # (scale, zero) of every slot: the ranges demotion gives rotated
        # N(0,1) + outlier tokens (scale ~ 7, zero ~ -10.5)
        g_sz = synth.generator(seed, 88)
        # (block, token slot, K|V, (scale, zero)): the pairs region of the
        # one-group format, token-major with K before V
        sz = np.empty((n_blocks, 16, 2, 2), np.float16)
        sz[..., 0] = g_sz.uniform(5.0, 9.0, size=(n_blocks, 16, 2)).astype(np.float16)
        sz[..., 1] = g_sz.uniform(-12.0, -9.0, size=(n_blocks, 16, 2)).astype(np.float16)
        blocks = self.pool.reshape(n_blocks, O.BLOCK_BYTES)
        blocks[:, O.SZ_OFFSET:] = sz.view(np.uint8).reshape(n_blocks, 128)
        # sink and recent tokens (first 64 and last 256 of each context)
        self.seg = []
        for b in range(self.B):
            n = int(self.sink_len[b] + self.recent_len[b])
            k = synth.activations(seed, (0, b, 0), n, self.outl)
            v = synth.activations(seed, (0, b, 1), n, self.outl)
            sl = int(self.sink_len[b])
            self.seg.append((k[:sl], v[:sl], k[sl:], v[sl:]))
        qo = np.repeat(self.outl, g, axis=0)
        self.q = np.stack([synth.activations(seed, (0, b, 2), 1, qo)[0] for b in range(self.B)])

    def sink(self):
        sk = np.zeros((self.B, self.sink_cap, self.n_kv, H.D), np.float32)
        sv = np.zeros_like(sk)
        for b, (k, v, _, _) in enumerate(self.seg):
            sk[b, :k.shape[0]] = k
            sv[b, :v.shape[0]] = v
        return sk, sv

    def ring(self):
        rk = np.zeros((self.B, self.recent_cap, self.n_kv, H.D), np.float32)
        rv = np.zeros_like(rk)
        for b, (_, _, k, v) in enumerate(self.seg):
            for i in range(k.shape[0]):
                slot = (int(self.recent_start[b]) + i) % self.recent_cap
                rk[b, slot] = k[i]
                rv[b, slot] = v[i]
        return rk, rv

    def expected(self, b):
        hl = int(self.hist_len[b])
        ck, sk, zk = O.load_history_bulk(self.pool, self.table, self.n_kv, b, hl, 0)
        cv, sv, zv = O.load_history_bulk(self.pool, self.table, self.n_kv, b, hl, 1)
        hist = dict(codes_k=ck, scale_k=sk, zero_k=zk, codes_v=cv, scale_v=sv, zero_v=zv)
        k_s, v_s, k_r, v_r = self.seg[b]
        return O.decode_attention(self.q[b].astype(np.float64), k_s, v_s, hist, k_r, v_r,
                                  self.rk32.astype(np.float64), self.rv32.astype(np.float64))


def _check_sampled(sc, out, requests):
    for b in requests:
        ref = sc.expected(b)
        err = H.relative_error(out[b], ref)
        assert np.all(np.isfinite(out[b]))
        assert err.max() <= TOL, "request %d: max relative error %.3g" % (b, err.max())


def test_qwen3_32b_layer_batch64_ragged_shared_prefix():
    ctxs = synth.ragged_lengths(1004, 64, 8192, 131072)
    sc = RandomHistory(1004, ctxs, n_kv=8, g=8, shared_prefix_hist=32768 - 64)
    # the shared prefix really is shared: page 0 is one physical page for all
    assert len(set(sc.table[:, 0].tolist())) == 1
    cache, q = H.to_device(sc)
    out, status = H.run_decode(cache, q)
    assert status == 0
    order = np.argsort(sc.hist_len)
    _check_sampled(sc, out, [int(order[0]), int(order[-1]), int(order[len(order) // 2]), 7])


def test_qwen3_4b_layer_batch28_100k_with_demotion():
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    sc = RandomHistory(1003, [100_000] * 28, n_kv=8, g=4)
    pool0 = sc.pool.copy()          # the oracle reads the history as generated
    cache, q = H.to_device(sc)
    out, status = H.run_decode(cache, q)
    assert status == 0
    sc.pool = pool0
    _check_sampled(sc, out, [0, 13, 27])
    # one demotion per request and step, eight steps, into history positions
    # hist_len .. hist_len + 7 (the tail page and the next); 28 x 8 tokens x
    # 8 KV heads x 128 codes, enough for the 1e-4 bound on mismatches
    n, steps = sc.B, 8
    xk = synth.activations(1003, (3, 0), n * steps, sc.outl)
    xv = synth.activations(1003, (3, 1), n * steps, sc.outl)
    dev = q.device
    k_src = torch.from_numpy(xk).to(torch.bfloat16).to(dev).contiguous()
    v_src = torch.from_numpy(xv).to(torch.bfloat16).to(dev).contiguous()
    dr = torch.arange(n, dtype=torch.int32, device=dev)
    for step in range(steps):
        si = torch.arange(step * n, (step + 1) * n, dtype=torch.int32, device=dev)
        dp = torch.from_numpy(sc.hist_len.copy() + step).to(dev)
        B.oscar_quantize_append(cache.desc(int(sc.hist_len.max()) + steps), k_src.view(torch.uint16),
                                v_src.view(torch.uint16), n * steps, sc.n_kv * 128, si, dr, dp, n, None, None)
    torch.cuda.synchronize()
    assert int(cache.dev_status.item()) == 0
    pool = cache.pages.cpu().numpy()
    for which, x, r32, tau in ((0, xk, sc.rk32, sc.tau_k), (1, xv, sc.rv32, sc.tau_v)):
        got = [O.load_history_bulk(pool, sc.table, sc.n_kv, b, int(sc.hist_len[b]) + steps, which) for b in range(n)]
        # token step * n + b went to request b, position hist_len[b] + step
        gc = np.stack([got[b][0][-steps + st] for st in range(steps) for b in range(n)])
        gs = np.stack([got[b][1][-steps + st] for st in range(steps) for b in range(n)])
        gz = np.stack([got[b][2][-steps + st] for st in range(steps) for b in range(n)])
        xr = np.stack([np.clip(x[:, h].astype(np.float64) @ r32[h].astype(np.float64), -tau, tau)
                       for h in range(sc.n_kv)], axis=1)
        rc, rs, rz = H.demote_heads(x, r32, tau)
        H.code_parity(xr, gc, gs, gz, rc, rs, rz, (xr.max(-1) - xr.min(-1)) / 3.0, xr.min(-1))


def test_bulk_demotion_128k_then_decode():
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    from bit_rotated_kv_split_gb300.cache import LayerCache
    seed, n_kv, g, ctx = 1005, 8, 4, 131_072
    outl = synth.outlier_channels(seed, 0, n_kv)
    rk32, rv32, tau_k, tau_v = H.rotations(seed, 0, n_kv, outl, n_q=1024, n_k=512)
    sl, hl, rl = synth.history_split(ctx)
    xk = synth.activations(seed, (0, 0, 0), ctx, outl)
    xv = synth.activations(seed, (0, 0, 1), ctx, outl)
    table, n_pages = synth.page_table(seed, [hl], n_extra_pages=0)
    dev = torch.device("cuda")
    cache = LayerCache(1, n_kv * g, n_kv, table.shape[1], n_pages, torch.from_numpy(rk32),
                       torch.from_numpy(rv32), tau_k, tau_v, device=dev)
    cache.page_table.copy_(torch.from_numpy(table))
    k_src = torch.from_numpy(xk).to(torch.bfloat16).to(dev).contiguous()
    v_src = torch.from_numpy(xv).to(torch.bfloat16).to(dev).contiguous()
    # contiguous source rows (the prefill buffer from its first history
    # token, no index): the tile-copy path of the bulk kernel
    dr = torch.zeros(hl, dtype=torch.int32, device=dev)
    dp = torch.arange(hl, dtype=torch.int32, device=dev)
    B.oscar_quantize_append(cache.desc(hl), k_src[sl:].view(torch.uint16), v_src[sl:].view(torch.uint16),
                            ctx - sl, n_kv * 128, None, dr, dp, hl, None, None)
    torch.cuda.synchronize()
    assert int(cache.dev_status.item()) == 0
    # demotion parity on every token
    pool = cache.pages.cpu().numpy()
    hist = {}
    for which, x, r32, tau, tag in ((0, xk, rk32, tau_k, "k"), (1, xv, rv32, tau_v, "v")):
        gc, gs, gz = O.load_history_bulk(pool, table, n_kv, 0, hl, which)
        xh = x[sl:sl + hl]
        xr = np.stack([np.clip(xh[:, h].astype(np.float64) @ r32[h].astype(np.float64), -tau, tau)
                       for h in range(n_kv)], axis=1)
        rc, rs, rz = H.demote_heads(xh, r32, tau)
        H.code_parity(xr, gc, gs, gz, rc, rs, rz, (xr.max(-1) - xr.min(-1)) / 3.0, xr.min(-1))
        hist.update({"codes_" + tag: rc, "scale_" + tag: rs, "zero_" + tag: rz})
    # decode over identical codes: the oracle's demotion placed in the pool
    # (the tolerance is stated for outputs computed from identical codes)
    pool_ref = np.zeros_like(pool)
    O.store_history_bulk(pool_ref, table, n_kv, 0, 0, O.pack(hist["codes_k"]), hist["scale_k"], hist["zero_k"], 0)
    O.store_history_bulk(pool_ref, table, n_kv, 0, 0, O.pack(hist["codes_v"]), hist["scale_v"], hist["zero_v"], 1)
    cache.pages.copy_(torch.from_numpy(pool_ref))
    cache.hist_len.fill_(hl)
    cache.sink_len.fill_(sl)
    cache.recent_len.fill_(rl)
    cache.recent_start.fill_(0)
    cache.sink_k[0, :sl] = k_src[:sl]
    cache.sink_v[0, :sl] = v_src[:sl]
    cache.recent_k[0, :rl] = k_src[sl + hl:]
    cache.recent_v[0, :rl] = v_src[sl + hl:]
    cache.max_hist = hl
    qo = np.repeat(outl, g, axis=0)
    qh = synth.activations(seed, (0, 0, 2), 1, qo)
    q = torch.from_numpy(qh).to(torch.bfloat16).to(dev)
    out, status = H.run_decode(cache, q)
    assert status == 0
    ref = O.decode_attention(qh[0].astype(np.float64), xk[:sl], xv[:sl], hist, xk[sl + hl:], xv[sl + hl:],
                             rk32.astype(np.float64), rv32.astype(np.float64))
    err = H.relative_error(out[0], ref)
    assert err.max() <= TOL, "max relative error %.3g" % err.max()
