"""GPU parity of oscar_quantize_append (rotate, clip, quantise, pack, place).

Codes, scales and zero points produced on the GPU are read back from the
page pool with the oracle's reader and compared with the oracle's demotion of
the same bf16 tokens under the same fp32 rotation, with the comparison rule in
`harness.code_parity`.
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


def _pre_rounding(x_rot_clipped):
    mn = x_rot_clipped.min(-1)
    mx = x_rot_clipped.max(-1)
    return (mx - mn) / 3.0, mn


def _run(seed, n_tok, n_kv, positions=None, with_new=False, canalized_block=None, first_row=None,
         groups=None, levels=None, scale=None, overlapped=False):
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    from bit_rotated_kv_split_gb300.cache import LayerCache
    outl = synth.outlier_channels(seed, 0, n_kv)
    if canalized_block is None:
        rk32, rv32, tau_k, tau_v = H.rotations(seed, 0, n_kv, outl, n_q=1024, n_k=512)
    else:
        rk32, rv32, tau_k, tau_v = H.canalized_rotations(seed, 0, n_kv, outl, canalized_block)
    xk = synth.activations(seed, (1, 0), n_tok, outl)
    xv = synth.activations(seed, (1, 1), n_tok, outl)
    if scale is not None:
        # rows scaled by a power of two (still bf16 values), thresholds with
        # them up to the largest the library accepts
        xk = xk * np.float32(scale)
        xv = xv * np.float32(scale)
        tau_k, tau_v = min(tau_k * scale, 65504.0), min(tau_v * scale, 65504.0)
    g = synth.generator(seed, 5)
    src_index = g.permutation(n_tok).astype(np.int32)
    if first_row is not None:
        # contiguous rows: item i reads row first_row + i of the buffer (no
        # index; the bulk kernel's tile copies)
        src_index = np.arange(first_row, first_row + n_tok, dtype=np.int32)
        xk = np.concatenate([synth.activations(seed, (1, 7), first_row, outl), xk])
        xv = np.concatenate([synth.activations(seed, (1, 8), first_row, outl), xv])
    if positions is None:
        positions = np.arange(n_tok)
    hist = int(positions.max()) + 1
    table, n_pages = synth.page_table(seed, [hist], n_extra_pages=0)
    gk, gv = groups if groups is not None else (128, 128)
    cache = LayerCache(1, n_kv * 4, n_kv, table.shape[1], n_pages, torch.from_numpy(rk32),
                       torch.from_numpy(rv32), tau_k, tau_v, quant_group_k=gk, quant_group_v=gv,
                       levels_k=None if levels is None else levels[0],
                       levels_v=None if levels is None else levels[1])
    cache.page_table.copy_(torch.from_numpy(table))
    dev = torch.device("cuda")
    k_src = torch.from_numpy(xk).to(torch.bfloat16).to(dev).contiguous()
    v_src = torch.from_numpy(xv).to(torch.bfloat16).to(dev).contiguous()
    si = None if first_row is not None else torch.from_numpy(src_index).to(dev)
    dr = torch.zeros(n_tok, dtype=torch.int32, device=dev)
    dp = torch.from_numpy(positions.astype(np.int32)).to(dev)
    new_k = new_v = None
    if with_new:
        nk = synth.activations(seed, (1, 2), n_tok, outl)
        nv = synth.activations(seed, (1, 3), n_tok, outl)
        new_k = torch.from_numpy(nk).to(torch.bfloat16).to(dev)
        new_v = torch.from_numpy(nv).to(torch.bfloat16).to(dev)
    k_in = k_src[first_row:] if first_row is not None else k_src
    v_in = v_src[first_row:] if first_row is not None else v_src
    append = B.oscar_quantize_append_overlapped if overlapped else B.oscar_quantize_append
    append(cache.desc(hist), k_in.view(torch.uint16), v_in.view(torch.uint16),
           k_in.shape[0], n_kv * 128, si, dr, dp, n_tok,
           None if new_k is None else new_k.view(torch.uint16),
           None if new_v is None else new_v.view(torch.uint16))
    torch.cuda.synchronize()
    assert int(cache.dev_status.item()) == 0
    pool = cache.pages.cpu().numpy()
    res = {}
    for which, x, r32, tau, gsz in ((0, xk, rk32, tau_k, gk), (1, xv, rv32, tau_v, gv)):
        xs = x[src_index]                                  # token written to position i
        xr = np.stack([np.clip(xs[:, h].astype(np.float64) @ r32[h].astype(np.float64), -tau, tau)
                       for h in range(n_kv)], axis=1)
        if groups is None:
            gc, gs, gz = O.load_history_bulk(pool, table, n_kv, 0, hist, which)
            gc, gs, gz = gc[positions], gs[positions], gz[positions]
            lv = None if levels is None else levels[which]
            if lv is None:
                rc, rs, rz = H.demote_heads(xs, r32, tau)
            else:
                rc, rs, rz = H.demote_heads_codebook(xs, r32, tau, lv)
            pre_s, pre_z = _pre_rounding(xr)
            res[which] = H.code_parity(xr, gc, gs, gz, rc, rs, rz, pre_s, pre_z, levels=lv)
            continue
        # groups: each group of gsz channels is compared as its own vector
        ng = 128 // gsz
        gc, gs, gz = O.load_history_groups(pool, table, n_kv, 0, hist, which, 128 // gk, 128 // gv)
        gc, gs, gz = gc[positions], gs[positions], gz[positions]
        rc, rs, rz = H.demote_heads(xs, r32, tau, gsz)
        shp = (n_tok, n_kv, ng, gsz)
        xg = xr.reshape(shp)
        pre_s, pre_z = _pre_rounding(xg)
        res[which] = H.code_parity(xg, gc.reshape(shp), gs, gz, rc.reshape(shp), rs, rz, pre_s, pre_z)
    if with_new:
        np.testing.assert_array_equal(k_src.float().cpu().numpy()[src_index], nk)
        np.testing.assert_array_equal(v_src.float().cpu().numpy()[src_index], nv)
    return res


def _lloyd_levels(seed, n_kv):
    """(levels_k, levels_v): the oracle's Lloyd-Max fit on seeded calibration rows."""
    outl = synth.outlier_channels(seed, 0, n_kv)
    rk32, rv32, tau_k, tau_v = H.rotations(seed, 0, n_kv, outl, n_q=1024, n_k=512)
    out = []
    for r32, tau, sub in ((rk32, tau_k, 0), (rv32, tau_v, 1)):
        x = synth.activations(seed, (3, sub), 256, outl)
        out.append(np.asarray(O.fit_codebook(x[:, 0].astype(np.float64), r32[0].astype(np.float64), tau),
                              np.float16))
    return tuple(out)


@pytest.mark.parametrize("variant", ["uniform", "groups32", "groups64x128", "levels", "bulk"])
def test_overlapped_entry_point_matches_oracle(variant):
    """oscar_quantize_append_overlapped (every kernel form it instantiates,
    and the tensor-core path it forwards to) under the same code rule."""
    if variant == "bulk":
        res = _run(2016, 1500, 2, overlapped=True)
    else:
        groups = {"groups32": (32, 32), "groups64x128": (64, 128)}.get(variant)
        levels = _lloyd_levels(2015, 4) if variant == "levels" else None
        res = _run(2015, 300, 4, with_new=True, groups=groups, levels=levels, overlapped=True)
    print(res)


def test_demote_tiny_config_tokens():
    # 1728 tokens: the tensor-core bulk path
    res = _run(2001, 1728, 1)
    print(res)


def test_demote_bulk_path_eight_heads_ragged_tail():
    # 3000 tokens (not a multiple of the 128-token tile), scattered positions
    g = synth.generator(4, 1)
    pos = g.permutation(5000)[:3000]
    res = _run(2004, 3000, 8, positions=pos)
    print(res)


def test_demote_bulk_path_contiguous_rows_ragged_tail():
    # 3000 contiguous rows starting at row 77 of the buffer (no index), so
    # the last 128-token tile is partial and the tile copies start mid-buffer
    g = synth.generator(6, 1)
    pos = g.permutation(4000)[:3000]
    res = _run(2005, 3000, 4, positions=pos, first_row=77)
    print(res)


def test_demote_eight_heads_scattered_positions():
    g = synth.generator(3, 1)
    pos = g.permutation(700)[:333]
    res = _run(2002, 333, 8, positions=pos)
    print(res)


def test_demote_writes_new_token_into_freed_rows():
    # 512 tokens x 4 KV heads: enough codes for the 1e-4 bound on mismatches
    _run(2003, 512, 4, with_new=True)


def test_append_then_decode_matches_oracle_steps():
    """Decode steps: demote the oldest recent token into history, write the new
    token into its ring slot, attend; the oracle replays the same steps with
    its own demotion."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    sc = H.Scenario(2004, [1000, 700], n_kv=2, g=4)
    cache, q = H.to_device(sc)
    dev = q.device
    steps = 5
    outl = sc.outl
    hist = [dict((k, v.copy()) for k, v in h.items()) for h in sc.hist]
    recents = [list(zip(*sc.segments(b)[2:])) for b in range(sc.B)]
    start = sc.recent_start.copy()
    hist_len = sc.hist_len.copy()
    for step in range(steps):
        newk = synth.activations(sc.seed, (7, step, 0), sc.B, outl)
        newv = synth.activations(sc.seed, (7, step, 1), sc.B, outl)
        src = torch.tensor([b * 256 + int(start[b]) for b in range(sc.B)], dtype=torch.int32, device=dev)
        dr = torch.arange(sc.B, dtype=torch.int32, device=dev)
        dp = torch.from_numpy(hist_len.astype(np.int32)).to(dev)
        B.oscar_quantize_append(cache.desc(int(hist_len.max()) + 1), cache.recent_k.view(torch.uint16),
                                cache.recent_v.view(torch.uint16), sc.B * 256, sc.n_kv * 128, src,
                                dr, dp, sc.B,
                                torch.from_numpy(newk).to(torch.bfloat16).to(dev).view(torch.uint16),
                                torch.from_numpy(newv).to(torch.bfloat16).to(dev).view(torch.uint16))
        for b in range(sc.B):
            ok, ov = recents[b].pop(0)
            ck, sk, zk = H.demote_heads(ok[None], sc.rk32, sc.tau_k)
            cv, sv, zv = H.demote_heads(ov[None], sc.rv32, sc.tau_v)
            for name, arr in (("codes_k", ck), ("scale_k", sk), ("zero_k", zk), ("codes_v", cv),
                              ("scale_v", sv), ("zero_v", zv)):
                hist[b][name] = np.concatenate([hist[b][name], arr])
            recents[b].append((newk[b], newv[b]))
        hist_len += 1
        start = (start + 1) % 256
        cache.hist_len.copy_(torch.from_numpy(hist_len))
        cache.recent_start.copy_(torch.from_numpy(start.astype(np.int32)))
        cache.max_hist = int(hist_len.max())
        out, status = H.run_decode(cache, q)
        assert status == 0
        ref = np.zeros_like(out)
        for b in range(sc.B):
            sk_, sv_, _, _ = sc.segments(b)
            rk = np.stack([x[0] for x in recents[b]])
            rv = np.stack([x[1] for x in recents[b]])
            ref[b] = O.decode_attention(sc.q[b].astype(np.float64), sk_, sv_, hist[b], rk, rv,
                                        sc.rk32.astype(np.float64), sc.rv32.astype(np.float64))
        err = H.relative_error(out, ref)
        assert err.max() <= 2e-3, (step, err.max())


@pytest.mark.parametrize("n_layers", [1, 2])
def test_overlapped_append_in_a_decode_chain(n_layers):
    """oscar_quantize_append_overlapped reads and rotates while the previous
    kernel (the attention of the layer before, or of the same layer one step
    earlier) still runs.  A chain of steps launched back to back with no
    host synchronisation gives the pages, rings and outputs of the same chain
    with oscar_quantize_append bit for bit, and the last step's output of
    layer 0 matches the oracle replaying the steps."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    steps = 4
    base = H.Scenario(2013, [1100, 600], n_kv=2, g=4)
    dev = torch.device("cuda", 0)
    newk = [[synth.activations(base.seed, (10, s, i, 0), base.B, base.outl) for i in range(n_layers)]
            for s in range(steps)]
    newv = [[synth.activations(base.seed, (10, s, i, 1), base.B, base.outl) for i in range(n_layers)]
            for s in range(steps)]
    results = []
    for overlapped in (False, True):
        append = B.oscar_quantize_append_overlapped if overlapped else B.oscar_quantize_append
        layers = [H.to_device(base) for _ in range(n_layers)]
        q = layers[0][1]
        # per-step lengths and ring starts, resident before the chain starts
        hl = [torch.from_numpy((base.hist_len + s).astype(np.int32)).to(dev) for s in range(steps + 1)]
        rs = [torch.from_numpy(((base.recent_start + s) % 256).astype(np.int32)).to(dev) for s in range(steps + 1)]
        src = [torch.tensor([b * 256 + (int(base.recent_start[b]) + s) % 256 for b in range(base.B)],
                            dtype=torch.int32, device=dev) for s in range(steps)]
        dr = torch.arange(base.B, dtype=torch.int32, device=dev)
        nk = [[torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in row] for row in newk]
        nv = [[torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in row] for row in newv]
        outs = [[torch.empty(q.shape, dtype=torch.float32, device=dev) for _ in range(n_layers)]
                for _ in range(steps)]
        # one workspace per launch (the chain keeps several in flight)
        wss = [torch.zeros(B.oscar_decode_workspace_bytes(layers[0][0].desc(int(base.hist_len.max()) + s + 1)),
                           dtype=torch.uint8, device=dev) for s in range(steps) for _ in range(n_layers)]
        torch.cuda.synchronize()
        for s in range(steps):
            for i, (cache, _) in enumerate(layers):
                da = cache.desc(int(base.hist_len.max()) + s + 1)
                da.hist_len, da.recent_start = hl[s].data_ptr(), rs[s].data_ptr()
                dd = cache.desc(int(base.hist_len.max()) + s + 1)
                dd.hist_len, dd.recent_start = hl[s + 1].data_ptr(), rs[s + 1].data_ptr()
                append(da, cache.recent_k.view(torch.uint16), cache.recent_v.view(torch.uint16), base.B * 256,
                       base.n_kv * 128, src[s], dr, hl[s], base.B, nk[s][i].view(torch.uint16),
                       nv[s][i].view(torch.uint16))
                ws = wss[s * n_layers + i]
                B.oscar_decode_attention(dd, q, outs[s][i], ws, ws.numel())
        torch.cuda.synchronize()
        for cache, _ in layers:
            assert int(cache.dev_status.item()) == 0
        results.append([o.cpu().numpy() for row in outs for o in row] +
                       [t.cpu().numpy() for cache, _ in layers
                        for t in (cache.pages, cache.recent_k.view(torch.uint16), cache.recent_v.view(torch.uint16))])
    for a, b in zip(*results):
        np.testing.assert_array_equal(a, b)
    # the oracle replays layer 0's steps with its own demotion
    hist = [dict((k, v.copy()) for k, v in h.items()) for h in base.hist]
    recents = [list(zip(*base.segments(b)[2:])) for b in range(base.B)]
    for s in range(steps):
        for b in range(base.B):
            ok, ov = recents[b].pop(0)
            ck, sk, zk = H.demote_heads(ok[None], base.rk32, base.tau_k)
            cv, sv, zv = H.demote_heads(ov[None], base.rv32, base.tau_v)
            for name, arr in (("codes_k", ck), ("scale_k", sk), ("zero_k", zk), ("codes_v", cv),
                              ("scale_v", sv), ("zero_v", zv)):
                hist[b][name] = np.concatenate([hist[b][name], arr])
            recents[b].append((newk[s][0][b], newv[s][0][b]))
    got = results[1][(steps - 1) * n_layers].astype(np.float64)
    ref = np.zeros_like(got)
    for b in range(base.B):
        sk_, sv_, _, _ = base.segments(b)
        rk = np.stack([x[0] for x in recents[b]])
        rv = np.stack([x[1] for x in recents[b]])
        ref[b] = O.decode_attention(base.q[b].astype(np.float64), sk_, sv_, hist[b], rk, rv,
                                    base.rk32.astype(np.float64), base.rv32.astype(np.float64))
    err = H.relative_error(got, ref)
    assert err.max() <= 2e-3, err.max()


def test_decode_step_equals_separate_calls():
    """oscar_decode_step (staged H2D copy, demotion, decode, D2H copy) gives the
    output of oscar_quantize_append + oscar_decode_attention bit for bit."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    sc = H.Scenario(2010, [1500, 900], n_kv=2, g=4)
    outs = []
    for fused in (False, True):
        cache, q = H.to_device(sc)
        dev = q.device
        newk = synth.activations(sc.seed, (8, 0), sc.B, sc.outl)
        newv = synth.activations(sc.seed, (8, 1), sc.B, sc.outl)
        host = torch.cat([q.cpu().flatten(), torch.from_numpy(newk).to(torch.bfloat16).flatten(),
                          torch.from_numpy(newv).to(torch.bfloat16).flatten()]).pin_memory()
        stage = torch.empty(host.numel(), dtype=torch.bfloat16, device=dev)
        nq, nk = q.numel(), newk.size
        q_s, nk_s, nv_s = stage[:nq].view_as(q), stage[nq:nq + nk], stage[nq + nk:]
        src = torch.tensor([b * 256 + int(sc.recent_start[b]) for b in range(sc.B)], dtype=torch.int32, device=dev)
        dr = torch.arange(sc.B, dtype=torch.int32, device=dev)
        dp = torch.from_numpy(sc.hist_len.astype(np.int32)).to(dev)
        desc = cache.desc(int(sc.hist_len.max()) + 1)
        nbytes = B.oscar_decode_workspace_bytes(desc)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        out = torch.empty(q.shape, dtype=torch.float32, device=dev)
        host_out = torch.zeros(q.shape, dtype=torch.float32).pin_memory()
        args = (cache.recent_k.view(torch.uint16), cache.recent_v.view(torch.uint16), sc.B * 256, sc.n_kv * 128,
                src, dr, dp, sc.B, nk_s.view(torch.uint16), nv_s.view(torch.uint16))
        if fused:
            B.oscar_decode_step(desc, host, stage, host.numel() * 2, *args, q_s, out, ws, nbytes, host_out)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(host_out.numpy(), out.cpu().numpy())
        else:
            stage.copy_(host)
            B.oscar_quantize_append(desc, *args)
            B.oscar_decode_attention(desc, q_s, out, ws, nbytes)
            torch.cuda.synchronize()
        assert int(cache.dev_status.item()) == 0
        outs.append((out.cpu().numpy(), cache.pages.cpu().numpy(), cache.recent_k.float().cpu().numpy()))
    for a, b in zip(outs[0], outs[1]):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("staged", [False, True])
def test_decode_step_overlap_flag_in_a_chain(staged):
    """oscar_decode_step calls launched back to back over two layers: with
    OSCAR_STEP_OVERLAP_PREVIOUS (the demotion overlaps the previous call's
    decode) the outputs, pages and rings equal those without it bit for bit,
    both with the inputs read straight from pinned host memory and with them
    staged by the copy kernel (host buffer off the device buffer's 16-byte
    alignment), where the flag must leave the demotion waiting first."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    steps, n_layers = 3, 2
    base = H.Scenario(2014, [900, 1400], n_kv=2, g=4)
    dev = torch.device("cuda", 0)
    results = []
    for flags in (0, B.OSCAR_STEP_OVERLAP_PREVIOUS):
        layers = [H.to_device(base) for _ in range(n_layers)]
        q = layers[0][1]
        hl = [torch.from_numpy((base.hist_len + s).astype(np.int32)).to(dev) for s in range(steps + 1)]
        rs = [torch.from_numpy(((base.recent_start + s) % 256).astype(np.int32)).to(dev) for s in range(steps + 1)]
        src = [torch.tensor([b * 256 + (int(base.recent_start[b]) + s) % 256 for b in range(base.B)],
                            dtype=torch.int32, device=dev) for s in range(steps)]
        dr = torch.arange(base.B, dtype=torch.int32, device=dev)
        # per (step, layer): q, new K, new V in one pinned buffer and its staging range
        nq, nk = q.numel(), base.B * base.n_kv * 128
        hosts, stages = [], []
        for s in range(steps):
            for i in range(n_layers):
                newk = synth.activations(base.seed, (11, s, i, 0), base.B, base.outl)
                newv = synth.activations(base.seed, (11, s, i, 1), base.B, base.outl)
                pad = torch.zeros(4 if staged else 0, dtype=torch.bfloat16)   # 8 bytes: off the grid
                hosts.append(torch.cat([pad, q.cpu().flatten(), torch.from_numpy(newk).to(torch.bfloat16).flatten(),
                                        torch.from_numpy(newv).to(torch.bfloat16).flatten()]).pin_memory())
                stages.append(torch.empty(nq + 2 * nk, dtype=torch.bfloat16, device=dev))
        host_outs = [torch.zeros(q.shape, dtype=torch.float32).pin_memory() for _ in range(steps * n_layers)]
        out = torch.empty(q.shape, dtype=torch.float32, device=dev)
        ws_bytes = B.oscar_decode_workspace_bytes(layers[0][0].desc(int(base.hist_len.max()) + steps))
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        for s in range(steps):
            for i, (cache, _) in enumerate(layers):
                k = s * n_layers + i
                st = stages[k]
                desc = cache.desc(int(base.hist_len.max()) + s + 1)
                desc.hist_len, desc.recent_start = hl[s + 1].data_ptr(), rs[s + 1].data_ptr()
                host_in = hosts[k].data_ptr() + (8 if staged else 0)
                B.oscar_decode_step(desc, host_in, st, st.numel() * 2, cache.recent_k.view(torch.uint16),
                                    cache.recent_v.view(torch.uint16), base.B * 256, base.n_kv * 128, src[s], dr,
                                    hl[s], base.B, st[nq:nq + nk].view(torch.uint16),
                                    st[nq + nk:].view(torch.uint16), st[:nq].view_as(q), out, ws, ws_bytes,
                                    host_outs[k], flags=flags)
        torch.cuda.synchronize()
        for cache, _ in layers:
            assert int(cache.dev_status.item()) == 0
        results.append([h.numpy().copy() for h in host_outs] +
                       [t.cpu().numpy() for cache, _ in layers
                        for t in (cache.pages, cache.recent_k.view(torch.uint16), cache.recent_v.view(torch.uint16))])
    for a, b in zip(*results):
        np.testing.assert_array_equal(a, b)


def test_decode_step_output_to_unaligned_host_buffer():
    """host_out off the 16-byte grid: the output goes through the copy
    kernel instead of the decode kernel's own stores; same bytes, and the
    bytes around it untouched."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    sc = H.Scenario(2012, [1300, 700], n_kv=1, g=4)
    cache, q = H.to_device(sc)
    ref, _ = H.run_decode(cache, q)
    desc = cache.desc()
    nbytes = B.oscar_decode_workspace_bytes(desc)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    big = torch.zeros(q.numel() * 4 + 64, dtype=torch.uint8).pin_memory()
    for off in (4, 16):
        big.zero_()
        B.oscar_decode_step(desc, None, None, 0, None, None, 1, 128, None, None, None, 0, None, None, q, out, ws,
                            nbytes, big.data_ptr() + off)
        torch.cuda.synchronize()
        got = big.numpy()[off:off + q.numel() * 4].view(np.float32).reshape(q.shape)
        np.testing.assert_array_equal(got, ref.astype(np.float32))
        assert not big.numpy()[:off].any() and not big.numpy()[off + q.numel() * 4:].any()


def test_decode_step_stages_odd_sizes_and_offsets():
    """The staging copy of oscar_decode_step moves an odd number of bytes
    between addresses off the 16-byte grid exactly (byte path) and leaves the
    bytes around them alone; the decode result is unchanged (n = 0: no
    demotion)."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    sc = H.Scenario(2011, [1200], n_kv=1, g=4)
    cache, q = H.to_device(sc)
    ref, _ = H.run_decode(cache, q)
    g = synth.generator(2011, 9)
    host = torch.from_numpy(g.integers(0, 256, size=1003).astype(np.uint8)).pin_memory()
    dev = torch.zeros(1024, dtype=torch.uint8, device=q.device)
    desc = cache.desc()
    nbytes = B.oscar_decode_workspace_bytes(desc)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    for off_h, off_d, n in ((1, 3, 997), (16, 32, 960), (0, 0, 5)):
        dev.zero_()
        B.oscar_decode_step(desc, host.data_ptr() + off_h, dev.data_ptr() + off_d, n, None, None, 1, 128, None,
                            None, None, 0, None, None, q, out, ws, nbytes, None)
        torch.cuda.synchronize()
        d = dev.cpu().numpy()
        np.testing.assert_array_equal(d[off_d:off_d + n], host.numpy()[off_h:off_h + n])
        assert not d[:off_d].any() and not d[off_d + n:].any()
        np.testing.assert_array_equal(out.cpu().numpy(), ref.astype(np.float32))


def _demote_rows(xk, xv, rk32, rv32, tau_k, tau_v, per_step, groups=(128, 128)):
    """Demote the bf16 rows xk, xv [n][n_kv][128] to history positions 0..n-1
    through one path: the tensor-core bulk kernel (one call, contiguous rows)
    or the per-token kernel (calls of at most 1000 rows).  Returns the pool
    and page table."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    from bit_rotated_kv_split_gb300.cache import LayerCache
    n, n_kv = xk.shape[0], xk.shape[1]
    table, n_pages = synth.page_table(77, [n], n_extra_pages=0)
    cache = LayerCache(1, n_kv * 4, n_kv, table.shape[1], n_pages, torch.from_numpy(rk32), torch.from_numpy(rv32),
                       tau_k, tau_v, quant_group_k=groups[0], quant_group_v=groups[1])
    cache.page_table.copy_(torch.from_numpy(table))
    dev = torch.device("cuda")
    k_src = torch.from_numpy(xk).to(torch.bfloat16).to(dev).contiguous()
    v_src = torch.from_numpy(xv).to(torch.bfloat16).to(dev).contiguous()
    chunks = [(0, n)] if not per_step else [(a, min(a + 1000, n)) for a in range(0, n, 1000)]
    for a, b in chunks:
        m = b - a
        assert per_step == (m < 1024)
        dr = torch.zeros(m, dtype=torch.int32, device=dev)
        dp = torch.arange(a, b, dtype=torch.int32, device=dev)
        B.oscar_quantize_append(cache.desc(n), k_src[a:b].view(torch.uint16), v_src[a:b].view(torch.uint16), m,
                                n_kv * 128, None, dr, dp, m, None, None)
    torch.cuda.synchronize()
    assert int(cache.dev_status.item()) == 0
    return cache.pages.cpu().numpy(), table


def _parity_of_pool(pool, table, xk, xv, rk32, rv32, tau_k, tau_v, groups=(128, 128)):
    n, n_kv = xk.shape[0], xk.shape[1]
    gk, gv = groups
    out = {}
    for which, x, r32, tau, gsz in ((0, xk, rk32, tau_k, gk), (1, xv, rv32, tau_v, gv)):
        xr = np.stack([np.clip(x[:, h].astype(np.float64) @ r32[h].astype(np.float64), -tau, tau)
                       for h in range(n_kv)], axis=1)
        ng = 128 // gsz
        if (gk, gv) == (128, 128):
            gc, gs, gz = O.load_history_bulk(pool, table, n_kv, 0, n, which)
            rc, rs, rz = H.demote_heads(x, r32, tau)
            pre_s, pre_z = _pre_rounding(xr)
            out[which] = (H.code_parity(xr, gc, gs, gz, rc, rs, rz, pre_s, pre_z), gc, gs, gz)
            continue
        gc, gs, gz = O.load_history_groups(pool, table, n_kv, 0, n, which, 128 // gk, 128 // gv)
        rc, rs, rz = H.demote_heads(x, r32, tau, gsz)
        shp = (n, n_kv, ng, gsz)
        xg = xr.reshape(shp)
        pre_s, pre_z = _pre_rounding(xg)
        out[which] = (H.code_parity(xg, gc.reshape(shp), gs, gz, rc.reshape(shp), rs, rz, pre_s, pre_z),
                      gc, gs, gz)
    return out


@pytest.mark.parametrize("groups", [(128, 128), (32, 64)])
def test_same_tokens_through_both_paths(groups):
    """The same 1500 tokens demoted by the tensor-core bulk kernel (one call
    of 1500) and by the per-token kernel (calls of 1000 and 500) both meet
    the code rule against the oracle; the two results differ, if at all,
    only in codes the rule allows to differ."""
    seed, n, n_kv = 2020, 1500, 4
    outl = synth.outlier_channels(seed, 0, n_kv)
    rk32, rv32, tau_k, tau_v = H.rotations(seed, 0, n_kv, outl, n_q=1024, n_k=512)
    xk = synth.activations(seed, (3, 0), n, outl)
    xv = synth.activations(seed, (3, 1), n, outl)
    res = {}
    for per_step in (False, True):
        pool, table = _demote_rows(xk, xv, rk32, rv32, tau_k, tau_v, per_step, groups)
        res[per_step] = _parity_of_pool(pool, table, xk, xv, rk32, rv32, tau_k, tau_v, groups)
    for which in (0, 1):
        d = int(np.sum(res[False][which][1] != res[True][which][1]))
        print("KV"[which], "codes differing between the paths:", d, res[False][which][0], res[True][which][0])
        assert d <= 2 * 1e-4 * res[False][which][1].size


@pytest.mark.parametrize("scale", [2.0 ** 12, 2.0 ** -20, 2.0 ** -60])
def test_rows_far_from_unit_magnitude_through_both_paths(scale):
    """Rows scaled by 2^12 (elements far beyond the fp16 range; thresholds
    capped at 65504), by 2^-20 (most elements below fp16's normal range) and
    by 2^-60 (every scale rounds to fp16 zero): the tensor-core kernel
    (contiguous rows) and the per-token kernel both meet the code rule
    against the oracle, which rotates the bf16 rows in float64."""
    seed, n, n_kv = 2022, 1200, 2
    outl = synth.outlier_channels(seed, 0, n_kv)
    rk32, rv32, tau_k, tau_v = H.rotations(seed, 0, n_kv, outl, n_q=1024, n_k=512)
    xk = synth.activations(seed, (5, 0), n, outl) * np.float32(scale)
    xv = synth.activations(seed, (5, 1), n, outl) * np.float32(scale)
    tau_k, tau_v = min(tau_k * scale, 65504.0), min(tau_v * scale, 65504.0)
    for per_step in (False, True):
        pool, table = _demote_rows(xk, xv, rk32, rv32, tau_k, tau_v, per_step)
        res = _parity_of_pool(pool, table, xk, xv, rk32, rv32, tau_k, tau_v)
        print("per-step" if per_step else "bulk", res[0][0], res[1][0])


@pytest.mark.parametrize("scale", [2.0 ** 12, 2.0 ** -20])
def test_bulk_gathered_rows_far_from_unit_magnitude(scale):
    # the tensor-core kernel's gathered-row loader (an index array)
    g = synth.generator(7, 1)
    pos = g.permutation(2500)[:2000]
    print(_run(2023, 2000, 2, positions=pos, scale=scale))


@pytest.mark.parametrize("groups", [(128, 128), (32, 32)])
def test_constant_groups_give_zero_scale_and_codes(groups):
    """Token-head vectors whose (group of) rotated values is constant - the
    zero vector, and vectors rotated far beyond +-tau so that the clip makes
    every value equal - get scale 0 and all codes 0 in both demotion
    kernels (bulk: 1100 tokens in one call; per-token: two calls)."""
    seed, n, n_kv = 2021, 1100, 2
    outl = synth.outlier_channels(seed, 0, n_kv)
    rk32, rv32, tau_k, tau_v = H.rotations(seed, 0, n_kv, outl, n_q=1024, n_k=512)
    xk = synth.activations(seed, (4, 0), n, outl)
    xv = synth.activations(seed, (4, 1), n, outl)
    g = groups[0]
    for x, r32, tau in ((xk, rk32, tau_k), (xv, rv32, tau_v)):
        for h in range(n_kv):
            rt = r32[h].astype(np.float64).T
            x[0, h] = 0.0                                                  # the zero vector
            x[1, h] = synth.to_bf16(np.full(128, 4.0 * tau) @ rt)         # all clipped to +tau
            x[2, h] = synth.to_bf16(np.full(128, -4.0 * tau) @ rt)        # all clipped to -tau
            target = np.concatenate([np.full(g, 4.0 * tau), np.linspace(-0.5, 0.5, 128 - g) * tau])
            x[3, h] = synth.to_bf16(target @ rt)                          # first group clipped flat
    for per_step in (False, True):
        pool, table = _demote_rows(xk, xv, rk32, rv32, tau_k, tau_v, per_step, groups)
        res = _parity_of_pool(pool, table, xk, xv, rk32, rv32, tau_k, tau_v, groups)
        for which in (0, 1):
            _, gc, gs, gz = res[which]
            gs = np.asarray(gs, dtype=np.float64).reshape(n, n_kv, -1)
            gcs = gc.reshape(n, n_kv, -1)
            assert np.all(gs[0:3] == 0) and np.all(gcs[0:3] == 0)
            assert np.all(gs[3, :, 0] == 0)
            if g < 128:
                assert np.all(gs[3, :, 1:] > 0)
