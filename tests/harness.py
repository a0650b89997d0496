"""Shared builders for the parity tests: seeded inputs -> oracle expectations.

Inputs come from `synth`; every expected value comes from `oracle`.  The INT2
history the GPU decode reads is quantised and packed by the oracle (never by
the CUDA path), so decode parity is measured on identical codes.
"""
from __future__ import annotations

import numpy as np

import oracle as O
import synth

D = 128


def rotations(seed: int, layer: int, n_kv: int, outl: np.ndarray, n_q: int = 4096, n_k: int = 2048):
    """Per-KV-head oracle rotations (as fp32, the precision uploaded) and per-layer taus."""
    rk, rv, ck, cv = [], [], [], []
    for h in range(n_kv):
        cal = synth.calibration_set(seed, layer, h, outl[h], n_q=n_q, n_k=n_k)
        rk.append(O.rotation_from_covariance(O.query_covariance(cal["q"])))
        rv.append(O.rotation_from_covariance(O.value_covariance(cal["q"], cal["k"], cal["v"])))
        ck.append(cal["k"])
        cv.append(cal["v"])
    rk32 = np.stack(rk).astype(np.float32)
    rv32 = np.stack(rv).astype(np.float32)
    tau_k = float(np.float32(O.clip_threshold(np.stack([ck[h] @ rk32[h].astype(np.float64)
                                                        for h in range(n_kv)]))))
    tau_v = float(np.float32(O.clip_threshold(np.stack([cv[h] @ rv32[h].astype(np.float64)
                                                        for h in range(n_kv)]))))
    return rk32, rv32, tau_k, tau_v


def canalized_rotations(seed: int, layer: int, n_kv: int, outl: np.ndarray, block: int,
                        n_q: int = 1024, n_k: int = 512):
    """The OScaR block-diagonal rotation for every KV head (K and V), as fp32,
    with per-layer taus from the calibration rows rotated by it."""
    r = O.canalized_rotation(128, block).astype(np.float32)
    r32 = np.stack([r] * n_kv)
    ck, cv = [], []
    for h in range(n_kv):
        cal = synth.calibration_set(seed, layer, h, outl[h], n_q=n_q, n_k=n_k)
        ck.append(cal["k"] @ r.astype(np.float64))
        cv.append(cal["v"] @ r.astype(np.float64))
    tau_k = float(np.float32(O.clip_threshold(np.stack(ck))))
    tau_v = float(np.float32(O.clip_threshold(np.stack(cv))))
    return r32, r32.copy(), tau_k, tau_v


def demote_heads(x: np.ndarray, r32: np.ndarray, tau: float, group: int = None):
    """Oracle demotion of x [T][n_kv][d] with per-head rotations: (codes, scale16, zero16).

    group None: one group per vector, scale/zero [T][n_kv]; group g: groups of
    g channels, scale/zero [T][n_kv][d / g].
    """
    t, n_kv, d = x.shape
    codes = np.zeros((t, n_kv, d), np.uint8)
    if group is None:
        s = np.zeros((t, n_kv), np.float16)
        z = np.zeros((t, n_kv), np.float16)
        for h in range(n_kv):
            codes[:, h], s[:, h], z[:, h] = O.demote(x[:, h].astype(np.float64), r32[h].astype(np.float64), tau)
        return codes, s, z
    s = np.zeros((t, n_kv, d // group), np.float16)
    z = np.zeros((t, n_kv, d // group), np.float16)
    for h in range(n_kv):
        codes[:, h], s[:, h], z[:, h] = O.quantize_groups(
            O.rotate(x[:, h].astype(np.float64), r32[h].astype(np.float64)), tau, group)
    return codes, s, z


def demote_heads_codebook(x: np.ndarray, r32: np.ndarray, tau: float, levels):
    """Oracle codebook demotion of x [T][n_kv][d]: (codes, scale16 [T][n_kv], zero16 [T][n_kv])."""
    t, n_kv, d = x.shape
    codes = np.zeros((t, n_kv, d), np.uint8)
    s = np.zeros((t, n_kv), np.float16)
    z = np.zeros((t, n_kv), np.float16)
    for h in range(n_kv):
        codes[:, h], s[:, h], z[:, h] = O.quantize_codebook(
            O.rotate(x[:, h].astype(np.float64), r32[h].astype(np.float64)), tau, levels)
    return codes, s, z


class Scenario:
    """A seeded batch of three-segment caches with oracle expectations."""

    def __init__(self, seed: int, ctxs, n_kv: int = 1, g: int = 4, shared_prefix_hist: int = 0,
                 cal=(1024, 512), ring_start=None, identity_pages: bool = False, rot=None,
                 sink_cap: int = 64, recent_cap: int = 256, groups=(128, 128), levels=None,
                 scales=(1.0, 1.0, 1.0)):
        # scales: powers of two applied to the keys, values and queries (bf16
        # values stay exact); the clip thresholds scale with K and V
        self.seed, self.ctxs, self.n_kv, self.g = seed, [int(c) for c in ctxs], n_kv, g
        self.gk, self.gv = int(groups[0]), int(groups[1])
        # levels: (levels_k, levels_v) of a Lloyd-Max codebook (fp16), or None
        self.levels = None if levels is None else tuple(np.asarray(l, np.float16) for l in levels)
        grouped = (self.gk, self.gv) != (D, D)
        ngk, ngv = D // self.gk, D // self.gv
        self.B = len(self.ctxs)
        self.h_q = n_kv * g
        self.sink_cap, self.recent_cap = sink_cap, recent_cap
        self.outl = synth.outlier_channels(seed, 0, n_kv)
        if rot is None:
            rot = rotations(seed, 0, n_kv, self.outl, n_q=cal[0], n_k=cal[1])
        self.rk32, self.rv32, self.tau_k, self.tau_v = rot
        sk_, sv_, sq_ = (float(x) for x in scales)
        self.tau_k, self.tau_v = self.tau_k * sk_, self.tau_v * sv_
        splits = [synth.history_split(c, sink_cap, recent_cap) for c in self.ctxs]
        self.sink_len = np.array([s[0] for s in splits], np.int32)
        self.hist_len = np.array([s[1] for s in splits], np.int32)
        self.recent_len = np.array([s[2] for s in splits], np.int32)
        gstart = synth.generator(seed, 77)
        if ring_start is None:
            self.recent_start = gstart.integers(0, max(recent_cap, 1), size=self.B).astype(np.int32)
        else:
            self.recent_start = np.full(self.B, ring_start, np.int32)
        self.table, self.n_pages = synth.page_table(seed, self.hist_len, n_extra_pages=1,
                                                    shared_prefix_tokens=shared_prefix_hist)
        if identity_pages:
            order = np.unique(self.table[self.table >= 0])
            remap = {int(p): i for i, p in enumerate(order)}
            self.table = np.vectorize(lambda p: remap.get(int(p), -1))(self.table).astype(np.int32)
        shared_ctx = sink_cap + shared_prefix_hist if shared_prefix_hist else 0
        self.k_tok, self.v_tok = [], []
        for b, c in enumerate(self.ctxs):
            k = synth.activations(seed, (0, b, 0), c, self.outl)
            v = synth.activations(seed, (0, b, 1), c, self.outl)
            if shared_ctx:
                m = min(shared_ctx, c)
                k[:m] = synth.activations(seed, (0, 9999, 0), shared_ctx, self.outl)[:m]
                v[:m] = synth.activations(seed, (0, 9999, 1), shared_ctx, self.outl)[:m]
            self.k_tok.append(k * sk_)
            self.v_tok.append(v * sv_)
        qo = np.repeat(self.outl, g, axis=0)
        self.q = np.stack([synth.activations(seed, (0, b, 2), 1, qo)[0] for b in range(self.B)]) * sq_
        # oracle history codes and the page pool holding them
        self.pool = np.zeros(self.n_pages * n_kv * O.block_bytes(ngk, ngv), np.uint8)
        self.hist = []
        for b in range(self.B):
            sl, hl = int(self.sink_len[b]), int(self.hist_len[b])
            xk = self.k_tok[b][sl:sl + hl]
            xv = self.v_tok[b][sl:sl + hl]
            if self.levels is not None:
                ck, sk, zk = demote_heads_codebook(xk, self.rk32, self.tau_k, self.levels[0])
                cv, sv, zv = demote_heads_codebook(xv, self.rv32, self.tau_v, self.levels[1])
            else:
                ck, sk, zk = demote_heads(xk, self.rk32, self.tau_k, self.gk if grouped else None)
                cv, sv, zv = demote_heads(xv, self.rv32, self.tau_v, self.gv if grouped else None)
            self.hist.append(dict(codes_k=ck, scale_k=sk, zero_k=zk, codes_v=cv, scale_v=sv, zero_v=zv))
            if self.levels is not None:
                self.hist[-1]["levels_k"], self.hist[-1]["levels_v"] = self.levels
            if hl and grouped:
                O.store_history_groups(self.pool, self.table, n_kv, b, 0, ck, sk, zk, 0, ngk, ngv)
                O.store_history_groups(self.pool, self.table, n_kv, b, 0, cv, sv, zv, 1, ngk, ngv)
            elif hl:
                O.store_history_bulk(self.pool, self.table, n_kv, b, 0, O.pack(ck), sk, zk, 0)
                O.store_history_bulk(self.pool, self.table, n_kv, b, 0, O.pack(cv), sv, zv, 1)

    def segments(self, b):
        sl, hl, rl = int(self.sink_len[b]), int(self.hist_len[b]), int(self.recent_len[b])
        k, v = self.k_tok[b], self.v_tok[b]
        return (k[:sl], v[:sl], k[sl + hl:sl + hl + rl], v[sl + hl:sl + hl + rl])

    def expected(self):
        out = np.zeros((self.B, self.h_q, D))
        for b in range(self.B):
            sk, sv, rk, rv = self.segments(b)
            out[b] = O.decode_attention(self.q[b].astype(np.float64), sk, sv, self.hist[b], rk, rv,
                                        self.rk32.astype(np.float64), self.rv32.astype(np.float64))
        return out

    def ring(self):
        """Recent tokens placed in ring slots (start + i) % cap: [B][cap][n_kv][d] float32."""
        rk = np.zeros((self.B, max(self.recent_cap, 1), self.n_kv, D), np.float32)
        rv = np.zeros_like(rk)
        for b in range(self.B):
            _, _, k, v = self.segments(b)
            for i in range(k.shape[0]):
                slot = (int(self.recent_start[b]) + i) % self.recent_cap
                rk[b, slot] = k[i]
                rv[b, slot] = v[i]
        return rk, rv

    def sink(self):
        sk = np.zeros((self.B, max(self.sink_cap, 1), self.n_kv, D), np.float32)
        sv = np.zeros_like(sk)
        for b in range(self.B):
            k, v, _, _ = self.segments(b)
            sk[b, :k.shape[0]] = k
            sv[b, :v.shape[0]] = v
        return sk, sv


REL = 1e-5        # the code rule's relative distance to a rounding boundary
MAX_FRACTION = 1e-4   # at most this fraction of codes may differ end to end


def code_parity(x_rot_clipped: np.ndarray, gpu_codes, gpu_s, gpu_z, ref_codes, ref_s, ref_z,
                pre_s: np.ndarray, pre_z: np.ndarray, levels=None, check: bool = True):
    """The demotion comparison rule (codes match except within 1e-5, relative,
    of a rounding boundary; at most 1e-4 of the codes differ).

    * codes: recomputed from the GPU's own scale/zero and the oracle's float64
      rotated value; a GPU code may differ from that only when
      u = (x - z) / s lies within 1e-5 * b of a rounding boundary b in
      {0.5, 1.5, 2.5} (with codebook `levels`: the midpoints of adjacent
      levels, and codes are nearest-level indices).  End to end at most 1e-4
      of the codes differ from the oracle's own.
    * scale/zero: fp16 bit-equal, or else the GPU's fp16 value is a rounding
      of a value within 1e-5 (relative) of the float64 pre-rounding value.
      The same rule, read in the unit of the code rule: the zero point is a
      position on the group's scale, so its distance is taken relative to
      max(|z|, s) (near z = 0 a distance relative to |z| alone would ask for
      more than any binary32 rotation holds), the scale's relative to s.
    With check=False nothing is asserted and the violation counts are
    returned with the rest.  Returns a dict of counts; raises AssertionError
    on a violation otherwise.
    """
    def fp16_check(g, r, pre, unit):
        g = g.astype(np.float16)
        r = r.astype(np.float16)
        bad = g.view(np.uint16) != r.view(np.uint16)
        if not bad.any():
            return 0, 0
        gb = g[bad].astype(np.float64)
        pb = pre[bad]
        tol = REL * unit[bad]
        # the interval of values that round to g (asymmetric at a binade edge)
        gh = g[bad]
        lo_edge = gb - (gb - np.nextafter(gh, np.float16(-np.inf)).astype(np.float64)) / 2
        hi_edge = gb + (np.nextafter(gh, np.float16(np.inf)).astype(np.float64) - gb) / 2
        ok = (pb >= lo_edge - tol) & (pb <= hi_edge + tol)
        if check and not np.all(ok):
            idx = np.argwhere(bad)[~ok][:4]
            raise AssertionError("scale/zero differ beyond the rounding rule: %d of %d differ; "
                                 "first (index, gpu, oracle, pre-rounding): %s"
                                 % (int((~ok).sum()), int(bad.size),
                                    [(tuple(int(v) for v in i), float(g[tuple(i)]), float(r[tuple(i)]),
                                      float(pre[tuple(i)])) for i in idx]))
        return int(bad.sum()), int((~ok).sum())

    pre_s = np.asarray(pre_s, dtype=np.float64)
    pre_z = np.asarray(pre_z, dtype=np.float64)
    n_s, bad_s = fp16_check(gpu_s, ref_s, pre_s, np.abs(pre_s))
    n_z, bad_z = fp16_check(gpu_z, ref_z, pre_z, np.maximum(np.abs(pre_z), np.abs(pre_s)))
    s = gpu_s.astype(np.float64)[..., None]
    z = gpu_z.astype(np.float64)[..., None]
    bounds = (0.5, 1.5, 2.5)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (x_rot_clipped - z) / s
        if levels is None:
            recomputed = np.where(s > 0, np.clip(np.rint(u), 0, 3), 0)
        else:
            lv = np.asarray(levels, dtype=np.float16).astype(np.float64)
            bounds = tuple((lv[:-1] + lv[1:]) / 2)
            recomputed = np.where(s > 0, (u > bounds[0]).astype(int) + (u > bounds[1]) + (u > bounds[2]), 0)
    diff = gpu_codes != recomputed
    far = 0
    worst = 0.0
    if diff.any():
        ud = u[diff]
        near = np.zeros(ud.shape, bool)
        dist = np.full(ud.shape, np.inf)
        for bnd in bounds:
            near |= np.abs(ud - bnd) <= REL * bnd
            dist = np.minimum(dist, np.abs(ud - bnd) / bnd)
        far = int((~near).sum())
        worst = float(dist.max())
        if check:
            assert far == 0, ("%d codes differ away from a rounding boundary (largest relative distance %.3g)"
                              % (far, worst))
    n_diff = int(np.sum(gpu_codes != ref_codes))
    e2e = n_diff / max(gpu_codes.size, 1)
    if check:
        assert n_diff <= MAX_FRACTION * gpu_codes.size, "code mismatch fraction %g (%d codes)" % (e2e, n_diff)
    return dict(scale_diff=n_s, zero_diff=n_z, boundary_codes=int(diff.sum()), e2e_fraction=e2e,
                scale_violations=bad_s, zero_violations=bad_z, far_codes=far, worst_distance=worst,
                e2e_codes=n_diff)


def relative_error(gpu: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per (request, head): max|gpu - ref| / max|ref| over the head_dim channels."""
    num = np.abs(gpu - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    return np.where(den > 0, num / np.maximum(den, 1e-300), num)


def to_device(sc: Scenario):
    """LayerCache + bf16 queries on cuda:0 holding the scenario's inputs."""
    import torch
    from bit_rotated_kv_split_gb300.cache import LayerCache
    dev = torch.device("cuda")
    cache = LayerCache(sc.B, sc.h_q, sc.n_kv, sc.table.shape[1], sc.n_pages,
                       torch.from_numpy(sc.rk32), torch.from_numpy(sc.rv32), sc.tau_k, sc.tau_v,
                       device=dev, sink_cap=sc.sink_cap, recent_cap=sc.recent_cap,
                       quant_group_k=getattr(sc, "gk", 128), quant_group_v=getattr(sc, "gv", 128),
                       levels_k=None if getattr(sc, "levels", None) is None else sc.levels[0],
                       levels_v=None if getattr(sc, "levels", None) is None else sc.levels[1])
    cache.pages.copy_(torch.from_numpy(sc.pool))
    cache.page_table.copy_(torch.from_numpy(sc.table))
    cache.hist_len.copy_(torch.from_numpy(sc.hist_len))
    cache.sink_len.copy_(torch.from_numpy(sc.sink_len))
    cache.recent_len.copy_(torch.from_numpy(sc.recent_len))
    cache.recent_start.copy_(torch.from_numpy(sc.recent_start))
    sk, sv = sc.sink()
    rk, rv = sc.ring()
    cache.sink_k.copy_(torch.from_numpy(sk).to(torch.bfloat16))
    cache.sink_v.copy_(torch.from_numpy(sv).to(torch.bfloat16))
    cache.recent_k.copy_(torch.from_numpy(rk).to(torch.bfloat16))
    cache.recent_v.copy_(torch.from_numpy(rv).to(torch.bfloat16))
    cache.max_hist = int(sc.hist_len.max()) if sc.B else 0
    q = torch.from_numpy(sc.q).to(torch.bfloat16).to(dev)
    return cache, q


def run_decode(cache, q, max_hist=None):
    """GPU decode through the C ABI; returns (out float32 numpy [B][H_q][d], dev_status)."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    desc = cache.desc(max_hist)
    nbytes = B.oscar_decode_workspace_bytes(desc)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    B.oscar_decode_attention(desc, q, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), int(cache.dev_status.item())
