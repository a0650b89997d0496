"""Pins of the float64 oracle against what the pages and mathematics fix.

Every check here compares the oracle with something other than itself: values
the pages print, hand-derived worked examples (tests/golden), closed forms,
textbook special cases, invariants, or brute force on tiny inputs.
"""
import math

import numpy as np
import pytest

import oracle as O
import synth
from conftest import golden_lines


def _orthogonal(d, seed):
    # Orthogonal matrix from a QR factorisation (a different library routine
    # from the eigensolver under test).
    g = synth.generator(seed, 99)
    q, r = np.linalg.qr(g.standard_normal((d, d)))
    return q * np.sign(np.diag(r))


# ---------------------------------------------------------------- Hadamard, P_br

@pytest.mark.parametrize("d", [2, 4, 8, 16, 128])
def test_hadamard_matches_sylvester_recursion(d):
    h = np.array([[1.0]])
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    np.testing.assert_array_equal(O.hadamard(d), h / math.sqrt(d))
    np.testing.assert_allclose(O.hadamard(d) @ O.hadamard(d), np.eye(d), atol=1e-14)


def test_bit_reversal_golden_and_involution():
    for line in golden_lines("bit_reversal.txt"):
        d, rest = line.split(":")
        d = int(d)
        want = [int(x) for x in rest.split()]
        p = O.bit_reversal_matrix(d)
        got = [int(np.argmax(p[i])) for i in range(d)]
        assert got == want
    p = O.bit_reversal_matrix(128)
    np.testing.assert_array_equal(p, p.T)
    np.testing.assert_array_equal(p @ p, np.eye(128))


# ---------------------------------------------------------------- eigenbasis, R

def test_eigenbasis_of_diagonal_is_sorted_permutation():
    diag = np.array([3.0, 7.0, 1.0, 5.0])
    u, w = O.eigenbasis(np.diag(diag))
    np.testing.assert_array_equal(w, [7.0, 5.0, 3.0, 1.0])
    want = np.zeros((4, 4))
    for col, row in enumerate([1, 3, 0, 2]):
        want[row, col] = 1.0
    np.testing.assert_array_equal(u, want)


def test_eigenbasis_recovers_constructed_spectrum():
    d = 128
    q = _orthogonal(d, 1)
    lam = np.linspace(400.0, 0.5, d) * (1 + 0.01 * np.arange(d) / d)  # distinct, gaps >= 1%
    perm = synth.generator(2, 0).permutation(d)
    c = q[:, perm] @ np.diag(lam[perm]) @ q[:, perm].T
    u, w = O.eigenbasis(c)
    np.testing.assert_allclose(w, lam, rtol=1e-12)
    for k in range(d):
        v = q[:, k].copy()
        j = int(np.argmax(np.abs(v)))
        v = v if v[j] > 0 else -v
        np.testing.assert_allclose(u[:, k], v, atol=1e-10)
    np.testing.assert_allclose(u.T @ u, np.eye(d), atol=1e-12)
    np.testing.assert_allclose(c @ u, u * w, atol=1e-12 * np.linalg.norm(c))


def test_rotation_of_diagonal_covariance_is_hadamard_then_bitreversal():
    # Descending diagonal C gives U = I, so R must be H . P_br elementwise:
    # R[i][j] = (-1)^popcount(i & br(j)) / sqrt(d).
    d = 16
    r = O.rotation_from_covariance(np.diag(np.arange(d, 0, -1, dtype=float)))
    br = [int(x) for x in golden_lines("bit_reversal.txt")[1].split(":")[1].split()]
    for i in range(d):
        for j in range(d):
            want = (-1.0) ** bin(i & br[j]).count("1") / 4.0
            assert r[i, j] == pytest.approx(want, abs=1e-15)


def _fwht(v):
    """Unnormalised fast Walsh-Hadamard transform by butterflies (Sylvester order)."""
    v = np.array(v, dtype=np.float64)
    h = 1
    while h < v.size:
        for i in range(0, v.size, 2 * h):
            a, b = v[i:i + h].copy(), v[i + h:i + 2 * h].copy()
            v[i:i + h], v[i + h:i + 2 * h] = a + b, a - b
        h *= 2
    return v


def test_canalized_rotation_golden_and_blockwise_transform():
    # [CSDN] section 4.2 (OScaR): rotation inside channel groups.  Golden for
    # d = 4, groups of 2: two copies of [[1, 1], [1, -1]] / sqrt(2) on the diagonal
    s = 1 / np.sqrt(2.0)
    golden = np.array([[s, s, 0, 0], [s, -s, 0, 0], [0, 0, s, s], [0, 0, s, -s]])
    np.testing.assert_array_equal(O.canalized_rotation(4, 2), golden)
    # x . R equals, group by group, the butterfly transform (a different
    # algorithm from the closed form) scaled by 1/sqrt(block)
    x = synth.generator(31, 0).standard_normal((3, 128))
    for block in (1, 8, 32, 128):
        r = O.canalized_rotation(128, block)
        want = np.concatenate([np.stack([_fwht(row[g:g + block]) for row in x]) for g in range(0, 128, block)],
                              axis=1) / np.sqrt(block)
        np.testing.assert_allclose(x @ r, want, rtol=0, atol=1e-12)
        np.testing.assert_allclose(r @ r.T, np.eye(128), rtol=0, atol=1e-12)
        mask = np.kron(np.eye(128 // block), np.ones((block, block)))
        assert np.all(r[mask == 0] == 0)
    np.testing.assert_array_equal(O.canalized_rotation(128, 128), O.hadamard(128))
    np.testing.assert_array_equal(O.canalized_rotation(16, 1), np.eye(16))
    with pytest.raises(ValueError):
        O.canalized_rotation(128, 48)


def test_rotation_is_orthogonal_and_composed_u_first():
    d = 128
    cal = synth.calibration_set(7, 0, 0, np.array([3, 40, 77, 100]), n_q=1024, n_k=256)
    c = O.query_covariance(cal["q"])
    r = O.rotation_from_covariance(c)
    np.testing.assert_allclose(r @ r.T, np.eye(d), atol=1e-12)
    np.testing.assert_allclose(r.T @ r, np.eye(d), atol=1e-12)
    u, _ = O.eigenbasis(c)
    hp = np.array([[(-1.0) ** bin(i & O.bit_reverse(j, 7)).count("1") for j in range(d)]
                   for i in range(d)]) / math.sqrt(d)
    np.testing.assert_allclose(r, u @ hp, atol=1e-13)


# ---------------------------------------------------------------- covariances

def test_query_covariance_brute_force():
    g = synth.generator(3, 0)
    q = g.standard_normal((5, 4))
    want = np.zeros((4, 4))
    for n in range(5):
        for i in range(4):
            for j in range(4):
                want[i, j] += q[n, i] * q[n, j] / 5
    np.testing.assert_allclose(O.query_covariance(q), want, atol=1e-15)


def test_score_weighted_values_brute_force_and_one_hot():
    g = synth.generator(4, 0)
    d = 4
    q = g.standard_normal((3, d))
    k = g.standard_normal((5, d))
    v = g.standard_normal((5, d))
    want = np.zeros((3, d))
    for n in range(3):
        s = [sum(q[n, c] * k[t, c] for c in range(d)) / 2.0 for t in range(5)]
        e = [math.exp(x) for x in s]
        for t in range(5):
            want[n] += e[t] / sum(e) * v[t]
    np.testing.assert_allclose(O.score_weighted_values(q, k, v), want, atol=1e-14)
    # S one-hot: each query matches exactly one key, so C_S = V_sel^T V_sel / N
    d = 8
    k = 100.0 * np.eye(d)
    sel = np.array([2, 5, 5, 0])
    q = 100.0 * np.eye(d)[sel]
    v = g.standard_normal((d, d))
    np.testing.assert_allclose(O.value_covariance(q, k, v), v[sel].T @ v[sel] / 4, atol=1e-12)


def test_clip_threshold_nearest_rank():
    g = synth.generator(5, 0)
    x = np.arange(1, 1001, dtype=float) * g.choice([-1.0, 1.0], size=1000)
    x = g.permutation(x).reshape(10, 100)
    assert O.clip_threshold(x, 0.999) == 999.0
    assert O.clip_threshold(x, 0.5) == 500.0
    assert O.clip_threshold(x, 1.0) == 1000.0


# ---------------------------------------------------------------- codec

def test_fp16_rounding_golden():
    for line in golden_lines("fp16_rounding.txt"):
        val, bits = [s.strip() for s in line.split("->")]
        got = np.array([float(val)]).astype(np.float16).view(np.uint16)[0]
        assert got == int(bits, 16), line


def test_pack_golden_and_round_trip():
    for line in golden_lines("pack_bytes.txt"):
        codes, byte = line.split("->")
        c = np.array([int(x) for x in codes.split()], dtype=np.uint8)
        assert O.pack(c)[0] == int(byte)
    allb = np.arange(256, dtype=np.uint8)
    np.testing.assert_array_equal(O.pack(O.unpack(allb[None, :])), allb[None, :])
    c = synth.generator(6, 0).integers(0, 4, size=(7, 128)).astype(np.uint8)
    np.testing.assert_array_equal(O.unpack(O.pack(c)), c)


def _worked_cases():
    d = 128
    x = -2.0 + 0.5 * (np.arange(d) % 4)
    shift = np.zeros((d, d))
    for i in range(d):
        shift[i, (i + 1) % d] = 1.0
    return x, {"shift": (shift, 8.0), "clip": (np.eye(d), 1.5),
               "bitrev": (O.bit_reversal_matrix(d), 8.0)}


def test_quantize_worked_examples():
    x, cases = _worked_cases()
    for line in golden_lines("quantize_worked.txt"):
        name, rest = line.split(":")
        toks = rest.split()
        want_bytes = []
        for t in toks[2:]:
            v, n = t.split("*")
            want_bytes += [int(v)] * int(n)
        r, tau = cases[name]
        codes, s16, z16 = O.demote(x[None, :], r, tau)
        assert s16.view(np.uint16)[0] == int(toks[0], 16), name
        assert z16.view(np.uint16)[0] == int(toks[1], 16), name
        np.testing.assert_array_equal(O.pack(codes)[0], want_bytes, err_msg=name)


def test_quantize_invariants_brute_force():
    g = synth.generator(8, 0)
    x = g.standard_normal((64, 128)) * g.uniform(0.1, 30, size=(64, 1))
    tau = 12.0
    codes, s16, z16 = O.quantize(x, tau)
    assert codes.max() <= 3
    xc = np.clip(x, -tau, tau)
    s = s16.astype(float)
    z = z16.astype(float)
    for r in range(64):
        assert codes[r, np.argmin(xc[r])] == 0
        assert codes[r, np.argmax(xc[r])] == 3
        for j in range(128):
            errs = [abs(xc[r, j] - (c * s[r] + z[r])) for c in range(4)]
            best = int(np.argmin(errs))
            if sorted(errs)[1] - sorted(errs)[0] > 1e-9 * s[r]:
                assert codes[r, j] == best
        xhat = codes[r] * s[r] + z[r]
        assert np.max(np.abs(xhat - xc[r])) <= s[r] / 2 + 2e-3 * (abs(z[r]) + 3 * s[r])


def test_constant_group_gives_zero_scale_and_codes():
    codes, s16, z16 = O.quantize(np.full((1, 128), 1.25), 8.0)
    assert s16[0] == 0 and z16[0] == np.float16(1.25)
    assert not codes.any()
    np.testing.assert_array_equal(O.dequantize(codes, s16, z16), np.full((1, 128), 1.25))


# ---------------------------------------------------------------- paged layout

def test_page_layout_offsets_and_round_trip():
    # The block of (page 3, KV head 1) with 2 KV heads starts at (3*2+1)*1152.
    # K code byte l of slot t at 32 t + l; V code byte l of slot t at
    # 512 + 64 (t // 2) + 4 (l // 2) + 2 (t % 2) + (l % 2); the (scale, zero)
    # pairs of slot t at 1024 + 8 t (K) and 1024 + 8 t + 4 (V).
    assert O.block_offset(3, 1, 2) == 8064
    assert O.block_bytes(1, 1) == O.BLOCK_BYTES == 1152
    assert O.block_bytes(4, 2) == 1024 + 16 * 4 * 6
    assert O.code_byte_offset(0, 5, 3) == 163
    assert O.code_byte_offset(1, 5, 0) == 642 and O.code_byte_offset(1, 5, 3) == 647
    assert O.code_byte_offset(1, 4, 3) == 512 + 128 + 4 + 1
    assert O.pair_offset(0, 5, 0) == 1064 and O.pair_offset(1, 5, 0) == 1068
    assert O.pair_offset(1, 5, 1, 4, 2) == 1024 + 24 * 5 + 4 * 5
    n_kv = 2
    table, n_pages = synth.page_table(9, [37], n_extra_pages=1)
    pool = np.zeros(n_pages * n_kv * O.BLOCK_BYTES, dtype=np.uint8)
    g = synth.generator(9, 1)
    packed = g.integers(0, 256, size=(37, n_kv, 32)).astype(np.uint8)
    s = g.uniform(0.1, 2, size=(37, n_kv)).astype(np.float16)
    z = g.uniform(-3, 0, size=(37, n_kv)).astype(np.float16)
    O.store_history_bulk(pool, table, n_kv, 0, 0, packed, s, z, which=1)
    for pos in (0, 15, 16, 36):
        for h in range(n_kv):
            pk, ss, zz = O.load_history(pool, table, n_kv, 0, pos, h, 1)
            np.testing.assert_array_equal(pk, packed[pos, h])
            assert ss == s[pos, h] and zz == z[pos, h]
            page, slot = table[0, pos // 16], pos % 16
            base = (page * n_kv + h) * 1152
            for l in range(32):
                # V rows of a slot pair alternate by 16-bit halves
                assert pool[base + 512 + 64 * (slot // 2) + 4 * (l // 2) + 2 * (slot % 2) + l % 2] == packed[pos, h, l]
            sz = pool[base + 1024 + 8 * slot + 4: base + 1024 + 8 * slot + 8].copy().view(np.float16)
            assert sz[0] == s[pos, h] and sz[1] == z[pos, h]
    codes, s2, z2 = O.load_history_bulk(pool, table, n_kv, 0, 37, 1)
    np.testing.assert_array_equal(O.pack(codes), packed)
    np.testing.assert_array_equal(s2, s)
    # the K rows and pairs were never written
    for pos in range(37):
        pk, ss, zz = O.load_history(pool, table, n_kv, 0, pos, 0, 0)
        assert not pk.any() and ss == 0 and zz == 0


def test_decode_operand_words_of_the_v_rows():
    # The 32-bit word at 512 + 64 a + 4 h of a block holds 16-bit half h of
    # slot 2a's V row (low) and of slot 2a + 1's (high): eight code positions
    # 8h .. 8h+7 of two consecutive tokens, as one tensor-core operand pair.
    n_kv = 1
    table = np.array([[0]], np.int32)
    pool = np.zeros(O.BLOCK_BYTES, np.uint8)
    g = synth.generator(9, 2)
    codes = g.integers(0, 4, size=(16, 1, 128)).astype(np.uint8)
    O.store_history_bulk(pool, table, n_kv, 0, 0, O.pack(codes), np.ones((16, 1), np.float16),
                         np.zeros((16, 1), np.float16), 1)
    for a in (0, 3, 7):
        for h in (0, 9, 15):
            w = int(pool[512 + 64 * a + 4 * h: 512 + 64 * a + 4 * h + 4].copy().view(np.uint32)[0])
            for half, t in ((0, 2 * a), (1, 2 * a + 1)):
                bits = (w >> (16 * half)) & 0xFFFF
                for i in range(8):
                    assert (bits >> (2 * i)) & 3 == codes[t, 0, 8 * h + i]


# ---------------------------------------------------------------- attention

def test_softmax_scale_closed_form():
    d = 128
    q = np.zeros(d); q[0] = 4.0
    keys = np.zeros((2, d)); keys[0, 0] = 2.0
    vals = np.zeros((2, d)); vals[0, 1] = 1.0
    w1 = 1.0 / (1.0 + math.exp(-8.0 / math.sqrt(128.0)))
    o = O.softmax_attention(q, keys, vals)
    assert o[1] == pytest.approx(w1, abs=1e-15)
    assert np.count_nonzero(o) == 1


def test_merge_equals_one_shot_softmax():
    g = synth.generator(10, 0)
    d = 8
    q = g.standard_normal(d) * 3
    keys = g.standard_normal((11, d)) * 3
    vals = g.standard_normal((11, d))
    one_shot = O.softmax_attention(q, keys, vals)
    for cuts in ([0, 11], [0, 4, 11], [0, 1, 2, 7, 11], [0, 0, 5, 5, 11]):
        states = [O.partial_state(q, keys[a:b], vals[a:b]) for a, b in zip(cuts, cuts[1:])]
        np.testing.assert_allclose(O.merge_states(states), one_shot, atol=1e-13)
    empty = O.partial_state(q, keys[:0], vals[:0])
    assert empty[0] == -math.inf and empty[1] == 0.0
    np.testing.assert_array_equal(O.merge_states([empty]), np.zeros(d))


def test_attention_special_cases():
    d = 16
    g = synth.generator(11, 0)
    q = g.standard_normal(d)
    same = np.tile(g.standard_normal(d), (9, 1))
    vals = g.standard_normal((9, d))
    np.testing.assert_allclose(O.softmax_attention(q, same, vals), vals.mean(0), atol=1e-14)
    keys = g.standard_normal((9, d))
    keys[4] = 60.0 * q / np.linalg.norm(q) * math.sqrt(d)
    np.testing.assert_allclose(O.softmax_attention(q, keys, vals), vals[4], atol=1e-12)


def _tiny_state(seed, n_kv=2, g=2, d=128, ls=3, lh=21, lr=5, tau=6.0):
    rng = synth.generator(seed, 0)
    rk = np.stack([_orthogonal(d, seed * 10 + h) for h in range(n_kv)])
    rv = np.stack([_orthogonal(d, seed * 10 + 5 + h) for h in range(n_kv)])
    hk = rng.standard_normal((lh, n_kv, d)) * 3
    hv = rng.standard_normal((lh, n_kv, d)) * 3
    hist = {}
    for name, x, r in (("k", hk, rk), ("v", hv, rv)):
        codes = np.zeros((lh, n_kv, d), np.uint8)
        sc = np.zeros((lh, n_kv), np.float16)
        ze = np.zeros((lh, n_kv), np.float16)
        for h in range(n_kv):
            codes[:, h], sc[:, h], ze[:, h] = O.demote(x[:, h], r[h], tau)
        hist["codes_" + name], hist["scale_" + name], hist["zero_" + name] = codes, sc, ze
    st = dict(q=rng.standard_normal((n_kv * g, d)) * 2,
              sink_k=rng.standard_normal((ls, n_kv, d)), sink_v=rng.standard_normal((ls, n_kv, d)),
              recent_k=rng.standard_normal((lr, n_kv, d)), recent_v=rng.standard_normal((lr, n_kv, d)),
              hist=hist, r_k=rk, r_v=rv)
    return st


def test_history_token_equals_same_token_in_bf16_segment():
    # A dequantised history token, rotated back with R^T, must act exactly like
    # the same vector stored unquantised: pins the inverse rotation's direction.
    st = _tiny_state(12)
    hist = st["hist"]
    kv_keys = []
    for name, r in (("k", st["r_k"]), ("v", st["r_v"])):
        x = O.dequantize(hist["codes_" + name][-1:], hist["scale_" + name][-1:],
                         hist["zero_" + name][-1:])            # [1][n_kv][d] rotated
        kv_keys.append(np.einsum("thd,hed->the", x, r))        # x . R^T per head
    a = O.decode_attention(st["q"], st["sink_k"], st["sink_v"], hist, st["recent_k"],
                           st["recent_v"], st["r_k"], st["r_v"])
    short = {k: v[:-1] for k, v in hist.items()}
    b = O.decode_attention(st["q"], st["sink_k"], st["sink_v"], short,
                           np.concatenate([st["recent_k"], kv_keys[0]]),
                           np.concatenate([st["recent_v"], kv_keys[1]]), st["r_k"], st["r_v"])
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_rotation_invariance_of_attention():
    g = synth.generator(13, 0)
    d = 128
    r = _orthogonal(d, 13)
    q = g.standard_normal(d)
    keys = g.standard_normal((17, d))
    vals = g.standard_normal((17, d))
    plain = O.softmax_attention(q, keys, vals)
    rotated = O.softmax_attention(q @ r, keys @ r, vals @ r) @ r.T
    np.testing.assert_allclose(rotated, plain, atol=1e-12)


def test_gqa_head_mapping_and_empty_segments():
    d = 128
    n_kv, g = 2, 3
    z = lambda n: np.zeros((n, n_kv, d))
    hist = {"codes_k": np.zeros((0, n_kv, d), np.uint8), "codes_v": np.zeros((0, n_kv, d), np.uint8),
            "scale_k": np.zeros((0, n_kv), np.float16), "zero_k": np.zeros((0, n_kv), np.float16),
            "scale_v": np.zeros((0, n_kv), np.float16), "zero_v": np.zeros((0, n_kv), np.float16)}
    rv = z(4)
    rv[:, 0] = 1.0
    rv[:, 1] = 2.0
    q = synth.generator(14, 0).standard_normal((n_kv * g, d))
    eye = np.stack([np.eye(d)] * n_kv)
    out = O.decode_attention(q, z(0), z(0), hist, synth.generator(14, 1).standard_normal((4, n_kv, d)),
                             rv, eye, eye)
    np.testing.assert_allclose(out[:g], 1.0, atol=1e-14)
    np.testing.assert_allclose(out[g:], 2.0, atol=1e-14)


def test_three_segments_equal_one_shot_over_concatenation():
    st = _tiny_state(15)
    hist = st["hist"]
    out = O.decode_attention(st["q"], st["sink_k"], st["sink_v"], hist, st["recent_k"],
                             st["recent_v"], st["r_k"], st["r_v"])
    g = st["q"].shape[0] // st["r_k"].shape[0]
    for h in range(st["q"].shape[0]):
        kv = h // g
        parts = []
        parts.append(O.partial_state(st["q"][h], st["sink_k"][:, kv], st["sink_v"][:, kv]))
        kh = O.dequantize(hist["codes_k"][:, kv], hist["scale_k"][:, kv], hist["zero_k"][:, kv])
        vh = O.dequantize(hist["codes_v"][:, kv], hist["scale_v"][:, kv], hist["zero_v"][:, kv])
        # history partial in the rotated domain: q.R_K against c*s+z, output rotated back once
        m, l, o = O.partial_state(st["q"][h] @ st["r_k"][kv], kh, vh)
        parts.append((m, l, o @ st["r_v"][kv].T))
        parts.append(O.partial_state(st["q"][h], st["recent_k"][:, kv], st["recent_v"][:, kv]))
        np.testing.assert_allclose(O.merge_states(parts), out[h], atol=1e-11)


# ---------------------------------------------------------------- accounting

def test_effective_bits_match_printed_values():
    for line in golden_lines("effective_bits.txt"):
        ctx, printed = line.split("->")
        assert round(O.effective_bits_per_element(int(ctx)), 2) == float(printed)
    # 576 B per history token-layer (8 KV heads) against 4096 B in BF16: 7.11x
    assert O.kv_bytes_per_history_token(8) == 576
    assert 4096 / O.kv_bytes_per_history_token(8) == pytest.approx(7.111, abs=1e-3)


# ---------------------------------------------------------------- quantisation groups

def test_quantize_groups_with_one_group_is_quantize():
    g = synth.generator(7, 70)
    x = g.standard_normal((9, 128)) * 2.0
    c, s, z = O.quantize(x, 3.0)
    cg, sg, zg = O.quantize_groups(x, 3.0, 128)
    np.testing.assert_array_equal(cg, c)
    np.testing.assert_array_equal(sg[..., 0].view(np.uint16), s.view(np.uint16))
    np.testing.assert_array_equal(zg[..., 0].view(np.uint16), z.view(np.uint16))


@pytest.mark.parametrize("group", [32, 64])
def test_quantize_groups_arithmetic_progressions_closed_form(group):
    # Group q holds a + k delta (k = 0..3 repeated) with a, delta exact in
    # fp16 and every distance exact: codes are k, scale delta, zero a.
    ng = 128 // group
    a = np.array([-1.5, 0.25, 2.0, -0.125])[:ng]
    delta = np.array([0.5, 0.125, 0.25, 1.0])[:ng]
    k = np.tile(np.arange(4), group // 4)
    x = np.concatenate([a[q] + delta[q] * k for q in range(ng)])
    c, s, z = O.quantize_groups(x, 10.0, group)
    np.testing.assert_array_equal(c, np.tile(k, ng))
    np.testing.assert_array_equal(s.astype(np.float64), delta)
    np.testing.assert_array_equal(z.astype(np.float64), a)


@pytest.mark.parametrize("group", [32, 64])
def test_quantize_groups_locality(group):
    # A group's codes and (scale, zero) depend on its own channels only: an
    # outlier planted in another group changes nothing in this one, while a
    # single 128-channel group is changed by it.
    g = synth.generator(8, 71)
    x = g.standard_normal((5, 128))
    y = x.copy()
    y[:, 127] = 40.0
    cx, sx, zx = O.quantize_groups(x, 50.0, group)
    cy, sy, zy = O.quantize_groups(y, 50.0, group)
    keep = 128 - group
    np.testing.assert_array_equal(cx[:, :keep], cy[:, :keep])
    np.testing.assert_array_equal(sx[:, :-1], sy[:, :-1])
    np.testing.assert_array_equal(zx[:, :-1], zy[:, :-1])
    assert not np.array_equal(O.quantize(x, 50.0)[1], O.quantize(y, 50.0)[1])
    # dequantisation error within half a step of the channel's own group
    xr = O.dequantize_groups(cy, sy, zy)
    step = np.repeat(sy.astype(np.float64), group, axis=-1)
    assert np.all(np.abs(xr - y) <= step / 2 + 1e-3 * step + 1e-12)


def test_bit_reversal_balances_groups():
    # The pages' stated purpose of P_br: with channels ordered by decreasing
    # variance (an eigenbasis order), contiguous groups of 32 without P_br put
    # all high-variance channels together; with P_br every group gets the
    # same spread.  With one 128-channel group P_br only permutes the codes.
    g = synth.generator(9, 72)
    sd = 8.0 * 0.96 ** np.arange(128)
    x = g.standard_normal((4000, 128)) * sd
    xp = x @ O.bit_reversal_matrix(128)
    _, s_plain, _ = O.quantize_groups(x, 1e4, 32)
    _, s_br, _ = O.quantize_groups(xp, 1e4, 32)
    ratio_plain = s_plain.astype(np.float64).mean(0).max() / s_plain.astype(np.float64).mean(0).min()
    ratio_br = s_br.astype(np.float64).mean(0).max() / s_br.astype(np.float64).mean(0).min()
    assert ratio_plain > 10.0 and ratio_br < 1.5
    c1, s1, z1 = O.quantize(x[:50], 1e4)
    c2, s2, z2 = O.quantize(xp[:50], 1e4)
    np.testing.assert_array_equal(s1.view(np.uint16), s2.view(np.uint16))
    np.testing.assert_array_equal(c1 @ O.bit_reversal_matrix(128), c2)


def test_storage_channel_golden_and_permutation():
    # hand-derived from the format definition (K: p = 32 t + 8 e + j,
    # V: p = 16 a + 8 e + m)
    assert O.storage_channel(0, 4, 51) == 54     # t 1, e 2, j 3: group 1, 16 + 4 + 2
    assert O.storage_channel(0, 2, 51) == 54     # j 3 < 4: group 0, 48 + 4 + 2
    assert O.storage_channel(0, 2, 6) == 96      # t 0, e 0, j 6: group 1, 64 + 32
    assert O.storage_channel(1, 2, 61) == 87     # a 3, e 1, m 5: group 1, 64 + 16 + 7
    assert O.storage_channel(1, 4, 15) == 113    # a 0, e 1, m 7: group 3, 96 + 16 + 1
    for which in (0, 1):
        assert list(O.storage_order(which, 1)) == list(range(128))
        for ng in (2, 4):
            assert sorted(O.storage_order(which, ng)) == list(range(128))


@pytest.mark.parametrize("ng", [2, 4])
def test_storage_order_makes_mma_operands_group_pure(ng):
    # K: the 16 codes a tensor-core contraction step takes together sit at
    # positions {32 t + 8 e + j : t, e < 4} for one j; V: a 16-row tile takes
    # {16 a + 8 e + m : a < 8, e < 2} for one m.  Each such set must hold 16
    # consecutive channels of one group.
    gs = 128 // ng
    for j in range(8):
        ch = sorted(O.storage_channel(0, ng, 32 * t + 8 * e + j) for t in range(4) for e in range(4))
        assert ch == list(range(ch[0], ch[0] + 16)) and ch[0] // gs == ch[-1] // gs
    for m in range(8):
        ch = sorted(O.storage_channel(1, ng, 16 * a + 8 * e + m) for a in range(8) for e in range(2))
        assert ch == list(range(ch[0], ch[0] + 16)) and ch[0] // gs == ch[-1] // gs


@pytest.mark.parametrize("ng_k,ng_v", [(1, 1), (2, 2), (4, 4), (4, 1), (1, 4)])
def test_grouped_page_format_round_trip_and_offsets(ng_k, ng_v):
    assert O.block_bytes(1, 1) == 1152 and O.block_bytes(2, 2) == 1280 and O.block_bytes(4, 4) == 1536
    n_kv, n_pages = 2, 4
    table = np.array([[3, 1, 0, 2]], np.int32)
    pool = np.zeros(n_pages * n_kv * O.block_bytes(ng_k, ng_v), np.uint8)
    g = synth.generator(10, 73)
    t = 40
    data = {}
    for which, ng in ((0, ng_k), (1, ng_v)):
        c = g.integers(0, 4, size=(t, n_kv, 128)).astype(np.uint8)
        s = g.standard_normal((t, n_kv, ng)).astype(np.float16)
        z = g.standard_normal((t, n_kv, ng)).astype(np.float16)
        O.store_history_groups(pool, table, n_kv, 0, 0, c, s, z, which, ng_k, ng_v)
        data[which] = (c, s, z)
    for which in (0, 1):
        c, s, z = O.load_history_groups(pool, table, n_kv, 0, t, which, ng_k, ng_v)
        np.testing.assert_array_equal(c, data[which][0])
        np.testing.assert_array_equal(s.view(np.uint16), data[which][1].view(np.uint16))
        np.testing.assert_array_equal(z.view(np.uint16), data[which][2].view(np.uint16))
    # bytes located by hand: token 21 (page 1, slot 5), KV head 1, V codes at
    # 512 + 64 * 2 + 4 * (byte // 2) + 2 * 1 + byte % 2; position p (byte
    # p // 4) holds the code of channel storage_channel(1, ng_v, p)
    blk = O.block_bytes(ng_k, ng_v)
    base = (1 * n_kv + 1) * blk
    c_v = data[1][0]
    for p in (0, 37, 127):
        byte = pool[base + 512 + 128 + 4 * ((p // 4) // 2) + 2 + (p // 4) % 2]
        assert (byte >> (2 * (p % 4))) & 3 == c_v[21, 1, O.storage_channel(1, ng_v, p)]
    # the last V pair of slot 5 sits after its ng_k K pairs and ng_v - 1 V pairs
    so = base + 1024 + 4 * (ng_k + ng_v) * 5 + 4 * (ng_k + ng_v - 1)
    pair = pool[so:so + 4].copy().view(np.float16)
    assert pair[0] == data[1][1][21, 1, ng_v - 1] and pair[1] == data[1][2][21, 1, ng_v - 1]
    # K code rows are plain token rows: token 21's byte 7 at 32 * 5 + 7
    c_k = data[0][0]
    byte = pool[base + 32 * 5 + 7]
    for i in range(4):
        assert (byte >> (2 * i)) & 3 == c_k[21, 1, O.storage_channel(0, ng_k, 28 + i)]
    if (ng_k, ng_v) == (1, 1):
        # the grouped writer with one group is the original format
        pool2 = np.zeros_like(pool)
        for which in (0, 1):
            c, s, z = data[which]
            O.store_history_bulk(pool2, table, n_kv, 0, 0, O.pack(c), s[..., 0], z[..., 0], which)
        np.testing.assert_array_equal(pool, pool2)


def test_grouped_decode_reduces_to_plain_dequantisation():
    # With ng groups whose (scale, zero) are all equal, grouped decode equals
    # the one-group decode; with distinct pairs it equals the plain softmax
    # over keys/values dequantised channel by channel.
    g = synth.generator(11, 74)
    n_kv, hq, lh = 2, 8, 30
    r = np.stack([_orthogonal(128, 5), _orthogonal(128, 6)])
    codes = g.integers(0, 4, size=(lh, n_kv, 128)).astype(np.uint8)
    s1 = (np.abs(g.standard_normal((lh, n_kv))) * 0.3 + 0.05).astype(np.float16)
    z1 = (g.standard_normal((lh, n_kv)) * 0.2).astype(np.float16)
    q = g.standard_normal((hq, 128))
    empty = np.zeros((0, n_kv, 128))
    one = dict(codes_k=codes, scale_k=s1, zero_k=z1, codes_v=codes[::-1], scale_v=s1, zero_v=z1)
    four = dict(codes_k=codes, scale_k=np.repeat(s1[..., None], 4, -1), zero_k=np.repeat(z1[..., None], 4, -1),
                codes_v=codes[::-1], scale_v=np.repeat(s1[..., None], 4, -1), zero_v=np.repeat(z1[..., None], 4, -1))
    a = O.decode_attention(q, empty, empty, one, empty, empty, r, r)
    b = O.decode_attention(q, empty, empty, four, empty, empty, r, r)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
    s4 = (np.abs(g.standard_normal((lh, n_kv, 4))) * 0.3 + 0.05).astype(np.float16)
    z4 = (g.standard_normal((lh, n_kv, 4)) * 0.2).astype(np.float16)
    h = dict(codes_k=codes, scale_k=s4, zero_k=z4, codes_v=codes, scale_v=s4, zero_v=z4)
    got = O.decode_attention(q, empty, empty, h, empty, empty, r, r)
    for kv in range(n_kv):
        deq = np.empty((lh, 128))
        for t in range(lh):
            for c in range(128):
                deq[t, c] = codes[t, kv, c] * float(s4[t, kv, c // 32]) + float(z4[t, kv, c // 32])
        keys = deq @ r[kv].T
        for hh in range(kv * 4, kv * 4 + 4):
            sc = keys @ q[hh] / math.sqrt(128)
            p = np.exp(sc - sc.max())
            np.testing.assert_allclose(got[hh], (p / p.sum()) @ keys, rtol=1e-12, atol=1e-12)


def test_grouped_storage_cost_closed_form():
    # 2-bit codes plus one 32-bit (scale, zero) pair per group: 2 + 32 / g bits
    assert O.effective_bits_per_element(10 ** 9, group=32) == pytest.approx(3.0, abs=1e-5)
    assert O.effective_bits_per_element(10 ** 9, group=64) == pytest.approx(2.5, abs=1e-5)
    assert O.kv_bytes_per_history_token(8, group_k=32, group_v=32) == 8 * (64 + 32)
    assert O.kv_bytes_per_history_token(8) == 576


# ---------------------------------------------------------------- Lloyd-Max codebook

def test_lloyd_max_uniform_density_closed_form():
    # For a uniform density on [0, 3] the optimal 4-level quantiser has equal
    # cells: levels (k + 1/2) 3 / 4.
    u = (np.arange(240000) + 0.5) / 240000 * 3.0
    np.testing.assert_allclose(O.lloyd_max_levels(u, 2000), [0.375, 1.125, 1.875, 2.625], atol=2e-5)


def test_lloyd_max_gaussian_matches_max_1960():
    norm = pytest.importorskip("scipy.stats").norm
    want = {}
    for line in golden_lines("lloyd_max_gaussian.txt"):
        k, v = line.split(":")
        want[k.strip()] = np.array([float(x) for x in v.split()])
    g = norm.ppf((np.arange(400000) + 0.5) / 400000)
    lv = O.lloyd_max_levels(g, 3000, init=(-1.5, -0.5, 0.5, 1.5))
    np.testing.assert_allclose(lv, want["levels"], atol=6e-4)
    np.testing.assert_allclose((lv[:-1] + lv[1:]) / 2, want["thresholds"], atol=6e-4)


def test_lloyd_max_affine_equivariance_and_fixed_point():
    g = synth.generator(12, 75)
    u = np.concatenate([g.gamma(2.0, 0.4, 5000), 3.0 - g.gamma(3.0, 0.3, 3000)]).clip(0, 3)
    lv = O.lloyd_max_levels(u, 500)
    lv2 = O.lloyd_max_levels(2.5 * u - 1.0, 500, init=tuple(2.5 * np.array([0.0, 1.0, 2.0, 3.0]) - 1.0))
    np.testing.assert_allclose(lv2, 2.5 * lv - 1.0, rtol=1e-9, atol=1e-9)
    # centroid condition: every level is the mean of the samples nearest to it
    near = np.argmin(np.abs(u[:, None] - lv[None, :]), axis=1)
    for k in range(4):
        if np.any(near == k):
            assert abs(u[near == k].mean() - lv[k]) < 1e-9


def test_codebook_code_is_nearest_level_brute_force():
    g = synth.generator(13, 76)
    x = g.standard_normal((200, 128)) * 1.5
    levels = np.array([0.3, 1.05, 1.9, 2.75], np.float16)
    c, s, z = O.quantize_codebook(x, 4.0, levels)
    xc = np.clip(x, -4.0, 4.0)
    lv = levels.astype(np.float64)
    u = (xc - z.astype(np.float64)[:, None]) / s.astype(np.float64)[:, None]
    want = np.argmin(np.abs(u[..., None] - lv), axis=-1)       # lowest index on a tie
    np.testing.assert_array_equal(c, want)
    # scale and zero are the uniform codec's; uniform levels give its codes
    _, s0, z0 = O.quantize(x, 4.0)
    np.testing.assert_array_equal(s.view(np.uint16), s0.view(np.uint16))
    np.testing.assert_array_equal(z.view(np.uint16), z0.view(np.uint16))
    cu, _, _ = O.quantize_codebook(x, 4.0, np.array([0, 1, 2, 3], np.float16))
    np.testing.assert_array_equal(cu, O.quantize(x, 4.0)[0])    # no exact ties in this draw
    # reconstruction error: within half the widest cell, in units of s
    xr = O.dequantize_codebook(c, s, z, levels)
    width = np.max(np.diff(np.concatenate([[0.0], (lv[:-1] + lv[1:]) / 2, [3.0]])))
    assert np.all(np.abs(xr - xc) <= np.maximum(width, 2 * lv[0], ) * s.astype(np.float64)[:, None] + 1e-9)


def test_codebook_decode_equals_plain_dequantisation():
    g = synth.generator(14, 77)
    n_kv, hq, lh = 1, 4, 25
    r = _orthogonal(128, 7)[None]
    codes = g.integers(0, 4, size=(lh, n_kv, 128)).astype(np.uint8)
    s = (np.abs(g.standard_normal((lh, n_kv))) * 0.3 + 0.05).astype(np.float16)
    z = (g.standard_normal((lh, n_kv)) * 0.2).astype(np.float16)
    lk = np.array([0.2, 0.9, 2.1, 2.8], np.float16)
    lvv = np.array([0.4, 1.2, 1.7, 2.6], np.float16)
    q = g.standard_normal((hq, 128))
    empty = np.zeros((0, n_kv, 128))
    h = dict(codes_k=codes, scale_k=s, zero_k=z, codes_v=codes[::-1].copy(), scale_v=s[::-1].copy(),
             zero_v=z[::-1].copy(), levels_k=lk, levels_v=lvv)
    got = O.decode_attention(q, empty, empty, h, empty, empty, r, r)
    keys = np.array([[float(z[t, 0]) + float(s[t, 0]) * float(lk[codes[t, 0, c]]) for c in range(128)]
                     for t in range(lh)]) @ r[0].T
    vals = np.array([[float(z[::-1][t, 0]) + float(s[::-1][t, 0]) * float(lvv[codes[::-1][t, 0, c]])
                      for c in range(128)] for t in range(lh)]) @ r[0].T
    for hh in range(hq):
        sc = keys @ q[hh] / math.sqrt(128)
        p = np.exp(sc - sc.max())
        np.testing.assert_allclose(got[hh], (p / p.sum()) @ vals, rtol=1e-12, atol=1e-12)


def test_fit_codebook_levels_stay_in_range_for_two_valued_rows():
    # rows taking only their min and max: every u is 0 or 3 up to the fp16
    # rounding of scale and zero; the two outer levels sit at the ends and
    # stay inside [0, 3]
    g = synth.generator(15, 78)
    x = np.where(g.random((400, 128)) < 0.5, -1.2345, 2.71828) * (1 + 0.1 * g.random((400, 1)))
    lv = O.fit_codebook(x, np.eye(128), 10.0).astype(np.float64)
    assert lv[0] >= 0.0 and lv[3] <= 3.0
    assert lv[0] == pytest.approx(0.0, abs=2e-3) and lv[3] == pytest.approx(3.0, abs=2e-3)
