"""CPU checks of the C-ABI library: it loads, exports every declared symbol,
rejects bad arguments before any launch, and its host-side rotation routines
agree with the oracle (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O
import synth
from conftest import ROOT


def _declared():
    with open(os.path.join(ROOT, "include", "oscar.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\w[\w\s\*]*?\b(oscar_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol(built_lib):
    lib = ctypes.CDLL(built_lib)
    names = _declared()
    assert "oscar_decode_attention" in names and "oscar_quantize_append" in names
    assert "oscar_build_rotation" in names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    assert B.oscar_abi_version() == 4
    assert B.oscar_status_string(0) == "ok"
    assert B.oscar_status_string(3).startswith("workspace")


def _desc(**over):
    from bit_rotated_kv_split_gb300.binding import LayerDesc
    d = LayerDesc()
    d.batch, d.n_q_heads, d.n_kv_heads, d.head_dim = 1, 4, 1, 128
    d.sink_cap, d.recent_cap, d.max_pages_per_seq, d.max_hist = 64, 256, 8, 100
    d.n_pages, d.tau_k, d.tau_v = 8, 10.0, 10.0
    fake = 1 << 20   # 128-byte aligned fake addresses: never dereferenced on rejection
    for name in ("pages", "page_table", "hist_len", "sink_k", "sink_v", "sink_len", "recent_k",
                 "recent_v", "recent_len", "recent_start", "r_k", "r_v"):
        setattr(d, name, fake)
    for k, v in over.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("over,status", [
    (dict(head_dim=64), 1), (dict(batch=0), 1), (dict(n_q_heads=6, n_kv_heads=4), 1),
    (dict(sink_cap=10), 1), (dict(tau_k=0.0), 1), (dict(tau_v=float("inf")), 1),
    (dict(tau_k=float("nan")), 1), (dict(tau_v=70000.0), 1), (dict(max_hist=8 * 16 + 1), 1),
    (dict(pages=0), 1), (dict(page_table=0), 1), (dict(hist_len=0), 1),
    (dict(pages=(1 << 20) + 64), 2), (dict(r_k=(1 << 20) + 4), 2), (dict(sink_k=(1 << 20) + 2), 2),
    (dict(quant_group_k=16), 1), (dict(quant_group_v=96), 1), (dict(quant_group_k=-32), 1),
])
def test_decode_rejects_bad_descriptors_before_launch(built_lib, over, status):
    from bit_rotated_kv_split_gb300 import binding as B
    size = ctypes.c_size_t(0)
    got = B.lib.oscar_decode_attention(ctypes.byref(_desc(**over)), None, None, None,
                                       ctypes.byref(size), None)
    assert got == status


def test_decode_unsupported_group(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    size = ctypes.c_size_t(0)
    got = B.lib.oscar_decode_attention(ctypes.byref(_desc(n_q_heads=2)), None, None, None,
                                       ctypes.byref(size), None)
    assert got == 6


@pytest.mark.parametrize("kw,status", [
    (dict(n=-1), 1), (dict(k_src=0), 1), (dict(row_stride=100), 1), (dict(row_stride=64), 1),
    (dict(src_rows=0), 1), (dict(src_rows=3), 1),
    (dict(new_k=1 << 20), 1), (dict(k_src=(1 << 20) + 8), 2), (dict(dst_pos=(1 << 20) + 2), 2),
])
@pytest.mark.parametrize("entry", ["oscar_quantize_append", "oscar_quantize_append_overlapped"])
def test_quantize_append_rejects_bad_arguments(built_lib, kw, status, entry):
    from bit_rotated_kv_split_gb300 import binding as B
    args = dict(k_src=1 << 20, v_src=1 << 20, src_rows=16, row_stride=128, src_index=None,
                dst_req=1 << 20, dst_pos=1 << 20, n=4, new_k=None, new_v=None)
    args.update(kw)
    got = getattr(B.lib, entry)(ctypes.byref(_desc()), args["k_src"], args["v_src"],
                                args["src_rows"], args["row_stride"], args["src_index"],
                                args["dst_req"],
                                args["dst_pos"], args["n"], args["new_k"], args["new_v"], None)
    assert got == status


@pytest.mark.parametrize("entry", ["oscar_quantize_append", "oscar_quantize_append_overlapped"])
def test_quantize_append_zero_items_is_noop(built_lib, entry):
    from bit_rotated_kv_split_gb300 import binding as B
    assert getattr(B.lib, entry)(ctypes.byref(_desc()), None, None, 0, 0, None, None, None, 0,
                                 None, None, None) == 0


# ---------------------------------------------------------------- host rotation routines

def test_build_rotation_matches_oracle(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    outl = synth.outlier_channels(31, 0, 1)
    cal = synth.calibration_set(31, 0, 0, outl[0], n_q=2048, n_k=256)
    r_lib, w_lib = B.oscar_build_rotation(cal["q"])
    c = O.query_covariance(cal["q"])
    u, w = O.eigenbasis(c)
    assert np.min(np.abs(np.diff(w))) > 1e-7 * w[0]      # separated: U unique to ~1e-10
    np.testing.assert_allclose(w_lib, w, rtol=1e-10, atol=1e-12 * w[0])
    np.testing.assert_allclose(r_lib, O.compose_rotation(u), atol=1e-9)
    np.testing.assert_allclose(r_lib @ r_lib.T, np.eye(128), atol=1e-12)


def test_build_rotation_value_covariance_matches_oracle(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    # outlier-scaled calibration data makes S nearly one-hot and C_S rank
    # deficient (eigenvectors not unique); plain N(0,1) data over 256 keys
    # gives a full-rank C_S with separated eigenvalues, so U is unique
    outl = synth.outlier_channels(32, 0, 1)
    cal = synth.calibration_set(32, 0, 0, outl[0], n_q=512, n_k=256)
    sv_lib = B.oscar_score_weighted_rows(cal["q"], cal["k"], cal["v"])
    np.testing.assert_allclose(sv_lib, O.score_weighted_values(cal["q"], cal["k"], cal["v"]),
                               rtol=1e-11, atol=1e-11)
    g = synth.generator(32, 1)
    q, k, v = g.standard_normal((2048, 128)) * 2, g.standard_normal((256, 128)), g.standard_normal((256, 128))
    c = O.value_covariance(q, k, v)
    _, w = O.eigenbasis(c)
    assert np.min(np.abs(np.diff(w))) > 1e-7 * w[0]
    r_lib, _ = B.oscar_build_rotation(B.oscar_score_weighted_rows(q, k, v))
    np.testing.assert_allclose(r_lib, O.rotation_from_covariance(c), atol=1e-8)


def test_build_rotation_rejects_bad_dims(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    x = np.ones((4, 12))
    with pytest.raises(B.OscarError):
        B.oscar_build_rotation(x)


def test_clip_threshold_matches_oracle(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    g = synth.generator(33, 0)
    acts = g.standard_normal((3, 200, 16)) * 4
    r = np.stack([np.linalg.qr(g.standard_normal((16, 16)))[0] for _ in range(3)])
    tau = B.oscar_clip_threshold(acts, r, 0.999)
    ref = O.clip_threshold(np.stack([acts[h] @ r[h] for h in range(3)]), 0.999)
    assert tau == pytest.approx(ref, rel=1e-14)


def test_canalized_rotation_matches_oracle(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    for d, block in ((128, 32), (128, 128), (64, 8), (16, 1)):
        np.testing.assert_array_equal(B.oscar_build_canalized_rotation(d, block), O.canalized_rotation(d, block))
    for d, block in ((128, 48), (128, 256), (96, 32), (128, 0)):
        with pytest.raises(B.OscarError) as err:
            B.oscar_build_canalized_rotation(d, block)
        assert err.value.status == 1


def test_rotation_from_covariance_matches_row_builder(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    outl = synth.outlier_channels(41, 0, 1)
    cal = synth.calibration_set(41, 0, 0, outl[0], n_q=2048, n_k=256)
    r_rows, w_rows = B.oscar_build_rotation(cal["q"])
    r_cov, w_cov = B.oscar_build_rotation_from_covariance(O.query_covariance(cal["q"]))
    np.testing.assert_allclose(w_cov, w_rows, rtol=1e-12, atol=1e-12 * w_rows[0])
    np.testing.assert_allclose(r_cov, r_rows, atol=1e-9)
    bad = O.query_covariance(cal["q"])
    bad[3, 5] = np.nan
    with pytest.raises(B.OscarError) as err:
        B.oscar_build_rotation_from_covariance(bad)
    assert err.value.status == 1


def test_covariance_rejects_bad_arguments(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    lib = B.lib
    size = ctypes.c_size_t(0)
    assert lib.oscar_covariance(None, 0, 128, 128, None, None, ctypes.byref(size), None) == 1
    assert lib.oscar_covariance(None, 10, 64, 128, None, None, ctypes.byref(size), None) == 1
    assert lib.oscar_covariance(None, 10, 128, 128, None, None, None, None) == 1
    assert lib.oscar_covariance(None, 5000, 128, 128, None, None, ctypes.byref(size), None) == 0
    assert size.value == 3 * 128 * 128 * 4
    small = ctypes.c_size_t(size.value - 1)
    assert lib.oscar_covariance(ctypes.c_void_p(256), 5000, 128, 128, ctypes.c_void_p(256), ctypes.c_void_p(256),
                                ctypes.byref(small), None) == 3


def test_value_covariance_rejects_bad_arguments(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    lib = B.lib
    size = ctypes.c_size_t(0)
    f = lib.oscar_value_covariance
    assert f(None, 0, None, None, 1, 128, 128, None, None, ctypes.byref(size), None) == 1
    assert f(None, 10, None, None, 0, 128, 128, None, None, ctypes.byref(size), None) == 1
    assert f(None, 10, None, None, 1, 64, 128, None, None, ctypes.byref(size), None) == 1
    assert f(None, 10, None, None, 1, 128, 100, None, None, ctypes.byref(size), None) == 1
    assert f(None, 10, None, None, 1, 128, 128, None, None, None, None) == 1
    # the S V rows (fp32, padded to 256 bytes) and one 128 x 128 fp32
    # partial per 256 rows
    assert f(None, 1000, None, None, 1, 128, 128, None, None, ctypes.byref(size), None) == 0
    assert size.value == 1000 * 512 + 4 * 128 * 128 * 4
    assert B.oscar_value_covariance_workspace_bytes(1000) == size.value
    small = ctypes.c_size_t(size.value - 1)
    a = ctypes.c_void_p(256)
    assert f(a, 1000, a, a, 1, 128, 128, a, a, ctypes.byref(small), None) == 3
    ok = ctypes.c_size_t(size.value)
    # a row stride that is not a whole number of 16-byte units
    assert f(a, 1000, a, a, 1, 128, 132, a, a, ctypes.byref(ok), None) == 2
    assert f(ctypes.c_void_p(258), 1000, a, a, 1, 128, 128, a, a, ctypes.byref(ok), None) == 2


def test_block_bytes_match_the_format(built_lib):
    # the library's block size equals the oracle's grouped format for every
    # valid pair of group sizes (0 means 128), and 0 for anything else
    from bit_rotated_kv_split_gb300 import binding as B
    for gk in (0, 32, 64, 128):
        for gv in (0, 32, 64, 128):
            ngk, ngv = 128 // (gk or 128), 128 // (gv or 128)
            assert B.oscar_block_bytes(gk, gv) == O.block_bytes(ngk, ngv)
    assert B.oscar_block_bytes(128, 128) == 1152 == O.BLOCK_BYTES
    for bad in (16, 48, 96, 256, -1):
        assert B.oscar_block_bytes(bad, 128) == 0 and B.oscar_block_bytes(128, bad) == 0


def test_append_rejects_bad_group_before_launch(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    fake = 1 << 20
    got = B.lib.oscar_quantize_append(ctypes.byref(_desc(quant_group_v=48)), fake, fake, 4, 128, None,
                                      fake, fake, 4, None, None, None)
    assert got == 1


def test_fit_codebook_matches_oracle(built_lib):
    # the library's Lloyd-Max fit on seeded calibration rows equals the
    # oracle's (fp16 levels; the float64 sums may differ in order only)
    from bit_rotated_kv_split_gb300 import binding as B
    outl = synth.outlier_channels(5, 0, 1)
    cal = synth.calibration_set(5, 0, 0, outl[0], n_q=64, n_k=1500)
    r = O.rotation_from_covariance(O.query_covariance(cal["k"]))
    tau = O.clip_threshold(cal["k"] @ r)
    want = O.fit_codebook(cal["k"], r, tau)
    got = B.oscar_fit_codebook(cal["k"], r, tau)
    ulp = np.abs(got.astype(np.float16).view(np.uint16).astype(int) - want.view(np.uint16).astype(int))
    assert ulp.max() <= 1, (got, want)
    assert np.all(np.diff(got) > 0) and got[0] > 0 and got[3] < 3


@pytest.mark.parametrize("over,status", [
    (dict(codebook=2), 1),
    (dict(codebook=1, levels_k=(0.5, 0.25, 2.0, 2.5), levels_v=(0.5, 1.0, 2.0, 2.5)), 1),   # not increasing
    (dict(codebook=1, levels_k=(0.1, 1.0, 2.0, 2.5), levels_v=(0.5, 1.0, 2.0, 2.5)), 1),    # 0.1 is no fp16 value
    (dict(codebook=1, levels_k=(0.5, 1.0, 2.0, 3.5), levels_v=(0.5, 1.0, 2.0, 2.5)), 1),    # above 3
])
def test_decode_rejects_bad_codebook(built_lib, over, status):
    from bit_rotated_kv_split_gb300 import binding as B
    d = _desc()
    for k, v in over.items():
        if k.startswith("levels"):
            for i in range(4):
                getattr(d, k)[i] = v[i]
        else:
            setattr(d, k, v)
    size = ctypes.c_size_t(0)
    assert B.lib.oscar_decode_attention(ctypes.byref(d), None, None, None, ctypes.byref(size), None) == status


def test_codebook_with_groups_is_unsupported(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    d = _desc(codebook=1, quant_group_k=32)
    for i, v in enumerate((0.25, 1.0, 2.0, 2.75)):
        d.levels_k[i] = v
        d.levels_v[i] = v
    fake = 1 << 20
    got = B.lib.oscar_quantize_append(ctypes.byref(d), fake, fake, 4, 128, None, fake, fake, 4, None, None, None)
    assert got == 6


def test_decode_step_rejects_before_any_copy(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    fake = 1 << 20
    args = lambda desc, host_in, dev_in, nbytes, ws: (  # noqa: E731
        ctypes.byref(desc), host_in, dev_in, nbytes, fake, fake, 4, 128, None, fake, fake, 1, None, None,
        fake, fake, ws, 1 << 20, None, 0, None)
    # staged bytes without both buffers
    assert B.lib.oscar_decode_step(*args(_desc(), None, fake, 64, fake)) == 1
    assert B.lib.oscar_decode_step(*args(_desc(), fake, None, 64, fake)) == 1
    # no workspace
    assert B.lib.oscar_decode_step(*args(_desc(), None, None, 0, None)) == 3
    # a bad descriptor
    assert B.lib.oscar_decode_step(*args(_desc(head_dim=64), None, None, 0, fake)) == 1
    # unknown flag bits
    bad = list(args(_desc(), None, None, 0, fake))
    bad[-2] = 2
    assert B.lib.oscar_decode_step(*bad) == 1


def test_fit_codebook_arguments_and_single_round(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    g = synth.generator(6, 3)
    x = g.standard_normal((300, 128))
    eye = np.eye(128)
    # one Lloyd round from {0, 1, 2, 3}: the cell means, as the oracle's
    want = O.fit_codebook(x, eye, 3.0, iters=1)
    got = B.oscar_fit_codebook(x, eye, 3.0, iters=1)
    ulp = np.abs(got.astype(np.float16).view(np.uint16).astype(int) - want.view(np.uint16).astype(int))
    assert ulp.max() <= 1
    out = np.zeros(4, np.float32)
    bad = [
        (x.ctypes.data, 300, 64, eye.ctypes.data, 3.0, 10),     # d != 128
        (x.ctypes.data, 0, 128, eye.ctypes.data, 3.0, 10),      # no rows
        (x.ctypes.data, 300, 128, eye.ctypes.data, 0.0, 10),    # tau <= 0
        (x.ctypes.data, 300, 128, eye.ctypes.data, 3.0, 0),     # iters < 1
        (None, 300, 128, eye.ctypes.data, 3.0, 10),             # no rows pointer
    ]
    for a in bad:
        assert B.lib.oscar_fit_codebook(*a, out.ctypes.data) == 1
    # constant rows: every scale is 0, no usable row
    c = np.ones((10, 128))
    assert B.lib.oscar_fit_codebook(c.ctypes.data, 10, 128, eye.ctypes.data, 3.0, 10, out.ctypes.data) == 1


def test_fit_codebook_leaves_output_untouched_when_levels_collapse(built_lib):
    """Rows whose normalised values sit just below and just above u = 1.5
    give two fitted levels that round to the same fp16 value: the fit is
    rejected and the output buffer keeps its contents."""
    from bit_rotated_kv_split_gb300 import binding as B
    row = np.concatenate([[0.0, 3.0], np.full(63, 1.5 - 1e-4), np.full(63, 1.5 + 1e-4)])
    x = np.tile(row, (20, 1))
    eye = np.eye(128)
    out = np.full(4, -7.0, np.float32)
    assert B.lib.oscar_fit_codebook(x.ctypes.data, 20, 128, eye.ctypes.data, 3.0, 50, out.ctypes.data) == 1
    np.testing.assert_array_equal(out, np.full(4, -7.0, np.float32))


def test_calls_are_traced_as_nvtx_ranges(tmp_path):
    """Every library call shows as one named NVTX range: a recording NVTX
    injection library (tests/nvtx/record_ranges.c, built here with gcc)
    sees a push named after each host call and a matching pop."""
    import shutil
    import subprocess
    import sys
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    from bit_rotated_kv_split_gb300 import build as _b
    lib_path = _b.ensure_built()
    inj = tmp_path / "librecord.so"
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(_b._nvcc())), "include")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "nvtx", "record_ranges.c")
    subprocess.run([gcc, "-shared", "-fPIC", "-O1", "-I", cuda_inc, src, "-o", str(inj)], check=True)
    log = tmp_path / "ranges.txt"
    code = (
        "import ctypes, numpy as np\n"
        "lib = ctypes.CDLL(%r)\n"
        "x = np.random.default_rng(0).standard_normal((64, 8))\n"
        "r = np.zeros((8, 8)); e = np.zeros(8)\n"
        "assert lib.oscar_build_rotation(x.ctypes.data, ctypes.c_int64(64), 8, r.ctypes.data, e.ctypes.data) == 0\n"
        "assert lib.oscar_build_canalized_rotation(8, 4, r.ctypes.data) == 0\n" % str(lib_path))
    env = dict(os.environ, NVTX_INJECTION64_PATH=str(inj), OSCAR_NVTX_LOG=str(log))
    subprocess.run([sys.executable, "-c", code], check=True, env=env)
    lines = log.read_text().split("\n")
    assert "push oscar_build_rotation" in lines and "push oscar_build_canalized_rotation" in lines
    assert lines.count("pop") == sum(1 for ln in lines if ln.startswith("push "))


def _q_orthogonal(g, d):
    q, r = np.linalg.qr(g.standard_normal((d, d)))
    return q * np.sign(np.diag(r))


def test_rotation_file_round_trip_and_damage(tmp_path, built_lib):
    """A rotation file written with the library reads back bit for bit; a
    flipped byte, a cut-short file, a foreign file and a dimension mismatch
    are refused before any output is written."""
    from bit_rotated_kv_split_gb300 import binding as B
    g = synth.generator(12, 1)
    n_layers, n_kv, d = 3, 2, 128
    rk = np.stack([np.stack([_q_orthogonal(g, d) for _ in range(n_kv)]) for _ in range(n_layers)]).astype(np.float32)
    rv = np.stack([np.stack([_q_orthogonal(g, d) for _ in range(n_kv)]) for _ in range(n_layers)]).astype(np.float32)
    tk = g.uniform(5, 20, n_layers).astype(np.float32)
    tv = g.uniform(5, 20, n_layers).astype(np.float32)
    path = str(tmp_path / "rot.bin")
    B.oscar_rotation_file_write(path, rk, rv, tk, tv)
    raw = open(path, "rb").read()
    assert raw[:8] == b"OSCARROT" and len(raw) == 8 + 16 + n_layers * (8 + 8 * n_kv * d * d) + 8
    assert np.frombuffer(raw[8:24], np.uint32).tolist() == [1, n_layers, n_kv, d]
    got = B.oscar_rotation_file_read(path)
    for a, b in zip(got, (rk, rv, tk, tv)):
        np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))
    # layer 1, KV head 0, R_K[5][7] sits at a fixed offset
    off = 24 + (8 + 8 * n_kv * d * d) + 8 + 4 * (5 * d + 7)
    assert np.frombuffer(raw[off:off + 4], np.float32)[0] == rk[1, 0, 5, 7]
    out = np.full(n_layers, -1.0, np.float32)
    big = np.zeros((n_layers, n_kv, d, d), np.float32)
    damaged = [bytearray(raw), raw[:-9], b"NOTAROTATIONFILE" + raw[16:]]
    damaged[0][1000] ^= 0x10
    for i, bad in enumerate(damaged):
        p = str(tmp_path / ("bad%d.bin" % i))
        open(p, "wb").write(bytes(bad))
        st = B.lib.oscar_rotation_file_read(os.fsencode(p), n_layers, n_kv, d, big.ctypes.data, big.ctypes.data,
                                            out.ctypes.data, out.ctypes.data)
        assert st == 7, (i, st)
        assert np.all(out == -1.0) and not big.any()
    assert B.lib.oscar_rotation_file_read(os.fsencode(path), n_layers, n_kv + 1, d, big.ctypes.data,
                                          big.ctypes.data, out.ctypes.data, out.ctypes.data) == 1
    assert B.lib.oscar_rotation_file_read(os.fsencode(str(tmp_path / "missing.bin")), n_layers, n_kv, d,
                                          big.ctypes.data, big.ctypes.data, out.ctypes.data, out.ctypes.data) == 7


def test_page_wait_limit_setting(built_lib):
    from bit_rotated_kv_split_gb300 import binding as B
    prev = B.oscar_set_page_wait_limit(12345)
    try:
        assert B.oscar_set_page_wait_limit(0) == 12345          # 0 restores the default
        assert B.oscar_set_page_wait_limit(-5) == 1_000_000_000
    finally:
        B.oscar_set_page_wait_limit(prev)
