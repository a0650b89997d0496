"""Plain, slow, float64 restatement of OSCAR's rotation, codec and decode attention.

TEST INFRASTRUCTURE ONLY: only the tests, `__graft_entry__.smoke()` and the
CPU-baseline leg of `bench.py` may import this module.  It shares no code,
header, table or constant generator with the CUDA library and never imports
it.  Every function is the plain definition or the pages' steps in the pages'
order; numpy routines (matmul, eigh, sort) serve as single steps and nothing
is blocked, fused or reordered beyond what the definition states.

Sources (three web pages about the same paper, cited by title and section):
  [GIST]  gist.science, "OSCAR: Offline Spectral Covariance-Aware Rotation for
          2-bit KV Cache Quantization", Technical summary, sections 2.1 (theory),
          2.2 A (offline calibration) and 2.2 B (online serving).
  [ZAKER] myzaker.com article on OSCAR (Together AI / USYD / UIUC), parts
          "OSCAR 把旋转对准 attention" (rotation) and
          "从离线校准到在线推理的 pipeline" (token pool, demotion, decode).
  [CSDN]  aicoding.csdn.net explainer of OSCAR / OScaR, section 三 (OSCAR):
          三.1 (offline and inference stages).

Readings where the pages are silent or garbled (the full list, with reasons,
is kept with the design notes):
  * Row-vector convention: a rotated key is k~ = k . R, with R = U . H . P.
  * Eigenvectors ordered by descending eigenvalue; each column's sign is set so
    that its largest-magnitude entry is positive (ties: lowest index).
  * Hadamard is Sylvester's, normalised by 1/sqrt(d).
  * Covariances are uncentred; C_S pools the rows of S.V with
    S = row-softmax(Q K^T / sqrt(d)); the query covariance of a KV head pools
    the queries of its whole GQA group.
  * Clip: symmetric clamp to [-tau, tau] after rotation; tau is the
    nearest-rank quantile (0.999) of |x . R| over a layer's calibration rows,
    pooled over its KV heads (our procedure: parity unpinned beyond the
    library agreeing with this function).
  * One quantisation group = one token's 128 rotated channels of one KV head;
    scale s = fp16((max - min) / 3), zero z = fp16(min) (round to nearest
    even); code = clamp(rint((x - z) / s), 0, 3) with ties to even; s == 0
    gives code 0.  Dequantised value: c * s + z.
  * Four codes per byte, channel 4j+i in bits 2i..2i+1 of byte j.
  * Lloyd-Max codebook: the group keeps its (scale, zero) from min and max;
    the normalised value u = (x - z) / s in [0, 3] takes the index of the
    nearest of four fp16 levels l_0 < l_1 < l_2 < l_3 fitted per layer (K and
    V apart) by Lloyd's iteration on calibration values, ties to the lower
    level; dequantised value z + s l[c].  Levels {0, 1, 2, 3} are the
    uniform codec.
  * Smaller quantisation groups (32 or 64 channels, K and V chosen apart):
    group q of a token-head is the contiguous run of rotated channels
    [q g, (q + 1) g), so the bit-reversal inside R decides which channels
    share a group; each group has its own fp16 (scale, zero) by the rule
    above.  With several groups the page stores a token's codes in a fixed
    channel order of this build's format (`storage_channel`); one group per
    token-head keeps channel order.
"""
from __future__ import annotations

import math

import numpy as np

D_DEFAULT = 128
PAGE_TOKENS = 16
SINK_CAP = 64
RECENT_CAP = 256
# Page block of one (physical page, KV head): 16 K code rows of 32 bytes, 16
# V code rows of 32 bytes (interleaved by token pair), then the (scale, zero)
# fp16 pairs of the 16 tokens (section 3).
CODE_BYTES = 32
CODES_BYTES = PAGE_TOKENS * CODE_BYTES                      # 512 per K or V
SZ_OFFSET = 2 * CODES_BYTES                                  # 1024
BLOCK_BYTES = SZ_OFFSET + PAGE_TOKENS * 2 * 4                # 1152 (one group each)


# --------------------------------------------------------------------------
# 1. rotation construction   [GIST] 2.1 and 2.2 A; [ZAKER] "OSCAR 把旋转对准 attention"
# --------------------------------------------------------------------------

def hadamard(d: int) -> np.ndarray:
    """Orthonormal Sylvester Hadamard matrix: H[i][j] = (-1)^popcount(i & j) / sqrt(d).

    [GIST] 2.2 A (H_Had spreads outlier energy across channels).
    """
    if d <= 0 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.empty((d, d), dtype=np.float64)
    for i in range(d):
        for j in range(d):
            h[i, j] = -1.0 if bin(i & j).count("1") % 2 else 1.0
    return h / math.sqrt(d)


def bit_reverse(i: int, bits: int) -> int:
    """i with its lowest `bits` bits in reverse order."""
    r = 0
    for _ in range(bits):
        r = (r << 1) | (i & 1)
        i >>= 1
    return r


def bit_reversal_matrix(d: int) -> np.ndarray:
    """Permutation P_br with P[i][br(i)] = 1, so (x . P)[j] = x[br(j)].

    [GIST] 2.2 A (P_br interleaves high- and low-variance channels).
    """
    bits = int(round(math.log2(d)))
    p = np.zeros((d, d), dtype=np.float64)
    for i in range(d):
        p[i, bit_reverse(i, bits)] = 1.0
    return p


def canalized_rotation(d: int, block: int) -> np.ndarray:
    """Block-diagonal rotation of the OScaR variant: R = I_(d/block) (x) H_block.

    [CSDN] section 四.2 (OScaR): the K/V channels are split into groups and
    rotated within each group, with no matrix inversion and no iteration.
    The pages name no in-group rotation; the plainest fixed orthogonal choice
    is taken, the orthonormal Sylvester Hadamard of the group size.  The
    variant's per-token scaling is already carried by this codec's per-token
    (scale, zero) pair, so it adds nothing to R.
    """
    if d <= 0 or d & (d - 1) or block <= 0 or block & (block - 1) or block > d:
        raise ValueError("d and block must be powers of two with block <= d")
    r = np.zeros((d, d), dtype=np.float64)
    hb = hadamard(block)
    for g in range(d // block):
        r[g * block:(g + 1) * block, g * block:(g + 1) * block] = hb
    return r


def query_covariance(q: np.ndarray) -> np.ndarray:
    """C_Q = (1/N) sum_n q_n^T q_n over the N calibration query rows.   [GIST] 2.2 A."""
    q = np.asarray(q, dtype=np.float64)
    return q.T @ q / q.shape[0]


def score_weighted_values(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Rows of S . V with S = row-softmax(Q K^T / sqrt(d)): [N_q][d].  [GIST] 2.1, 2.2 A."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = q @ k.T / math.sqrt(q.shape[1])
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ v


def value_covariance(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """C_S = (1/N) V^T S^T S V = (1/N) (S V)^T (S V).   [GIST] 2.1, 2.2 A."""
    sv = score_weighted_values(q, k, v)
    return sv.T @ sv / sv.shape[0]


def eigenbasis(c: np.ndarray):
    """(U, eigenvalues): columns of U are eigenvectors of the symmetric C.

    Ordered by descending eigenvalue, so the strongest query directions come
    first; each column's largest-|entry| made positive (ties: lowest index).
    [GIST] 2.2 A (eigendecomposition gives U_Q / U_S).
    """
    c = np.asarray(c, dtype=np.float64)
    w, u = np.linalg.eigh(c)
    order = np.argsort(-w, kind="stable")
    w = w[order]
    u = u[:, order].copy()
    for col in range(u.shape[1]):
        j = int(np.argmax(np.abs(u[:, col])))
        if u[j, col] < 0:
            u[:, col] = -u[:, col]
    return u, w


def compose_rotation(u: np.ndarray) -> np.ndarray:
    """R = U . H_Had . P_br.   [GIST] 2.2 A formula; [ZAKER] R = U . Hadamard . bit-reversal."""
    d = u.shape[0]
    return u @ hadamard(d) @ bit_reversal_matrix(d)


def rotation_from_covariance(c: np.ndarray) -> np.ndarray:
    u, _ = eigenbasis(c)
    return compose_rotation(u)


def clip_threshold(rotated: np.ndarray, quantile: float = 0.999) -> float:
    """Nearest-rank `quantile` of |x| over every element of the rotated rows.

    [GIST] 2.2 A (per-layer clip thresholds estimated from rotated calibration
    activations; the procedure itself is this build's choice).
    """
    a = np.sort(np.abs(np.asarray(rotated, dtype=np.float64)).ravel())
    rank = int(math.ceil(quantile * a.size))
    rank = min(max(rank, 1), a.size)
    return float(a[rank - 1])


# --------------------------------------------------------------------------
# 2. demotion codec   [ZAKER] pipeline part; [CSDN] 三.1 inference stage
# --------------------------------------------------------------------------

def rotate(x: np.ndarray, r: np.ndarray) -> np.ndarray:
    """x . R for row vectors x[..., d] (float64)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(r, dtype=np.float64)


def quantize(x_rot: np.ndarray, tau: float):
    """Clip to [-tau, tau], then asymmetric 2-bit scale/zero quantisation per group.

    x_rot[..., d]: one group per trailing vector.  Returns (codes uint8 in
    0..3, scale float16, zero float16).  Codes are decided from the fp16
    scale and zero that dequantisation will use.
    [ZAKER] pipeline part (rotate, clip, quantize, pack; scale/zero point).
    """
    xc = np.clip(np.asarray(x_rot, dtype=np.float64), -tau, tau)
    mn = xc.min(axis=-1)
    mx = xc.max(axis=-1)
    s16 = ((mx - mn) / 3.0).astype(np.float16)
    z16 = mn.astype(np.float16)
    s = s16.astype(np.float64)[..., None]
    z = z16.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (xc - z) / s
        c = np.where(s > 0, np.clip(np.rint(u), 0, 3), 0)
    return c.astype(np.uint8), s16, z16


def dequantize(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """x^ = c * s + z (float64).   [ZAKER] pipeline part (scale/zero dequantisation)."""
    return (codes.astype(np.float64) * np.asarray(scale, dtype=np.float64)[..., None]
            + np.asarray(zero, dtype=np.float64)[..., None])


def quantize_groups(x_rot: np.ndarray, tau: float, group: int):
    """`quantize` applied to each run of `group` consecutive rotated channels.

    Returns (codes uint8 [..., d], scale float16 [..., d / group], zero
    float16 [..., d / group]); group == d gives `quantize`'s values with a
    trailing group axis of length 1.  [GIST] 2.2 A (bit-reversal balances the
    dynamic range inside each quantisation group); [ZAKER] "OSCAR 把旋转对准
    attention" (bit-reversal keeps an INT2 group from being ruled by a few
    outlier channels).
    """
    x_rot = np.asarray(x_rot, dtype=np.float64)
    d = x_rot.shape[-1]
    if group <= 0 or d % group:
        raise ValueError("group must divide the head dimension")
    parts = [quantize(x_rot[..., q * group:(q + 1) * group], tau) for q in range(d // group)]
    codes = np.concatenate([c for c, _, _ in parts], axis=-1)
    scale = np.stack([s for _, s, _ in parts], axis=-1)
    zero = np.stack([z for _, _, z in parts], axis=-1)
    return codes, scale, zero


def dequantize_groups(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """x^ = c * s_q + z_q with q the group of the channel (float64)."""
    codes = np.asarray(codes)
    ng = np.asarray(scale).shape[-1]
    g = codes.shape[-1] // ng
    s = np.repeat(np.asarray(scale, dtype=np.float64), g, axis=-1)
    z = np.repeat(np.asarray(zero, dtype=np.float64), g, axis=-1)
    return codes.astype(np.float64) * s + z


def lloyd_max_levels(u: np.ndarray, iters: int = 100, init=(0.0, 1.0, 2.0, 3.0)) -> np.ndarray:
    """Four-level Lloyd-Max quantiser of the samples u (float64).

    Lloyd's iteration from `init`: thresholds at the midpoints of adjacent
    levels; each level becomes the mean of the samples in its cell (u <=
    t_1, t_1 < u <= t_2, ...; an empty cell keeps its level); stops after
    `iters` rounds or when no level moves.  [ZAKER] "OSCAR 把旋转对准
    attention" closing part (the code repo pairs the rotation with a
    Lloyd-Max codebook).
    """
    u = np.sort(np.asarray(u, dtype=np.float64).ravel())
    lv = np.array(init, dtype=np.float64)
    for _ in range(iters):
        t = (lv[:-1] + lv[1:]) / 2.0
        cell = np.searchsorted(t, u, side="left")      # number of thresholds below u
        new = lv.copy()
        for k in range(4):
            sel = u[cell == k]
            if sel.size:
                new[k] = sel.mean()
        if np.array_equal(new, lv):
            break
        lv = new
    return lv


def normalised_values(x_rot: np.ndarray, tau: float) -> np.ndarray:
    """u = (x - z) / s of every channel of rows with s > 0, with the codec's
    fp16 (scale, zero) of one group per row (the calibration input of the
    codebook fit)."""
    xc = np.clip(np.asarray(x_rot, dtype=np.float64), -tau, tau)
    _, s16, z16 = quantize(xc, tau)
    s = s16.astype(np.float64)
    z = z16.astype(np.float64)
    keep = s > 0
    return ((xc[keep] - z[keep][:, None]) / s[keep][:, None]).ravel()


def fit_codebook(x: np.ndarray, r: np.ndarray, tau: float, iters: int = 100) -> np.ndarray:
    """fp16 Lloyd-Max levels (as float16) of one layer from calibration rows
    x [n][d] (rotated by r, clipped at tau, normalised per row).  The levels
    are clamped to [0, 3] before rounding (the fp16 scale and zero can put u
    a rounding step outside it)."""
    lv = lloyd_max_levels(normalised_values(rotate(x, r), tau), iters)
    return np.clip(lv, 0.0, 3.0).astype(np.float16)


def quantize_codebook(x_rot: np.ndarray, tau: float, levels):
    """Clip, then (scale, zero) as in `quantize` and the nearest-level code.

    code = number of thresholds t_k = (l_(k-1) + l_k) / 2 strictly below
    u = (x - z) / s (so a tie takes the lower level); s == 0 gives code 0.
    """
    lv = np.asarray(levels, dtype=np.float16).astype(np.float64)
    xc = np.clip(np.asarray(x_rot, dtype=np.float64), -tau, tau)
    _, s16, z16 = quantize(xc, tau)
    s = s16.astype(np.float64)[..., None]
    z = z16.astype(np.float64)[..., None]
    t = (lv[:-1] + lv[1:]) / 2.0
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (xc - z) / s
        c = (u > t[0]).astype(np.uint8) + (u > t[1]) + (u > t[2])
    c = np.where(s > 0, c, 0)
    return c.astype(np.uint8), s16, z16


def dequantize_codebook(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray, levels) -> np.ndarray:
    """x^ = z + s l[c] (float64)."""
    lv = np.asarray(levels, dtype=np.float16).astype(np.float64)
    return (lv[np.asarray(codes)] * np.asarray(scale, dtype=np.float64)[..., None]
            + np.asarray(zero, dtype=np.float64)[..., None])


def demote(x: np.ndarray, r: np.ndarray, tau: float):
    """Rotate -> clip -> quantise one or many token vectors x[..., d] with one R."""
    return quantize(rotate(x, r), tau)


def pack(codes: np.ndarray) -> np.ndarray:
    """Four 2-bit codes per byte: byte j = c[4j] | c[4j+1]<<2 | c[4j+2]<<4 | c[4j+3]<<6.

    [ZAKER] pipeline part (the codes are packed four to a byte).
    """
    c = np.asarray(codes, dtype=np.uint8)
    c = c.reshape(c.shape[:-1] + (c.shape[-1] // 4, 4))
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def unpack(packed: np.ndarray) -> np.ndarray:
    b = np.asarray(packed, dtype=np.uint8)
    out = np.stack([(b >> (2 * i)) & 3 for i in range(4)], axis=-1)
    return out.reshape(b.shape[:-1] + (b.shape[-1] * 4,)).astype(np.uint8)


# --------------------------------------------------------------------------
# 3. paged history layout (this build's format; the pages fix only "paged")
# --------------------------------------------------------------------------
#
# Block of one (physical page, KV head) with G_K groups per K vector and G_V
# per V vector (1, 2 or 4 each), 1024 + 64 (G_K + G_V) bytes:
#   K codes  [0, 512):     token slot t, code byte l at 32 t + l;
#   V codes  [512, 1024):  token slot t, code byte l at
#                          512 + 64 (t // 2) + 4 (l // 2) + 2 (t % 2) + (l % 2),
#                          i.e. the two tokens of a slot pair alternate by
#                          16-bit halves (8 codes each);
#   pairs    [1024, ...):  token slot t holds its G_K K (scale, zero) fp16
#                          pairs, then its G_V V pairs, at 1024 + 4 (G_K + G_V) t.
# Code byte l of a token row holds code positions 4l .. 4l+3 (bits 2i..2i+1);
# position p holds rotated channel storage_channel(which, G, p).


def block_bytes(ng_k: int = 1, ng_v: int = 1) -> int:
    """Bytes of one (page, KV head) block with ng_k / ng_v groups per vector."""
    return SZ_OFFSET + PAGE_TOKENS * 4 * (ng_k + ng_v)


def block_offset(page_id: int, kv_head: int, n_kv: int, ng_k: int = 1, ng_v: int = 1) -> int:
    """Byte offset of the block of (physical page, KV head) inside the pool."""
    return (int(page_id) * n_kv + int(kv_head)) * block_bytes(ng_k, ng_v)


def code_byte_offset(which: int, slot, byte):
    """Offset within a block of code byte `byte` of token `slot`; which 0 = K, 1 = V."""
    slot = np.asarray(slot)
    byte = np.asarray(byte)
    if which == 0:
        return slot * CODE_BYTES + byte
    return CODES_BYTES + 64 * (slot // 2) + 4 * (byte // 2) + 2 * (slot % 2) + (byte % 2)


def pair_offset(which: int, slot, q, ng_k: int = 1, ng_v: int = 1):
    """Offset within a block of the (scale, zero) pair of group q of token `slot`."""
    first = 0 if which == 0 else ng_k
    return SZ_OFFSET + 4 * (ng_k + ng_v) * np.asarray(slot) + 4 * (first + np.asarray(q))


def storage_channel(which: int, ng: int, p: int) -> int:
    """Rotated channel whose code sits at position p (byte p // 4, bits 2 (p % 4)).

    This build's format; the pages fix none.  ng == 1: channel p.  ng > 1:
    K (which 0): p = 32 t + 8 e + j (t, e < 4; j < 8) holds channel
    (j // J) (128 / ng) + (j % J) 16 + 4 t + e with J = 8 / ng.
    V (which 1): p = 16 a + 8 e + m (a < 8; e < 2; m < 8) holds channel
    (m // M) (128 / ng) + (m % M) 16 + 2 a + e with M = 8 / ng.
    Either way a channel's group is decided by j (K) or m (V) alone.
    """
    if ng == 1:
        return p
    gs = D_DEFAULT // ng
    if which == 0:
        t, e, j = p // 32, (p // 8) % 4, p % 8
        jj = 8 // ng
        return (j // jj) * gs + (j % jj) * 16 + 4 * t + e
    a, e, m = p // 16, (p // 8) % 2, p % 8
    mm = 8 // ng
    return (m // mm) * gs + (m % mm) * 16 + 2 * a + e


def storage_order(which: int, ng: int) -> np.ndarray:
    """perm[p] = storage_channel(which, ng, p) for p < 128."""
    return np.array([storage_channel(which, ng, p) for p in range(D_DEFAULT)], dtype=np.int64)


def _block_bases(page_table, n_kv, b, pos, ng_k, ng_v):
    pages = page_table[b, pos // PAGE_TOKENS].astype(np.int64)
    return (pages[:, None] * n_kv + np.arange(n_kv)[None, :]) * block_bytes(ng_k, ng_v)   # [T][n_kv]


def store_history_groups(pool: np.ndarray, page_table: np.ndarray, n_kv: int, b: int, pos0: int,
                         codes: np.ndarray, scale16: np.ndarray, zero16: np.ndarray, which: int,
                         ng_k: int, ng_v: int) -> None:
    """Tokens pos0 .. pos0+T-1 of all KV heads (history positions of request b).

    codes [T][n_kv][128] in channel order, scale16 / zero16 [T][n_kv][ng].
    The page is page_table[b][pos // 16], the slot pos % 16.  [GIST] 2.2 B
    (paged KV cache).
    """
    ng = ng_k if which == 0 else ng_v
    pos = pos0 + np.arange(np.asarray(codes).shape[0])
    slots = (pos % PAGE_TOKENS)[:, None, None]
    base = _block_bases(page_table, n_kv, b, pos, ng_k, ng_v)[..., None]
    packed = pack(np.asarray(codes)[..., storage_order(which, ng)])              # [T][n_kv][32]
    pool[base + code_byte_offset(which, slots, np.arange(CODE_BYTES))] = packed
    pair = np.stack([np.asarray(scale16).reshape(packed.shape[0], n_kv, ng),
                     np.asarray(zero16).reshape(packed.shape[0], n_kv, ng)], axis=-1)
    pair = pair.astype(np.float16).view(np.uint8).reshape(packed.shape[0], n_kv, 4 * ng)
    so = base + pair_offset(which, slots, 0, ng_k, ng_v)
    pool[so + np.arange(4 * ng)] = pair


def load_history_groups(pool: np.ndarray, page_table: np.ndarray, n_kv: int, b: int,
                        hist_len: int, which: int, ng_k: int, ng_v: int):
    """(codes [T][n_kv][128] channel order, scale [T][n_kv][ng], zero [T][n_kv][ng])."""
    ng = ng_k if which == 0 else ng_v
    pos = np.arange(hist_len)
    slots = (pos % PAGE_TOKENS)[:, None, None]
    base = _block_bases(page_table, n_kv, b, pos, ng_k, ng_v)[..., None]
    stored = unpack(pool[base + code_byte_offset(which, slots, np.arange(CODE_BYTES))])
    codes = np.empty_like(stored)
    codes[..., storage_order(which, ng)] = stored
    so = base + pair_offset(which, slots, 0, ng_k, ng_v)
    sz = pool[so + np.arange(4 * ng)].copy().view(np.float16)
    sz = sz.reshape(sz.shape[0], sz.shape[1], ng, 2)
    return codes, sz[..., 0], sz[..., 1]


def store_history_bulk(pool: np.ndarray, page_table: np.ndarray, n_kv: int, b: int,
                       pos0: int, packed: np.ndarray, scale16: np.ndarray,
                       zero16: np.ndarray, which: int) -> None:
    """One group per vector: packed[T][n_kv][32] codes, scale16 / zero16 [T][n_kv]."""
    store_history_groups(pool, page_table, n_kv, b, pos0, unpack(packed), np.asarray(scale16)[..., None],
                         np.asarray(zero16)[..., None], which, 1, 1)


def load_history_bulk(pool: np.ndarray, page_table: np.ndarray, n_kv: int, b: int,
                      hist_len: int, which: int):
    """(codes [T][n_kv][d] uint8, scale [T][n_kv] f16, zero [T][n_kv] f16) for positions < hist_len."""
    codes, s, z = load_history_groups(pool, page_table, n_kv, b, hist_len, which, 1, 1)
    return codes, s[..., 0], z[..., 0]


def store_history(pool: np.ndarray, page_table: np.ndarray, n_kv: int, b: int, pos: int,
                  kv_head: int, which: int, packed: np.ndarray, scale16, zero16) -> None:
    """One token's packed codes [32] and (scale, zero) of one KV head at history position `pos`."""
    base = block_offset(page_table[b, pos // PAGE_TOKENS], kv_head, n_kv)
    slot = pos % PAGE_TOKENS
    pool[base + code_byte_offset(which, slot, np.arange(CODE_BYTES))] = packed
    so = base + int(pair_offset(which, slot, 0))
    pool[so: so + 4] = np.array([scale16, zero16], dtype=np.float16).view(np.uint8)


def load_history(pool: np.ndarray, page_table: np.ndarray, n_kv: int, b: int, pos: int,
                 kv_head: int, which: int):
    """(packed[32], scale float16, zero float16) stored for a history position."""
    base = block_offset(page_table[b, pos // PAGE_TOKENS], kv_head, n_kv)
    slot = pos % PAGE_TOKENS
    packed = pool[base + code_byte_offset(which, slot, np.arange(CODE_BYTES))].copy()
    so = base + int(pair_offset(which, slot, 0))
    sz = pool[so: so + 4].copy().view(np.float16)
    return packed, sz[0], sz[1]


# --------------------------------------------------------------------------
# 4. three-segment decode attention   [ZAKER] pipeline part; [GIST] 2.2 B
# --------------------------------------------------------------------------

def softmax_attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray) -> np.ndarray:
    """o = softmax(q . K^T / sqrt(d)) . V for one query row (float64)."""
    q = np.asarray(q, dtype=np.float64)
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1], dtype=np.float64)
    s = np.asarray(keys, dtype=np.float64) @ q / math.sqrt(q.shape[0])
    s = s - s.max()
    p = np.exp(s)
    return (p / p.sum()) @ np.asarray(values, dtype=np.float64)


def decode_attention(q: np.ndarray, sink_k: np.ndarray, sink_v: np.ndarray,
                     hist: dict, recent_k: np.ndarray, recent_v: np.ndarray,
                     r_k: np.ndarray, r_v: np.ndarray) -> np.ndarray:
    """Decode attention of one request over BF16 sink | INT2 history | BF16 recent.

    q: [H_q][d]; sink_k/v: [Ls][H_kv][d]; recent_k/v: [Lr][H_kv][d] (logical
    order; attention does not depend on it); hist: dict with codes_k/codes_v
    [Lh][H_kv][d], scale_k/zero_k/scale_v/zero_v [Lh][H_kv]; r_k, r_v:
    [H_kv][d][d].  Query head h reads KV head h // (H_q / H_kv).

    The plain definition: every history token is dequantised and rotated back
    with R^T, the three segments are concatenated and one softmax is taken.
    [ZAKER] pipeline part (BF16 sink 64 | INT2 history | BF16 recent 256);
    [GIST] 2.2 B (inverse rotation inside attention); [CSDN] 三.1.
    With several quantisation groups, scale_* / zero_* carry a trailing group
    axis [Lh][H_kv][ng] and each channel uses its group's pair.  With a
    Lloyd-Max codebook, hist also holds levels_k / levels_v (four fp16
    levels each) and a history value is z + s l[c].
    """
    n_q = q.shape[0]
    n_kv = r_k.shape[0]
    g = n_q // n_kv
    out = np.zeros((n_q, q.shape[1]), dtype=np.float64)

    def deq(which, kv):
        c, s, z = hist["codes_" + which][:, kv], hist["scale_" + which][:, kv], hist["zero_" + which][:, kv]
        if "levels_" + which in hist:
            return dequantize_codebook(c, s, z, hist["levels_" + which])
        return dequantize_groups(c, s, z) if np.ndim(s) == 2 else dequantize(c, s, z)

    for kv in range(n_kv):
        k_hist = deq("k", kv) @ np.asarray(r_k[kv], dtype=np.float64).T
        v_hist = deq("v", kv) @ np.asarray(r_v[kv], dtype=np.float64).T
        keys = np.concatenate([np.asarray(sink_k[:, kv], dtype=np.float64), k_hist,
                               np.asarray(recent_k[:, kv], dtype=np.float64)], axis=0)
        vals = np.concatenate([np.asarray(sink_v[:, kv], dtype=np.float64), v_hist,
                               np.asarray(recent_v[:, kv], dtype=np.float64)], axis=0)
        for h in range(kv * g, (kv + 1) * g):
            out[h] = softmax_attention(q[h], keys, vals)
    return out


def partial_state(q: np.ndarray, keys: np.ndarray, values: np.ndarray):
    """(m, l, o) of one segment: m = max score, l = sum exp(s - m), o = sum exp(s - m) v.

    An empty segment is (-inf, 0, 0).   [ZAKER] pipeline part (online softmax merge).
    """
    d = values.shape[1]
    if keys.shape[0] == 0:
        return -math.inf, 0.0, np.zeros(d)
    s = np.asarray(keys, dtype=np.float64) @ np.asarray(q, dtype=np.float64) / math.sqrt(len(q))
    m = float(s.max())
    p = np.exp(s - m)
    return m, float(p.sum()), p @ np.asarray(values, dtype=np.float64)


def merge_states(states) -> np.ndarray:
    """Online-softmax merge of segment states into the normalised output.

    m = max m_i, l = sum l_i e^(m_i - m), o = sum o_i e^(m_i - m) / l; empty
    segments (l = 0) are skipped and an all-empty merge gives zeros.
    """
    live = [(m, l, o) for (m, l, o) in states if l > 0]
    if not live:
        return np.zeros_like(states[0][2])
    m = max(s[0] for s in live)
    l = sum(s[1] * math.exp(s[0] - m) for s in live)
    o = sum(s[2] * math.exp(s[0] - m) for s in live)
    return o / l


# --------------------------------------------------------------------------
# 5. storage accounting   [ZAKER] "小模型也能守住高难推理"; [GIST] 4 (memory)
# --------------------------------------------------------------------------

def kv_bytes_per_history_token(n_kv: int, d: int = D_DEFAULT, group_k: int = D_DEFAULT,
                               group_v: int = D_DEFAULT) -> int:
    """Bytes per INT2 history token per layer: n_kv x (K and V: d/4 codes + 4 per group)."""
    return n_kv * (2 * (d // 4) + 4 * (d // group_k) + 4 * (d // group_v))


def effective_bits_per_element(ctx: int, d: int = D_DEFAULT,
                               sink: int = SINK_CAP, recent: int = RECENT_CAP,
                               group: int = D_DEFAULT) -> float:
    """Average stored bits per K (or V) element over a context of `ctx` tokens
    (history: 2-bit codes plus a 32-bit (scale, zero) pair per group)."""
    bf16_tokens = min(ctx, sink + recent)
    hist = ctx - bf16_tokens
    bits = bf16_tokens * d * 16 + hist * (2 * d + 32 * (d // group))
    return bits / (ctx * d)
