"""Seeded synthetic inputs for the OSCAR two-bit KV-cache decode path.

This module is shared test and benchmark infrastructure.  It serves both the
float64 oracle tests and the CUDA path tests, and it holds none of the
method's arithmetic: no rotation, no clipping, no quantisation, no packing and
no attention.  It only draws seeded random numbers and arranges them into the
shapes of the workloads.

Value recipe.  The pages evaluate Qwen3 / GLM models on real prompts; neither
weights nor datasets exist here, so Qwen3-shaped tensors stand in for them.
Every query/key/value element is N(0, 1), except four fixed "outlier" channels
per (layer, KV head), drawn without replacement from the seed, that are scaled
by 20.  Q, K and V of one (layer, KV head) share the same outlier channels.
Values are rounded to bfloat16 (round to nearest even) because the cache and
the queries are bfloat16 on the decode path.

Host data comes from numpy PCG64 streams keyed by (seed, stream id...).  Bulk
device data for the benchmark comes from torch's CUDA Philox generator, keyed
the same way; its values are copied back to the host whenever a test needs to
compare them with the oracle.
"""
from __future__ import annotations

import math

import numpy as np

HEAD_DIM = 128
PAGE_TOKENS = 16
SINK_TOKENS = 64
RECENT_TOKENS = 256
N_OUTLIERS = 4
OUTLIER_SCALE = 20.0

# stream ids (first element of the spawn key)
_S_OUTLIER = 1
_S_ACT = 2
_S_CAL = 3
_S_PAGES = 4
_S_LENS = 5
_S_BYTES = 6


def generator(seed: int, *stream: int) -> np.random.Generator:
    """A PCG64 generator for the sub-stream `stream` of `seed`."""
    return np.random.Generator(
        np.random.PCG64(np.random.SeedSequence(int(seed), spawn_key=tuple(int(s) for s in stream))))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """The float32 values of bfloat16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 and return float32 values."""
    return bf16_value(bf16_bits(x))


def outlier_channels(seed: int, layer: int, n_kv: int, d: int = HEAD_DIM,
                     n: int = N_OUTLIERS) -> np.ndarray:
    """int64 [n_kv][n]: the outlier channels of each KV head of one layer, sorted."""
    out = np.empty((n_kv, n), dtype=np.int64)
    for h in range(n_kv):
        g = generator(seed, _S_OUTLIER, layer, h)
        out[h] = np.sort(g.choice(d, size=n, replace=False))
    return out


def activations(seed: int, stream: tuple, n_rows: int, outliers: np.ndarray,
                d: int = HEAD_DIM, scale: float = OUTLIER_SCALE) -> np.ndarray:
    """float32 [n_rows][n_heads][d], bfloat16-valued: N(0,1) with outlier channels scaled.

    `outliers` is [n_heads][n] (one row per KV head whose channels are boosted).
    """
    n_heads = outliers.shape[0]
    g = generator(seed, _S_ACT, *stream)
    x = g.standard_normal((n_rows, n_heads, d), dtype=np.float32)
    for h in range(n_heads):
        x[:, h, outliers[h]] *= np.float32(scale)
    return to_bf16(x)


def calibration_set(seed: int, layer: int, kv_head: int, outliers: np.ndarray,
                    n_q: int = 4096, n_k: int = 2048, d: int = HEAD_DIM) -> dict:
    """Calibration activations for one (layer, KV head), float64, bfloat16-valued.

    q: [n_q][d] queries pooled over the KV head's query group; k, v: [n_k][d]
    keys and values of one calibration context.  `outliers` is the head's [n].
    """
    g = generator(seed, _S_CAL, layer, kv_head)
    out = {}
    for name, rows in (("q", n_q), ("k", n_k), ("v", n_k)):
        x = g.standard_normal((rows, d), dtype=np.float32)
        x[:, outliers] *= np.float32(OUTLIER_SCALE)
        out[name] = to_bf16(x).astype(np.float64)
    return out


def page_table(seed: int, hist_lens, n_extra_pages: int = 0,
               shared_prefix_tokens: int = 0, page: int = PAGE_TOKENS):
    """A random physical page assignment for a batch of histories.

    Returns (table int32 [B][max_pages], n_pages).  Each request gets
    ceil(hist_len / page) + n_extra_pages private pages (room for appends),
    except that the first floor(shared_prefix_tokens / page) history pages
    are one shared set, referenced by every request whose history covers the
    whole page (the radix prefix-cache case).  A request's partial tail page
    is always private, so appending never writes into a shared page.  Physical
    page ids are a seeded permutation, so logical order never equals storage
    order.  Unused table entries are -1.
    """
    hist_lens = [int(h) for h in hist_lens]
    b = len(hist_lens)
    shared = int(shared_prefix_tokens) // page
    shared = min(shared, max([h // page for h in hist_lens] + [0]))
    per_req = []
    for h in hist_lens:
        n = -(-h // page) + n_extra_pages
        per_req.append(n)
    max_pages = max(per_req + [1])
    n_private = sum(n - min(shared, h // page) for n, h in zip(per_req, hist_lens))
    n_pages = shared + n_private
    perm = generator(seed, _S_PAGES).permutation(max(n_pages, 1)).astype(np.int32)
    table = np.full((b, max_pages), -1, dtype=np.int32)
    nxt = shared
    for r, n in enumerate(per_req):
        for p in range(n):
            if p < shared and (p + 1) * page <= hist_lens[r]:
                table[r, p] = perm[p]
            else:
                table[r, p] = perm[nxt]
                nxt += 1
    return table, max(n_pages, 1)


def ragged_lengths(seed: int, b: int, lo: int, hi: int) -> np.ndarray:
    """int64 [b]: context lengths uniform in [lo, hi]."""
    return generator(seed, _S_LENS).integers(lo, hi + 1, size=b).astype(np.int64)


def random_bytes(seed: int, stream: tuple, n: int) -> np.ndarray:
    return generator(seed, _S_BYTES, *stream).integers(0, 256, size=n, dtype=np.uint8)


def history_split(ctx: int, sink: int = SINK_TOKENS, recent: int = RECENT_TOKENS):
    """(sink_len, hist_len, recent_len) of a context of `ctx` tokens.

    The sink holds the first 64 tokens, the recent window the last 256, and the
    INT2 history the rest; short contexts fill the sink first, then the window.
    """
    s = min(ctx, sink)
    r = min(ctx - s, recent)
    return s, ctx - s - r, r


# --------------------------------------------------------------------------
# device-side bulk generation (benchmark inputs; torch is imported lazily)
# --------------------------------------------------------------------------

def _torch_seed(seed: int, stream: tuple) -> int:
    ss = np.random.SeedSequence(int(seed), spawn_key=tuple(int(s) for s in stream))
    return int(ss.generate_state(1, dtype=np.uint64)[0] & 0x7FFFFFFFFFFFFFFF)


def activations_device(seed: int, stream: tuple, n_rows: int, outliers: np.ndarray,
                       device, d: int = HEAD_DIM, scale: float = OUTLIER_SCALE):
    """torch bfloat16 [n_rows][n_heads][d] on `device`, same recipe as `activations`.

    Drawn with torch's Philox generator on the device (bulk benchmark data);
    the values differ from the numpy stream but follow the same distribution.
    """
    import torch
    n_heads = outliers.shape[0]
    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(seed, (_S_ACT,) + tuple(stream)))
    x = torch.randn((n_rows, n_heads, d), generator=g, device=device, dtype=torch.float32)
    scale_vec = torch.ones((n_heads, d), device=device, dtype=torch.float32)
    for h in range(n_heads):
        scale_vec[h, torch.as_tensor(outliers[h], device=device)] = float(scale)
    x.mul_(scale_vec)
    return x.to(torch.bfloat16)


def ceil_div(a: int, b: int) -> int:
    return -(-int(a) // int(b))


def log2_int(d: int) -> int:
    n = int(round(math.log2(d)))
    if 1 << n != d:
        raise ValueError("not a power of two: %d" % d)
    return n
