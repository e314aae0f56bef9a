"""Masked softmax attention over a paged E5M2 KV cache, in float64.

Test infrastructure only (see the package docstring).

What it computes is the plain definition of one decode step of grouped-query
attention (page "[Kernel][SM70] Pipeline batched E5M2 XQA decode", section
"Purpose": decoding many long sequences at once over an FP8 E5M2 KV cache;
section "Pending work and gates": checks with pages placed at random and with
edge-case context lengths).
The pages print no formula, so the following readings are taken:

* q head ``h`` reads kv head ``h // G`` with ``G = Hq / Hkv`` (consecutive groups);
* logical token ``t`` of sequence ``b`` lives in physical page
  ``block_tables[b, t // BS]``, slot ``t % BS``; cache layout [NB, Hkv, BS, D]
  ("hnd", the default) or [NB, BS, Hkv, D] ("nhd");
* ``k = k_scale * decode(K code)``, ``v = v_scale * decode(V code)`` with the
  E5M2 decode (default) or the E4M3 decode;
* ``s_t = sm_scale * <q, k_t>`` with ``sm_scale = 1/sqrt(D)`` unless given;
* ``out = sum_t softmax(s)_t v_t`` over ``t < ctx_b`` only (tokens past the
  context are never read); ``ctx_b == 0`` gives a zero output row.

The result is the exact attention value up to float64 rounding, not an
approximation; the output is left in float64 (no fp16 rounding).
"""
from __future__ import annotations

import math

import numpy as np

from . import e4m3, e5m2


def code_table(kv_dtype: str) -> np.ndarray:
    """float64 value of all 256 codes of the KV format."""
    if kv_dtype == "e5m2":
        return e5m2.lut()
    if kv_dtype == "e4m3":
        return e4m3.lut()
    raise ValueError(kv_dtype)


def gather_sequence_kv(cache: np.ndarray, block_tables: np.ndarray, b: int, ctx: int, kv_head: int,
                       kv_layout: str = "hnd") -> np.ndarray:
    """Codes of tokens 0..ctx-1 of sequence ``b``, kv head ``kv_head``: uint8 [ctx, D]."""
    if kv_layout == "hnd":
        num_blocks, _, bs, d = cache.shape
    elif kv_layout == "nhd":
        num_blocks, bs, _, d = cache.shape
    else:
        raise ValueError(kv_layout)
    npages = (ctx + bs - 1) // bs
    pages = np.asarray(block_tables[b, :npages], dtype=np.int64)
    if np.any(pages < 0) or np.any(pages >= num_blocks):
        raise ValueError(f"sequence {b}: block id out of range in the first {npages} table entries")
    if kv_layout == "hnd":
        return cache[pages, kv_head].reshape(npages * bs, d)[:ctx]
    return cache[pages, :, kv_head].reshape(npages * bs, d)[:ctx]


def paged_decode_attention(
    q: np.ndarray,
    k_cache: np.ndarray,
    v_cache: np.ndarray,
    block_tables: np.ndarray,
    context_lens: np.ndarray,
    k_scale: float,
    v_scale: float,
    sm_scale: float | None = None,
    kv_dtype: str = "e5m2",
    kv_layout: str = "hnd",
) -> np.ndarray:
    """One decode step: float64 [B, Hq, D] attention output."""
    batch, hq, d = q.shape
    hkv = k_cache.shape[1] if kv_layout == "hnd" else k_cache.shape[2]
    d2 = k_cache.shape[3]
    if d2 != d or hq % hkv != 0:
        raise ValueError("shape mismatch")
    group = hq // hkv
    if sm_scale is None or sm_scale <= 0.0:
        sm_scale = 1.0 / math.sqrt(d)
    table = code_table(kv_dtype)
    out = np.zeros((batch, hq, d), dtype=np.float64)
    for b in range(batch):
        ctx = int(context_lens[b])
        if ctx < 0:
            raise ValueError("negative context length")
        if ctx == 0:
            continue
        for g in range(hkv):
            k = float(k_scale) * table[gather_sequence_kv(k_cache, block_tables, b, ctx, g, kv_layout)]
            v = float(v_scale) * table[gather_sequence_kv(v_cache, block_tables, b, ctx, g, kv_layout)]
            heads = slice(g * group, (g + 1) * group)
            qh = q[b, heads].astype(np.float64)
            s = float(sm_scale) * (qh @ k.T)  # [G, ctx]
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[b, heads] = p @ v
    return out


def paged_decode_attention_rows(
    q: np.ndarray,
    k_cache: np.ndarray,
    v_cache: np.ndarray,
    block_tables: np.ndarray,
    context_lens: np.ndarray,
    k_scale: float,
    v_scale: float,
    rows,
    sm_scale: float | None = None,
    kv_dtype: str = "e5m2",
    kv_layout: str = "hnd",
) -> np.ndarray:
    """The same definition evaluated for selected (b, h) rows only: float64 [len(rows), D]."""
    batch, hq, d = q.shape
    hkv = k_cache.shape[1] if kv_layout == "hnd" else k_cache.shape[2]
    group = hq // hkv
    if sm_scale is None or sm_scale <= 0.0:
        sm_scale = 1.0 / math.sqrt(d)
    table = code_table(kv_dtype)
    res = np.zeros((len(rows), d), dtype=np.float64)
    for i, (b, h) in enumerate(rows):
        ctx = int(context_lens[b])
        if ctx == 0:
            continue
        g = h // group
        k = float(k_scale) * table[gather_sequence_kv(k_cache, block_tables, b, ctx, g, kv_layout)]
        v = float(v_scale) * table[gather_sequence_kv(v_cache, block_tables, b, ctx, g, kv_layout)]
        s = float(sm_scale) * (k @ q[b, h].astype(np.float64))
        s = s - s.max()
        p = np.exp(s)
        res[i] = (p / p.sum()) @ v
    return res


def paged_decode_attention_multi(
    q: np.ndarray,
    k_cache: np.ndarray,
    v_cache: np.ndarray,
    block_tables: np.ndarray,
    context_lens: np.ndarray,
    k_scale: float,
    v_scale: float,
    sm_scale: float | None = None,
    kv_dtype: str = "e5m2",
    kv_layout: str = "hnd",
) -> np.ndarray:
    """Decode of T new tokens per sequence: float64 [B, T, Hq, D].

    ``q`` is [B, T, Hq, D]; ``context_lens[b]`` counts the T new tokens, whose
    keys and values are already in the cache. New token i sits at position
    ``ctx_b - T + i`` and attends causally to tokens ``0 .. ctx_b - T + i``
    (none if that is negative: a zero row). Reading: the pages name multi-token
    (MTP) decode only as a variant their target excluded ("no MTP", page
    "[Kernel][SM70] Pipeline batched E5M2 XQA decode", section "Purpose").
    Each new token is therefore a single-token decode over its causal prefix.
    """
    batch, t_new = q.shape[0], q.shape[1]
    out = np.zeros(q.shape, dtype=np.float64)
    ctx = np.asarray(context_lens, dtype=np.int64)
    for i in range(t_new):
        visible = np.maximum(ctx - t_new + i + 1, 0).astype(np.int32)
        out[:, i] = paged_decode_attention(q[:, i], k_cache, v_cache, block_tables, visible,
                                           k_scale, v_scale, sm_scale, kv_dtype, kv_layout)
    return out
