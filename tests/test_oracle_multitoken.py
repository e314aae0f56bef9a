"""Pins of the multi-token (T new tokens per sequence) oracle (CPU only).

Brute force with an explicit causal mask in Python loops, reduction to the
single-token oracle, and planted mistakes (an off-by-one causal limit, new
tokens attending in reverse order) that the brute force must reject.
"""
import inspect
import math
import types

import numpy as np
import pytest

import oracle.attention as attn
import oracle.e4m3 as e4m3_mod
import oracle.e5m2 as e5m2_mod
from paged_fp8_kv_gqa_gb300 import workloads as wl


def _brute_multi(w, d_limit=None):
    """Explicit loops: new token i of sequence b sees tokens t <= ctx - T + i."""
    B, T, hq, D = w.q.shape
    hkv = w.num_kv_heads
    G = hq // hkv
    dec = lambda c: float(e5m2_mod.decode_closed_form(np.array([c], np.uint8))[0])
    out = np.zeros(w.q.shape)
    for b in range(B):
        ctx = int(w.context_lens[b])
        for i in range(T):
            lim = ctx - T + i  # last visible token (inclusive)
            for h in range(hq):
                g = h // G
                toks = list(range(0, lim + 1))
                if not toks:
                    continue
                logits = []
                for t in toks:
                    p, slot = int(w.block_tables[b, t // 16]), t % 16
                    dot = sum(float(w.q[b, i, h, j]) * w.k_scale * dec(w.k_cache[p, g, slot, j])
                              for j in range(D if d_limit is None else d_limit))
                    logits.append(dot / math.sqrt(D))
                mx = max(logits)
                ws = [math.exp(x - mx) for x in logits]
                tot = sum(ws)
                for j in range(D if d_limit is None else d_limit):
                    acc = 0.0
                    for wt, t in zip(ws, toks):
                        p, slot = int(w.block_tables[b, t // 16]), t % 16
                        acc += wt * w.v_scale * dec(w.v_cache[p, g, slot, j])
                    out[b, i, h, j] = acc / tot
    return out


def _small_multi(seed=3, ctxs=(3, 18, 2), T=3):
    w = wl.make_custom(list(ctxs), 4, 2, seed=seed, q_len=T)
    # zero the dims past 8 of q so an 8-dim brute force is exact for the dot product
    w.q[..., 8:] = 0
    return w


def test_multi_token_matches_brute_force():
    w = _small_multi()
    got = attn.paged_decode_attention_multi(w.q, w.k_cache, w.v_cache, w.block_tables,
                                            w.context_lens, w.k_scale, w.v_scale)
    ref = _brute_multi(w)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    # ctx 2 < T 3: the first new token sees nothing and gives a zero row
    assert np.all(got[2, 0] == 0)


def test_one_new_token_is_the_single_token_decode():
    w = wl.make_custom([17, 300], 8, 2, seed=5, q_len=1)
    multi = attn.paged_decode_attention_multi(w.q[:, None], w.k_cache, w.v_cache, w.block_tables,
                                              w.context_lens, 1.0, 1.0)
    single = attn.paged_decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables,
                                         w.context_lens, 1.0, 1.0)
    assert np.array_equal(multi[:, 0], single)


def test_last_new_token_sees_the_whole_context():
    w = wl.make_custom([40, 77], 16, 2, seed=6, q_len=4)
    multi = attn.paged_decode_attention_multi(w.q, w.k_cache, w.v_cache, w.block_tables,
                                              w.context_lens, 1.0, 1.0)
    single = attn.paged_decode_attention(w.q[:, 3], w.k_cache, w.v_cache, w.block_tables,
                                         w.context_lens, 1.0, 1.0)
    assert np.array_equal(multi[:, 3], single)


@pytest.mark.parametrize("old,new", [
    ("np.maximum(ctx - t_new + i + 1, 0)", "np.maximum(ctx - t_new + i, 0)"),
    ("np.maximum(ctx - t_new + i + 1, 0)", "np.maximum(ctx - i, 0)"),
    ("out[:, i] = paged_decode_attention(q[:, i]", "out[:, i] = paged_decode_attention(q[:, t_new - 1 - i]"),
])
def test_planted_causal_mistakes_are_caught(old, new):
    src = inspect.getsource(attn)
    assert src.count(old) == 1
    mod = types.ModuleType("oracle_mutant")
    mod.__dict__.update(e5m2=e5m2_mod, e4m3=e4m3_mod)
    exec(compile(src.replace("from . import e4m3, e5m2", "").replace(old, new), "m", "exec"),
         mod.__dict__)
    w = _small_multi(seed=9)
    got = mod.paged_decode_attention_multi(w.q, w.k_cache, w.v_cache, w.block_tables,
                                           w.context_lens, w.k_scale, w.v_scale)
    assert not np.allclose(got, _brute_multi(w), rtol=1e-9, atol=1e-9)
