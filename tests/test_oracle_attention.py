"""Pins of the oracle's paged GQA attention (CPU only).

Each pin ties the float64 oracle to something other than itself:

* single-token context: the output is exactly ``v_scale * V[0]``;
* constant V: the output is exactly that constant, whatever q and K are;
* q = 0: every token weighs the same, so the output is the mean of V;
* brute force: explicit per-token Python loops (math.exp) on tiny sizes;
* torch's scaled_dot_product_attention in float64 on KV gathered by loops here;
* GQA head mapping and masking, with poisoned pages and tail slots;
* page permutation: relocating pages leaves the output bitwise unchanged (the
  page "[Kernel][SM70] Pipeline batched E5M2 XQA decode", section "Pending work
  and gates", requires bit-identical results under random page placement).

The mutation tests at the end plant plausible mistakes in the oracle's own
source (a dropped scale, a transposed head mapping, an off-by-one gather, ...)
and check that at least one pin rejects every mutant.
"""
import inspect
import math
import types

import numpy as np
import pytest
import torch

import oracle.attention as attn
import oracle.e4m3 as e4m3_mod
import oracle.e5m2 as e5m2_mod
from paged_fp8_kv_gqa_gb300 import workloads as wl

ORACLE = attn.paged_decode_attention


def _tiny_paged(seed, ctxs, hq, hkv, d=16, bs=4, nb=None, scale_k=1.0, scale_v=1.0):
    """Small random paged inputs with arbitrary D and BS (oracle is generic)."""
    rng = np.random.default_rng(seed)
    ctxs = np.asarray(ctxs, np.int32)
    npages = (ctxs + bs - 1) // bs
    mbs = max(1, int(npages.max()))
    nb = nb or int(npages.sum()) + 3
    perm = rng.permutation(nb)
    bt = np.full((len(ctxs), mbs), -1, np.int32)
    off = 0
    for b, n in enumerate(npages):
        bt[b, :n] = perm[off:off + n]
        off += n
    finite = wl.finite_e5m2_codes()
    # moderate codes only (|x| <= 4) so brute-force exp stays tame
    mod = finite[np.abs(e5m2_mod.decode_fp16_view(finite)) <= 4.0]
    kc = np.full((nb, hkv, bs, d), wl.POISON_CODE, np.uint8)
    vc = np.full((nb, hkv, bs, d), wl.POISON_CODE, np.uint8)
    for b, n in enumerate(ctxs):
        for t in range(n):
            p, slot = bt[b, t // bs], t % bs
            kc[p, :, slot] = rng.choice(mod, size=(hkv, d))
            vc[p, :, slot] = rng.choice(mod, size=(hkv, d))
    q = rng.standard_normal((len(ctxs), hq, d)).astype(np.float16)
    return q, kc, vc, bt, ctxs, scale_k, scale_v


def _decode(code):
    return float(e5m2_mod.decode_closed_form(np.array([code], np.uint8))[0])


def _brute(q, kc, vc, bt, ctxs, ks, vs):
    """Per-token loops in Python floats; no numpy linear algebra."""
    B, hq, d = q.shape
    hkv, bs = kc.shape[1], kc.shape[2]
    G = hq // hkv
    out = np.zeros((B, hq, d))
    for b in range(B):
        n = int(ctxs[b])
        for h in range(hq):
            g = h // G
            logits = []
            for t in range(n):
                p, slot = int(bt[b, t // bs]), t % bs
                dot = 0.0
                for i in range(d):
                    dot += float(q[b, h, i]) * ks * _decode(kc[p, g, slot, i])
                logits.append(dot / math.sqrt(d))
            if n == 0:
                continue
            mx = max(logits)
            w = [math.exp(x - mx) for x in logits]
            tot = sum(w)
            for i in range(d):
                acc = 0.0
                for t in range(n):
                    p, slot = int(bt[b, t // bs]), t % bs
                    acc += w[t] * vs * _decode(vc[p, g, slot, i])
                out[b, h, i] = acc / tot
    return out


def _sdpa(q, kc, vc, bt, ctxs, ks, vs):
    B, hq, d = q.shape
    hkv, bs = kc.shape[1], kc.shape[2]
    table = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e5m2).to(torch.float64)
    out = np.zeros((B, hq, d))
    for b in range(B):
        n = int(ctxs[b])
        if n == 0:
            continue
        idx = [(int(bt[b, t // bs]), t % bs) for t in range(n)]
        K = torch.stack([table[torch.from_numpy(kc[p, :, s].astype(np.int64))] for p, s in idx], 1) * ks
        V = torch.stack([table[torch.from_numpy(vc[p, :, s].astype(np.int64))] for p, s in idx], 1) * vs
        K = K.repeat_interleave(hq // hkv, dim=0)
        V = V.repeat_interleave(hq // hkv, dim=0)
        Q = torch.from_numpy(q[b].astype(np.float64))[:, None, :]
        o = torch.nn.functional.scaled_dot_product_attention(Q[None], K[None], V[None])
        out[b] = o[0, :, 0].numpy()
    return out


# --------------------------------------------------------------------------
# pins, written as predicates over an oracle implementation
# --------------------------------------------------------------------------

def pin_single_token(fn):
    ok = True
    for seed, (ks, vs) in enumerate([(1.0, 1.0), (0.5, 0.5), (2.0**-12, 2.0**-12), (3.0, 0.25)]):
        q, kc, vc, bt, ctxs, _, _ = _tiny_paged(seed, [1, 1], 4, 2)
        out = fn(q, kc, vc, bt, ctxs, ks, vs)
        for b in range(2):
            for h in range(4):
                g = h // 2
                want = vs * e5m2_mod.decode_closed_form(vc[bt[b, 0], g, 0])
                ok &= bool(np.array_equal(out[b, h], want))
    return ok


def pin_constant_v(fn):
    q, kc, vc, bt, ctxs, _, _ = _tiny_paged(7, [5, 9, 13], 4, 2)
    vc = np.full_like(vc, 0x3E)  # 1.5 everywhere (poisoned slots too: never read)
    out = fn(q, kc, vc, bt, ctxs, 0.75, 0.5)
    return bool(np.allclose(out, 0.75, rtol=0, atol=1e-15))


def pin_zero_query_is_mean(fn):
    q, kc, vc, bt, ctxs, _, _ = _tiny_paged(11, [3, 6, 10], 4, 2)
    q = np.zeros_like(q)
    out = fn(q, kc, vc, bt, ctxs, 1.0, 2.0)
    ok = True
    for b, n in enumerate(ctxs):
        for h in range(4):
            g = h // 2
            rows = [vc[bt[b, t // 4], g, t % 4] for t in range(n)]
            mean = 2.0 * np.mean(e5m2_mod.decode_closed_form(np.array(rows)), axis=0)
            ok &= bool(np.allclose(out[b, h], mean, rtol=1e-14, atol=1e-14))
    return ok


def pin_brute_force(fn):
    ok = True
    for seed, (ctxs, hq, hkv) in enumerate([([5, 9], 4, 2), ([1, 4, 7], 2, 1), ([12], 6, 3)]):
        args = _tiny_paged(100 + seed, ctxs, hq, hkv, scale_k=0.5, scale_v=2.0)
        ok &= bool(np.allclose(fn(*args), _brute(*args), rtol=1e-12, atol=1e-12))
    return ok


def pin_sdpa(fn):
    args = _tiny_paged(200, [3, 17, 31, 64], 8, 2, d=32, bs=8, scale_k=0.25, scale_v=4.0)
    return bool(np.allclose(fn(*args), _sdpa(*args), rtol=1e-12, atol=1e-12))


def pin_gqa_mapping(fn):
    # kv head g carries V == g + 1 everywhere: q head h must read kv head h // G
    q, kc, vc, bt, ctxs, _, _ = _tiny_paged(300, [6, 11], 6, 3)
    one, two, three = 0x3C, 0x40, 0x42  # 1.0, 2.0, 3.0
    for g, code in enumerate((one, two, three)):
        vc[:, g] = code
    out = fn(q, kc, vc, bt, ctxs, 1.0, 1.0)
    want = np.repeat(np.array([1.0, 2.0, 3.0]), 2)[None, :, None]
    return bool(np.allclose(out, np.broadcast_to(want, out.shape), rtol=0, atol=1e-15))


def pin_masking(fn):
    # tail slots and unreferenced pages hold finite codes that would change the
    # result if read; the output must equal the clean (NaN-poisoned) run
    args = list(_tiny_paged(400, [5, 10, 3], 4, 2, nb=12))
    clean = fn(*args)
    kc, vc, bt, ctxs = args[1], args[2], args[3], args[4]
    kc2, vc2 = kc.copy(), vc.copy()
    used = set()
    for b, n in enumerate(ctxs):
        for t in range((n + 3) // 4 * 4):
            p, slot = int(bt[b, t // 4]), t % 4
            used.add(p)
            if t >= n:
                kc2[p, :, slot] = 0x7B
                vc2[p, :, slot] = 0x7B
    for p in range(kc.shape[0]):
        if p not in used:
            kc2[p] = 0x7B
            vc2[p] = 0x7B
    args[1], args[2] = kc2, vc2
    return bool(np.all(np.isfinite(clean))) and bool(np.array_equal(fn(*args), clean))


def pin_page_permutation(fn):
    w = wl.make_custom([17, 40, 1, 33], 8, 2, seed=5)
    w2 = wl.relocate_pages(w, seed=6)
    a = fn(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.k_scale, w.v_scale)
    b = fn(w2.q, w2.k_cache, w2.v_cache, w2.block_tables, w2.context_lens, w2.k_scale, w2.v_scale)
    return bool(np.all(np.isfinite(a))) and bool(np.array_equal(a, b))


PINS = [
    pin_single_token,
    pin_constant_v,
    pin_zero_query_is_mean,
    pin_brute_force,
    pin_sdpa,
    pin_gqa_mapping,
    pin_masking,
    pin_page_permutation,
]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    assert pin(ORACLE)


def test_zero_context_gives_zero_row_and_rows_api_agrees():
    w = wl.make_custom([0, 20, 3], 8, 2, seed=9)
    out = ORACLE(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.k_scale, w.v_scale)
    assert np.all(out[0] == 0.0)
    rows = [(1, 0), (1, 7), (2, 3), (0, 5)]
    got = attn.paged_decode_attention_rows(
        w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.k_scale, w.v_scale, rows)
    for i, (b, h) in enumerate(rows):
        assert np.allclose(got[i], out[b, h], rtol=1e-13, atol=1e-13)


def test_out_of_range_block_id_is_rejected():
    w = wl.make_custom([20], 8, 2, seed=3)
    w.block_tables[0, 1] = w.num_blocks
    with pytest.raises(ValueError):
        ORACLE(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1.0, 1.0)


def test_sm_scale_argument():
    # sm_scale -> tiny makes the softmax uniform: output -> mean of V
    q, kc, vc, bt, ctxs, _, _ = _tiny_paged(12, [7], 2, 1)
    out = ORACLE(q, kc, vc, bt, ctxs, 1.0, 1.0, sm_scale=1e-300)
    rows = [vc[bt[0, t // 4], 0, t % 4] for t in range(7)]
    mean = np.mean(e5m2_mod.decode_closed_form(np.array(rows)), axis=0)
    assert np.allclose(out[0, 0], mean, rtol=1e-14, atol=1e-14)


# --------------------------------------------------------------------------
# mutation tests: every planted mistake must fail at least one pin
# --------------------------------------------------------------------------

MUTATIONS = {
    "drop_k_scale": ("float(k_scale) * table", "table"),
    "drop_v_scale": ("float(v_scale) * table", "table"),
    "strided_head_mapping": ("heads = slice(g * group, (g + 1) * group)", "heads = slice(g, hq, hkv)"),
    "wrong_sm_scale": ("1.0 / math.sqrt(d)", "1.0 / d"),
    "softmax_over_heads": ("p / p.sum(axis=1, keepdims=True)", "p / p.sum(axis=0, keepdims=True)"),
    "qv_logits": ("(qh @ k.T)", "(qh @ v.T)"),
    "pk_output": ("out[b, heads] = p @ v", "out[b, heads] = p @ k"),
    "gather_off_by_one": ("[:ctx]", "[1 : ctx + 1]"),
    "gather_one_short": ("[:ctx]", "[: max(ctx - 1, 1)]"),
    "no_max_subtraction_wrong_sign": ("s = s - s.max(axis=1, keepdims=True)", "s = s.max(axis=1, keepdims=True) - s"),
}


def _mutant(old, new):
    src = inspect.getsource(attn)
    assert src.count(old) >= 1, old
    mod = types.ModuleType("oracle_mutant")
    mod.__dict__["__name__"] = "oracle_mutant"
    mod.__dict__["e5m2"] = e5m2_mod
    mod.__dict__["e4m3"] = e4m3_mod
    code = src.replace("from . import e4m3, e5m2", "")
    exec(compile(code.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod.paged_decode_attention


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_every_planted_mistake_is_caught(name):
    old, new = MUTATIONS[name]
    fn = _mutant(old, new)
    caught = []
    for pin in PINS:
        try:
            passed = pin(fn)
        except Exception:
            passed = False
        if not passed:
            caught.append(pin.__name__)
    assert caught, f"mutation {name} survived every pin"


@pytest.mark.parametrize("old,new", [("(e - 15)", "(e - 16)"), ("m / 4.0", "m / 2.0")])
def test_planted_decode_mistake_is_caught(old, new):
    src = inspect.getsource(e5m2_mod.decode_closed_form)
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    codes = np.arange(256, dtype=np.uint8)
    bad = ns["decode_closed_form"](codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e5m2).to(torch.float64).numpy()
    fin = np.isfinite(ref)
    assert not np.array_equal(bad[fin], ref[fin])
