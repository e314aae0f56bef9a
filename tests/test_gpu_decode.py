"""GPU parity tests of xqa_decode against the float64 oracle (through the C ABI).

Tolerance: every fp16 output element must satisfy |gpu - ref| <= 2e-3 + 1e-2*|ref|
(ref = unrounded float64 oracle). Plus bitwise properties: page relocation
invariance and poisoned-memory invariance (the page "[Kernel][SM70] Pipeline
batched E5M2 XQA decode", section "Pending work and gates", gates its kernel on
bit-identical output when pages are placed at random, and on edge-case context
lengths), CUDA-graph replay with changed
inputs (the changed-input graph replays on the page "[Kernel][WIP] Follow up
FlashNext batch HC fusion and QSA route audit", section "Test Result"),
determinism, and the device-side error paths.
"""
import functools

import numpy as np
import pytest
import torch

import paged_fp8_kv_gqa_gb300 as xqa
from gpu_helpers import Dev, assert_close, oracle_of, oracle_out, run, to_dev, workload
from oracle import e5m2, plan
from paged_fp8_kv_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("merge_mode", [0, 1])
@pytest.mark.parametrize("name", wl.WORKLOADS)
def test_workload_matches_oracle(name, merge_mode):
    out = run(workload(name), merge_mode=merge_mode)
    stats = assert_close(out, oracle_out(name), name)
    print(name, merge_mode, stats)


@pytest.mark.parametrize("name", ["b16_ragged_ctx16384_19200", "b12_boundary"])
def test_in_kernel_merge_equals_combine_kernel_bitwise(name):
    a = run(workload(name), merge_mode=0)
    b = run(workload(name), merge_mode=1)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


@pytest.mark.parametrize("merge_mode", [0, 1])
@pytest.mark.parametrize("max_ctas", [0, 1])
def test_large_batch_plan_read_from_planner(merge_mode, max_ctas):
    # 700 sequences x 4 kv heads: the segment table no longer fits in shared
    # memory, so the partial kernel reads the planner's table and copies its
    # range's window of it into shared memory; with a single CTA the window is
    # the whole table, too large, and the kernel reads the table in place
    rng = np.random.default_rng(77)
    ctx = rng.integers(0, 120, size=700)
    ctx[::37] = 0
    w = wl.make_custom(ctx, 32, 4, seed=77)
    assert_close(run(w, merge_mode=merge_mode, max_ctas=max_ctas), oracle_of(w), "large batch")


@pytest.mark.parametrize("name", ["b4_uniform_ctx1024", "b12_boundary"])
def test_page_relocation_is_bitwise_invariant(name):
    w = workload(name)
    a = run(w)
    b = run(wl.relocate_pages(w, seed=1234))
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_poisoned_memory_is_never_read():
    w = workload("b12_boundary")
    clean = run(w)
    p = w.copy()
    rng = np.random.default_rng(5)
    used = set()
    for b in range(p.batch):
        n = (int(p.context_lens[b]) + 15) // 16
        used.update(p.block_tables[b, :n].tolist())
        # unused table entries: garbage, including out-of-range ids
        tail = p.block_tables[b, n:]
        tail[:] = rng.integers(-(2**31), 2**31 - 1, size=tail.shape, dtype=np.int64).astype(np.int32)
    unused = np.setdiff1d(np.arange(p.num_blocks), sorted(used))
    finite = wl.finite_e5m2_codes()
    # unused pages and last-page tail slots: large finite codes instead of NaN
    p.k_cache[unused] = 0x7B
    p.v_cache[unused] = 0xFB
    for b in range(p.batch):
        ctx = int(p.context_lens[b])
        if ctx % 16:
            last = p.block_tables[b, (ctx + 15) // 16 - 1]
            p.k_cache[last, :, ctx % 16:] = rng.choice(finite, size=p.k_cache[last, :, ctx % 16:].shape)
            p.v_cache[last, :, ctx % 16:] = 0x7B
    got = run(p)
    assert np.array_equal(clean.view(np.uint16), got.view(np.uint16))


def test_deterministic():
    d = Dev(workload("b12_boundary"))
    d.run()
    a = d.result().copy()
    d.run()
    b = d.result()
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


@pytest.mark.parametrize("merge_mode", [0, 1])
@pytest.mark.parametrize("max_ctas,min_pages", [(1, 0), (2, 0), (7, 1), (37, 3), (0, 1), (300, 1)])
def test_split_count_does_not_change_the_result(max_ctas, min_pages, merge_mode):
    name = "b12_boundary"
    out = run(workload(name), max_ctas=max_ctas, min_pages=min_pages, merge_mode=merge_mode)
    assert_close(out, oracle_out(name), f"{name} max_ctas={max_ctas}")


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_ctas_with_only_switch_cost_on_the_line(merge_mode):
    # tiny segments and one CTA per page: several CTAs' shares of the cost line
    # fall inside a segment's switch cost and hold no page (they exit early)
    w = wl.make_custom([16, 1, 15, 16, 40, 3], 4, 2, seed=62)
    starts = plan.plan(w.context_lens, 2, w.max_blocks_per_seq, 300, 1)
    n, cc = starts["num_ctas"], starts["seg_cc"]
    empty = [i for i in range(n) if np.subtract(*plan.cta_range(i, starts["seg_start"], cc, n)) == 0]
    assert len(empty) > 0
    out = run(w, max_ctas=300, min_pages=1, merge_mode=merge_mode)
    assert_close(out, oracle_of(w), "empty cost-line shares")


@functools.lru_cache(maxsize=None)
def _long_sequence(q_len: int):
    # one 131 072-token sequence: every kv head's segment is split over about
    # 38 CTAs, so the final merge takes its pieces in several batches
    w = wl.make_custom([131072], 32, 4, seed=63, q_len=q_len)
    return w, oracle_of(w)


@pytest.mark.parametrize("q_len", [1, 2])
def test_one_long_sequence_split_over_every_cta(q_len):
    w, ref = _long_sequence(q_len)
    a = run(w, merge_mode=0)
    b = run(w, merge_mode=1)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    assert_close(a, ref, f"one 128K sequence, {q_len} new tokens")


@pytest.mark.parametrize("hq,ctas", [(8, 300), (16, 300), (4, 1000)])
def test_staged_merge_in_several_batches(hq, ctas):
    # one sequence, one kv head, hundreds of CTAs: the final merge stages more
    # pieces than fit in shared memory at once (47 per batch for G = 8, 24 for
    # G = 16, 91 for G = 4), so it runs in several batches
    w = wl.make_custom([32768], hq, 1, seed=64)
    a = run(w, max_ctas=ctas, min_pages=1, merge_mode=0)
    b = run(w, max_ctas=ctas, min_pages=1, merge_mode=1)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    assert_close(a, oracle_of(w), f"G={hq} over {ctas} CTAs")


def test_single_token_context_is_the_v_row_by_value():
    w = wl.make_custom([1, 1, 1], 16, 2, seed=21, k_scale=0.5, v_scale=0.25)
    out = run(w)
    for b in range(3):
        for h in range(16):
            g = h // 8
            page = w.block_tables[b, 0]
            want = (e5m2.decode_fp16_view(w.v_cache[page, g, 0]) * w.v_scale).astype(np.float16)
            # exact value equality (a -0 code comes out as +0: the accumulator starts at +0)
            assert np.array_equal(out[b, h].astype(np.float64), want.astype(np.float64))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (16, 4), (8, 1), (24, 3), (2, 2), (32, 2), (16, 1)])
def test_group_sizes(hq, hkv):
    # G up to 8 fills one 8-column MMA tile; G = 16 takes two
    w = wl.make_custom([1, 16, 17, 300, 2049], hq, hkv, seed=hq * 100 + hkv)
    assert_close(run(w), oracle_of(w), f"G={hq // hkv}")


def test_zero_and_max_contexts():
    w = wl.make_custom([0, 33, 0, 64], 8, 2, seed=3)
    # the table row length equals the longest context exactly (ctx = MBS*16)
    assert w.max_blocks_per_seq * 16 == 64
    out = run(w)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert_close(out, oracle_of(w), "zero/max ctx")


def test_all_contexts_zero():
    w = wl.make_custom([0, 0], 8, 1, seed=4)
    out = run(w)
    assert np.all(out == 0)


def test_custom_sm_scale():
    w = wl.make_custom([100, 7], 8, 1, seed=8)
    assert_close(run(w, sm_scale=0.02), oracle_of(w, sm_scale=0.02), "sm_scale")


@pytest.mark.parametrize("planner", [False, True])
def test_plan_matches_oracle_bit_exactly(planner):
    # planner=False: the plan the partial kernel derives itself (its CTA 0
    # publishes it); planner=True: the planner kernel, launched on request
    for ctxs, hkv, mbs_extra, max_ctas, minp in [
        ([256], 1, 0, 0, 0),
        (list(wl.BOUNDARY_CONTEXTS), 4, 0, 0, 0),
        ([5, 0, 17, 1000, 3], 2, 3, 5, 2),
        (list(range(0, 3000, 97)), 3, 0, 152, 1),
        ([None, 70, None, 16], 2, 0, 0, 0),  # None: an invalid context length
    ]:
        w = wl.make_custom([1 if c is None else c for c in ctxs], hkv * 2, hkv, seed=1)
        for i, c in enumerate(ctxs):
            if c is None:  # negative, then longer than the table row
                w.context_lens[i] = -4 if i == 0 else w.max_blocks_per_seq * 16 + 1
        d = Dev(w, max_ctas=max_ctas, min_pages=minp)
        if planner:
            xqa.xqa_plan(d.lens, d.ws, d.shape)
        else:
            d.run()
        got = xqa.xqa_read_plan(d.ws, d.shape)
        n_max = max_ctas or torch.cuda.get_device_properties(0).multi_processor_count
        ref = plan.plan(w.context_lens, hkv, w.max_blocks_per_seq, n_max, minp or 16)
        if not planner:
            assert got["ctas_launched"] == n_max
        assert np.array_equal(got["seg_start"], ref["seg_start"])
        assert np.array_equal(got["seg_cc"], ref["seg_cc"])
        assert np.array_equal(got["seg_bad"].astype(bool), ref["seg_bad"])
        assert got["num_ctas"] == ref["num_ctas"]
        assert got["total_pages"] == ref["total_pages"]
        assert got["num_segments"] == ref["num_segments"]


def _tickets(d: Dev) -> np.ndarray:
    """The workspace's merge-ticket words (bytes 64 .. 64 + 8*1024: two per
    possible CTA)."""
    torch.cuda.synchronize()
    return d.ws[64:64 + 8 * 1024].cpu().numpy().view(np.int32)


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_merge_tickets_are_zero_after_every_call(merge_mode):
    # the workspace is zeroed once; every call (good, with a bad block id, or a
    # bad context length) must leave the tickets at zero for the next one
    w = wl.make_custom([40, 300, 5000, 17, 2049], 8, 2, seed=71)
    d = Dev(w, max_ctas=9, merge_mode=merge_mode)  # most segments split
    ref = oracle_of(w)
    d.run()
    assert np.all(_tickets(d) == 0)
    assert_close(d.result(), ref, "first call")
    d.bt[2, 7] = w.num_blocks + 1  # a split segment meets a bad page
    d.run()
    assert d.status() == xqa.XQA_ERR_BAD_BLOCK_ID
    assert np.all(_tickets(d) == 0)
    assert np.all(np.isnan(d.result()[2].astype(np.float32)))
    d.bt.copy_(to_dev(w.block_tables))
    d.lens[1] = w.max_blocks_per_seq * 16 + 5
    d.run()
    assert d.status() == xqa.XQA_ERR_CTX_TOO_LONG
    assert np.all(_tickets(d) == 0)
    d.lens.copy_(to_dev(w.context_lens))
    d.run()
    assert d.status() == xqa.XQA_OK
    assert_close(d.result(), ref, "after the bad calls")


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_long_segments_of_few_pieces_with_a_bad_page(merge_mode):
    # segments of 563 and 750 pages split into 2-3 pieces over 8 CTAs: the
    # last piece to arrive merges them; a bad block id in one must give NaN
    # in its rows only, and every call must leave the tickets at zero
    w = wl.make_custom([9000, 12000, 40], 8, 2, seed=75)
    ref = oracle_of(w)
    d = Dev(w, max_ctas=8, merge_mode=merge_mode)
    d.run()
    assert d.status() == xqa.XQA_OK
    assert np.all(_tickets(d) == 0)
    assert_close(d.result(), ref, "long segments, few pieces")
    d.bt[1, 400] = w.num_blocks + 2
    d.run()
    assert d.status() == xqa.XQA_ERR_BAD_BLOCK_ID
    out = d.result()
    assert np.all(np.isnan(out[1].astype(np.float32)))
    assert_close(out[[0, 2]], ref[[0, 2]], "beside the bad sequence")
    assert np.all(_tickets(d) == 0)


@pytest.mark.parametrize("hq,hkv,q_len", [(8, 1, 1), (16, 1, 1), (4, 1, 1), (8, 2, 2), (32, 4, 1)])
def test_final_merge_shared_by_the_last_ctas(hq, hkv, q_len):
    # long sequences over one CTA per SM: a segment of many pieces is merged by
    # its last CTAs to finish, each taking every nh-th output row; results
    # equal the combine kernel's bit for bit and the tickets end at zero
    w = wl.make_custom([20000, 9000, 3], hq, hkv, seed=36, q_len=q_len)
    d = Dev(w, merge_mode=0)
    d.run()
    a = d.result()
    assert d.status() == xqa.XQA_OK
    assert np.all(_tickets(d) == 0)
    b = run(w, merge_mode=1)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    assert_close(a, oracle_of(w), f"shared final merge G={hq // hkv} q_len={q_len}")


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_bad_block_id_in_a_segment_merged_by_several_ctas(merge_mode):
    w = wl.make_custom([20000, 300], 8, 1, seed=37)
    ref = oracle_of(w)
    d = Dev(w, merge_mode=merge_mode)
    d.bt[0, 700] = w.num_blocks + 3
    d.run()
    assert d.status() == xqa.XQA_ERR_BAD_BLOCK_ID
    out = d.result()
    assert np.all(np.isnan(out[0].astype(np.float32)))
    assert_close(out[[1]], ref[[1]], "the sequence beside")
    assert np.all(_tickets(d) == 0)
    d.bt.copy_(to_dev(w.block_tables))
    d.run()
    assert d.status() == xqa.XQA_OK
    assert_close(d.result(), ref, "after the bad call")


def _hints(d: Dev) -> torch.Tensor:
    """The workspace's first-page hint words (16 per possible CTA), after the
    header, the merge tickets and the status words."""
    off = 64 + 8 * 1024 + 4 * 1024
    return d.ws[off:off + 4 * 16 * 1024].view(torch.int32)


@pytest.mark.parametrize("layout", ["hnd", "nhd"])
def test_first_page_hints_never_change_results(layout):
    # the hint words only steer an L2 prefetch before the wait: any content
    # (negative, huge, rows of other pages) leaves every result bit and the
    # status unchanged
    w = workload("b12_boundary")
    if layout == "nhd":
        w = wl.to_nhd(w)
    d = Dev(w)
    d.run()
    ref = d.result()
    assert d.status() == xqa.XQA_OK
    hints = _hints(d)
    assert int((hints >= 0).sum()) > 0  # the call recorded its first pages
    gen = torch.Generator().manual_seed(5)
    for fill in ("random", "max", "zero", "minus_one", "shifted"):
        if fill == "random":
            vals = torch.randint(-2**31, 2**31 - 1, (hints.numel(),), generator=gen, dtype=torch.int64)
            hints.copy_(vals.to(torch.int32).to(hints.device))
        elif fill == "max":
            hints.fill_(2**31 - 1)
        elif fill == "zero":
            hints.zero_()
        elif fill == "minus_one":
            hints.fill_(-1)
        else:  # the hints of other CTAs
            hints.copy_(torch.roll(hints.clone(), 16 * 5))
        d.run()
        assert np.array_equal(d.result().view(np.uint16), ref.view(np.uint16)), fill
        assert d.status() == xqa.XQA_OK


def test_one_workspace_serves_several_shapes():
    # the ticket and status regions sit at fixed offsets, so a workspace sized
    # for the largest shape can be used by calls of different shapes in turn
    ws_list = [wl.make_custom([3000, 20, 700], 32, 4, seed=72),
               wl.make_custom([1, 16, 17, 4097, 9000, 33, 64, 2], 16, 2, seed=73),
               wl.make_custom([5000], 8, 8, seed=74)]
    devs = [Dev(w, max_ctas=m) for w, m in zip(ws_list, (0, 37, 5))]
    shared = torch.zeros(max(d.ws.numel() for d in devs), dtype=torch.uint8, device="cuda")
    for rnd in range(2):
        for d in devs:
            d.ws = shared[:d.ws.numel()]
            d.out.fill_(float("nan"))
            d.run()
            assert d.status() == xqa.XQA_OK
            assert_close(d.result(), oracle_of(d.w), f"round {rnd}")
            assert np.all(_tickets(d) == 0)


def test_cuda_graph_replay_with_changed_inputs():
    w = workload("b12_boundary")
    d = Dev(w)
    d.run()
    eager_first = d.result().copy()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        d.run(stream=s)  # warm-up on the capture stream
        torch.cuda.current_stream().synchronize()
        with torch.cuda.graph(g, stream=s):
            d.run(stream=s)
    torch.cuda.synchronize()
    # 1) replay on unchanged inputs
    d.out.fill_(float("nan"))
    g.replay()
    assert np.array_equal(d.result().view(np.uint16), eager_first.view(np.uint16))
    # 2) change q, KV contents and context lengths in place (the plan changes)
    # same shapes and scales (the scales are captured launch arguments)
    w2 = wl.make_custom([5, 1, 4097, 32, 1025, 16385, 16, 17, 0, 3000, 1, 32768], 32, 4,
                        seed=99, num_blocks=w.num_blocks, k_scale=w.k_scale, v_scale=w.v_scale,
                        code_premul=4096.0)
    assert w2.block_tables.shape == w.block_tables.shape
    d.q.copy_(to_dev(w2.q))
    d.k.copy_(to_dev(w2.k_cache))
    d.v.copy_(to_dev(w2.v_cache))
    d.bt.copy_(to_dev(w2.block_tables))
    d.lens.copy_(to_dev(w2.context_lens))
    d.out.fill_(float("nan"))
    g.replay()
    replayed = d.result().copy()
    d.out.fill_(float("nan"))
    d.run()
    eager = d.result()
    assert np.array_equal(replayed.view(np.uint16), eager.view(np.uint16))
    assert_close(replayed, oracle_of(w2), "graph replay")


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_inputs_written_by_the_previous_kernel_are_seen(merge_mode):
    # q and the context lengths are rewritten by ordinary kernels on the same
    # stream right before every decode, with no synchronisation in between: the
    # planner (a programmatic dependent of whatever ran before) must wait for
    # those kernels before the partial kernel reads anything
    w = wl.make_custom([700, 33, 5000, 2049], 32, 4, seed=61)
    w2 = w.copy()
    w2.q = -w.q
    w2.context_lens = np.array([650, 1, 4000, 17], dtype=np.int32)
    refs = [oracle_of(w), oracle_of(w2)]
    d = Dev(w, merge_mode=merge_mode)
    srcs = [(to_dev(w.q), to_dev(w.context_lens)), (to_dev(w2.q), to_dev(w2.context_lens))]
    outs = []
    for it in range(12):
        q_src, lens_src = srcs[it % 2]
        torch.mul(q_src, 1.0, out=d.q)
        torch.add(lens_src, 0, out=d.lens)
        d.run()
        outs.append(d.out.clone())
    torch.cuda.synchronize()
    assert d.status() == xqa.XQA_OK
    for it, o in enumerate(outs):
        assert_close(o.cpu().numpy(), refs[it % 2], f"iteration {it}")


# --------------------------------------------------------------------------
# error paths
# --------------------------------------------------------------------------

def test_host_side_errors():
    w = workload("tiny_b1_ctx256")
    d = Dev(w)
    with pytest.raises(xqa.XqaError) as e:
        bad = xqa.XqaShape(1, 8, 1, 64, 16, 16, 16, 0.0, 0, 0)
        xqa.xqa_workspace_size(bad)
    assert e.value.code == xqa.XQA_ERR_SHAPE
    with pytest.raises(xqa.XqaError) as e:
        xqa.xqa_decode(d.q, d.k, d.v, d.bt, d.lens, 1.0, 1.0, out=d.out, workspace=d.ws[:64],
                       shape=d.shape)
    assert e.value.code == xqa.XQA_ERR_WORKSPACE
    qbuf = torch.zeros(d.q.numel() + 8, dtype=torch.float16, device="cuda")
    q_mis = qbuf[1:1 + d.q.numel()].view(d.q.shape)
    with pytest.raises(xqa.XqaError) as e:
        xqa.xqa_decode(q_mis, d.k, d.v, d.bt, d.lens, 1.0, 1.0, out=d.out, workspace=d.ws,
                       shape=d.shape)
    assert e.value.code == xqa.XQA_ERR_ALIGN
    lib = xqa.load_library()
    rc = lib.xqa_decode(None, d.k.data_ptr(), d.v.data_ptr(), d.bt.data_ptr(), d.lens.data_ptr(),
                        1.0, 1.0, d.out.data_ptr(), d.shape, d.ws.data_ptr(), d.ws.numel(), None)
    assert rc == xqa.XQA_ERR_NULL
    gqa32 = xqa.XqaShape(1, 32, 1, 128, 16, 16, 16, 0.0, 0, 0)
    with pytest.raises(xqa.XqaError) as e:
        xqa.xqa_workspace_size(gqa32)
    assert e.value.code == xqa.XQA_ERR_SHAPE


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_bad_block_id_is_reported_and_contained(merge_mode):
    w = wl.make_custom([40, 300, 5000], 8, 2, seed=31)
    ref = oracle_of(w)
    w.block_tables[1, 3] = w.num_blocks + 7  # sequence 1 is bad, the others are not
    d = Dev(w, max_ctas=7, merge_mode=merge_mode)  # the bad sequence is split over CTAs
    d.run()
    out = d.result()
    assert d.status() == xqa.XQA_ERR_BAD_BLOCK_ID
    assert np.all(np.isnan(out[1].astype(np.float32)))
    assert_close(out[[0, 2]], ref[[0, 2]], "rows beside a bad block id")
    # a later good call clears the status
    d.bt.copy_(to_dev(wl.make_custom([40, 300, 5000], 8, 2, seed=31).block_tables))
    d.run()
    assert d.status() == xqa.XQA_OK


def test_negative_block_id_is_reported():
    w = wl.make_custom([40, 70], 8, 2, seed=32)
    w.block_tables[0, 0] = -5
    d = Dev(w, max_ctas=1)
    d.run()
    out = d.result()
    assert d.status() == xqa.XQA_ERR_BAD_BLOCK_ID
    assert np.all(np.isnan(out[0].astype(np.float32)))
    assert np.all(np.isfinite(out[1].astype(np.float32)))


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_context_longer_than_table_is_reported(merge_mode):
    w = wl.make_custom([40, 70, 16], 8, 2, seed=33)
    ref = oracle_of(w)
    w.context_lens[1] = w.max_blocks_per_seq * 16 + 1
    d = Dev(w, merge_mode=merge_mode)
    d.run()
    out = d.result()
    assert d.status() == xqa.XQA_ERR_CTX_TOO_LONG
    assert np.all(np.isnan(out[1].astype(np.float32)))
    assert_close(out[[0, 2]], ref[[0, 2]], "rows beside a bad context length")
    w.context_lens[1] = -3
    d.lens.copy_(to_dev(w.context_lens))
    d.run()
    assert d.status() == xqa.XQA_ERR_CTX_TOO_LONG


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_group16_split_segments(merge_mode):
    # G = 16 (64 q heads / 4 kv heads) fills both 8-column MMA tiles for a
    # single new token; long contexts over few CTAs split every segment
    w = wl.make_custom([3000, 5000, 17, 1, 900], 64, 4, seed=91)
    a = run(w, max_ctas=23, merge_mode=merge_mode)
    assert_close(a, oracle_of(w), "G=16")
    b = run(wl.to_nhd(w), max_ctas=23, merge_mode=merge_mode)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
