"""Decode steps with 2B-like heads (16 key heads, 16 value heads, d = 128):
24 independent layer instances (own weights, state and tail) stepped one
after another, one row per stream, at 1, 4, 8 and 16 streams; every layer's
output and updated state checked against the oracle."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
from gated_deltanet_speculative_gb300 import synth

from harness import Case, check_state, check_y, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

LAYERS = 24


@pytest.mark.parametrize("n_streams", [1, 4, 8, 16])
def test_decode_24_layers(n_streams):
    cases = [Case(synth.LIKE_2B, [1] * n_streams, seed=1 + 100 * layer) for layer in range(LAYERS)]
    dims = cases[0].dims_gpu()
    dev_in = [(c.dev_weights(), c.dev_cache(), c.dev_rows(), dev(c.slots)) for c in cases]
    for w, cache, rows, slot in dev_in:   # the layers in order, one step each
        gdn.step(dims, w, cache, slot, rows)
    assert gdn.get_device_error() == 0
    for c, (w, cache, rows, slot) in zip(cases, dev_in):
        y = host_bits(rows["y"])
        st = cache["state"].cpu().numpy()
        tl = host_bits(cache["tail"])
        for s in range(n_streams):
            ref = c.oracle_stream(s)
            sl = int(c.slots[s])
            check_y(y[s:s + 1], ref["y"], what=f"decode y stream {s}")
            check_state(st[sl], ref["rec_state"][0], what=f"decode state stream {s}")
            assert np.array_equal(tl[sl], ref["rec_tail"][0])


@pytest.mark.parametrize("n_streams", [1, 4])
def test_dependent_steps_captured_in_a_graph_equal_eager_bitwise(n_streams):
    """Steps are launched as programmatic dependents of the kernel before
    them and wait for it before touching memory.  Eight consecutive steps on
    the same slots (each reads the state and tail the one before wrote),
    captured in a graph and replayed, equal eight eager steps bit for bit
    (2B-like heads: sliced, clustered steps)."""
    g = synth.LIKE_2B
    T = 8
    c = Case(g, [1] * (n_streams * T), seed=151 + n_streams, n_slots=n_streams + 1,
             slots=np.arange(n_streams * T, dtype=np.int32) % n_streams)
    d, w = c.dims_gpu(), c.dev_weights()
    slot = dev(np.arange(n_streams, dtype=np.int32))
    rows_t = []
    for t in range(T):
        sel = slice(t * n_streams, (t + 1) * n_streams)
        r = {k: dev_bf16(c.rows[k][sel]) for k in ("mixed", "z", "a", "b")}
        r["y"] = torch.zeros((n_streams, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device="cuda")
        rows_t.append(r)
    base_state, base_tail = dev(c.cache["state"]), dev_bf16(c.cache["tail"])

    cache = {"state": base_state.clone(), "tail": base_tail.clone()}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        gdn.step(d, w, {"state": base_state.clone(), "tail": base_tail.clone()}, slot,
                 dict(rows_t[0], y=torch.zeros_like(rows_t[0]["y"])), side)   # warm, outside the capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            for t in range(T):
                gdn.step(d, w, cache, slot, rows_t[t], side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    cache["state"].copy_(base_state)
    cache["tail"].copy_(base_tail)
    for r in rows_t:
        r["y"].zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    got_y = [host_bits(r["y"]) for r in rows_t]
    got_s, got_t = cache["state"].cpu().numpy().view(np.uint32), host_bits(cache["tail"])

    e_cache = {"state": base_state.clone(), "tail": base_tail.clone()}
    for t in range(T):
        e_rows = dict(rows_t[t], y=torch.zeros_like(rows_t[t]["y"]))
        gdn.step(d, w, e_cache, slot, e_rows)
        assert np.array_equal(host_bits(e_rows["y"]), got_y[t]), f"y of step {t}"
    torch.cuda.synchronize()
    assert np.array_equal(e_cache["state"].cpu().numpy().view(np.uint32), got_s)
    assert np.array_equal(host_bits(e_cache["tail"]), got_t)


@pytest.mark.parametrize("g,n_streams", [(synth.LIKE_2B, 1), (synth.LIKE_2B, 4), (synth.LIKE_2B, 16),
                                         (synth.Geometry(2, 6, 128, 128), 1), (synth.Geometry(2, 6, 128, 128), 5),
                                         (synth.Geometry(2, 4, 64, 64), 3), (synth.Geometry(2, 4, 32, 32), 2)],
                         ids=["2b-1", "2b-4", "2b-16", "g3-1", "g3-5", "d64-3", "d32-2"])
def test_early_state_steps_of_24_layers_equal_plain_steps_bitwise(g, n_streams):
    """gdn_step_ex with GDN_STEP_EARLY_STATE over 24 layers (each step's
    previous kernel is the step of another layer, so the promise holds),
    eager and captured in a graph, equals plain gdn_step calls bit for bit:
    y, every layer's state and tail (sliced and unsliced steps, clusters of
    one and of three value heads, d = 32, 64 and 128)."""
    cases = [Case(g, [1] * n_streams, seed=7 + 100 * layer) for layer in range(LAYERS)]
    dims = cases[0].dims_gpu()

    def layers():
        return [(c.dev_weights(), c.dev_cache(), c.dev_rows(), dev(c.slots)) for c in cases]

    def results(ls):
        torch.cuda.synchronize()
        return [(host_bits(r["y"]), cache["state"].cpu().numpy().view(np.uint32), host_bits(cache["tail"]))
                for _, cache, r, _ in ls]

    plain = layers()
    for w, cache, rows, slot in plain:
        gdn.step(dims, w, cache, slot, rows)
    want = results(plain)
    early = layers()
    for w, cache, rows, slot in early:
        gdn.step_ex(dims, w, cache, slot, rows, gdn.STEP_EARLY_STATE)
    assert gdn.get_device_error() == 0
    for l, (a, b) in enumerate(zip(results(early), want)):
        for x, y_, what in zip(a, b, ("y", "state", "tail")):
            assert np.array_equal(x, y_), f"eager layer {l} {what}"
    graphed = layers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    warm = layers()
    with torch.cuda.stream(side):
        for w, cache, rows, slot in warm:   # warm, outside the capture
            gdn.step_ex(dims, w, cache, slot, rows, gdn.STEP_EARLY_STATE, side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            for w, cache, rows, slot in graphed:
                gdn.step_ex(dims, w, cache, slot, rows, gdn.STEP_EARLY_STATE, side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    fresh = layers()   # the capture did not run the steps: reset the graphed buffers to the start
    for (_, c0, r0, _), (_, c1, r1, _) in zip(graphed, fresh):
        c0["state"].copy_(c1["state"])
        c0["tail"].copy_(c1["tail"])
        r0["y"].copy_(r1["y"])
    graph.replay()
    assert gdn.get_device_error() == 0
    for l, (a, b) in enumerate(zip(results(graphed), want)):
        for x, y_, what in zip(a, b, ("y", "state", "tail")):
            assert np.array_equal(x, y_), f"graphed layer {l} {what}"


def test_prepared_steps_equal_direct_calls_bitwise():
    """gdn.prepare checks and marshals a call once; calling the prepared
    steps of 24 layers (twice, the rows' contents changed in between) gives
    what direct gdn_step / gdn_step_ex calls give, bit for bit."""
    cases = [Case(synth.LIKE_2B, [1] * 2, seed=41 + 100 * layer) for layer in range(LAYERS)]
    dims = cases[0].dims_gpu()
    direct = [(c.dev_weights(), c.dev_cache(), c.dev_rows(), dev(c.slots)) for c in cases]
    prep = [(c.dev_weights(), c.dev_cache(), c.dev_rows(), dev(c.slots)) for c in cases]
    calls = [gdn.prepare(gdn.step_ex, dims, w, cache, slot, rows, gdn.STEP_EARLY_STATE) if i % 2
             else gdn.prepare(gdn.step, dims, w, cache, slot, rows)
             for i, (w, cache, rows, slot) in enumerate(prep)]
    for rnd in range(2):
        if rnd:   # new inputs in the same buffers
            for (_, _, r0, _), (_, _, r1, _) in zip(direct, prep):
                for k in ("mixed", "z", "a", "b"):
                    r0[k].copy_(torch.roll(r0[k], 1, dims=-1))
                    r1[k].copy_(r0[k])
        for i, (w, cache, rows, slot) in enumerate(direct):
            if i % 2:
                gdn.step_ex(dims, w, cache, slot, rows, gdn.STEP_EARLY_STATE)
            else:
                gdn.step(dims, w, cache, slot, rows)
        for call in calls:
            call()
        torch.cuda.synchronize()
        assert gdn.get_device_error() == 0
        for l, ((_, c0, r0, _), (_, c1, r1, _)) in enumerate(zip(direct, prep)):
            assert np.array_equal(host_bits(r0["y"]), host_bits(r1["y"])), f"round {rnd} layer {l} y"
            assert np.array_equal(c0["state"].cpu().numpy().view(np.uint32), c1["state"].cpu().numpy().view(np.uint32))
            assert np.array_equal(host_bits(c0["tail"]), host_bits(c1["tail"]))


def test_early_state_step_with_a_bad_slot_skips_only_that_stream():
    """gdn_step_ex with GDN_STEP_EARLY_STATE reads slot[] before it waits;
    a slot out of range still sets the slot bit of the error word, leaves
    that stream's y unwritten, and the other streams equal plain steps."""
    g = synth.LIKE_2B
    c = Case(g, [1, 1, 1], seed=239, n_slots=3, slots=[0, 1, 2])
    d = c.dims_gpu()
    bad = np.array([0, 7, 2], np.int32)   # stream 1's slot is out of range
    want_cache, want_rows = c.dev_cache(), c.dev_rows()
    gdn.step(d, c.dev_weights(), want_cache, dev(np.array([0, 1, 2], np.int32)), want_rows)
    assert gdn.get_device_error() == 0
    cache, rows = c.dev_cache(), c.dev_rows()
    gdn.step_ex(d, c.dev_weights(), cache, dev(bad), rows, gdn.STEP_EARLY_STATE)
    assert gdn.get_device_error() & 1
    y, wy = host_bits(rows["y"]), host_bits(want_rows["y"])
    assert np.all(np.isnan(synth.bf16_bits_to_f32(y[1])))
    for s in (0, 2):
        assert np.array_equal(y[s], wy[s]), f"stream {s}"
    st, wst = cache["state"].cpu().numpy(), want_cache["state"].cpu().numpy()
    for sl in (0, 2):
        assert np.array_equal(st[sl].view(np.uint32), wst[sl].view(np.uint32))
    assert np.array_equal(st[1].view(np.uint32), c.cache["state"][1].view(np.uint32))
