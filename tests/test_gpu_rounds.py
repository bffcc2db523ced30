"""Shared verify rounds of every shape, one captured graph for all shapes, and
prompt passes resumed at a chunk-grid point.

* Randomised shared rounds (TensorFold #747, first note: the engine's checks
  cover chain and tree windows and rounds shared by 2 to 16 streams, at most
  256 rows, packed at every possible offset): each round is compared with the
  oracle.
* One CUDA graph of gdn_window / gdn_tree / gdn_commit captured for the
  largest shape serves every smaller shape: the kernels read the true row
  counts from the device (TensorFold #932, drafter note: the row counts are
  read on the device, not baked into the launch), so replays with new row_ptr / parent /
  keep_row contents equal eager calls bit for bit.
* A prompt split at a multiple of the chunk (a grid point) and resumed from
  the kept state ends bit-identical to one pass (TensorFold #747, kept state
  note: resuming at a grid point gives the same result as an uninterrupted
  pass).
"""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
from gated_deltanet_speculative_gb300 import synth

from harness import Case, check_state, check_y, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("round_id", range(12))
def test_randomised_shared_rounds_against_oracle(round_id):
    rng = np.random.default_rng(1000 + round_id)
    S = int(rng.integers(2, 17))
    lengths = rng.integers(1, 17, size=S).tolist()
    tree = bool(round_id % 2)
    g = synth.Geometry(4, 12, 128, 128) if round_id % 3 else synth.Geometry(2, 8, 64, 64)
    pad = int(rng.integers(0, 7))           # unrelated rows packed in front
    c = Case(g, [pad] + lengths, seed=2000 + round_id, tree=tree, n_slots=S + 3)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    rs, rt = c.dev_records()
    if tree:
        gdn.tree(d, w, cache, dev(c.slots), dev(c.row_ptr), dev(c.parent), rows, rs, rt)
    else:
        gdn.window(d, w, cache, dev(c.slots), dev(c.row_ptr), rows, rs, rt)
    assert gdn.get_device_error() == 0
    y, rsn, rtn = host_bits(rows["y"]), rs.cpu().numpy(), host_bits(rt)
    for s in range(1, c.S):
        lo, hi = c.stream_rows(s)
        ref = c.oracle_stream(s)
        check_y(y[lo:hi], ref["y"], what=f"round {round_id} stream {s}")
        check_state(rsn[lo:hi], ref["rec_state"], what=f"round {round_id} stream {s}")
        assert np.array_equal(rtn[lo:hi], ref["rec_tail"])


def test_one_graph_serves_every_round_shape():
    g = synth.Geometry(4, 12, 128, 128)
    S, W = 16, 16
    R = S * W
    c = Case(g, [W] * S, seed=77, tree=True)
    d = c.dims_gpu()
    w = c.dev_weights()
    base_state = dev(c.cache["state"])
    base_tail = dev_bf16(c.cache["tail"])
    rows = c.dev_rows(poison=False)
    slot = dev(c.slots)
    rp = torch.zeros(S + 1, dtype=torch.int32, device="cuda")
    par = torch.zeros(R, dtype=torch.int32, device="cuda")
    keep = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    rs = torch.zeros((R, g.n_v_heads, g.d_v, g.d_k), dtype=torch.float32, device="cuda")
    rt = torch.zeros((R, 3, g.channels), dtype=torch.bfloat16, device="cuda")
    cache = {"state": base_state.clone(), "tail": base_tail.clone()}

    def round_():
        gdn.tree(d, w, cache, slot, rp, par, rows, rs, rt)
        gdn.commit(d, cache, slot, rp, keep, rs, rt)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        round_()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            round_()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    rng = np.random.default_rng(78)
    for trial in range(4):
        lengths = rng.integers(0, W + 1, size=S)
        rp_h = synth.row_ptr(lengths)
        par_h = np.zeros(R, np.int32)
        for s in range(S):
            par_h[rp_h[s]:rp_h[s + 1]] = synth.random_tree(int(lengths[s]), rng)
        keep_h = np.array([rp_h[s] + rng.integers(0, lengths[s]) if lengths[s] else -1 for s in range(S)], np.int32)
        # graph replay
        rp.copy_(torch.from_numpy(rp_h))
        par.copy_(torch.from_numpy(par_h))
        keep.copy_(torch.from_numpy(keep_h))
        cache["state"].copy_(base_state)
        cache["tail"].copy_(base_tail)
        rows["y"].zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.get_device_error() == 0
        got_y, got_s, got_t = host_bits(rows["y"]), cache["state"].cpu().numpy(), host_bits(cache["tail"])
        got_rs = rs.cpu().numpy()
        # the same round eagerly, into fresh buffers
        e_cache = {"state": base_state.clone(), "tail": base_tail.clone()}
        e_rows = dict(rows, y=torch.zeros_like(rows["y"]))
        e_rs, e_rt = torch.zeros_like(rs), torch.zeros_like(rt)
        gdn.tree(d, w, e_cache, slot, dev(rp_h), dev(par_h), e_rows, e_rs, e_rt)
        gdn.commit(d, e_cache, slot, dev(rp_h), dev(keep_h), e_rs, e_rt)
        torch.cuda.synchronize()
        n_live = int(rp_h[-1])
        assert np.array_equal(got_y[:n_live], host_bits(e_rows["y"])[:n_live])
        assert np.array_equal(got_rs[:n_live].view(np.uint32), e_rs.cpu().numpy()[:n_live].view(np.uint32))
        assert np.array_equal(got_s.view(np.uint32), e_cache["state"].cpu().numpy().view(np.uint32))
        assert np.array_equal(got_t, host_bits(e_cache["tail"]))


@pytest.mark.parametrize("cut", [64, 128, 192])
def test_prefill_resumed_at_a_grid_point_is_bit_identical(cut):
    g = synth.LIKE_27B
    whole = Case(g, [300], seed=81, zero_state=True)
    d = whole.dims_gpu()
    w = whole.dev_weights()

    def run(pieces):
        cache = whole.dev_cache()
        slot = dev(whole.slots)
        ys = []
        for lo, hi in pieces:
            rows = {k: dev_bf16(v[lo:hi]) for k, v in whole.rows.items() if k != "y"}
            rows["y"] = torch.empty((hi - lo, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device="cuda")
            ws = torch.empty(gdn.prefill_workspace_size(d, 1, hi - lo), dtype=torch.uint8, device="cuda")
            gdn.prefill(d, w, cache, slot, dev(np.array([0, hi - lo], np.int32)), rows, ws)
            ys.append(host_bits(rows["y"]))
        assert gdn.get_device_error() == 0
        return np.concatenate(ys), cache["state"].cpu().numpy(), host_bits(cache["tail"])

    y1, s1, t1 = run([(0, 300)])
    y2, s2, t2 = run([(0, cut), (cut, 300)])
    assert np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    assert np.array_equal(t1, t2)
    assert np.array_equal(y1, y2)


def test_kept_state_saved_to_host_and_restored_resumes_bit_identical():
    """A stream's kept state in host memory (TensorFold #888: a kept state is
    the stream's full recurrent state with its conv history, held in host
    memory and restored later).  Round 1 is verified and committed; the
    slot's state and tail are copied to pinned host memory, the device slot
    is overwritten with garbage, then restored with plain async copies; round
    2 from the restored slot equals round 2 of an uninterrupted run, bit for
    bit (the library keeps nothing else between calls)."""
    g = synth.LIKE_27B
    S, W = 4, 16
    c1 = Case(g, [W] * S, seed=131, n_slots=6)
    c2 = Case(g, [W] * S, seed=137, n_slots=6)   # round 2's rows (same weights and slots as round 1)
    d, w = c1.dims_gpu(), c1.dev_weights()
    slot, rp = dev(c1.slots), dev(c1.row_ptr)
    keep = dev(np.array([c1.row_ptr[s] + (5 * s + 3) % W for s in range(S)], np.int32))

    def round_(cache, c):
        rows = c.dev_rows()
        rs, rt = c.dev_records()
        gdn.window(d, w, cache, slot, rp, rows, rs, rt)
        gdn.commit(d, cache, slot, rp, keep, rs, rt)
        return rows

    # uninterrupted: round 1, round 2
    cache_a = c1.dev_cache()
    round_(cache_a, c1)
    rows_a = round_(cache_a, c2)
    # interrupted: round 1, save to pinned host memory, poison, restore, round 2
    cache_b = c1.dev_cache()
    round_(cache_b, c1)
    host_state = torch.empty(cache_b["state"].shape, dtype=torch.float32).pin_memory()
    host_tail = torch.empty(cache_b["tail"].shape, dtype=torch.bfloat16).pin_memory()
    host_state.copy_(cache_b["state"], non_blocking=True)
    host_tail.copy_(cache_b["tail"], non_blocking=True)
    torch.cuda.synchronize()
    cache_b["state"].fill_(float("nan"))
    cache_b["tail"].fill_(float("nan"))
    cache_b["state"].copy_(host_state, non_blocking=True)
    cache_b["tail"].copy_(host_tail, non_blocking=True)
    rows_b = round_(cache_b, c2)
    assert gdn.get_device_error() == 0
    assert np.array_equal(host_bits(rows_b["y"]), host_bits(rows_a["y"]))
    assert np.array_equal(cache_b["state"].cpu().numpy().view(np.uint32), cache_a["state"].cpu().numpy().view(np.uint32))
    assert np.array_equal(host_bits(cache_b["tail"]), host_bits(cache_a["tail"]))
