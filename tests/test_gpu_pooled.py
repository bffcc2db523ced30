"""Pooled records and the commit by index (gdn_window_pooled, gdn_tree_pooled,
gdn_commit_swap) against the recorded path (gdn_window / gdn_tree with
rec_state, rec_tail, then the copy commit gdn_commit), bit for bit.

The pooled calls record row r straight into cache entry rec_slot[r]; the
commit then only changes stream s's slot to the kept row's entry.  Every
value a caller can see must be what the recorded path gives: y, each row's
recorded state and tail, and the next round run from the committed slots.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
from gated_deltanet_speculative_gb300 import synth

from harness import Case, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def pool_of(c: Case, extra: int):
    """A device pool of c.n_slots + extra entries; the first c.n_slots hold c's
    committed states and tails, the rest NaN poison."""
    g = c.g
    n_pool = c.n_slots + extra
    st = np.full((n_pool, g.n_v_heads, g.d_v, g.d_k), np.nan, np.float32)
    tl = np.full((n_pool, 3, g.channels), 0x7FC0, np.uint16)
    st[:c.n_slots] = c.cache["state"]
    tl[:c.n_slots] = c.cache["tail"]
    return {"state": dev(st), "tail": dev_bf16(tl)}, n_pool


def run_recorded(c: Case, tree: bool):
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    rs, rt = c.dev_records()
    if tree:
        gdn.tree(d, w, cache, dev(c.slots), dev(c.row_ptr), dev(c.parent), rows, rs, rt)
    else:
        gdn.window(d, w, cache, dev(c.slots), dev(c.row_ptr), rows, rs, rt)
    assert gdn.get_device_error() == 0
    return w, cache, rows, rs, rt


@pytest.mark.parametrize("tree", [False, True], ids=["window", "tree"])
@pytest.mark.parametrize("g", [synth.Geometry(2, 4, 32, 32), synth.Geometry(2, 6, 128, 128)], ids=["d32", "d128"])
def test_pooled_records_equal_recorded_bitwise(g, tree):
    c = Case(g, [16, 5, 1, 9], seed=151, n_slots=6, tree=tree)
    _, _, rows, rs, rt = run_recorded(c, tree)
    d = c.dims_gpu()
    pool, n_pool = pool_of(c, c.R + 3)
    rec_slot = (c.n_slots + np.random.default_rng(5).permutation(c.R + 3)[:c.R]).astype(np.int32)
    prow = c.dev_rows()
    if tree:
        gdn.tree_pooled(d, c.dev_weights(), pool, dev(c.slots), dev(c.row_ptr), dev(c.parent), prow, dev(rec_slot))
    else:
        gdn.window_pooled(d, c.dev_weights(), pool, dev(c.slots), dev(c.row_ptr), prow, dev(rec_slot))
    assert gdn.get_device_error() == 0
    assert np.array_equal(host_bits(prow["y"]), host_bits(rows["y"]))
    pst, ptl = pool["state"].cpu().numpy(), host_bits(pool["tail"])
    rs_h, rt_h = rs.cpu().numpy(), host_bits(rt)
    for r in range(c.R):
        assert np.array_equal(pst[rec_slot[r]].view(np.uint32), rs_h[r].view(np.uint32)), f"state of row {r}"
        assert np.array_equal(ptl[rec_slot[r]], rt_h[r]), f"tail of row {r}"
    # the committed entries are read, never written
    assert np.array_equal(pst[:c.n_slots].view(np.uint32), c.cache["state"].view(np.uint32))
    assert np.array_equal(ptl[:c.n_slots], c.cache["tail"])


def test_commit_swap_then_next_round_equals_copy_commit_bitwise():
    """Round 1 pooled + swap against round 1 recorded + copy commit, then a
    second round from the committed slots on both sides."""
    g = synth.Geometry(2, 6, 128, 128)
    c = Case(g, [16, 7, 3, 12], seed=157, n_slots=5)
    rng = np.random.default_rng(157)
    acc = np.array([0, 7, 1, 5], np.int32)   # accepted lengths: nothing, all, one, part
    keep = np.where(acc > 0, c.row_ptr[:-1] + acc - 1, -1).astype(np.int32)
    d = c.dims_gpu()
    # recorded path
    w, cache, rows, rs, rt = run_recorded(c, False)
    gdn.commit(d, cache, dev(c.slots), dev(c.row_ptr), dev(keep), rs, rt)
    # pooled path
    pool, n_pool = pool_of(c, c.R + 2)
    rec_slot = (c.n_slots + rng.permutation(c.R + 2)[:c.R]).astype(np.int32)
    slot_t = dev(c.slots.copy())
    gdn.window_pooled(d, c.dev_weights(), pool, slot_t, dev(c.row_ptr), c.dev_rows(), dev(rec_slot))
    freed = torch.full((c.S,), 99, dtype=torch.int32, device="cuda")
    gdn.commit_swap(d, pool, slot_t, dev(c.row_ptr), dev(keep), dev(rec_slot), freed)
    assert gdn.get_device_error() == 0
    new_slot = slot_t.cpu().numpy()
    exp_slot = np.where(keep >= 0, rec_slot[np.maximum(keep, 0)], c.slots)
    assert np.array_equal(new_slot, exp_slot)
    assert np.array_equal(freed.cpu().numpy(), np.where(keep >= 0, c.slots, -1))
    st, tl = cache["state"].cpu().numpy(), host_bits(cache["tail"])
    pst, ptl = pool["state"].cpu().numpy(), host_bits(pool["tail"])
    for s in range(c.S):
        assert np.array_equal(pst[new_slot[s]].view(np.uint32), st[c.slots[s]].view(np.uint32)), f"stream {s}"
        assert np.array_equal(ptl[new_slot[s]], tl[c.slots[s]])
    # round 2: new rows from the committed states
    c2 = Case(g, [4, 16, 2, 9], seed=163, n_slots=5)
    rows2 = c2.dev_rows()
    rs2, rt2 = c2.dev_records()
    gdn.window(d, w, cache, dev(c.slots), dev(c2.row_ptr), rows2, rs2, rt2)
    free = sorted(set(range(n_pool)) - set(int(x) for x in new_slot))
    rec2 = np.array(free[:c2.R], np.int32)
    prow2 = c2.dev_rows()
    gdn.window_pooled(d, c.dev_weights(), pool, slot_t, dev(c2.row_ptr), prow2, dev(rec2))
    assert gdn.get_device_error() == 0
    assert np.array_equal(host_bits(prow2["y"]), host_bits(rows2["y"]))
    pst = pool["state"].cpu().numpy()
    rs2_h = rs2.cpu().numpy()
    for r in range(c2.R):
        assert np.array_equal(pst[rec2[r]].view(np.uint32), rs2_h[r].view(np.uint32)), f"round 2 row {r}"


def test_pooled_rounds_with_a_free_list_equal_recorded_rounds():
    """Five rounds of random accepted lengths on 8 streams, the pool's free
    entries recycled on the host from freed[] and the unkept rows."""
    g = synth.Geometry(2, 4, 64, 64)
    S, W = 8, 16
    base = Case(g, [W] * S, seed=167, n_slots=S)
    d = base.dims_gpu()
    w = base.dev_weights()
    cache = base.dev_cache()
    slots = np.arange(S, dtype=np.int32)
    pool, n_pool = pool_of(base, S * W + 4)
    pslot = dev(slots.copy())
    free = list(range(S, n_pool))
    rng = np.random.default_rng(167)
    for rnd in range(5):
        lengths = rng.integers(1, W + 1, size=S)
        c = Case(g, lengths, seed=200 + rnd, n_slots=S)
        acc = rng.integers(0, lengths + 1)
        keep = np.where(acc > 0, c.row_ptr[:-1] + acc - 1, -1).astype(np.int32)
        rows = c.dev_rows()
        rs, rt = c.dev_records()
        gdn.window(d, w, cache, dev(slots), dev(c.row_ptr), rows, rs, rt)
        gdn.commit(d, cache, dev(slots), dev(c.row_ptr), dev(keep), rs, rt)
        rec = np.array(free[:c.R], np.int32)
        free = free[c.R:]
        prow = c.dev_rows()
        gdn.window_pooled(d, w, pool, pslot, dev(c.row_ptr), prow, dev(rec))
        freed = torch.empty(S, dtype=torch.int32, device="cuda")
        gdn.commit_swap(d, pool, pslot, dev(c.row_ptr), dev(keep), dev(rec), freed)
        assert gdn.get_device_error() == 0
        assert np.array_equal(host_bits(prow["y"]), host_bits(rows["y"])), f"y round {rnd}"
        kept = set(int(rec[k]) for k in keep if k >= 0)
        free += [int(x) for x in rec if int(x) not in kept] + [int(x) for x in freed.cpu().numpy() if x >= 0]
        cur = pslot.cpu().numpy()
        st, pst = cache["state"].cpu().numpy(), pool["state"].cpu().numpy()
        for s in range(S):
            assert np.array_equal(pst[cur[s]].view(np.uint32), st[slots[s]].view(np.uint32)), f"round {rnd} stream {s}"
    assert len(set(free)) == len(free) == n_pool - S


def test_pooled_index_checks_skip_the_stream():
    g = synth.Geometry(2, 4, 32, 32)
    c = Case(g, [3, 2], seed=173, n_slots=2)
    d = c.dims_gpu()
    pool, n_pool = pool_of(c, 8)
    rows = c.dev_rows()
    # stream 1's second row is recorded outside the pool: stream 1 is skipped
    rec = np.array([2, 3, 4, 5, n_pool], np.int32)
    gdn.window_pooled(d, c.dev_weights(), pool, dev(c.slots), dev(c.row_ptr), rows, dev(rec))
    assert gdn.get_device_error() & 1
    y = synth.bf16_bits_to_f32(host_bits(rows["y"]))
    assert np.all(np.isfinite(y[0:3])) and np.all(np.isnan(y[3:5]))
    # a row recorded onto its own stream's slot
    rows = c.dev_rows()
    rec = np.array([2, 3, 4, int(c.slots[1]), 6], np.int32)
    gdn.window_pooled(d, c.dev_weights(), pool, dev(c.slots), dev(c.row_ptr), rows, dev(rec))
    assert gdn.get_device_error() & 1
    assert np.all(np.isnan(synth.bf16_bits_to_f32(host_bits(rows["y"]))[3:5]))
    # a kept row outside the stream's rows, and a kept entry out of range
    slot_t = dev(c.slots.copy())
    freed = torch.empty(2, dtype=torch.int32, device="cuda")
    gdn.commit_swap(d, pool, slot_t, dev(c.row_ptr), dev(np.array([3, 4], np.int32)), dev(np.array([2, 3, 4, 5, n_pool + 1], np.int32)), freed)
    bits = gdn.get_device_error()
    assert bits & 8 and bits & 1
    assert np.array_equal(slot_t.cpu().numpy(), c.slots)
    assert np.array_equal(freed.cpu().numpy(), [-1, -1])


def test_pooled_full_round_16x16_then_swap_against_oracle():
    """The round the benchmark times, at its size: 16 streams x 16 rows,
    27B-like heads, a pool of 16 + 256 + 16 entries with the round's entries
    taken in a shuffled order, every row recorded into its entry
    (gdn_window_pooled), then random accepted lengths committed by index
    (gdn_commit_swap).  y and every recorded state and tail against the
    oracle; each committed slot's entry holds the oracle's state and tail
    after the stream's last accepted row."""
    from harness import check_state, check_y
    g = synth.LIKE_27B
    c = Case(g, [16] * 16, seed=181)
    d = c.dims_gpu()
    n_pool = c.S + c.R + c.S
    rng = np.random.default_rng(181)
    free = c.S + rng.permutation(c.R + c.S).astype(np.int32)
    rec_slot = free[:c.R].copy()
    slots = np.arange(c.S, dtype=np.int32)
    ps = torch.full((n_pool, g.n_v_heads, g.d_v, g.d_k), float("nan"), dtype=torch.float32, device="cuda")
    pt = torch.full((n_pool, 3, g.channels), float("nan"), dtype=torch.bfloat16, device="cuda")
    ps[:c.S].copy_(torch.from_numpy(c.cache["state"][c.slots]))
    pt[:c.S].copy_(torch.from_numpy(c.cache["tail"][c.slots].view(np.int16)).view(torch.bfloat16))
    pool = {"state": ps, "tail": pt}
    rows = c.dev_rows()
    slot_t = dev(slots)
    gdn.window_pooled(d, c.dev_weights(), pool, slot_t, dev(c.row_ptr), rows, dev(rec_slot))
    acc = synth.accepted_lengths(c.S, 16, rng)
    keep = np.where(acc > 0, c.row_ptr[:-1] + acc - 1, -1).astype(np.int32)
    freed = torch.empty(c.S, dtype=torch.int32, device="cuda")
    gdn.commit_swap(d, pool, slot_t, dev(c.row_ptr), dev(keep), dev(rec_slot), freed)
    assert gdn.get_device_error() == 0
    y = host_bits(rows["y"])
    new_slot = slot_t.cpu().numpy()
    assert np.array_equal(new_slot, np.where(keep >= 0, rec_slot[np.maximum(keep, 0)], slots))
    assert np.array_equal(freed.cpu().numpy(), np.where(keep >= 0, slots, -1))
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        ref = c.oracle_stream(s)
        ent = rec_slot[lo:hi]
        check_y(y[lo:hi], ref["y"], what=f"y stream {s}")
        check_state(ps[torch.from_numpy(ent).long().cuda()].cpu().numpy(), ref["rec_state"],
                    what=f"recorded states stream {s}")
        assert np.array_equal(host_bits(pt[torch.from_numpy(ent).long().cuda()]), ref["rec_tail"]), f"tails {s}"
        e = int(new_slot[s])
        if keep[s] >= 0:
            k = int(keep[s]) - lo
            check_state(ps[e].cpu().numpy()[None], ref["rec_state"][k][None], what=f"committed state {s}")
            assert np.array_equal(host_bits(pt[e]), ref["rec_tail"][k]), f"committed tail {s}"
        else:
            assert np.array_equal(ps[e].cpu().numpy().view(np.uint32),
                                  c.cache["state"][c.slots[s]].view(np.uint32)), f"untouched slot {s}"


def test_pooled_round_swap_then_step_back_to_back_equals_copy_path():
    """window_pooled, commit_swap and a one-row step of every stream, queued
    back to back with no host synchronisation in between (the swap and the
    step are programmatic dependents of the kernel before them and read the
    slot words only after it ends), against gdn_window + gdn_commit +
    gdn_step, bit for bit."""
    g = synth.Geometry(2, 6, 128, 128)
    c = Case(g, [16, 9, 4, 1], seed=191, n_slots=4, slots=[0, 1, 2, 3])
    acc = np.array([16, 0, 2, 1], np.int32)
    keep = np.where(acc > 0, c.row_ptr[:-1] + acc - 1, -1).astype(np.int32)
    step_rows = synth.row_inputs(g, c.S, 193)
    d = c.dims_gpu()

    def dev_step_rows():
        r = {k: dev_bf16(step_rows[k]) for k in ("mixed", "z", "a", "b")}
        r["y"] = torch.full((c.S, g.n_v_heads, g.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        return r

    # copy path
    w, cache, rows, rs, rt = run_recorded(c, False)
    gdn.commit(d, cache, dev(c.slots), dev(c.row_ptr), dev(keep), rs, rt)
    sr = dev_step_rows()
    gdn.step(d, w, cache, dev(c.slots), sr)
    assert gdn.get_device_error() == 0
    # pooled path, one stream, no synchronisation
    pool, n_pool = pool_of(c, c.R)
    rec_slot = (c.n_slots + np.arange(c.R)).astype(np.int32)
    slot_t = dev(c.slots.copy())
    prow, psr = c.dev_rows(), dev_step_rows()
    gdn.window_pooled(d, c.dev_weights(), pool, slot_t, dev(c.row_ptr), prow, dev(rec_slot))
    gdn.commit_swap(d, pool, slot_t, dev(c.row_ptr), dev(keep), dev(rec_slot))
    gdn.step(d, c.dev_weights(), pool, slot_t, psr)
    assert gdn.get_device_error() == 0
    assert np.array_equal(host_bits(psr["y"]), host_bits(sr["y"]))
    cur = slot_t.cpu().numpy()
    st, pst = cache["state"].cpu().numpy(), pool["state"].cpu().numpy()
    tl, ptl = host_bits(cache["tail"]), host_bits(pool["tail"])
    for s in range(c.S):
        assert np.array_equal(pst[cur[s]].view(np.uint32), st[c.slots[s]].view(np.uint32)), f"state {s}"
        assert np.array_equal(ptl[cur[s]], tl[c.slots[s]]), f"tail {s}"


def test_prepared_pooled_rounds_equal_direct_calls_bitwise():
    """Three pooled rounds (window + index commit) through prepared calls,
    the rows, pool entries and keep rows refilled in the same buffers each
    round, against the same rounds through direct calls."""
    g = synth.Geometry(2, 6, 128, 128)
    S, W = 4, 16
    base = Case(g, [W] * S, seed=197, n_slots=S)
    d = base.dims_gpu()
    rng = np.random.default_rng(197)
    sides = []
    for _ in range(2):
        pool, n_pool = pool_of(base, 3 * S * W)
        sides.append({"w": base.dev_weights(), "pool": pool, "slot": dev(base.slots.copy()),
                      "rp": dev(base.row_ptr), "rows": base.dev_rows(),
                      "rec": torch.zeros(S * W, dtype=torch.int32, device="cuda"),
                      "keep": torch.zeros(S, dtype=torch.int32, device="cuda")})
    p = sides[1]
    win = gdn.prepare(gdn.window_pooled, d, p["w"], p["pool"], p["slot"], p["rp"], p["rows"], p["rec"])
    swap = gdn.prepare(gdn.commit_swap, d, p["pool"], p["slot"], p["rp"], p["keep"], p["rec"])
    for rnd in range(3):
        c = Case(g, [W] * S, seed=300 + rnd, n_slots=S)
        acc = rng.integers(0, W + 1, size=S)
        keep = np.where(acc > 0, c.row_ptr[:-1] + acc - 1, -1).astype(np.int32)
        rec = (S + rnd * S * W + rng.permutation(S * W)).astype(np.int32)   # fresh entries each round
        for side in sides:
            for k, v in c.dev_rows().items():
                side["rows"][k].copy_(v)
            side["rec"].copy_(dev(rec))
            side["keep"].copy_(dev(keep))
        q = sides[0]
        gdn.window_pooled(d, q["w"], q["pool"], q["slot"], q["rp"], q["rows"], q["rec"])
        gdn.commit_swap(d, q["pool"], q["slot"], q["rp"], q["keep"], q["rec"])
        win()
        swap()
        torch.cuda.synchronize()
        assert gdn.get_device_error() == 0
        assert np.array_equal(host_bits(q["rows"]["y"]), host_bits(p["rows"]["y"])), f"y round {rnd}"
        assert np.array_equal(q["slot"].cpu().numpy(), p["slot"].cpu().numpy())
        cur = p["slot"].cpu().numpy()
        a, b = q["pool"]["state"].cpu().numpy(), p["pool"]["state"].cpu().numpy()
        for s_ in range(S):
            assert np.array_equal(a[cur[s_]].view(np.uint32), b[cur[s_]].view(np.uint32)), f"round {rnd} stream {s_}"
