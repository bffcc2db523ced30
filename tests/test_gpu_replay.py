"""Logged windows and replay commit (TensorFold #932, tree note: per-row logs
of the decay, the write vector and the key replace the recorded states, and
the commit re-applies the accepted rows to the committed state in one pass).

gdn_window_log must give gdn_window's y and tails bit for bit, its logs must
be the oracle's per-row decay and key (to tolerance) and satisfy
S_r = a_r S_{r-1} + u_r k_r^T against the recorded states, and
gdn_commit_replay must leave every slot exactly as gdn_commit does."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
import oracle
from gated_deltanet_speculative_gb300 import synth

from harness import Case, check_state, check_y, dev, host_bits

pytestmark = pytest.mark.gpu


def _logs(c: Case):
    g = c.g
    R = max(c.R, 1)
    return (torch.full((R, g.n_v_heads), float("nan"), device="cuda"),
            torch.full((R, g.n_v_heads, g.d_v), float("nan"), device="cuda"),
            torch.full((R, g.n_k_heads, g.d_k), float("nan"), device="cuda"),
            torch.full((R, 3, g.channels), float("nan"), dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("g", [synth.LIKE_27B, synth.Geometry(2, 4, 64, 64), synth.Geometry(2, 2, 32, 32)])
def test_logged_window_and_replay_commit_equal_recorded_path(g):
    lengths = [16, 5, 1, 16, 9, 0, 12]
    c = Case(g, lengths, seed=91, n_slots=9)
    d = c.dims_gpu()
    w = c.dev_weights()
    slot, rp = dev(c.slots), dev(c.row_ptr)
    rng = np.random.default_rng(91)
    acc = synth.accepted_lengths(c.S, 16, rng)
    acc = np.minimum(acc, np.array(lengths))
    acc[0], acc[3] = 0, 16
    keep = np.where(acc > 0, c.row_ptr[:-1] + acc - 1, -1).astype(np.int32)

    # recorded path
    cache_r, rows_r = c.dev_cache(), c.dev_rows()
    rs, rt = c.dev_records()
    gdn.window(d, w, cache_r, slot, rp, rows_r, rs, rt)
    gdn.commit(d, cache_r, slot, rp, dev(keep), rs, rt)
    # logged path
    cache_l, rows_l = c.dev_cache(), c.dev_rows()
    la, lu, lk, lt = _logs(c)
    gdn.window_log(d, w, cache_l, slot, rp, rows_l, la, lu, lk, lt)
    gdn.commit_replay(d, cache_l, slot, rp, dev(keep), la, lu, lk, lt)
    assert gdn.get_device_error() == 0

    assert np.array_equal(host_bits(rows_l["y"])[:c.R], host_bits(rows_r["y"])[:c.R])
    assert np.array_equal(host_bits(lt)[:c.R], host_bits(rt)[:c.R])
    assert np.array_equal(cache_l["state"].cpu().numpy().view(np.uint32), cache_r["state"].cpu().numpy().view(np.uint32))
    assert np.array_equal(host_bits(cache_l["tail"]), host_bits(cache_r["tail"]))

    # the logs themselves: decay and key against the oracle, and the rank-1
    # step against the recorded states
    la_n, lu_n, lk_n, rs_n = la.cpu().numpy(), lu.cpu().numpy(), lk.cpu().numpy(), rs.cpu().numpy()
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        if hi == lo:
            continue
        r = c.rows
        sl = int(c.slots[s])
        ref = oracle.gdn_rows(c.dims_oracle(), c.w, c.cache["state"][sl], c.cache["tail"][sl], r["mixed"][lo:hi],
                              r["z"][lo:hi], r["a"][lo:hi], r["b"][lo:hi], extras=True)
        np.testing.assert_allclose(la_n[lo:hi], ref["decay"], rtol=1e-5, atol=1e-7)
        for hh in range(g.n_v_heads):
            kh = hh // g.group
            np.testing.assert_allclose(lk_n[lo:hi, kh], ref["k"][:, hh], rtol=0, atol=2e-6)
        prev = c.cache["state"][sl].astype(np.float64)
        for t in range(lo, hi):
            kk = lk_n[t][np.arange(g.n_v_heads) // g.group]            # [Hv, dk]
            step = la_n[t][:, None, None] * prev + lu_n[t][:, :, None] * kk[:, None, :]
            scale = np.abs(rs_n[t]).max()
            assert np.abs(step - rs_n[t]).max() <= 1e-6 * scale
            prev = rs_n[t].astype(np.float64)


def test_replay_commit_rejects_keep_outside_the_stream_window():
    g = synth.Geometry(2, 4, 32, 32)
    c = Case(g, [4, 3], seed=93)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    la, lu, lk, lt = _logs(c)
    gdn.window_log(d, w, cache, dev(c.slots), dev(c.row_ptr), rows, la, lu, lk, lt)
    before = cache["state"].cpu().numpy().copy()
    bad = np.array([5, -1], np.int32)   # row 5 belongs to stream 1, not stream 0
    gdn.commit_replay(d, cache, dev(c.slots), dev(c.row_ptr), dev(bad), la, lu, lk, lt)
    assert gdn.get_device_error() & 8
    assert np.array_equal(cache["state"].cpu().numpy(), before)


def _tree_case(g, seed):
    """Trees of several shapes in one call: random recursive trees, a star, a
    window with several roots (nodes that follow the committed slot), a
    chain with late branches, a single node and an empty window."""
    lengths = [16, 5, 1, 16, 9, 0, 12, 16]
    c = Case(g, lengths, seed=seed, n_slots=10, tree=True)
    shapes = {
        3: [-1] + [0] * 15,                                   # star under node 0
        4: [-1, 0, -1, 2, 1, -1, 5, 3, 0],                    # three roots
        6: [-1, 0, 1, 2, 3, 4, 5, 6, 7, 8, 2, 10],            # chain, then a branch from node 2
    }
    for s, par in shapes.items():
        lo, hi = c.stream_rows(s)
        c.parent[lo:hi] = np.asarray(par, np.int32)
    return c


def _kept_nodes(c: Case, rng):
    keep = np.full(c.S, -1, np.int32)
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        if hi == lo or s == 2:          # stream 2 accepts nothing: its slot must keep its bits
            continue
        par = c.parent[lo:hi]
        node = synth.random_leaf(par, rng) if s % 2 == 0 else int(rng.integers(0, hi - lo))
        keep[s] = lo + node
    return keep


@pytest.mark.parametrize("g", [synth.LIKE_27B, synth.Geometry(2, 4, 64, 64), synth.Geometry(2, 2, 32, 32)])
def test_logged_tree_and_replay_commit_equal_recorded_tree(g):
    """gdn_tree_log gives gdn_tree's y and tails bit for bit (a node whose
    parent is not the node visited before it rebuilds the parent's state by
    replaying logs from the slot), and gdn_commit_replay_tree leaves every
    slot exactly as gdn_commit of the recorded node does."""
    c = _tree_case(g, 95)
    d = c.dims_gpu()
    w = c.dev_weights()
    slot, rp, par = dev(c.slots), dev(c.row_ptr), dev(c.parent)
    keep = _kept_nodes(c, np.random.default_rng(95))

    cache_r, rows_r = c.dev_cache(), c.dev_rows()
    rs, rt = c.dev_records()
    gdn.tree(d, w, cache_r, slot, rp, par, rows_r, rs, rt)
    gdn.commit(d, cache_r, slot, rp, dev(keep), rs, rt)
    cache_l, rows_l = c.dev_cache(), c.dev_rows()
    la, lu, lk, lt = _logs(c)
    gdn.tree_log(d, w, cache_l, slot, rp, par, rows_l, la, lu, lk, lt)
    gdn.commit_replay_tree(d, cache_l, slot, rp, par, dev(keep), la, lu, lk, lt)
    assert gdn.get_device_error() == 0

    assert np.array_equal(host_bits(rows_l["y"])[:c.R], host_bits(rows_r["y"])[:c.R])
    assert np.array_equal(host_bits(lt)[:c.R], host_bits(rt)[:c.R])
    assert np.array_equal(cache_l["state"].cpu().numpy().view(np.uint32), cache_r["state"].cpu().numpy().view(np.uint32))
    assert np.array_equal(host_bits(cache_l["tail"]), host_bits(cache_r["tail"]))

    # each node's log is one rank-1 step from its parent's recorded state (or
    # the committed slot) to its own
    la_n, lu_n, lk_n, rs_n = la.cpu().numpy(), lu.cpu().numpy(), lk.cpu().numpy(), rs.cpu().numpy()
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        sl = int(c.slots[s])
        for t in range(lo, hi):
            p_loc = int(c.parent[t])
            prev = (c.cache["state"][sl] if p_loc < 0 else rs_n[lo + p_loc]).astype(np.float64)
            kk = lk_n[t][np.arange(g.n_v_heads) // g.group]
            step = la_n[t][:, None, None] * prev + lu_n[t][:, :, None] * kk[:, None, :]
            assert np.abs(step - rs_n[t]).max() <= 1e-6 * np.abs(rs_n[t]).max()


def test_logged_tree_round_16x16_against_oracle():
    """The bench's tree round (16 streams x 16-node random trees, 27B-like
    heads): y within tolerance of the oracle, and the replayed commit of a
    random leaf per stream equal to the oracle's state at that node."""
    g = synth.LIKE_27B
    c = Case(g, [16] * 16, seed=97, tree=True)
    d = c.dims_gpu()
    slot, rp, par = dev(c.slots), dev(c.row_ptr), dev(c.parent)
    rng = np.random.default_rng(97)
    keep = np.array([c.row_ptr[s] + synth.random_leaf(c.parent[c.row_ptr[s]:c.row_ptr[s + 1]], rng)
                     for s in range(c.S)], np.int32)
    cache, rows = c.dev_cache(), c.dev_rows()
    la, lu, lk, lt = _logs(c)
    gdn.tree_log(d, c.dev_weights(), cache, slot, rp, par, rows, la, lu, lk, lt)
    gdn.commit_replay_tree(d, cache, slot, rp, par, dev(keep), la, lu, lk, lt)
    assert gdn.get_device_error() == 0
    y = host_bits(rows["y"])
    st = cache["state"].cpu().numpy()
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        ref = c.oracle_stream(s)
        check_y(y[lo:hi], ref["y"], f"stream {s} y")
        check_state(st[c.slots[s]], ref["rec_state"][keep[s] - lo], f"stream {s} committed state")


def test_tree_replay_commit_rejects_bad_parent_and_keep():
    g = synth.Geometry(2, 4, 32, 32)
    c = Case(g, [4, 3], seed=99, tree=True)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    la, lu, lk, lt = _logs(c)
    par = dev(c.parent)
    gdn.tree_log(d, w, cache, dev(c.slots), dev(c.row_ptr), par, rows, la, lu, lk, lt)
    assert gdn.get_device_error() == 0
    before = cache["state"].cpu().numpy().copy()
    bad_par = c.parent.copy()
    bad_par[3] = 3                          # node 3 of stream 0 names itself as its parent
    gdn.commit_replay_tree(d, cache, dev(c.slots), dev(c.row_ptr), dev(bad_par), dev(np.array([3, -1], np.int32)),
                           la, lu, lk, lt)
    assert gdn.get_device_error() & 4
    gdn.commit_replay_tree(d, cache, dev(c.slots), dev(c.row_ptr), par, dev(np.array([5, -1], np.int32)),
                           la, lu, lk, lt)   # row 5 belongs to stream 1
    assert gdn.get_device_error() & 8
    assert np.array_equal(cache["state"].cpu().numpy(), before)


@pytest.mark.parametrize("round_id", range(8))
def test_randomised_rounds_logged_equal_recorded_bitwise(round_id):
    """Shared rounds of random shape (2 to 16 streams, windows of 0 to 16
    rows, a stream of unrelated rows packed in front, chains or trees,
    d = 64 or 128,
    random kept rows, some streams keeping nothing): the logged window and
    its replay commit equal the recorded window and its copy commit, bit for
    bit, in y, tails and the committed slots."""
    rng = np.random.default_rng(3000 + round_id)
    S = int(rng.integers(2, 17))
    lengths = rng.integers(0, 17, size=S).tolist()
    tree = bool(round_id % 2)
    g = synth.Geometry(4, 12, 128, 128) if round_id % 4 < 2 else synth.Geometry(2, 8, 64, 64)
    pad = int(rng.integers(0, 5))
    c = Case(g, [pad] + lengths, seed=4000 + round_id, tree=tree, n_slots=S + 4)
    keep = np.full(c.S, -1, np.int32)
    for s in range(1, c.S):
        lo, hi = c.stream_rows(s)
        if hi > lo and rng.random() < 0.8:
            keep[s] = lo + int(rng.integers(0, hi - lo))
    d, w = c.dims_gpu(), c.dev_weights()
    slot, rp, kp = dev(c.slots), dev(c.row_ptr), dev(keep)
    par = dev(c.parent) if tree else None

    cache_r, rows_r = c.dev_cache(), c.dev_rows()
    rs, rt = c.dev_records()
    if tree:
        gdn.tree(d, w, cache_r, slot, rp, par, rows_r, rs, rt)
    else:
        gdn.window(d, w, cache_r, slot, rp, rows_r, rs, rt)
    gdn.commit(d, cache_r, slot, rp, kp, rs, rt)
    cache_l, rows_l = c.dev_cache(), c.dev_rows()
    la, lu, lk, lt = _logs(c)
    if tree:
        gdn.tree_log(d, w, cache_l, slot, rp, par, rows_l, la, lu, lk, lt)
        gdn.commit_replay_tree(d, cache_l, slot, rp, par, kp, la, lu, lk, lt)
    else:
        gdn.window_log(d, w, cache_l, slot, rp, rows_l, la, lu, lk, lt)
        gdn.commit_replay(d, cache_l, slot, rp, kp, la, lu, lk, lt)
    assert gdn.get_device_error() == 0

    assert np.array_equal(host_bits(rows_l["y"])[:c.R], host_bits(rows_r["y"])[:c.R])
    assert np.array_equal(host_bits(lt)[:c.R], host_bits(rt)[:c.R])
    assert np.array_equal(cache_l["state"].cpu().numpy().view(np.uint32), cache_r["state"].cpu().numpy().view(np.uint32))
    assert np.array_equal(host_bits(cache_l["tail"]), host_bits(cache_r["tail"]))


@pytest.mark.parametrize("g,n_round", [(synth.LIKE_2B, 5), (synth.LIKE_27B, 2)])
@pytest.mark.parametrize("mode", ["tree", "window_log", "tree_log"])
def test_sliced_trees_and_logged_windows_equal_unsliced_bitwise(mode, g, n_round):
    """Trees and logged windows of few streams split each head's state rows
    over a cluster (a lone 2B-like stream: 8 slices; a lone 27B-like one: 2),
    as recording windows do.  A stream alone equals the same stream in an
    unsliced round, bit for bit: y, tails, and the recorded states or the
    logs."""
    tree = mode != "window_log"
    c = Case(g, [16, 11] + [16] * (n_round - 2), seed=227, n_slots=n_round + 1, tree=tree)

    def run(case):
        d, w = case.dims_gpu(), case.dev_weights()
        cache, rows = case.dev_cache(), case.dev_rows()
        slot, rp = dev(case.slots), dev(case.row_ptr)
        if mode == "tree":
            rs, rt = case.dev_records()
            gdn.tree(d, w, cache, slot, rp, dev(case.parent), rows, rs, rt)
            extra = [rs.cpu().numpy().view(np.uint32)]
        else:
            la, lu, lk, rt = _logs(case)
            if mode == "tree_log":
                gdn.tree_log(d, w, cache, slot, rp, dev(case.parent), rows, la, lu, lk, rt)
            else:
                gdn.window_log(d, w, cache, slot, rp, rows, la, lu, lk, rt)
            extra = [x.cpu().numpy().view(np.uint32) for x in (la, lu, lk)]
        assert gdn.get_device_error() == 0
        return [host_bits(rows["y"]), host_bits(rt)] + extra

    full = run(c)
    for s in range(2):
        lo, hi = c.stream_rows(s)
        solo = Case(g, [hi - lo], seed=227, slots=[0], tree=tree)
        solo.w = c.w
        sl = c.slots[s]
        solo.cache = {"state": c.cache["state"][sl:sl + 1], "tail": c.cache["tail"][sl:sl + 1]}
        solo.rows = {k: v[lo:hi] for k, v in c.rows.items()}
        if tree:
            solo.parent = c.parent[lo:hi].copy()
        alone = run(solo)
        for i, (a, b) in enumerate(zip(alone, full)):
            assert np.array_equal(a[:hi - lo], b[lo:hi]), f"stream {s}: output {i} differs"
