"""GPU parity of gdn_step / gdn_window / gdn_tree / gdn_commit against the
CPU oracle, element by element, through the C ABI; plus the bit-exact
structural invariants between the GPU kernels themselves (window rows equal
one-row steps, a tree node equals the chain along its path, a stream alone
equals the same stream inside a full round, any packing offset gives the
same bits)."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
from gated_deltanet_speculative_gb300 import synth

from harness import Case, check_state, check_y, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    gdn.load()
    gdn.get_device_error()   # start from a clean error word
    yield


def run_window(c: Case, tree=False, poison=True):
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows(poison)
    rs, rt = c.dev_records(poison)
    slot, rp = dev(c.slots), dev(c.row_ptr)
    if tree:
        gdn.tree(d, w, cache, slot, rp, dev(c.parent), rows, rs, rt)
    else:
        gdn.window(d, w, cache, slot, rp, rows, rs, rt)
    assert gdn.get_device_error() == 0
    return {"y": host_bits(rows["y"]), "rec_state": rs.cpu().numpy(), "rec_tail": host_bits(rt),
            "state": cache["state"].cpu().numpy(), "tail": host_bits(cache["tail"])}


def compare_with_oracle(c: Case, out, streams=None):
    for s in (range(c.S) if streams is None else streams):
        lo, hi = c.stream_rows(s)
        if hi == lo:
            continue
        ref = c.oracle_stream(s)
        check_y(out["y"][lo:hi], ref["y"], what=f"y stream {s}")
        check_state(out["rec_state"][lo:hi], ref["rec_state"], what=f"rec_state stream {s}")
        assert np.array_equal(out["rec_tail"][lo:hi], ref["rec_tail"]), f"rec_tail stream {s}"


# ---- parity against the oracle -------------------------------------------

def test_tiny_chain_window():
    """Tiny geometry: 1 stream, 2 key heads, 4 value heads, d = 32, window of 4, seed 0."""
    c = Case(synth.TINY, [4], seed=0)
    out = run_window(c)
    compare_with_oracle(c, out)
    # the committed slot is read-only in a window
    assert np.array_equal(out["state"], c.cache["state"]) and np.array_equal(out["tail"], c.cache["tail"])


@pytest.mark.parametrize("g", [synth.Geometry(2, 4, 32, 32), synth.Geometry(4, 8, 64, 64),
                               synth.Geometry(2, 16, 128, 128), synth.Geometry(3, 3, 64, 64)])
def test_window_geometries_ragged(g):
    c = Case(g, [5, 16, 1, 0, 9], seed=3, n_slots=7)
    compare_with_oracle(c, run_window(c))


def test_window_27b_ragged_streams():
    c = Case(synth.LIKE_27B, [16, 1, 7, 0, 13, 3], seed=5, n_slots=9)
    compare_with_oracle(c, run_window(c))


def test_window_full_round_16x16():
    """The shared verify round at full size: 16 streams x 16 rows, 27B-like heads."""
    c = Case(synth.LIKE_27B, [16] * 16, seed=2)
    compare_with_oracle(c, run_window(c))


def test_tree_full_round_16x16():
    c = Case(synth.LIKE_27B, [16] * 16, seed=3, tree=True)
    compare_with_oracle(c, run_window(c, tree=True))


def test_tree_geometries_ragged():
    c = Case(synth.Geometry(2, 4, 32, 32), [16, 3, 1, 11], seed=13, tree=True, n_slots=6)
    compare_with_oracle(c, run_window(c, tree=True))


def test_identity_gates_keep_state_bits():
    """A_log = -inf gives decay 1 and b = -inf gives beta 0: the recorded
    state equals the committed one bit for bit."""
    c = Case(synth.Geometry(2, 4, 64, 64), [5, 2], seed=17)
    c.w["A_log"][:] = -np.inf
    c.rows["b"][:] = synth.to_bf16_bits(np.full(c.rows["b"].shape, -np.inf, np.float32))
    out = run_window(c)
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        for r in range(lo, hi):
            assert np.array_equal(out["rec_state"][r], c.cache["state"][c.slots[s]])
    compare_with_oracle(c, out)


# ---- bit-exact invariants between GPU kernels ----------------------------

def steps_along(c: Case, s, rows_idx):
    """Run one-row gdn_step calls for stream s over the given packed rows, in order."""
    d = c.dims_gpu()
    w = c.dev_weights()
    sl = int(c.slots[s])
    cache = {"state": dev(c.cache["state"][sl:sl + 1]), "tail": dev_bf16(c.cache["tail"][sl:sl + 1])}
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys, states, tails = [], [], []
    for r in rows_idx:
        rows = {k: dev_bf16(c.rows[k][r:r + 1]) for k in ("mixed", "z", "a", "b")}
        rows["y"] = torch.full((1, c.g.n_v_heads, c.g.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        gdn.step(d, w, cache, slot, rows)
        ys.append(host_bits(rows["y"])[0])
        states.append(cache["state"][0].cpu().numpy())
        tails.append(host_bits(cache["tail"])[0])
    assert gdn.get_device_error() == 0
    return np.stack(ys), np.stack(states), np.stack(tails)


def test_window_rows_equal_one_row_steps_bitwise():
    c = Case(synth.LIKE_27B, [16, 5], seed=21)
    out = run_window(c)
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        y, st, tl = steps_along(c, s, range(lo, hi))
        assert np.array_equal(y, out["y"][lo:hi])
        assert np.array_equal(st.view(np.uint32), out["rec_state"][lo:hi].view(np.uint32))
        assert np.array_equal(tl, out["rec_tail"][lo:hi])


@pytest.mark.parametrize("g,n_streams", [(synth.LIKE_2B, 1), (synth.LIKE_2B, 4), (synth.LIKE_2B, 8),
                                          (synth.LIKE_2B, 16), (synth.TINY, 1), (synth.TINY, 2)])
def test_sliced_steps_equal_window_rows_bitwise(g, n_streams):
    """Steps of few streams split each head's state rows over up to 8 CTAs of
    a cluster (2B-like: 8, 4, 2, 1 slices at 1, 4, 8, 16 streams); a step must
    still equal the one-row window of the same inputs bit for bit."""
    c = Case(g, [1] * n_streams, seed=29 + n_streams, n_slots=n_streams + 2)
    out = run_window(c)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    gdn.step(d, w, cache, dev(c.slots), rows)
    assert gdn.get_device_error() == 0
    y, st, tl = host_bits(rows["y"]), cache["state"].cpu().numpy(), host_bits(cache["tail"])
    for s in range(c.S):
        sl = int(c.slots[s])
        assert np.array_equal(y[s], out["y"][s]), f"y stream {s}"
        assert np.array_equal(st[sl].view(np.uint32), out["rec_state"][s].view(np.uint32)), f"state stream {s}"
        assert np.array_equal(tl[sl], out["rec_tail"][s]), f"tail stream {s}"


def test_step_against_oracle_many_streams():
    c = Case(synth.LIKE_2B, [1] * 8, seed=23, n_slots=11)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    gdn.step(d, w, cache, dev(c.slots), rows)
    assert gdn.get_device_error() == 0
    y = host_bits(rows["y"])
    st = cache["state"].cpu().numpy()
    tl = host_bits(cache["tail"])
    touched = set(int(x) for x in c.slots)
    for s in range(c.S):
        ref = c.oracle_stream(s)
        sl = int(c.slots[s])
        check_y(y[s:s + 1], ref["y"], what=f"step y {s}")
        check_state(st[sl], ref["rec_state"][0], what=f"step state {s}")
        assert np.array_equal(tl[sl], ref["rec_tail"][0])
    for sl in range(c.n_slots):
        if sl not in touched:
            assert np.array_equal(st[sl].view(np.uint32), c.cache["state"][sl].view(np.uint32))
            assert np.array_equal(tl[sl], c.cache["tail"][sl])


def test_tree_node_equals_chain_along_path_bitwise():
    c = Case(synth.LIKE_27B, [16, 12], seed=29, tree=True)
    tree = run_window(c, tree=True)
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        par = c.parent[lo:hi]
        for node in range(hi - lo):
            path = []
            x = node
            while x >= 0:
                path.append(lo + x)
                x = par[x]
            path = path[::-1]
            chain = Case(c.g, [len(path)], seed=29, slots=[0])
            chain.w = c.w
            chain.cache = {"state": c.cache["state"][c.slots[s]:c.slots[s] + 1],
                           "tail": c.cache["tail"][c.slots[s]:c.slots[s] + 1]}
            chain.rows = {k: v[path] for k, v in c.rows.items()}
            ch = run_window(chain)
            assert np.array_equal(ch["y"][-1], tree["y"][lo + node])
            assert np.array_equal(ch["rec_state"][-1].view(np.uint32), tree["rec_state"][lo + node].view(np.uint32))
            assert np.array_equal(ch["rec_tail"][-1], tree["rec_tail"][lo + node])


def test_solo_stream_equals_stream_in_full_round_bitwise():
    """Every stream of the full 16 x 16 round (768 (stream, head) CTAs, 2.5
    waves) equals the same stream run alone (48 CTAs), bit for bit: y, every
    recorded state and every recorded tail."""
    c = Case(synth.LIKE_27B, [16] * 16, seed=31)
    full = run_window(c)
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        solo = Case(c.g, [16], seed=31, slots=[0])
        solo.w = c.w
        sl = c.slots[s]
        solo.cache = {"state": c.cache["state"][sl:sl + 1], "tail": c.cache["tail"][sl:sl + 1]}
        solo.rows = {k: v[lo:hi] for k, v in c.rows.items()}
        out = run_window(solo)
        assert np.array_equal(out["y"], full["y"][lo:hi]), f"y stream {s}"
        assert np.array_equal(out["rec_state"].view(np.uint32), full["rec_state"][lo:hi].view(np.uint32)), \
            f"rec_state stream {s}"
        assert np.array_equal(out["rec_tail"], full["rec_tail"][lo:hi]), f"rec_tail stream {s}"


@pytest.mark.parametrize("offset", [1, 3, 8, 13])
def test_packing_offset_does_not_change_bits(offset):
    """The same windows packed after `offset` unrelated rows give the same bits."""
    c = Case(synth.Geometry(4, 8, 128, 128), [7, 16, 2], seed=37)
    base = run_window(c)
    shifted = Case(c.g, [offset] + c.lengths, seed=37, slots=np.concatenate([[c.n_slots], c.slots]),
                   n_slots=c.n_slots + 1)
    shifted.w = c.w
    shifted.cache = {"state": np.concatenate([c.cache["state"], c.cache["state"][:1]]),
                     "tail": np.concatenate([c.cache["tail"], c.cache["tail"][:1]])}
    junk = synth.row_inputs(c.g, offset, 99)
    shifted.rows = {k: np.concatenate([junk[k], c.rows[k]]) for k in c.rows}
    out = run_window(shifted)
    assert np.array_equal(out["y"][offset:], base["y"])
    assert np.array_equal(out["rec_state"][offset:].view(np.uint32), base["rec_state"].view(np.uint32))
    assert np.array_equal(out["rec_tail"][offset:], base["rec_tail"])


# ---- commit ---------------------------------------------------------------

def test_commit_accepted_lengths_then_step():
    """Random accepted length 0..16 per stream: slots take the kept row's
    state and tail bit for bit (length 0 leaves them untouched); a step
    after the commit equals the window's next row."""
    c = Case(synth.LIKE_27B, [16] * 16, seed=41)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    rs, rt = c.dev_records()
    slot, rp = dev(c.slots), dev(c.row_ptr)
    gdn.window(d, w, cache, slot, rp, rows, rs, rt)
    rng = np.random.default_rng(41)
    acc = synth.accepted_lengths(c.S, 16, rng)
    acc[0], acc[1] = 0, 16
    keep = np.where(acc > 0, c.row_ptr[:-1] + acc - 1, -1).astype(np.int32)
    gdn.commit(d, cache, slot, rp, dev(keep), rs, rt)
    assert gdn.get_device_error() == 0
    st, tl = cache["state"].cpu().numpy(), host_bits(cache["tail"])
    rsn, rtn = rs.cpu().numpy(), host_bits(rt)
    for s in range(c.S):
        sl = c.slots[s]
        if keep[s] < 0:
            assert np.array_equal(st[sl].view(np.uint32), c.cache["state"][sl].view(np.uint32))
            assert np.array_equal(tl[sl], c.cache["tail"][sl])
        else:
            assert np.array_equal(st[sl].view(np.uint32), rsn[keep[s]].view(np.uint32))
            assert np.array_equal(tl[sl], rtn[keep[s]])
    # commit(n) then one step == row n of the window (n < 16)
    sel = [s for s in range(c.S) if 0 <= acc[s] < 16]
    nxt = np.array([c.row_ptr[s] + acc[s] for s in sel])
    step_rows = {k: dev_bf16(c.rows[k][nxt]) for k in ("mixed", "z", "a", "b")}
    step_rows["y"] = torch.empty((len(sel), c.g.n_v_heads, c.g.d_v), dtype=torch.bfloat16, device="cuda")
    gdn.step(d, w, cache, dev(c.slots[sel]), step_rows)
    assert gdn.get_device_error() == 0
    ys = host_bits(step_rows["y"])
    st2 = cache["state"].cpu().numpy()
    yw = host_bits(rows["y"])
    for i, s in enumerate(sel):
        assert np.array_equal(ys[i], yw[nxt[i]])
        assert np.array_equal(st2[c.slots[s]].view(np.uint32), rsn[nxt[i]].view(np.uint32))


# ---- device-side index checks ---------------------------------------------

def test_device_index_errors_skip_the_stream():
    """Out-of-range slot, over-long window and bad parent set the error word
    and leave that stream's outputs unwritten (the poison stays)."""
    c = Case(synth.Geometry(2, 4, 32, 32), [3, 2], seed=43, tree=True)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    rs, rt = c.dev_records()
    bad_slot = c.slots.copy()
    bad_slot[1] = 99
    gdn.window(d, w, cache, dev(bad_slot), dev(c.row_ptr), rows, rs, rt)
    assert gdn.get_device_error() & 1
    y = host_bits(rows["y"])
    assert np.all(np.isnan(synth.bf16_bits_to_f32(y[3:5])))
    assert np.all(np.isfinite(synth.bf16_bits_to_f32(y[0:3])))
    bad_parent = c.parent.copy()
    bad_parent[2] = 2   # own index: not an earlier row
    gdn.tree(d, w, cache, dev(c.slots), dev(c.row_ptr), dev(bad_parent), rows, rs, rt)
    assert gdn.get_device_error() & 4
    long_rp = np.array([0, 17, 17], np.int32)
    big = Case(c.g, [17], seed=43)
    rows2 = big.dev_rows()
    rs2, rt2 = big.dev_records()
    gdn.window(d, w, cache, dev(np.array([0, 1], np.int32)), dev(long_rp), rows2, rs2, rt2)
    assert gdn.get_device_error() & 2
    assert torch.isnan(rs2).all()
    keep = np.array([5, -1], np.int32)   # row 5 does not exist (R = 5 rows -> max index 4)
    gdn.commit(d, cache, dev(c.slots), dev(c.row_ptr), dev(keep), rs, rt)
    assert gdn.get_device_error() & 8
    assert np.array_equal(cache["state"].cpu().numpy(), c.cache["state"])


def test_commit_refuses_a_row_of_another_streams_window():
    """Each stream keeps only its own accepted rows: stream 0 naming row 3
    (stream 1's first row) and stream 1 naming row 0 (stream 0's) set the
    keep bit and leave both slots bit-unchanged, while a third stream's
    valid kept row is committed in the same call."""
    c = Case(synth.Geometry(2, 4, 64, 64), [3, 2, 4], seed=47, n_slots=5)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    rs, rt = c.dev_records()
    gdn.window(d, w, cache, dev(c.slots), dev(c.row_ptr), rows, rs, rt)
    assert gdn.get_device_error() == 0
    keep = np.array([3, 0, 7], np.int32)
    gdn.commit(d, cache, dev(c.slots), dev(c.row_ptr), dev(keep), rs, rt)
    assert gdn.get_device_error() & 8
    st, tl = cache["state"].cpu().numpy(), host_bits(cache["tail"])
    for s in (0, 1):
        sl = int(c.slots[s])
        assert np.array_equal(st[sl].view(np.uint32), c.cache["state"][sl].view(np.uint32)), f"slot of stream {s}"
        assert np.array_equal(tl[sl], c.cache["tail"][sl])
    sl = int(c.slots[2])
    assert np.array_equal(st[sl].view(np.uint32), rs[7].cpu().numpy().view(np.uint32))
    assert np.array_equal(tl[sl], host_bits(rt)[7])


@pytest.mark.parametrize("polls", [0, 1000])
def test_bounded_wait_timeout_sets_the_error_word_and_the_context_stays_usable(polls):
    """Failure detection without a hang or a fault: the kernels' bounded
    mbarrier wait, run on a phase that nothing completes, gives up after
    `polls` polls and sets the timeout bit; reading the word clears it, and
    the next call on the same context still matches the oracle."""
    gdn.debug_wait_timeout(polls)
    assert gdn.get_device_error() & 32
    assert gdn.get_device_error() == 0
    c = Case(synth.Geometry(2, 4, 32, 32), [4, 2], seed=101)
    compare_with_oracle(c, run_window(c))


@pytest.mark.parametrize("g", [synth.Geometry(2, 4, 64, 64), synth.Geometry(2, 6, 128, 128)])
@pytest.mark.parametrize("lengths", [[1], [3], [2, 1], [15]])
def test_calls_with_fewer_rows_than_a_staging_box(g, lengths):
    """The window's inputs are staged in boxes of up to 16 rows; a call whose
    packed buffer holds fewer rows (1 to 15) uses shorter boxes.  Chains and
    trees against the oracle."""
    c = Case(g, lengths, seed=103 + sum(lengths), n_slots=len(lengths) + 1)
    compare_with_oracle(c, run_window(c))
    t = Case(g, lengths, seed=107 + sum(lengths), n_slots=len(lengths) + 1, tree=True)
    compare_with_oracle(t, run_window(t, tree=True))


@pytest.mark.parametrize("tree", [False, True])
def test_many_streams_in_one_call(tree):
    """200 streams in one call (the ABI allows up to 65535; the bench's round
    has 16), windows of 0 to 16 rows: sampled streams against the oracle and,
    bit for bit, against the same stream run alone."""
    g = synth.Geometry(2, 4, 64, 64)
    rng = np.random.default_rng(211 + tree)
    lengths = rng.integers(0, 17, size=200).tolist()
    c = Case(g, lengths, seed=213 + tree, tree=tree, n_slots=203)
    out = run_window(c, tree=tree)
    sample = [s for s in (0, 1, 57, 123, 198, 199) if lengths[s] > 0]
    compare_with_oracle(c, out, streams=sample)
    for s in sample:
        lo, hi = c.stream_rows(s)
        solo = Case(g, [hi - lo], seed=213 + tree, slots=[0], tree=tree)
        solo.w = c.w
        sl = c.slots[s]
        solo.cache = {"state": c.cache["state"][sl:sl + 1], "tail": c.cache["tail"][sl:sl + 1]}
        solo.rows = {k: v[lo:hi] for k, v in c.rows.items()}
        if tree:
            solo.parent = c.parent[lo:hi].copy()
        alone = run_window(solo, tree=tree)
        assert np.array_equal(alone["y"], out["y"][lo:hi]), f"y stream {s}"
        assert np.array_equal(alone["rec_state"].view(np.uint32), out["rec_state"][lo:hi].view(np.uint32))
        assert np.array_equal(alone["rec_tail"], out["rec_tail"][lo:hi])


@pytest.mark.parametrize("g,n_round", [(synth.LIKE_2B, 5), (synth.Geometry(2, 6, 128, 128), 13),
                                       (synth.Geometry(2, 4, 64, 64), 20), (synth.LIKE_27B, 2)])
def test_sliced_windows_equal_unsliced_bitwise(g, n_round):
    """A window of few streams splits each head's state rows over a cluster of
    2 to 8 CTAs (a lone 2B-like stream: 8; a lone 27B-like stream: 2); a round
    of n_round streams has enough (stream, head) units to run unsliced.  Each
    stream alone equals the same stream in the round, bit for bit."""
    c = Case(g, [16, 9, 1] + [16] * (n_round - 3), seed=223, n_slots=n_round + 1)
    full = run_window(c)
    for s in range(3):
        lo, hi = c.stream_rows(s)
        solo = Case(g, [hi - lo], seed=223, slots=[0])
        solo.w = c.w
        sl = c.slots[s]
        solo.cache = {"state": c.cache["state"][sl:sl + 1], "tail": c.cache["tail"][sl:sl + 1]}
        solo.rows = {k: v[lo:hi] for k, v in c.rows.items()}
        out = run_window(solo)
        assert np.array_equal(out["y"], full["y"][lo:hi]), f"y stream {s}"
        assert np.array_equal(out["rec_state"].view(np.uint32), full["rec_state"][lo:hi].view(np.uint32))
        assert np.array_equal(out["rec_tail"], full["rec_tail"][lo:hi])
