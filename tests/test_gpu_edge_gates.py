"""GPU parity at the edges of the gates, on every entry point that runs the
recurrence (gdn_step, gdn_window, gdn_tree, gdn_prefill), against the oracle.

The gates are a_t = exp(-exp(A_log) softplus(a + dt_bias)) and
b_t = sigmoid(b).  Random N(0, 1) inputs keep both well inside (0, 1); these
cases push them to their ends:

* identity: A_log = -inf and b = -inf give a_t = 1 and b_t = 0 exactly, so
  the state must come out bit for bit as it went in (the layer's
  "a = 1, b = 0 leaves the state unchanged" invariant) and o = S q;
* strong decay: A_log = 4, a = 8 (+ noise) give log a_t near -440 a row, so
  a_t is 0 in fp32 and the chunk form's gamma_t = exp(G_t) underflows from
  the first row of a chunk on, while Gamma_ts = exp(G_t - G_s) is 1 on the
  diagonal and 0 below it;
* graded decay: log a_t spread over about [-60, -1], so gamma_t underflows
  part-way through a chunk and Gamma_ts is a mix of tiny and ordinary
  values;
* beta one: b = +inf gives b_t = 1 exactly, the delta rule's exact-write
  case S_t k_t = v_t for unit k_t.

Prompts end with a chunk of one row (65 and 129 tokens) beside whole and
ragged chunks.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
from gated_deltanet_speculative_gb300 import synth

from harness import Case, check_state, check_y, dev, host_bits
from test_gpu_prefill import compare as compare_prefill
from test_gpu_prefill import run_prefill
from test_gpu_rows import compare_with_oracle, run_window

pytestmark = pytest.mark.gpu

KINDS = ["identity", "strong_decay", "graded_decay", "beta_one"]


def set_gates(c: Case, kind: str, seed: int = 0):
    rng = np.random.default_rng(seed)
    a_shape = c.rows["a"].shape
    if kind == "identity":
        c.w["A_log"][:] = -np.inf
        c.rows["b"][:] = synth.to_bf16_bits(np.full(c.rows["b"].shape, -np.inf, np.float32))
    elif kind == "strong_decay":
        c.w["A_log"][:] = 4.0
        c.rows["a"][:] = synth.to_bf16_bits((8.0 + 0.25 * rng.normal(size=a_shape)).astype(np.float32))
    elif kind == "graded_decay":
        c.w["A_log"][:] = rng.uniform(0.0, 3.0, size=c.w["A_log"].shape).astype(np.float32)
        c.rows["a"][:] = synth.to_bf16_bits(rng.uniform(-1.0, 3.0, size=a_shape).astype(np.float32))
    elif kind == "beta_one":
        c.rows["b"][:] = synth.to_bf16_bits(np.full(c.rows["b"].shape, np.inf, np.float32))
    else:
        raise ValueError(kind)


@pytest.mark.parametrize("kind", KINDS)
def test_step_edge_gates(kind):
    c = Case(synth.LIKE_2B, [1] * 4, seed=131, n_slots=6)
    set_gates(c, kind, 1)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    gdn.step(d, w, cache, dev(c.slots), rows)
    assert gdn.get_device_error() == 0
    y, st, tl = host_bits(rows["y"]), cache["state"].cpu().numpy(), host_bits(cache["tail"])
    for s in range(c.S):
        sl = int(c.slots[s])
        ref = c.oracle_stream(s)
        check_y(y[s:s + 1], ref["y"], what=f"{kind} step y {s}")
        check_state(st[sl], ref["rec_state"][0], what=f"{kind} step state {s}")
        assert np.array_equal(tl[sl], ref["rec_tail"][0])
        if kind == "identity":
            assert np.array_equal(st[sl].view(np.uint32), c.cache["state"][sl].view(np.uint32))


@pytest.mark.parametrize("tree", [False, True], ids=["window", "tree"])
@pytest.mark.parametrize("kind", KINDS)
def test_window_and_tree_edge_gates(kind, tree):
    c = Case(synth.Geometry(2, 6, 128, 128), [16, 7, 1], seed=137, n_slots=4, tree=tree)
    set_gates(c, kind, 2)
    out = run_window(c, tree=tree)
    compare_with_oracle(c, out)
    if kind == "identity":
        for s in range(c.S):
            lo, hi = c.stream_rows(s)
            ref_bits = c.cache["state"][c.slots[s]].view(np.uint32)
            for r in range(lo, hi):
                assert np.array_equal(out["rec_state"][r].view(np.uint32), ref_bits), f"row {r}"


@pytest.mark.parametrize("g", [synth.Geometry(2, 4, 64, 64), synth.Geometry(2, 6, 128, 128)],
                         ids=["d64", "d128"])
@pytest.mark.parametrize("kind", KINDS)
def test_prefill_edge_gates(kind, g):
    """Prompts of 129, 64, 1 and 200 tokens (the first ends with a one-row
    chunk) from a nonzero kept state, y and the final state and tail
    against the oracle's sequential recurrence; with identity gates the
    final state is the kept one bit for bit."""
    c = Case(g, [129, 64, 1, 200], seed=139, n_slots=5)
    set_gates(c, kind, 3)
    out = run_prefill(c)
    compare_prefill(c, out)
    if kind == "identity":
        for s in range(c.S):
            sl = int(c.slots[s])
            assert np.array_equal(out["state"][sl].view(np.uint32), c.cache["state"][sl].view(np.uint32))


def test_prefill_27b_prompt_ending_in_a_one_row_chunk():
    """27B-like heads, one prompt of 3 x 64 + 1 tokens from a zero state."""
    c = Case(synth.LIKE_27B, [193], seed=149, zero_state=True)
    compare_prefill(c, run_prefill(c))
