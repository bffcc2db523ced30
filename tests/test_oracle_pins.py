"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something it does not compute itself:
hand-worked values, closed forms, algebraic invariants of the gated delta
rule, special cases that reduce to numpy/scipy library routines, and brute
force with explicit matrices on tiny inputs.  Together they are chosen so
that a dropped term, a wrong sign, a wrong index or a transposed operand in
any part of the oracle fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
from gated_deltanet_speculative_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _unit(rng, n):
    x = rng.normal(size=n)
    return x / np.linalg.norm(x)


# ---- a5: the gated delta rule -------------------------------------------

def test_delta_rule_hand_worked_golden():
    with open(os.path.join(GOLDEN, "delta_rule_hand.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        S, o = oracle.delta_rule(np.array(c["S"], float), c["q"], c["k"], c["v"], c["a"], c["b"])
        np.testing.assert_allclose(S, np.array(c["S_new"], float), rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(o, np.array(c["o"], float), rtol=0, atol=1e-12, err_msg=c["name"])


@pytest.mark.parametrize("dv,dk", [(3, 5), (5, 3), (8, 8), (4, 32)])
def test_delta_rule_brute_force_matrices(dv, dk):
    """S' = a S (I - b k k^T) + b v k^T with the d_k x d_k matrix formed
    explicitly and multiplied with numpy; o = S' q."""
    rng = np.random.default_rng(dv * 100 + dk)
    for _ in range(5):
        S = rng.normal(size=(dv, dk))
        q, k, v = rng.normal(size=dk), rng.normal(size=dk), rng.normal(size=dv)
        a, b = rng.uniform(0, 1), rng.uniform(0, 1)
        M = np.eye(dk) - b * np.outer(k, k)
        S_ref = a * (S @ M) + b * np.outer(v, k)
        S_new, o = oracle.delta_rule(S, q, k, v, a, b)
        np.testing.assert_allclose(S_new, S_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(o, S_ref @ q, rtol=0, atol=1e-12)


def test_delta_rule_single_rank1_closed_form():
    """From S0 = 0 with a unit key: S1 = b v k^T and o = b (k.q) v."""
    rng = np.random.default_rng(7)
    dv, dk = 6, 10
    k = _unit(rng, dk)
    q, v = rng.normal(size=dk), rng.normal(size=dv)
    for a, b in [(0.3, 0.7), (1.0, 1.0), (0.9, 0.1)]:
        S1, o = oracle.delta_rule(np.zeros((dv, dk)), q, k, v, a, b)
        np.testing.assert_allclose(S1, b * np.outer(v, k), atol=1e-14)
        np.testing.assert_allclose(o, b * (k @ q) * v, atol=1e-14)


def test_delta_rule_write_invariant():
    """For a unit key, S' k = a (1 - b) S k + b v; at b = 1 the state maps
    k exactly to v (the delta rule's defining property)."""
    rng = np.random.default_rng(11)
    dv, dk = 7, 9
    for trial in range(6):
        S = rng.normal(size=(dv, dk))
        k = _unit(rng, dk)
        q, v = rng.normal(size=dk), rng.normal(size=dv)
        a = rng.uniform(0.05, 1.0)
        b = 1.0 if trial % 2 else rng.uniform(0, 1)
        S_new, _ = oracle.delta_rule(S, q, k, v, a, b)
        np.testing.assert_allclose(S_new @ k, a * (1 - b) * (S @ k) + b * v, atol=1e-12)
        if b == 1.0:
            np.testing.assert_allclose(S_new @ k, v, atol=1e-12)


def test_delta_rule_identity_case():
    """a = 1, b = 0 leaves the state unchanged (bit for bit) and o = S q."""
    rng = np.random.default_rng(3)
    S = rng.normal(size=(4, 6))
    q, k, v = rng.normal(size=6), rng.normal(size=6), rng.normal(size=4)
    S_new, o = oracle.delta_rule(S, q, k, v, 1.0, 0.0)
    assert np.array_equal(S_new, S)
    np.testing.assert_allclose(o, S @ q, atol=1e-14)


# ---- a3 / a4 / a7: norms and gates --------------------------------------

def test_gates_hand_worked_golden():
    with open(os.path.join(GOLDEN, "gates_hand.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        d, b = oracle.gates(c["A_log"], c["dt_bias"], c["a"], c["b"])
        assert d == pytest.approx(c["decay"], abs=1e-15)
        assert b == pytest.approx(c["beta"], abs=1e-15)


def test_gates_against_library_routines():
    """softplus = numpy.logaddexp(0, x); sigmoid = scipy.special.expit."""
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.normal(0, 3, 50), [-60.0, -25.0, -1e-3, 0.0, 1e-3, 25.0, 60.0]])
    for x in xs:
        A_log = rng.uniform(0, 2)
        dt = rng.normal(0, 0.1)
        d, b = oracle.gates(A_log, dt, x, x)
        d_ref = np.exp(-np.exp(A_log) * np.logaddexp(0.0, x + dt))
        assert d == pytest.approx(d_ref, rel=1e-13, abs=1e-300)
        assert b == pytest.approx(expit(x), rel=1e-13, abs=1e-300)
        assert 0.0 <= d <= 1.0 and 0.0 <= b <= 1.0


def test_gates_limits():
    """A_log = -inf gives decay 1 exactly; b = -inf gives beta 0 exactly."""
    d, b = oracle.gates(-np.inf, 0.3, 1.7, -np.inf)
    assert d == 1.0 and b == 0.0


def test_l2norm_unit_length_and_direction():
    rng = np.random.default_rng(9)
    for n in (4, 32, 128):
        x = rng.normal(size=n)
        y = oracle.l2norm(x, eps=1e-6, scale=0.5)
        ss = x @ x
        assert np.linalg.norm(y) == pytest.approx(0.5 * np.sqrt(ss / (ss + 1e-6)), rel=1e-13)
        np.testing.assert_allclose(y / np.linalg.norm(y), x / np.linalg.norm(x), atol=1e-14)
    assert np.all(oracle.l2norm(np.zeros(8)) == 0.0)


def test_gated_rmsnorm_special_cases():
    rng = np.random.default_rng(13)
    dv = 16
    z, w = rng.normal(size=dv), rng.normal(1, 0.1, size=dv)
    silu = z * expit(z)
    # constant o: the normalised value is c / sqrt(c^2 + eps), i.e. 1 to 1e-6
    y = oracle.gated_rmsnorm(np.full(dv, 2.0), z, w, eps=1e-6)
    np.testing.assert_allclose(y, w * silu * 2.0 / np.sqrt(4.0 + 1e-6), rtol=1e-13)
    # scale invariance at eps = 0, and sign follows o
    o = rng.normal(size=dv)
    y1 = oracle.gated_rmsnorm(o, z, w, eps=0.0)
    y2 = oracle.gated_rmsnorm(37.5 * o, z, w, eps=0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-13)
    # z = 0 silences the output (SiLU(0) = 0); normalised |o| has mean square 1
    assert np.all(oracle.gated_rmsnorm(o, np.zeros(dv), w, eps=0.0) == 0.0)
    y3 = oracle.gated_rmsnorm(o, np.full(dv, 50.0), np.ones(dv), eps=0.0)   # SiLU(50) = 50 to 1e-20
    assert np.mean((y3 / 50.0) ** 2) == pytest.approx(1.0, rel=1e-12)


# ---- a2 and the layer: conv taps, tail, head mapping ----------------------

def _layer_inputs(g, n, seed, tail_seed=None):
    w = synth.layer_weights(g, seed)
    cache = synth.slot_cache(g, 1, seed if tail_seed is None else tail_seed)
    rows = synth.row_inputs(g, n, seed)
    return w, cache["state"][0], cache["tail"][0], rows


def _dims(g, **kw):
    return oracle.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v, **kw)


def _conv_w_tap(g, j):
    w = np.zeros((g.channels, 4), np.float32)
    w[:, j] = 1.0
    return synth.to_bf16_bits(w)


def test_conv_current_tap_reduces_to_silu_and_library_norm():
    """conv weight e_3 makes the conv the identity on the current row, so
    q = L2(SiLU(x_q)) * q_scale, k = L2(SiLU(x_k)), v = SiLU(x_v), with SiLU
    from scipy.special.expit and the norm from numpy.linalg.norm."""
    g = synth.Geometry(2, 4, 8, 6)
    w, s0, t0, r = _layer_inputs(g, 3, 21)
    w["conv_w"] = _conv_w_tap(g, 3)
    dims = _dims(g, eps_l2=0.0)
    out = oracle.gdn_rows(dims, w, s0, t0, r["mixed"], r["z"], r["a"], r["b"], extras=True)
    x = synth.bf16_bits_to_f32(r["mixed"]).astype(np.float64)
    silu = x * expit(x)
    Hk, dk, dv = g.n_k_heads, g.d_k, g.d_v
    for t in range(3):
        for h in range(g.n_v_heads):
            kh = h // g.group
            qx = silu[t, kh * dk:(kh + 1) * dk]
            kx = silu[t, Hk * dk + kh * dk: Hk * dk + (kh + 1) * dk]
            vx = silu[t, 2 * Hk * dk + h * dv: 2 * Hk * dk + (h + 1) * dv]
            np.testing.assert_allclose(out["q"][t, h], qx / np.linalg.norm(qx) * dk ** -0.5, rtol=1e-12)
            np.testing.assert_allclose(out["k"][t, h], kx / np.linalg.norm(kx), rtol=1e-12)
            np.testing.assert_allclose(out["v"][t, h], vx, rtol=1e-12)


@pytest.mark.parametrize("tap", [0, 1, 2])
def test_conv_past_taps_follow_the_tail(tap):
    """conv weight e_j selects the input 3 - j rows back: for early rows that
    input is the kept tail (oldest first), later it is an earlier window row."""
    g = synth.Geometry(1, 1, 4, 4)
    n = 5
    w, s0, t0, r = _layer_inputs(g, n, 31)
    w["conv_w"] = _conv_w_tap(g, tap)
    out = oracle.gdn_rows(_dims(g), w, s0, t0, r["mixed"], r["z"], r["a"], r["b"], extras=True)
    history = np.concatenate([t0, r["mixed"]])     # [3 + n, CH], oldest first
    x = synth.bf16_bits_to_f32(history).astype(np.float64)
    back = 3 - tap
    for t in range(n):
        src = x[3 + t - back]
        vx = src[2 * g.d_k:]
        np.testing.assert_allclose(out["v"][t, 0], vx * expit(vx), rtol=1e-13)
    # recorded tail after row t: the three newest inputs, oldest first
    for t in range(n):
        assert np.array_equal(out["rec_tail"][t], history[t + 1:t + 4])


def test_grouped_head_mapping():
    """Value head h reads key head h // G: changing key head 1's k inputs
    changes exactly the value heads of group 1; changing v of head 2 changes
    head 2 only."""
    g = synth.Geometry(2, 6, 8, 8)
    w, s0, t0, r = _layer_inputs(g, 2, 41)
    dims = _dims(g)
    base = oracle.gdn_rows(dims, w, s0, t0, r["mixed"], r["z"], r["a"], r["b"])["y"]
    m = r["mixed"].copy()
    f = synth.bf16_bits_to_f32(m)
    k0 = g.n_k_heads * g.d_k + 1 * g.d_k
    f[:, k0:k0 + g.d_k] += 1.0
    m2 = synth.to_bf16_bits(f)
    y = oracle.gdn_rows(dims, w, s0, t0, m2, r["z"], r["a"], r["b"])["y"]
    changed = [h for h in range(g.n_v_heads) if not np.array_equal(y[:, h], base[:, h])]
    assert changed == [3, 4, 5]
    f = synth.bf16_bits_to_f32(r["mixed"]).copy()
    v2 = 2 * g.n_k_heads * g.d_k + 2 * g.d_v
    f[:, v2:v2 + g.d_v] += 1.0
    y = oracle.gdn_rows(dims, w, s0, t0, synth.to_bf16_bits(f), r["z"], r["a"], r["b"])["y"]
    changed = [h for h in range(g.n_v_heads) if not np.array_equal(y[:, h], base[:, h])]
    assert changed == [2]


def test_layer_recurrence_matches_explicit_matrix_chain():
    """The layer's state after each row equals an explicit-matrix recurrence
    (numpy) driven by the per-row q, k, v, a, b the oracle reports."""
    g = synth.Geometry(1, 2, 8, 4)
    w, s0, t0, r = _layer_inputs(g, 6, 51)
    out = oracle.gdn_rows(_dims(g), w, s0, t0, r["mixed"], r["z"], r["a"], r["b"], extras=True)
    for h in range(g.n_v_heads):
        S = s0[h].astype(np.float64)
        for t in range(6):
            k, q, v = out["k"][t, h], out["q"][t, h], out["v"][t, h]
            a, b = out["decay"][t, h], out["beta"][t, h]
            S = a * S @ (np.eye(g.d_k) - b * np.outer(k, k)) + b * np.outer(v, k)
            np.testing.assert_allclose(out["rec_state"][t, h], S, atol=1e-12)


def test_layer_output_is_gated_rmsnorm_of_its_own_head():
    """y[t, h] is assembled from head h's own o_t = S_t q_t, z[t, h] and the
    shared w_norm element by element: recomputed with numpy from the state
    and q the oracle reports, y = o / sqrt(mean(o^2) + eps) * w_norm * SiLU(z)
    with SiLU from scipy.special.expit.  Hk = 2, Hv = 6 puts value heads and
    key heads at different indices, and a random w_norm is not symmetric, so
    a z read at the key head's index or a reversed w_norm fails here."""
    g = synth.Geometry(2, 6, 8, 8)
    n = 6
    w, s0, t0, r = _layer_inputs(g, n, 57)
    dims = _dims(g)
    out = oracle.gdn_rows(dims, w, s0, t0, r["mixed"], r["z"], r["a"], r["b"], extras=True)
    z = oracle.bf16_to_f64(r["z"])
    wn = oracle.bf16_to_f64(w["norm_w"])
    assert not np.allclose(wn, wn[::-1])
    for t in range(n):
        for h in range(g.n_v_heads):
            o = out["rec_state"][t, h] @ out["q"][t, h]
            zz = z[t, h]
            y = o / np.sqrt(np.mean(o * o) + dims.eps_rms) * wn * (zz * expit(zz))
            np.testing.assert_allclose(out["y"][t, h], y, rtol=0, atol=1e-12 * max(1.0, np.abs(y).max()))


# ---- structural invariants of the verify path ---------------------------

def test_window_rows_equal_one_row_steps():
    g = synth.Geometry(2, 4, 16, 16)
    n = 7
    w, s0, t0, r = _layer_inputs(g, n, 61)
    dims = _dims(g)
    win = oracle.gdn_rows(dims, w, s0, t0, r["mixed"], r["z"], r["a"], r["b"])
    S, T = s0, t0
    for t in range(n):
        sl = slice(t, t + 1)
        st = oracle.gdn_rows(dims, w, S, T, r["mixed"][sl], r["z"][sl], r["a"][sl], r["b"][sl],
                             record=False, final=True)
        # the carried state passes through fp32 (the committed-state format)
        scale = np.abs(win["rec_state"][t]).max()
        np.testing.assert_allclose(st["y"][0], win["y"][t], rtol=0, atol=1e-5)
        np.testing.assert_allclose(st["final_state"], win["rec_state"][t], rtol=0, atol=1e-6 * scale)
        assert np.array_equal(st["final_tail"], win["rec_tail"][t])
        S, T = st["final_state"].astype(np.float32), st["final_tail"]


def test_tree_node_equals_chain_along_its_path():
    g = synth.Geometry(2, 4, 16, 16)
    n = 12
    rng = np.random.default_rng(71)
    parent = synth.random_tree(n, rng)
    w, s0, t0, r = _layer_inputs(g, n, 71)
    dims = _dims(g)
    tree = oracle.gdn_rows(dims, w, s0, t0, r["mixed"], r["z"], r["a"], r["b"], parent=parent)
    for node in range(n):
        path = []
        x = node
        while x >= 0:
            path.append(x)
            x = parent[x]
        path = path[::-1]
        ch = oracle.gdn_rows(dims, w, s0, t0, r["mixed"][path], r["z"][path], r["a"][path], r["b"][path])
        assert np.array_equal(ch["rec_state"][-1], tree["rec_state"][node])
        assert np.array_equal(ch["y"][-1], tree["y"][node])
        assert np.array_equal(ch["rec_tail"][-1], tree["rec_tail"][node])


def test_tree_of_roots_is_independent_steps():
    """parent = -1 everywhere: every node is one step from the committed slot."""
    g = synth.Geometry(1, 2, 8, 8)
    n = 4
    w, s0, t0, r = _layer_inputs(g, n, 81)
    dims = _dims(g)
    tree = oracle.gdn_rows(dims, w, s0, t0, r["mixed"], r["z"], r["a"], r["b"], parent=np.full(n, -1, np.int32))
    for t in range(n):
        sl = slice(t, t + 1)
        st = oracle.gdn_rows(dims, w, s0, t0, r["mixed"][sl], r["z"][sl], r["a"][sl], r["b"][sl])
        assert np.array_equal(st["rec_state"][0], tree["rec_state"][t])


def test_commit_then_step_equals_longer_chain():
    g = synth.Geometry(2, 4, 16, 16)
    n = 6
    w, s0, t0, r = _layer_inputs(g, n, 91)
    dims = _dims(g)
    win = oracle.gdn_rows(dims, w, s0, t0, r["mixed"], r["z"], r["a"], r["b"])
    keep = 3
    S, T = oracle.commit(win["rec_state"], win["rec_tail"], keep, s0, t0)
    sl = slice(keep + 1, keep + 2)
    st = oracle.gdn_rows(dims, w, S.astype(np.float32), T, r["mixed"][sl], r["z"][sl], r["a"][sl], r["b"][sl])
    scale = np.abs(win["rec_state"][keep + 1]).max()
    np.testing.assert_allclose(st["rec_state"][0], win["rec_state"][keep + 1], rtol=0, atol=1e-6 * scale)
    S0, T0 = oracle.commit(win["rec_state"], win["rec_tail"], -1, s0, t0)
    assert S0 is s0 and T0 is t0


# ---- a10: the chunk algebra -----------------------------------------------

@pytest.mark.parametrize("L,C", [(1, 1), (9, 1), (37, 4), (64, 64), (130, 64), (77, 16)])
def test_chunked_form_equals_sequential_recurrence(L, C):
    rng = np.random.default_rng(L * 7 + C)
    dv, dk = 6, 8
    S0 = rng.normal(0, 0.5, size=(dv, dk))
    Q = np.stack([_unit(rng, dk) for _ in range(L)]) * dk ** -0.5
    K = np.stack([_unit(rng, dk) for _ in range(L)])
    V = rng.normal(size=(L, dv))
    g = -rng.uniform(0.01, 3.0, size=L)
    beta = rng.uniform(0, 1, size=L)
    S = S0.copy()
    O_ref = np.empty((L, dv))
    for t in range(L):
        S, O_ref[t] = oracle.delta_rule(S, Q[t], K[t], V[t], np.exp(g[t]), beta[t])
    S_c, O_c = oracle.chunked_rule(S0, Q, K, V, g, beta, C)
    scale = max(1.0, np.abs(S).max())
    np.testing.assert_allclose(S_c, S, atol=1e-12 * scale)
    np.testing.assert_allclose(O_c, O_ref, atol=1e-12 * max(1.0, np.abs(O_ref).max()))
