"""A speculative-decoding loop against the oracle over several rounds:
each round verifies a window of draft rows per stream (gdn_window_pooled,
every row recorded into a fresh cache entry), commits a random accepted
length by index (gdn_commit_swap), then takes one decode step from the
committed state (gdn_step), all queued back to back on one stream.  The
oracle runs each stream's rows one by one from the state it kept itself
(rounded to fp32 where a committed state becomes the next call's input),
so the loop's y, recorded states, committed slots and step outputs are all
checked against the definition, round after round."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
import oracle
from gated_deltanet_speculative_gb300 import synth

from harness import check_state, check_y, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("g", [synth.Geometry(2, 6, 128, 128), synth.Geometry(2, 4, 64, 64)], ids=["d128", "d64"])
def test_verify_commit_step_rounds_against_oracle(g):
    S, W, ROUNDS = 4, 16, 3
    rng = np.random.default_rng(211)
    w = synth.layer_weights(g, 211)
    cache0 = synth.slot_cache(g, S, 211)
    od = oracle.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    d = gdn.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    dw = {"conv_w": dev_bf16(w["conv_w"]), "A_log": dev(w["A_log"]), "dt_bias": dev(w["dt_bias"]),
          "norm_w": dev_bf16(w["norm_w"])}
    n_pool = S + ROUNDS * S * W
    ps = torch.full((n_pool, g.n_v_heads, g.d_v, g.d_k), float("nan"), dtype=torch.float32, device="cuda")
    pt = torch.full((n_pool, 3, g.channels), float("nan"), dtype=torch.bfloat16, device="cuda")
    ps[:S].copy_(torch.from_numpy(cache0["state"]))
    pt[:S].copy_(torch.from_numpy(cache0["tail"].view(np.int16)).view(torch.bfloat16))
    pool = {"state": ps, "tail": pt}
    slot_t = dev(np.arange(S, dtype=np.int32))
    # the oracle's own kept state and tail per stream
    o_state = [cache0["state"][s].astype(np.float32) for s in range(S)]
    o_tail = [cache0["tail"][s].copy() for s in range(S)]
    for rnd in range(ROUNDS):
        lengths = rng.integers(1, W + 1, size=S)
        R = int(lengths.sum())
        rp = synth.row_ptr(lengths)
        rows = synth.row_inputs(g, R, 400 + rnd)
        acc = rng.integers(0, lengths + 1)
        keep = np.where(acc > 0, rp[:-1] + acc - 1, -1).astype(np.int32)
        rec = (S + rnd * S * W + rng.permutation(R)).astype(np.int32)
        step_rows = synth.row_inputs(g, S, 500 + rnd)
        dr = {k: dev_bf16(rows[k]) for k in ("mixed", "z", "a", "b")}
        dr["y"] = torch.full((R, g.n_v_heads, g.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        sr = {k: dev_bf16(step_rows[k]) for k in ("mixed", "z", "a", "b")}
        sr["y"] = torch.full((S, g.n_v_heads, g.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        gdn.window_pooled(d, dw, pool, slot_t, dev(rp), dr, dev(rec))
        gdn.commit_swap(d, pool, slot_t, dev(rp), dev(keep), dev(rec))
        gdn.step(d, dw, pool, slot_t, sr)
        torch.cuda.synchronize()
        assert gdn.get_device_error() == 0
        y = host_bits(dr["y"])
        sy = host_bits(sr["y"])
        pst, ptl = ps.cpu().numpy(), host_bits(pt)
        cur = slot_t.cpu().numpy()
        for s in range(S):
            lo, hi = int(rp[s]), int(rp[s + 1])
            ref = oracle.gdn_rows(od, w, o_state[s], o_tail[s], rows["mixed"][lo:hi], rows["z"][lo:hi],
                                  rows["a"][lo:hi], rows["b"][lo:hi], threads=8)
            check_y(y[lo:hi], ref["y"], what=f"round {rnd} stream {s} window y")
            if keep[s] >= 0:
                k = int(keep[s]) - lo
                assert cur[s] == rec[keep[s]]
                o_state[s] = ref["rec_state"][k].astype(np.float32)
                o_tail[s] = ref["rec_tail"][k].copy()
            # the step from the committed state, on the GPU and in the oracle
            st = oracle.gdn_rows(od, w, o_state[s], o_tail[s], step_rows["mixed"][s:s + 1], step_rows["z"][s:s + 1],
                                 step_rows["a"][s:s + 1], step_rows["b"][s:s + 1], threads=8)
            check_y(sy[s:s + 1], st["y"], what=f"round {rnd} stream {s} step y")
            check_state(pst[cur[s]], st["rec_state"][0], what=f"round {rnd} stream {s} state after the step")
            assert np.array_equal(ptl[cur[s]], st["rec_tail"][0]), f"round {rnd} stream {s} tail after the step"
            o_state[s] = st["rec_state"][0].astype(np.float32)
            o_tail[s] = st["rec_tail"][0].copy()


def test_prefill_then_verify_rounds_against_oracle():
    """The same loop started from prompts: gdn_prefill of four prompts
    (300, 65, 1 and 130 tokens, zero initial state) into the streams'
    entries, then two verify / commit / step rounds; the oracle runs each
    prompt token by token and continues from its own final state."""
    g = synth.Geometry(2, 6, 128, 128)
    S, W, ROUNDS = 4, 16, 2
    prompt = [300, 65, 1, 130]
    rng = np.random.default_rng(223)
    w = synth.layer_weights(g, 223)
    od = oracle.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    d = gdn.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    dw = {"conv_w": dev_bf16(w["conv_w"]), "A_log": dev(w["A_log"]), "dt_bias": dev(w["dt_bias"]),
          "norm_w": dev_bf16(w["norm_w"])}
    n_pool = S + ROUNDS * S * W
    ps = torch.full((n_pool, g.n_v_heads, g.d_v, g.d_k), float("nan"), dtype=torch.float32, device="cuda")
    pt = torch.full((n_pool, 3, g.channels), float("nan"), dtype=torch.bfloat16, device="cuda")
    ps[:S].zero_()
    pt[:S].zero_()
    pool = {"state": ps, "tail": pt}
    slot_t = dev(np.arange(S, dtype=np.int32))
    T = sum(prompt)
    cu = synth.row_ptr(prompt)
    prows = synth.row_inputs(g, T, 227)
    pr = {k: dev_bf16(prows[k]) for k in ("mixed", "z", "a", "b")}
    pr["y"] = torch.full((T, g.n_v_heads, g.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(gdn.prefill_workspace_size(d, S, T), dtype=torch.uint8, device="cuda")
    gdn.prefill(d, dw, pool, slot_t, dev(cu), pr, ws)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    py = host_bits(pr["y"])
    zs = np.zeros((g.n_v_heads, g.d_v, g.d_k), np.float32)
    zt = np.zeros((3, g.channels), np.uint16)
    o_state, o_tail = [], []
    for s in range(S):
        lo, hi = int(cu[s]), int(cu[s + 1])
        ref = oracle.gdn_rows(od, w, zs, zt, prows["mixed"][lo:hi], prows["z"][lo:hi], prows["a"][lo:hi],
                              prows["b"][lo:hi], record=False, final=True, threads=8)
        check_y(py[lo:hi], ref["y"], what=f"prompt {s} y")
        o_state.append(ref["final_state"].astype(np.float32))
        o_tail.append(ref["final_tail"].copy())
    for rnd in range(ROUNDS):
        lengths = rng.integers(1, W + 1, size=S)
        R = int(lengths.sum())
        rp = synth.row_ptr(lengths)
        rows = synth.row_inputs(g, R, 600 + rnd)
        acc = rng.integers(0, lengths + 1)
        keep = np.where(acc > 0, rp[:-1] + acc - 1, -1).astype(np.int32)
        rec = (S + rnd * S * W + rng.permutation(R)).astype(np.int32)
        step_rows = synth.row_inputs(g, S, 700 + rnd)
        dr = {k: dev_bf16(rows[k]) for k in ("mixed", "z", "a", "b")}
        dr["y"] = torch.full((R, g.n_v_heads, g.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        sr = {k: dev_bf16(step_rows[k]) for k in ("mixed", "z", "a", "b")}
        sr["y"] = torch.full((S, g.n_v_heads, g.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        gdn.window_pooled(d, dw, pool, slot_t, dev(rp), dr, dev(rec))
        gdn.commit_swap(d, pool, slot_t, dev(rp), dev(keep), dev(rec))
        gdn.step(d, dw, pool, slot_t, sr)
        torch.cuda.synchronize()
        assert gdn.get_device_error() == 0
        y, sy = host_bits(dr["y"]), host_bits(sr["y"])
        pst, ptl = ps.cpu().numpy(), host_bits(pt)
        cur = slot_t.cpu().numpy()
        for s in range(S):
            lo, hi = int(rp[s]), int(rp[s + 1])
            ref = oracle.gdn_rows(od, w, o_state[s], o_tail[s], rows["mixed"][lo:hi], rows["z"][lo:hi],
                                  rows["a"][lo:hi], rows["b"][lo:hi], threads=8)
            check_y(y[lo:hi], ref["y"], what=f"round {rnd} stream {s} window y")
            if keep[s] >= 0:
                k = int(keep[s]) - lo
                o_state[s] = ref["rec_state"][k].astype(np.float32)
                o_tail[s] = ref["rec_tail"][k].copy()
            st = oracle.gdn_rows(od, w, o_state[s], o_tail[s], step_rows["mixed"][s:s + 1], step_rows["z"][s:s + 1],
                                 step_rows["a"][s:s + 1], step_rows["b"][s:s + 1], threads=8)
            check_y(sy[s:s + 1], st["y"], what=f"round {rnd} stream {s} step y")
            check_state(pst[cur[s]], st["rec_state"][0], what=f"round {rnd} stream {s} state after the step")
            assert np.array_equal(ptl[cur[s]], st["rec_tail"][0]), f"round {rnd} stream {s} tail after the step"
            o_state[s] = st["rec_state"][0].astype(np.float32)
            o_tail[s] = st["rec_tail"][0].copy()
