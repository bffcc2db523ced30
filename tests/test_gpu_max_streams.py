"""The ABI's largest stream count, 65535, in one call (tiny heads, so the
whole cache fits easily): a one-row step of every stream, a one-row
pooled window of every stream and its index commit.  Sampled streams are
checked against the oracle; the grid's second dimension is at its limit."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
import oracle
from gated_deltanet_speculative_gb300 import synth

from harness import check_state, check_y, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

S_MAX = 65535
SAMPLE = (0, 1, 4097, 32767, 65533, 65534)


def test_step_window_and_commit_at_the_maximum_stream_count():
    g = synth.Geometry(2, 4, 32, 32)
    w = synth.layer_weights(g, 229)
    cache = synth.slot_cache(g, S_MAX, 229)
    rows = synth.row_inputs(g, S_MAX, 231)
    od = oracle.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    d = gdn.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    dw = {"conv_w": dev_bf16(w["conv_w"]), "A_log": dev(w["A_log"]), "dt_bias": dev(w["dt_bias"]),
          "norm_w": dev_bf16(w["norm_w"])}
    # slot s -> entry S_MAX - 1 - s, so that no index equals its stream's
    slots = (S_MAX - 1 - np.arange(S_MAX)).astype(np.int32)

    # one step of every stream
    dc = {"state": dev(cache["state"]), "tail": dev_bf16(cache["tail"])}
    dr = {k: dev_bf16(rows[k]) for k in ("mixed", "z", "a", "b")}
    dr["y"] = torch.full((S_MAX, g.n_v_heads, g.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdn.step(d, dw, dc, dev(slots), dr)
    assert gdn.get_device_error() == 0
    y = host_bits(dr["y"])
    st = dc["state"].cpu().numpy()
    for s in SAMPLE:
        sl = int(slots[s])
        ref = oracle.gdn_rows(od, w, cache["state"][sl], cache["tail"][sl], rows["mixed"][s:s + 1],
                              rows["z"][s:s + 1], rows["a"][s:s + 1], rows["b"][s:s + 1])
        check_y(y[s:s + 1], ref["y"], what=f"step y stream {s}")
        check_state(st[sl], ref["rec_state"][0], what=f"step state stream {s}")
    del dc, st

    # a one-row pooled window of every stream, then the index commit
    n_pool = 2 * S_MAX
    pool = {"state": torch.empty((n_pool, g.n_v_heads, g.d_v, g.d_k), dtype=torch.float32, device="cuda"),
            "tail": torch.empty((n_pool, 3, g.channels), dtype=torch.bfloat16, device="cuda")}
    pool["state"][:S_MAX].copy_(dev(cache["state"]))
    pool["tail"][:S_MAX].copy_(dev_bf16(cache["tail"]))
    rp = np.arange(S_MAX + 1, dtype=np.int32)
    rec = (S_MAX + np.arange(S_MAX)).astype(np.int32)
    keep = np.where(np.arange(S_MAX) % 3 == 0, -1, np.arange(S_MAX)).astype(np.int32)
    slot_t = dev(slots.copy())
    dr["y"].fill_(float("nan"))
    gdn.window_pooled(d, dw, pool, slot_t, dev(rp), dr, dev(rec))
    gdn.commit_swap(d, pool, slot_t, dev(rp), dev(keep), dev(rec))
    assert gdn.get_device_error() == 0
    y2 = host_bits(dr["y"])
    assert np.array_equal(y2, y), "a one-row window equals the step, bit for bit"
    cur = slot_t.cpu().numpy()
    assert np.array_equal(cur, np.where(keep >= 0, rec, slots))
    pst = pool["state"]
    for s in SAMPLE:
        sl = int(slots[s])
        ref = oracle.gdn_rows(od, w, cache["state"][sl], cache["tail"][sl], rows["mixed"][s:s + 1],
                              rows["z"][s:s + 1], rows["a"][s:s + 1], rows["b"][s:s + 1])
        check_state(pst[int(rec[s])].cpu().numpy(), ref["rec_state"][0], what=f"recorded state stream {s}")
