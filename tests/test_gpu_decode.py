"""Decode steps with 2B-like heads (16 key heads, 16 value heads, d = 128):
24 independent layer instances (own weights, state and tail) stepped one
after another, one row per stream, at 1, 4, 8 and 16 streams; every layer's
output and updated state checked against the oracle."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
from gated_deltanet_speculative_gb300 import synth

from harness import Case, check_state, check_y, dev, host_bits

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
