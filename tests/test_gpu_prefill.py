"""GPU parity of the chunked prefill (gdn_prefill) against the oracle's
sequential recurrence: every token's y, and the slot's final state and conv
tail, for ragged packed prompts, resumed prompts, and the full prompt shapes
(one 4722-token prompt; 512/1024/2048/4096 in one pass)."""
import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
import oracle
from gated_deltanet_speculative_gb300 import synth

from harness import Case, check_state, check_y, dev, host_bits

pytestmark = pytest.mark.gpu


def run_prefill(c: Case):
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    ws = torch.empty(gdn.prefill_workspace_size(d, c.S, rows["mixed"].shape[0]), dtype=torch.uint8, device="cuda")
    ws.fill_(0xff)   # NaN poison: the kernels must not read what they did not write
    gdn.prefill(d, w, cache, dev(c.slots), dev(c.row_ptr), rows, ws)
    assert gdn.get_device_error() == 0
    return {"y": host_bits(rows["y"]), "state": cache["state"].cpu().numpy(), "tail": host_bits(cache["tail"])}


def compare(c: Case, out, threads=16):
    for s in range(c.S):
        lo, hi = c.stream_rows(s)
        sl = int(c.slots[s])
        if hi == lo:
            assert np.array_equal(out["state"][sl].view(np.uint32), c.cache["state"][sl].view(np.uint32))
            assert np.array_equal(out["tail"][sl], c.cache["tail"][sl])
            continue
        r = c.rows
        ref = oracle.gdn_rows(c.dims_oracle(), c.w, c.cache["state"][sl], c.cache["tail"][sl], r["mixed"][lo:hi],
                              r["z"][lo:hi], r["a"][lo:hi], r["b"][lo:hi], record=False, final=True, threads=threads)
        check_y(out["y"][lo:hi], ref["y"], what=f"prefill y seq {s}")
        check_state(out["state"][sl], ref["final_state"], what=f"prefill state seq {s}")
        assert np.array_equal(out["tail"][sl], ref["final_tail"]), f"prefill tail seq {s}"


@pytest.mark.parametrize("g", [synth.Geometry(2, 4, 32, 32), synth.Geometry(2, 4, 64, 64),
                               synth.Geometry(2, 6, 128, 128)])
def test_prefill_ragged_prompts_resume_from_kept_state(g):
    """Lengths around the chunk edges (1, 2, 3, 63, 64, 65, 130) and an empty
    prompt, each starting from a nonzero kept state and tail."""
    c = Case(g, [1, 2, 3, 0, 63, 64, 65, 130], seed=51, n_slots=10)
    compare(c, run_prefill(c))


@pytest.mark.parametrize("hk,hv", [(4, 4), (2, 4), (2, 8), (1, 8)])
def test_prefill_value_heads_per_key_head(hk, hv):
    """d = 128 with 1, 2, 4 and 8 value heads per key head: the prep writes a
    key head's Q once, into the block of its first value head, and every
    value head's scan reads it from there (the rest of the workspace is NaN
    poison)."""
    c = Case(synth.Geometry(hk, hv, 128, 128), [1, 64, 65, 200], seed=59, n_slots=5)
    compare(c, run_prefill(c))


def test_prefill_27b_heads_zero_state():
    c = Case(synth.LIKE_27B, [200, 70, 1], seed=53, zero_state=True)
    compare(c, run_prefill(c))


def test_prefill_single_4722_token_prompt():
    """One 4722-token prompt, 27B-like heads, chunk 64, zero initial state."""
    c = Case(synth.LIKE_27B, [4722], seed=4, zero_state=True)
    compare(c, run_prefill(c))


def test_prefill_shared_pass_of_four_prompts():
    """512 / 1024 / 2048 / 4096 tokens packed into one pass."""
    c = Case(synth.LIKE_27B, [512, 1024, 2048, 4096], seed=4, zero_state=True)
    compare(c, run_prefill(c))


def test_prefill_split_at_chunk_and_off_chunk_points_matches_whole():
    """A prompt prefilled in two passes (split at 64, then at 100) ends in the
    same slot state as one pass over the whole prompt, to tolerance."""
    g = synth.Geometry(2, 4, 128, 128)
    whole = Case(g, [300], seed=57)
    out_whole = run_prefill(whole)
    for cut in (64, 100):
        d = whole.dims_gpu()
        w = whole.dev_weights()
        cache = whole.dev_cache()
        slot = dev(whole.slots)
        for lo, hi in ((0, cut), (cut, 300)):
            rows = {k: torch.from_numpy(np.ascontiguousarray(v[lo:hi]).view(np.int16)).view(torch.bfloat16).cuda()
                    for k, v in whole.rows.items()}
            rows["y"] = torch.empty((hi - lo, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device="cuda")
            ws = torch.empty(gdn.prefill_workspace_size(d, 1, hi - lo), dtype=torch.uint8, device="cuda")
            gdn.prefill(d, w, cache, slot, dev(np.array([0, hi - lo], np.int32)), rows, ws)
        sl = int(whole.slots[0])
        check_state(cache["state"].cpu().numpy()[sl], out_whole["state"][sl].astype(np.float64),
                    what=f"resume at {cut}")
        assert np.array_equal(host_bits(cache["tail"])[sl], out_whole["tail"][sl])


def test_prefill_matches_gpu_steps():
    """Prefill of L tokens equals L one-row gdn_step calls, to tolerance."""
    g = synth.Geometry(2, 4, 64, 64)
    c = Case(g, [77], seed=59)
    out = run_prefill(c)
    d = c.dims_gpu()
    w = c.dev_weights()
    sl = int(c.slots[0])
    cache = {"state": dev(c.cache["state"][sl:sl + 1]), "tail": torch.from_numpy(
        c.cache["tail"][sl:sl + 1].view(np.int16)).view(torch.bfloat16).cuda()}
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = []
    for t in range(77):
        rows = {k: torch.from_numpy(np.ascontiguousarray(v[t:t + 1]).view(np.int16)).view(torch.bfloat16).cuda()
                for k, v in c.rows.items()}
        rows["y"] = torch.empty((1, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device="cuda")
        gdn.step(d, w, cache, slot, rows)
        ys.append(synth.bf16_bits_to_f32(host_bits(rows["y"]))[0])
    # both sides are rounded to bf16: allow 2e-3 plus one ulp of the larger
    y_steps = np.stack(ys).astype(np.float64)
    y_pre = synth.bf16_bits_to_f32(out["y"][:77]).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.maximum(np.abs(y_pre), np.abs(y_steps)), 1e-30))) - 7)
    assert np.all(np.abs(y_pre - y_steps) <= 2e-3 + ulp)
    check_state(cache["state"].cpu().numpy()[0], out["state"][sl].astype(np.float64), what="prefill vs steps")


def test_prefill_bad_seqlens_sets_error_and_skips():
    g = synth.Geometry(2, 4, 32, 32)
    c = Case(g, [10, 5], seed=61)
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    ws = torch.empty(gdn.prefill_workspace_size(d, 2, 15), dtype=torch.uint8, device="cuda")
    gdn.prefill(d, w, cache, dev(c.slots), dev(np.array([0, 10, 99], np.int32)), rows, ws)
    assert gdn.get_device_error() & 16
    with pytest.raises(gdn.GdnError):
        gdn.prefill(d, w, cache, dev(c.slots), dev(c.row_ptr), rows, ws[:100])


def test_pipelined_prefill_equals_single_stream_bitwise():
    """For d = 128 gdn_prefill takes the chunks in groups: the scan of a
    group runs on a side stream while later groups' prep runs, and the state
    passes from one scan launch to the next through the slot (fp32, exact).
    gdn_prefill_noalloc runs the same kernels as one prep, one scan and one
    norm on the caller's stream; the two must agree bit for bit, with
    sequences that straddle group boundaries and a one-token sequence, and
    the caller's stream must see the finished result."""
    g = synth.Geometry(4, 12, 128, 128)
    c = Case(g, [700, 130, 64, 1], seed=67, n_slots=6)
    d = c.dims_gpu()
    T = c.R
    assert gdn.prefill_workspace_size(d, c.S, T) <= gdn.PREFILL_NOALLOC_SCRATCH_BYTES

    side = torch.cuda.Stream()   # a caller stream other than the default one
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    ws = torch.empty(gdn.prefill_workspace_size(d, c.S, T), dtype=torch.uint8, device="cuda")
    slot, cu = dev(c.slots), dev(c.row_ptr)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        gdn.prefill(d, w, cache, slot, cu, rows, ws, stream=side)
        out = {"y": rows["y"].clone(), "state": cache["state"].clone(), "tail": cache["tail"].clone()}
    side.synchronize()
    assert gdn.get_device_error() == 0

    w2, cache2, rows2 = c.dev_weights(), c.dev_cache(), c.dev_rows()
    gdn.prefill_noalloc(d, w2, cache2, slot, cu, rows2)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    assert np.array_equal(host_bits(out["y"]), host_bits(rows2["y"]))
    assert np.array_equal(out["state"].cpu().numpy().view(np.uint32), cache2["state"].cpu().numpy().view(np.uint32))
    assert np.array_equal(host_bits(out["tail"]), host_bits(cache2["tail"]))
    # and against the oracle
    compare(c, {"y": host_bits(out["y"]), "state": out["state"].cpu().numpy(), "tail": host_bits(out["tail"])})


def test_pipelined_prefill_captured_in_a_graph_equals_eager_bitwise():
    """The d = 128 prefill forks onto the library's side streams and joins
    back with events; captured in a CUDA graph on a caller stream, replays
    must equal eager calls bit for bit (new inputs copied in between)."""
    g = synth.Geometry(4, 12, 128, 128)
    c = Case(g, [700, 130, 64, 1], seed=73, n_slots=6)
    d = c.dims_gpu()
    T = c.R
    w = c.dev_weights()
    slot, cu = dev(c.slots), dev(c.row_ptr)
    base = c.dev_cache()
    cache = {"state": base["state"].clone(), "tail": base["tail"].clone()}
    rows = c.dev_rows(poison=False)
    ws = torch.empty(gdn.prefill_workspace_size(d, c.S, T), dtype=torch.uint8, device="cuda")

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        gdn.prefill(d, w, cache, slot, cu, rows, ws, stream=side)   # warm-up (makes the side streams)
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            gdn.prefill(d, w, cache, slot, cu, rows, ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    rng = np.random.default_rng(74)
    for trial in range(2):
        mixed = synth.to_bf16_bits(rng.standard_normal(c.rows["mixed"].shape).astype(np.float32))
        rows["mixed"].copy_(torch.from_numpy(mixed.view(np.int16)).view(torch.bfloat16))
        cache["state"].copy_(base["state"])
        cache["tail"].copy_(base["tail"])
        rows["y"].zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.get_device_error() == 0
        got = (host_bits(rows["y"]), cache["state"].cpu().numpy().view(np.uint32), host_bits(cache["tail"]))
        e_cache = {"state": base["state"].clone(), "tail": base["tail"].clone()}
        e_rows = dict(rows, y=torch.zeros_like(rows["y"]))
        gdn.prefill(d, w, e_cache, slot, cu, e_rows, ws)
        torch.cuda.synchronize()
        assert np.array_equal(got[0], host_bits(e_rows["y"]))
        assert np.array_equal(got[1], e_cache["state"].cpu().numpy().view(np.uint32))
        assert np.array_equal(got[2], host_bits(e_cache["tail"]))


def test_single_stream_prefill_with_several_items_per_cta_equals_pipelined_bitwise():
    """On the single-stream plan (gdn_prefill_noalloc) the prep grid is at
    most one CTA per SM, so with more (key head, chunk) items than SMs a CTA
    takes several items in turn, carrying its TMEM and barrier phases across
    them: 5000 tokens with 2 key heads are 158 items.  gdn_prefill must give
    the same bits.  (With one sequence gdn_prefill cuts groups in whole prep
    rounds, and with 2 key heads the first group already holds all 79
    chunks; the persistent preps of its later groups are covered by the
    4722-token test against the oracle.)"""
    g = synth.Geometry(2, 4, 128, 128)
    c = Case(g, [5000], seed=79, zero_state=True)
    d = c.dims_gpu()
    T = c.R
    assert gdn.prefill_workspace_size(d, 1, T) <= gdn.PREFILL_NOALLOC_SCRATCH_BYTES
    out = run_prefill(c)

    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    gdn.prefill_noalloc(d, w, cache, dev(c.slots), dev(c.row_ptr), rows)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    assert np.array_equal(out["y"], host_bits(rows["y"]))
    assert np.array_equal(out["state"].view(np.uint32), cache["state"].cpu().numpy().view(np.uint32))
    assert np.array_equal(out["tail"], host_bits(cache["tail"]))


def test_prefill_long_prompt_many_chunk_groups():
    """A 16,384-token prompt with 27B-like heads: 256 chunks, which the
    pipelined plan runs as 20 chunk groups (state handed from group to group
    through the slot), against the sequential oracle."""
    c = Case(synth.LIKE_27B, [16384], seed=233, zero_state=True)
    compare(c, run_prefill(c), threads=16)
