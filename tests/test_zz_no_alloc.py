"""gdn_prefill_noalloc: the prefill for callers that cannot allocate device
memory (their host runtime owns the device's memory, or a cudaMalloc would
synchronise the whole device in the middle of a serving loop).  It keeps its
scratch in a fixed 64 MiB device array inside the library instead of a
caller workspace.

Checked through the C ABI against gdn_prefill with a caller workspace, on two
calls in a row (the second call starts from whatever the first left in the
shared array), and its refusal of sizes beyond the array.  This file is
collected last so that a run stopping at the first failure has already run
every other test."""
import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_speculative_gb300 as gdn
from gated_deltanet_speculative_gb300 import _binding as B
from gated_deltanet_speculative_gb300 import synth

from harness import Case, check_state, dev, host_bits

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def _fn():
    fn = gdn.load().gdn_prefill_noalloc
    fn.argtypes = [ctypes.POINTER(B.c_dims), ctypes.POINTER(B.c_weights), ctypes.POINTER(B.c_cache),
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(B.c_rows),
                   ctypes.c_int32, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _noalloc_call(c: Case, slots=None, cu=None):
    """gdn_prefill_noalloc through the C ABI; sequences are c's streams unless
    ``slots`` / ``cu`` (host int32 arrays) give others."""
    slots = c.slots if slots is None else slots
    cu = c.row_ptr if cu is None else cu
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    T = rows["mixed"].shape[0]
    cw, cc, cr = B._weights(d, w), B._cache(d, cache), B._rows(d, rows, T)
    slot_t, cu_t = dev(slots), dev(cu)
    rc = _fn()(ctypes.byref(d.c()), ctypes.byref(cw), ctypes.byref(cc), ctypes.c_void_p(slot_t.data_ptr()),
               ctypes.c_void_p(cu_t.data_ptr()), len(slots), T, ctypes.byref(cr), 64,
               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, f"gdn_prefill_noalloc returned {rc}"
    assert gdn.get_device_error() == 0
    return {"y": host_bits(rows["y"]), "state": cache["state"].cpu().numpy(), "tail": host_bits(cache["tail"])}


def _workspace_call(c: Case, slots=None, cu=None):
    slots = c.slots if slots is None else slots
    cu = c.row_ptr if cu is None else cu
    d = c.dims_gpu()
    w, cache, rows = c.dev_weights(), c.dev_cache(), c.dev_rows()
    ws = torch.empty(gdn.prefill_workspace_size(d, len(slots), rows["mixed"].shape[0]), dtype=torch.uint8,
                     device="cuda")
    gdn.prefill(d, w, cache, dev(slots), dev(cu), rows, ws)
    assert gdn.get_device_error() == 0
    return {"y": host_bits(rows["y"]), "state": cache["state"].cpu().numpy(), "tail": host_bits(cache["tail"])}


def _assert_close(out, ref, c: Case, slots=None, rows=slice(None)):
    slots = c.slots if slots is None else slots
    y, y_ref = (synth.bf16_bits_to_f32(v[rows]).astype(np.float64) for v in (out["y"], ref["y"]))
    assert np.all(np.isfinite(y))
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.maximum(np.abs(y), np.abs(y_ref)), 1e-30))) - 7)
    assert np.all(np.abs(y - y_ref) <= 2e-3 + ulp)
    for s, sl in enumerate(slots):
        sl = int(sl)
        check_state(out["state"][sl], ref["state"][sl].astype(np.float64), what=f"no-alloc state seq {s}")
        assert np.array_equal(out["tail"][sl], ref["tail"][sl])


def test_prefill_noalloc_matches_prefill_on_two_calls_in_a_row():
    """A call on another case (other seed, lengths and head count) fills the
    shared array first; then two calls in a row of the case under test must
    each equal gdn_prefill with a workspace of its own, so no call reads what
    an earlier one left behind."""
    other = Case(synth.Geometry(1, 3, 128, 128), [250, 7], seed=83, n_slots=3)
    c = Case(synth.Geometry(2, 4, 128, 128), [100, 64, 3, 0, 129], seed=71, n_slots=6)
    d = c.dims_gpu()
    assert gdn.prefill_workspace_size(d, c.S, c.R) <= SCRATCH_BYTES
    _assert_close(_noalloc_call(other), _workspace_call(other), other)
    ref = _workspace_call(c)
    for _ in range(2):
        _assert_close(_noalloc_call(c), ref, c)


def test_prefill_noalloc_and_prefill_leave_rows_outside_every_sequence_alone():
    """cu_seqlens starting at 5 and ending 7 rows before the packed buffers'
    end: both entry points leave y of those 12 rows as it was (NaN poison)
    and agree on every other row."""
    base = Case(synth.Geometry(2, 4, 128, 128), [5, 100, 64, 3, 0, 129, 7], seed=89, n_slots=8)
    slots, cu = base.slots[1:-1], base.row_ptr[1:-1]
    lo, hi = int(cu[0]), int(cu[-1])
    assert lo == 5 and hi == base.R - 7
    ref = _workspace_call(base, slots, cu)
    _noalloc_call(Case(synth.Geometry(2, 4, 128, 128), [300], seed=97))   # leaves other values in the array
    out = _noalloc_call(base, slots, cu)
    for y in (ref["y"], out["y"]):
        outside = synth.bf16_bits_to_f32(np.concatenate([y[:lo], y[hi:]]))
        assert np.all(np.isnan(outside)), "a row outside every sequence was written"
    _assert_close(out, ref, base, slots, rows=slice(lo, hi))


def test_prefill_noalloc_refuses_sizes_beyond_its_scratch():
    """One 4722-token prompt with 27B-like heads needs ~640 MB of scratch:
    refused with GDN_EWORKSPACE on the host, before any launch."""
    d = gdn.Dims(16, 48, 128, 128)
    assert gdn.prefill_workspace_size(d, 1, 4722) > SCRATCH_BYTES
    a = ctypes.c_void_p(0x10000)
    w = B.c_weights(a, a, a, a)
    cc = B.c_cache(a, a, 1)
    cr = B.c_rows(a, a, a, a, a)
    rc = _fn()(ctypes.byref(d.c()), ctypes.byref(w), ctypes.byref(cc), a, a, 1, 4722, ctypes.byref(cr), 64, None)
    assert rc == -5
