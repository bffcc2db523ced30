"""The C ABI without a GPU: the library builds, loads, exports every entry
point include/gdn.h declares, and refuses bad arguments on the host before
touching CUDA (no call here reaches a kernel launch)."""
import ctypes
import os
import re

import pytest

import gated_deltanet_speculative_gb300 as gdn
from gated_deltanet_speculative_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    lib = gdn.load()
    names = declared_functions()
    assert {"gdn_step", "gdn_window", "gdn_tree", "gdn_commit", "gdn_status_string",
            "gdn_get_device_error"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"libgdn.so does not export {n}"


def test_binding_declares_every_entry_point():
    """The ctypes binding gives every declared entry point its argument
    types, and the package exposes a wrapper of the same name (without the
    gdn_ prefix) for each compute call."""
    names = declared_functions()
    assert names == set(B._SIGS), f"declared but not bound: {names - set(B._SIGS)}"
    for n in names - {"gdn_status_string", "gdn_get_device_error"}:
        assert callable(getattr(gdn, n[len("gdn_"):], None)), f"no wrapper for {n}"


def test_status_strings():
    lib = gdn.load()
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.gdn_status_string(code)
    assert lib.gdn_status_string(12345) == b"unknown status"


# fake device addresses: validation rejects every call below before any CUDA use
A16 = 0x10000
MIS = 0x10002


def _args(dims=None, **over):
    d = dims or B.c_dims(16, 48, 128, 128, 4, 128 ** -0.5, 1e-6, 1e-6)
    w = B.c_weights(A16, A16, A16, A16)
    c = B.c_cache(A16, A16, 4)
    r = B.c_rows(A16, A16, A16, A16, A16)
    for k, v in over.items():
        for s in (d, w, c, r):
            if hasattr(s, k):
                setattr(s, k, v)
    return d, w, c, r


def _window(d, w, c, r, n_streams=2, n_rows=4, slot=A16, row_ptr=A16, rec_state=A16, rec_tail=A16):
    lib = gdn.load()
    return lib.gdn_window(ctypes.byref(d), ctypes.byref(w), ctypes.byref(c), slot, row_ptr, n_streams, n_rows,
                          ctypes.byref(r), rec_state, rec_tail, None)


@pytest.mark.parametrize("field,value", [("n_k_heads", 0), ("n_v_heads", 47), ("d_k", 96), ("d_v", 64),
                                         ("conv_width", 3), ("n_v_heads", 16 * 9)])
def test_bad_geometry_is_einval(field, value):
    d, w, c, r = _args()
    setattr(d, field, value)
    assert _window(d, w, c, r) == -1


def test_bad_sizes_are_einval():
    d, w, c, r = _args()
    assert _window(d, w, c, r, n_streams=0) == -1
    assert _window(d, w, c, r, n_rows=0) == -1
    assert _window(d, w, c, r, n_streams=70000) == -1
    d2, w2, c2, r2 = _args(n_slots=0)
    assert _window(d2, w2, c2, r2) == -1
    d3, w3, c3, r3 = _args(eps_rms=float("nan"))
    assert _window(d3, w3, c3, r3) == -1


def test_null_pointers_are_enull():
    lib = gdn.load()
    d, w, c, r = _args()
    assert lib.gdn_window(None, ctypes.byref(w), ctypes.byref(c), A16, A16, 2, 4, ctypes.byref(r), A16, A16,
                          None) == -2
    assert _window(*_args(mixed=None)) == -2
    assert _window(*_args(A_log=None)) == -2
    assert _window(*_args(state=None)) == -2
    assert _window(d, w, c, r, slot=None) == -2
    assert _window(d, w, c, r, rec_state=None) == -2
    assert lib.gdn_tree(ctypes.byref(d), ctypes.byref(w), ctypes.byref(c), A16, A16, None, 2, 4, ctypes.byref(r),
                        A16, A16, None) == -2
    assert lib.gdn_commit(ctypes.byref(d), ctypes.byref(c), A16, A16, None, 2, 4, A16, A16, None) == -2
    assert lib.gdn_commit(ctypes.byref(d), ctypes.byref(c), A16, None, A16, 2, 4, A16, A16, None) == -2
    assert lib.gdn_step(ctypes.byref(d), ctypes.byref(w), ctypes.byref(c), None, 2, ctypes.byref(r), None) == -2
    assert lib.gdn_get_device_error(None, None) == -2


def test_misaligned_pointers_are_ealign():
    lib = gdn.load()
    assert _window(*_args(mixed=MIS)) == -3
    assert _window(*_args(state=MIS)) == -3
    assert _window(*_args(conv_w=MIS)) == -3
    d, w, c, r = _args()
    assert _window(d, w, c, r, rec_state=MIS) == -3
    assert _window(d, w, c, r, slot=A16 + 2) == -3
    assert lib.gdn_commit(ctypes.byref(d), ctypes.byref(c), A16, A16, A16, 2, 4, MIS, A16, None) == -3
    assert lib.gdn_commit(ctypes.byref(d), ctypes.byref(c), A16, A16 + 2, A16, 2, 4, A16, A16, None) == -3


def test_binding_checks_shapes_before_calling():
    torch = pytest.importorskip("torch")
    d = gdn.Dims(2, 4, 32, 32)
    bad = {"conv_w": torch.zeros(3, 4, dtype=torch.bfloat16)}
    with pytest.raises((TypeError, ValueError)):
        B._weights(d, {**bad, "A_log": torch.zeros(4), "dt_bias": torch.zeros(4),
                       "norm_w": torch.zeros(32, dtype=torch.bfloat16)})


def test_logged_tree_entry_points_validate_on_the_host():
    """gdn_tree_log and gdn_commit_replay_tree need the parent array (NULL is
    GDN_ENULL, a misaligned one GDN_EALIGN) and the logs, like their chain
    counterparts."""
    lib = gdn.load()
    d, w, c, r = _args()

    def tree_log(parent=A16, log_u=A16):
        return lib.gdn_tree_log(ctypes.byref(d), ctypes.byref(w), ctypes.byref(c), A16, A16, parent, 2, 4,
                                ctypes.byref(r), A16, log_u, A16, A16, None)

    def replay_tree(parent=A16, keep=A16, n_rows=4):
        return lib.gdn_commit_replay_tree(ctypes.byref(d), ctypes.byref(c), A16, A16, parent, keep, 2, n_rows,
                                          A16, A16, A16, A16, None)

    assert tree_log(parent=None) == -2
    assert tree_log(log_u=None) == -2
    assert tree_log(parent=A16 + 2) == -3
    assert tree_log(log_u=A16 + 4) == -3
    assert replay_tree(parent=None) == -2
    assert replay_tree(keep=None) == -2
    assert replay_tree(parent=A16 + 2) == -3
    assert replay_tree(n_rows=0) == -1


def test_debug_wait_timeout_bounds_its_polls():
    """The timeout hook refuses a poll count above the kernels' own limit
    (2^22) before launching anything."""
    lib = gdn.load()
    assert lib.gdn_debug_wait_timeout((1 << 22) + 1, None) == -1


def test_pooled_entry_points_refuse_bad_arguments_on_the_host():
    """gdn_window_pooled / gdn_tree_pooled / gdn_commit_swap: a missing
    rec_slot, row_ptr or keep_row is GDN_ENULL, a misaligned index array
    GDN_EALIGN, a non-positive size GDN_EINVAL, all before any CUDA call
    (the addresses below are never dereferenced)."""
    lib = gdn.load()
    d, w, c, r = _args()
    W, C, R = ctypes.byref(w), ctypes.byref(c), ctypes.byref(r)
    D = ctypes.byref(d)
    assert lib.gdn_window_pooled(D, W, C, A16, A16, 2, 4, R, None, None) == -2
    assert lib.gdn_window_pooled(D, W, C, A16, A16, 2, 4, R, A16 + 2, None) == -3
    assert lib.gdn_window_pooled(D, W, C, A16, A16, 0, 4, R, A16, None) == -1
    assert lib.gdn_window_pooled(D, W, None, A16, A16, 2, 4, R, A16, None) == -2
    assert lib.gdn_tree_pooled(D, W, C, A16, A16, None, 2, 4, R, A16, None) == -2
    assert lib.gdn_tree_pooled(D, W, C, A16, A16, A16, 2, 4, R, None, None) == -2
    assert lib.gdn_commit_swap(D, C, A16, A16, A16, None, 2, 4, None, None) == -2
    assert lib.gdn_commit_swap(D, C, A16, None, A16, A16, 2, 4, None, None) == -2
    assert lib.gdn_commit_swap(D, C, A16, A16, A16, A16, 2, 4, A16 + 1, None) == -3
    assert lib.gdn_commit_swap(D, C, A16, A16, A16, A16, 2, 0, None, None) == -1
    assert lib.gdn_commit_swap(D, C, A16, A16, A16, A16, 0, 4, None, None) == -1


def test_commit_refuses_a_missing_or_misaligned_row_ptr():
    lib = gdn.load()
    d, w, c, r = _args()
    assert lib.gdn_commit(ctypes.byref(d), ctypes.byref(c), A16, None, A16, 2, 4, A16, A16, None) == -2
    assert lib.gdn_commit(ctypes.byref(d), ctypes.byref(c), A16, A16 + 2, A16, 2, 4, A16, A16, None) == -3
    assert lib.gdn_prefill_workspace(ctypes.byref(d), 1, 4722, 64) == \
        lib.gdn_prefill_workspace_size(ctypes.byref(d), 1, 4722, 64) > 0


def test_step_ex_refuses_unknown_flags_and_bad_arguments():
    lib = gdn.load()
    d, w, c, r = _args()
    assert lib.gdn_step_ex(ctypes.byref(d), ctypes.byref(w), ctypes.byref(c), A16, 2, ctypes.byref(r), 2,
                           None) == -1
    assert lib.gdn_step_ex(ctypes.byref(d), ctypes.byref(w), ctypes.byref(c), A16, 2, ctypes.byref(r), 0x80000000,
                           None) == -1
    assert lib.gdn_step_ex(ctypes.byref(d), ctypes.byref(w), ctypes.byref(c), None, 2, ctypes.byref(r),
                           B.STEP_EARLY_STATE, None) == -2
    assert lib.gdn_step_ex(ctypes.byref(d), ctypes.byref(w), ctypes.byref(c), A16 + 2, 2, ctypes.byref(r),
                           B.STEP_EARLY_STATE, None) == -3
    assert lib.gdn_step_ex(ctypes.byref(d), ctypes.byref(w), ctypes.byref(c), A16, 0, ctypes.byref(r),
                           B.STEP_EARLY_STATE, None) == -1
