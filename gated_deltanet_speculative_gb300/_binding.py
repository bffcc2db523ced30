"""ctypes binding of libgdn.so (include/gdn.h): argument marshalling only.

Every function takes torch CUDA tensors, checks their shapes and dtypes
against the geometry, and passes raw device pointers and sizes to the C ABI
on the current (or given) CUDA stream.  All computation happens in the CUDA
kernels; there is no fallback: if the library cannot be loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

STATUS = {0: "GDN_OK", -1: "GDN_EINVAL", -2: "GDN_ENULL", -3: "GDN_EALIGN", -4: "GDN_ECUDA", -5: "GDN_EWORKSPACE"}
DERR = {1: "slot", 2: "rows", 4: "parent", 8: "keep_row", 16: "cu_seqlens", 32: "timeout"}
MAX_WINDOW = 16


class GdnError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({msg})")
        self.status = status


class c_dims(ctypes.Structure):
    _fields_ = [("n_k_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("conv_width", ctypes.c_int32), ("q_scale", ctypes.c_float),
                ("eps_l2", ctypes.c_float), ("eps_rms", ctypes.c_float)]


class c_weights(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("norm_w", ctypes.c_void_p)]


class c_cache(ctypes.Structure):
    _fields_ = [("state", ctypes.c_void_p), ("tail", ctypes.c_void_p), ("n_slots", ctypes.c_int32)]


class c_rows(ctypes.Structure):
    _fields_ = [("mixed", ctypes.c_void_p), ("z", ctypes.c_void_p), ("a", ctypes.c_void_p),
                ("b", ctypes.c_void_p), ("y", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIGS = {
    "gdn_step": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _I,
                 ctypes.POINTER(c_rows), _P],
    "gdn_step_ex": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _I,
                    ctypes.POINTER(c_rows), ctypes.c_uint32, _P],
    "gdn_window": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _P, _I, _I,
                   ctypes.POINTER(c_rows), _P, _P, _P],
    "gdn_tree": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _P, _P, _I, _I,
                 ctypes.POINTER(c_rows), _P, _P, _P],
    "gdn_commit": [ctypes.POINTER(c_dims), ctypes.POINTER(c_cache), _P, _P, _P, _I, _I, _P, _P, _P],
    "gdn_window_pooled": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _P, _I, _I,
                          ctypes.POINTER(c_rows), _P, _P],
    "gdn_tree_pooled": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _P, _P, _I,
                        _I, ctypes.POINTER(c_rows), _P, _P],
    "gdn_commit_swap": [ctypes.POINTER(c_dims), ctypes.POINTER(c_cache), _P, _P, _P, _P, _I, _I, _P, _P],
    "gdn_prefill": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _P, _I, _I,
                    ctypes.POINTER(c_rows), _I, _P, ctypes.c_size_t, _P],
    "gdn_prefill_workspace_size": [ctypes.POINTER(c_dims), _I, _I, _I],
    "gdn_prefill_workspace": [ctypes.POINTER(c_dims), _I, _I, _I],
    "gdn_prefill_noalloc": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _P, _I,
                            _I, ctypes.POINTER(c_rows), _I, _P],
    "gdn_window_log": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _P, _I, _I,
                       ctypes.POINTER(c_rows), _P, _P, _P, _P, _P],
    "gdn_commit_replay": [ctypes.POINTER(c_dims), ctypes.POINTER(c_cache), _P, _P, _P, _I, _I, _P, _P, _P, _P, _P],
    "gdn_tree_log": [ctypes.POINTER(c_dims), ctypes.POINTER(c_weights), ctypes.POINTER(c_cache), _P, _P, _P, _I, _I,
                     ctypes.POINTER(c_rows), _P, _P, _P, _P, _P],
    "gdn_commit_replay_tree": [ctypes.POINTER(c_dims), ctypes.POINTER(c_cache), _P, _P, _P, _P, _I, _I, _P, _P, _P,
                               _P, _P],
    "gdn_debug_wait_timeout": [ctypes.c_uint32, _P],
    "gdn_status_string": [ctypes.c_int],
    "gdn_get_device_error": [_P, ctypes.POINTER(ctypes.c_int32)],
}


def library_path() -> str:
    return _build.LIB


_capture = threading.local()   # prepare(): the recorder that stands in for the library


def load(build_if_missing: bool = True):
    """Load libgdn.so (building it first if it is missing or stale)."""
    global _lib
    rec = getattr(_capture, "rec", None)
    if rec is not None:
        return rec
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libgdn.so not found at {path}; build it with gated_deltanet_speculative_gb300.build")
            lib = ctypes.CDLL(path)
            for name, argtypes in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = {"gdn_status_string": ctypes.c_char_p,
                              "gdn_prefill_workspace_size": ctypes.c_size_t,
                              "gdn_prefill_workspace": ctypes.c_size_t}.get(name, ctypes.c_int)
            _lib = lib
    return _lib


class _Recorder:
    """Records the library call a binding function makes instead of making it."""

    def __init__(self, lib):
        self._lib = lib
        self.calls = []

    def __getattr__(self, name):
        fn = getattr(self._lib, name)

        def record(*cargs):
            self.calls.append((name, fn, cargs))
            return 0
        return record


class PreparedCall:
    """One entry point with its arguments checked and marshalled once.

    Calling it enqueues the same C call on the given stream (default: the
    current one) with a single ctypes call.  The tensors it was prepared
    with must stay allocated and keep their shapes; their contents may
    change between calls (new rows, new keep rows), as in a serving loop."""

    def __init__(self, name, cfn, cargs, keep):
        self.name, self._cfn, self._cargs, self._keep = name, cfn, cargs, keep

    def __call__(self, stream=None):
        _check(self.name, self._cfn(*self._cargs, _stream_ptr(stream)))


def prepare(fn, *args, **kwargs) -> PreparedCall:
    """Check and marshal the arguments of a compute call once, e.g.
    ``prepare(step, dims, weights, cache, slot, rows)``; the result enqueues
    that call when called (its stream is the C call's last argument)."""
    rec = _Recorder(load())
    _capture.rec = rec
    try:
        fn(*args, stream=0, **kwargs)
    finally:
        _capture.rec = None
    if len(rec.calls) != 1:
        raise ValueError(f"{getattr(fn, '__name__', fn)} is not a single compute call")
    name, cfn, cargs = rec.calls[0]
    return PreparedCall(name, cfn, cargs[:-1], (args, kwargs))


class Dims:
    """Head geometry and epsilons of one GDN layer (mirrors gdn_dims)."""

    def __init__(self, n_k_heads, n_v_heads, d_k, d_v, q_scale=None, eps_l2=1e-6, eps_rms=1e-6):
        self.n_k_heads, self.n_v_heads, self.d_k, self.d_v = int(n_k_heads), int(n_v_heads), int(d_k), int(d_v)
        self.q_scale = float(d_k) ** -0.5 if q_scale is None else float(q_scale)
        self.eps_l2, self.eps_rms = float(eps_l2), float(eps_rms)

    @property
    def channels(self) -> int:
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    def c(self) -> c_dims:
        return c_dims(self.n_k_heads, self.n_v_heads, self.d_k, self.d_v, 4, self.q_scale, self.eps_l2,
                      self.eps_rms)


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _weights(d: Dims, w: dict) -> c_weights:
    _need(w["conv_w"], "conv_w", torch.bfloat16, (d.channels, 4))
    _need(w["A_log"], "A_log", torch.float32, (d.n_v_heads,))
    _need(w["dt_bias"], "dt_bias", torch.float32, (d.n_v_heads,))
    _need(w["norm_w"], "norm_w", torch.bfloat16, (d.d_v,))
    return c_weights(w["conv_w"].data_ptr(), w["A_log"].data_ptr(), w["dt_bias"].data_ptr(), w["norm_w"].data_ptr())


def _cache(d: Dims, cache: dict) -> c_cache:
    st, tl = cache["state"], cache["tail"]
    _need(st, "state", torch.float32)
    n_slots = st.shape[0]
    _need(st, "state", torch.float32, (n_slots, d.n_v_heads, d.d_v, d.d_k))
    _need(tl, "tail", torch.bfloat16, (n_slots, 3, d.channels))
    return c_cache(st.data_ptr(), tl.data_ptr(), n_slots)


def _rows(d: Dims, rows: dict, n_rows: int) -> c_rows:
    _need(rows["mixed"], "mixed", torch.bfloat16, (n_rows, d.channels))
    _need(rows["z"], "z", torch.bfloat16, (n_rows, d.n_v_heads, d.d_v))
    _need(rows["a"], "a", torch.bfloat16, (n_rows, d.n_v_heads))
    _need(rows["b"], "b", torch.bfloat16, (n_rows, d.n_v_heads))
    _need(rows["y"], "y", torch.bfloat16, (n_rows, d.n_v_heads, d.d_v))
    return c_rows(*(rows[k].data_ptr() for k in ("mixed", "z", "a", "b", "y")))


def _check(fn, rc):
    if rc != 0:
        raise GdnError(fn, rc, load().gdn_status_string(rc).decode())


def step(dims: Dims, weights: dict, cache: dict, slot, rows: dict, stream=None):
    """One row per stream, state and tail of slot[s] advanced in place."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, S)
    _check("gdn_step", lib.gdn_step(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc), _ptr(slot), S,
                                    ctypes.byref(cr), _stream_ptr(stream)))


STEP_EARLY_STATE = 1


def step_ex(dims: Dims, weights: dict, cache: dict, slot, rows: dict, flags: int = 0, stream=None):
    """gdn_step with launch flags: STEP_EARLY_STATE promises that the kernel
    queued just before on the stream writes none of slot, the cache or the
    weights, so the step reads them while that kernel finishes."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, S)
    _check("gdn_step_ex", lib.gdn_step_ex(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc), _ptr(slot), S,
                                          ctypes.byref(cr), int(flags), _stream_ptr(stream)))


def window(dims: Dims, weights: dict, cache: dict, slot, row_ptr, rows: dict, rec_state, rec_tail, stream=None):
    """Chain verify windows, every row's state and tail recorded."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    R = rows["mixed"].shape[0]
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, R)
    _need(rec_state, "rec_state", torch.float32, (R, dims.n_v_heads, dims.d_v, dims.d_k))
    _need(rec_tail, "rec_tail", torch.bfloat16, (R, 3, dims.channels))
    _check("gdn_window", lib.gdn_window(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc), _ptr(slot),
                                        _ptr(row_ptr), S, R, ctypes.byref(cr), _ptr(rec_state), _ptr(rec_tail),
                                        _stream_ptr(stream)))


def tree(dims: Dims, weights: dict, cache: dict, slot, row_ptr, parent, rows: dict, rec_state, rec_tail,
         stream=None):
    """Tree verify windows given by window-local parent indices (-1 = slot)."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    R = rows["mixed"].shape[0]
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    _need(parent, "parent", torch.int32, (R,))
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, R)
    _need(rec_state, "rec_state", torch.float32, (R, dims.n_v_heads, dims.d_v, dims.d_k))
    _need(rec_tail, "rec_tail", torch.bfloat16, (R, 3, dims.channels))
    _check("gdn_tree", lib.gdn_tree(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc), _ptr(slot),
                                    _ptr(row_ptr), _ptr(parent), S, R, ctypes.byref(cr), _ptr(rec_state),
                                    _ptr(rec_tail), _stream_ptr(stream)))


def commit(dims: Dims, cache: dict, slot, row_ptr, keep_row, rec_state, rec_tail, stream=None):
    """Slot s takes recorded row keep_row[s], one of its own rows
    [row_ptr[s], row_ptr[s+1]) (-1: slot untouched)."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    _need(keep_row, "keep_row", torch.int32, (S,))
    cc = _cache(dims, cache)
    R = rec_state.shape[0]
    _need(rec_state, "rec_state", torch.float32, (R, dims.n_v_heads, dims.d_v, dims.d_k))
    _need(rec_tail, "rec_tail", torch.bfloat16, (R, 3, dims.channels))
    _check("gdn_commit", lib.gdn_commit(ctypes.byref(dims.c()), ctypes.byref(cc), _ptr(slot), _ptr(row_ptr),
                                        _ptr(keep_row), S, R, _ptr(rec_state), _ptr(rec_tail), _stream_ptr(stream)))


def window_pooled(dims: Dims, weights: dict, cache: dict, slot, row_ptr, rows: dict, rec_slot, stream=None):
    """Chain verify windows recording row r at cache entry rec_slot[r]."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    R = rows["mixed"].shape[0]
    _need(rec_slot, "rec_slot", torch.int32, (R,))
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, R)
    _check("gdn_window_pooled", lib.gdn_window_pooled(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc),
                                                      _ptr(slot), _ptr(row_ptr), S, R, ctypes.byref(cr),
                                                      _ptr(rec_slot), _stream_ptr(stream)))


def tree_pooled(dims: Dims, weights: dict, cache: dict, slot, row_ptr, parent, rows: dict, rec_slot, stream=None):
    """Tree verify windows recording node r at cache entry rec_slot[r]."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    R = rows["mixed"].shape[0]
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    _need(parent, "parent", torch.int32, (R,))
    _need(rec_slot, "rec_slot", torch.int32, (R,))
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, R)
    _check("gdn_tree_pooled", lib.gdn_tree_pooled(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc),
                                                  _ptr(slot), _ptr(row_ptr), _ptr(parent), S, R, ctypes.byref(cr),
                                                  _ptr(rec_slot), _stream_ptr(stream)))


def commit_swap(dims: Dims, cache: dict, slot, row_ptr, keep_row, rec_slot, freed=None, stream=None):
    """Slot s takes pool entry rec_slot[keep_row[s]] (-1: unchanged); its
    previous entry goes to freed[s] (-1 when nothing was committed)."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    _need(keep_row, "keep_row", torch.int32, (S,))
    _need(rec_slot, "rec_slot", torch.int32)
    if freed is not None:
        _need(freed, "freed", torch.int32, (S,))
    cc = _cache(dims, cache)
    _check("gdn_commit_swap", lib.gdn_commit_swap(ctypes.byref(dims.c()), ctypes.byref(cc), _ptr(slot), _ptr(row_ptr),
                                                  _ptr(keep_row), _ptr(rec_slot), S, rec_slot.numel(), _ptr(freed),
                                                  _stream_ptr(stream)))


def window_log(dims: Dims, weights: dict, cache: dict, slot, row_ptr, rows: dict, log_a, log_u, log_k, rec_tail,
               stream=None):
    """Chain verify windows logging each row's decay, write and key."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    R = rows["mixed"].shape[0]
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, R)
    _need(log_a, "log_a", torch.float32, (R, dims.n_v_heads))
    _need(log_u, "log_u", torch.float32, (R, dims.n_v_heads, dims.d_v))
    _need(log_k, "log_k", torch.float32, (R, dims.n_k_heads, dims.d_k))
    _need(rec_tail, "rec_tail", torch.bfloat16, (R, 3, dims.channels))
    _check("gdn_window_log", lib.gdn_window_log(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc),
                                                _ptr(slot), _ptr(row_ptr), S, R, ctypes.byref(cr), _ptr(log_a),
                                                _ptr(log_u), _ptr(log_k), _ptr(rec_tail), _stream_ptr(stream)))


def commit_replay(dims: Dims, cache: dict, slot, row_ptr, keep_row, log_a, log_u, log_k, rec_tail, stream=None):
    """Commit by replaying the logged chain up to keep_row[s] (-1: untouched)."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    _need(keep_row, "keep_row", torch.int32, (S,))
    cc = _cache(dims, cache)
    R = log_a.shape[0]
    _need(log_a, "log_a", torch.float32, (R, dims.n_v_heads))
    _need(log_u, "log_u", torch.float32, (R, dims.n_v_heads, dims.d_v))
    _need(log_k, "log_k", torch.float32, (R, dims.n_k_heads, dims.d_k))
    _need(rec_tail, "rec_tail", torch.bfloat16, (R, 3, dims.channels))
    _check("gdn_commit_replay", lib.gdn_commit_replay(ctypes.byref(dims.c()), ctypes.byref(cc), _ptr(slot),
                                                      _ptr(row_ptr), _ptr(keep_row), S, R, _ptr(log_a), _ptr(log_u),
                                                      _ptr(log_k), _ptr(rec_tail), _stream_ptr(stream)))


def tree_log(dims: Dims, weights: dict, cache: dict, slot, row_ptr, parent, rows: dict, log_a, log_u, log_k,
             rec_tail, stream=None):
    """Tree verify windows logging each node's decay, write and key."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    R = rows["mixed"].shape[0]
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    _need(parent, "parent", torch.int32, (R,))
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, R)
    _need(log_a, "log_a", torch.float32, (R, dims.n_v_heads))
    _need(log_u, "log_u", torch.float32, (R, dims.n_v_heads, dims.d_v))
    _need(log_k, "log_k", torch.float32, (R, dims.n_k_heads, dims.d_k))
    _need(rec_tail, "rec_tail", torch.bfloat16, (R, 3, dims.channels))
    _check("gdn_tree_log", lib.gdn_tree_log(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc), _ptr(slot),
                                            _ptr(row_ptr), _ptr(parent), S, R, ctypes.byref(cr), _ptr(log_a),
                                            _ptr(log_u), _ptr(log_k), _ptr(rec_tail), _stream_ptr(stream)))


def commit_replay_tree(dims: Dims, cache: dict, slot, row_ptr, parent, keep_row, log_a, log_u, log_k, rec_tail,
                       stream=None):
    """Commit by replaying the logged root-to-node path of keep_row[s] (-1: untouched)."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    _need(row_ptr, "row_ptr", torch.int32, (S + 1,))
    _need(keep_row, "keep_row", torch.int32, (S,))
    cc = _cache(dims, cache)
    R = log_a.shape[0]
    _need(parent, "parent", torch.int32, (R,))
    _need(log_a, "log_a", torch.float32, (R, dims.n_v_heads))
    _need(log_u, "log_u", torch.float32, (R, dims.n_v_heads, dims.d_v))
    _need(log_k, "log_k", torch.float32, (R, dims.n_k_heads, dims.d_k))
    _need(rec_tail, "rec_tail", torch.bfloat16, (R, 3, dims.channels))
    _check("gdn_commit_replay_tree",
           lib.gdn_commit_replay_tree(ctypes.byref(dims.c()), ctypes.byref(cc), _ptr(slot), _ptr(row_ptr),
                                      _ptr(parent), _ptr(keep_row), S, R, _ptr(log_a), _ptr(log_u), _ptr(log_k),
                                      _ptr(rec_tail), _stream_ptr(stream)))


def debug_wait_timeout(polls: int = 1000, stream=None):
    """Run the kernels' bounded mbarrier wait on a phase nothing completes;
    it gives up after ``polls`` polls and sets the timeout bit (32) of the
    device error word."""
    _check("gdn_debug_wait_timeout", load().gdn_debug_wait_timeout(int(polls), _stream_ptr(stream)))


PREFILL_CHUNK = 64


def prefill_workspace_size(dims: Dims, n_seqs: int, n_tokens: int, chunk: int = PREFILL_CHUNK) -> int:
    """Bytes of scratch gdn_prefill needs (0 for invalid sizes)."""
    return int(load().gdn_prefill_workspace_size(ctypes.byref(dims.c()), int(n_seqs), int(n_tokens), int(chunk)))


def prefill_workspace(dims: Dims, n_seqs: int, n_tokens: int, chunk: int = PREFILL_CHUNK) -> int:
    """The same size through the header's shorter name."""
    return int(load().gdn_prefill_workspace(ctypes.byref(dims.c()), int(n_seqs), int(n_tokens), int(chunk)))


def prefill(dims: Dims, weights: dict, cache: dict, slot, cu_seqlens, rows: dict, workspace, chunk: int = PREFILL_CHUNK,
            stream=None):
    """Chunked prompt prefill of packed sequences; slots advanced in place.

    ``workspace`` is a CUDA uint8 tensor of at least
    ``prefill_workspace_size(dims, n_seqs, n_tokens)`` bytes."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    _need(cu_seqlens, "cu_seqlens", torch.int32, (S + 1,))
    T = rows["mixed"].shape[0]
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, T)
    _need(workspace, "workspace", torch.uint8)
    _check("gdn_prefill", lib.gdn_prefill(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc), _ptr(slot),
                                          _ptr(cu_seqlens), S, T, ctypes.byref(cr), int(chunk), _ptr(workspace),
                                          workspace.numel(), _stream_ptr(stream)))


def prefill_noalloc(dims: Dims, weights: dict, cache: dict, slot, cu_seqlens, rows: dict,
                    chunk: int = PREFILL_CHUNK, stream=None):
    """gdn_prefill without a workspace: the library's fixed device scratch
    (PREFILL_NOALLOC_SCRATCH_BYTES) stands in for it, and every launch goes
    on the given stream.  Calls whose work overlaps on the GPU share that
    scratch and must be serialised by the caller."""
    lib = load()
    _need(slot, "slot", torch.int32)
    S = slot.numel()
    _need(cu_seqlens, "cu_seqlens", torch.int32, (S + 1,))
    T = rows["mixed"].shape[0]
    cw, cc, cr = _weights(dims, weights), _cache(dims, cache), _rows(dims, rows, T)
    _check("gdn_prefill_noalloc", lib.gdn_prefill_noalloc(ctypes.byref(dims.c()), ctypes.byref(cw), ctypes.byref(cc),
                                                          _ptr(slot), _ptr(cu_seqlens), S, T, ctypes.byref(cr),
                                                          int(chunk), _stream_ptr(stream)))


PREFILL_NOALLOC_SCRATCH_BYTES = 64 << 20


def get_device_error(stream=None) -> int:
    """Read and clear the device error word (synchronises the stream)."""
    lib = load()
    bits = ctypes.c_int32(0)
    _check("gdn_get_device_error", lib.gdn_get_device_error(_stream_ptr(stream), ctypes.byref(bits)))
    return bits.value
