"""CPU oracle for the gated-DeltaNet verify path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It wraps ``gdn_oracle.c`` (plain sequential C in
double precision) through ctypes and shares no code with the CUDA library.

Every function takes numpy arrays on the host: bf16 tensors are passed as
their raw ``uint16`` bit patterns, fp32 states as ``float32``; results are
``float64`` (states, outputs) or ``uint16`` (copied bf16 tails).

Sources (by page title): TensorFold #932 "deliver the first token before
drafting" (a causal conv and the gated delta rule in the CUDA glue; verify
windows of at most 16 rows with every row's state kept; tree windows whose
taps and recurrence follow each row's branch) and TensorFold #747 "reduce
repeated-prompt TTFT" (one verify round for at most 16 streams x 16 rows;
only the accepted rows of each stream are kept).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math) into oracle/_build."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dims(ctypes.Structure):
    _fields_ = [("n_k_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("q_scale", ctypes.c_double), ("eps_l2", ctypes.c_double),
                ("eps_rms", ctypes.c_double)]


def _configure(lib):
    P = ctypes.c_void_p
    lib.oracle_gdn_rows.restype = ctypes.c_int
    lib.oracle_gdn_rows.argtypes = [ctypes.POINTER(_Dims), P, P, P, P, ctypes.c_int32, P, P, P,
                                    P, P, P, P, ctypes.c_int32, ctypes.c_int32,
                                    P, P, P, P, P, P, P, P, P, P]
    lib.oracle_gates.restype = None
    lib.oracle_gates.argtypes = [ctypes.c_double] * 4 + [P, P]
    lib.oracle_delta_rule.restype = None
    lib.oracle_delta_rule.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P,
                                      ctypes.c_double, ctypes.c_double, P]
    lib.oracle_gated_rmsnorm.restype = None
    lib.oracle_gated_rmsnorm.argtypes = [ctypes.c_int, P, P, P, ctypes.c_double, P]
    lib.oracle_l2norm.restype = None
    lib.oracle_l2norm.argtypes = [ctypes.c_int, P, ctypes.c_double, ctypes.c_double]
    lib.oracle_chunked_rule.restype = None
    lib.oracle_chunked_rule.argtypes = [ctypes.c_int] * 4 + [P] * 7
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Route every oracle call through another build of gdn_oracle.c (the
    mutation tests use it to check that the pins catch planted mistakes)."""
    global _lib
    _load()
    with _lock:
        old, _lib = _lib, _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = old


def source_path() -> str:
    return _SRC


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Dims:
    """Layer geometry: key heads Hk, value heads Hv, head widths dk, dv."""

    def __init__(self, n_k_heads, n_v_heads, d_k, d_v, q_scale=None, eps_l2=1e-6, eps_rms=1e-6):
        self.n_k_heads, self.n_v_heads, self.d_k, self.d_v = n_k_heads, n_v_heads, d_k, d_v
        self.q_scale = d_k ** -0.5 if q_scale is None else q_scale
        self.eps_l2, self.eps_rms = eps_l2, eps_rms

    @property
    def channels(self):
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    def _c(self):
        return _Dims(self.n_k_heads, self.n_v_heads, self.d_k, self.d_v,
                     float(self.q_scale), float(self.eps_l2), float(self.eps_rms))


# ---- scalar / single-head definitions (exposed for the pins) ---------------

def gates(A_log, dt_bias, a_in, b_in):
    """(decay a_t, beta b_t) of one (row, value head)."""
    lib = _load()
    d, b = ctypes.c_double(), ctypes.c_double()
    lib.oracle_gates(float(A_log), float(dt_bias), float(a_in), float(b_in), ctypes.byref(d), ctypes.byref(b))
    return d.value, b.value


def delta_rule(S, q, k, v, decay, beta):
    """One gated-delta-rule row: returns (S', o) for S [dv, dk] in float64."""
    lib = _load()
    S = _c(S, np.float64).copy()
    dv, dk = S.shape
    o = np.empty(dv, np.float64)
    lib.oracle_delta_rule(dv, dk, _ptr(S), _ptr(_c(q, np.float64)), _ptr(_c(k, np.float64)),
                          _ptr(_c(v, np.float64)), float(decay), float(beta), _ptr(o))
    return S, o


def gated_rmsnorm(o, z, w, eps=1e-6):
    lib = _load()
    o = _c(o, np.float64)
    y = np.empty_like(o)
    lib.oracle_gated_rmsnorm(o.size, _ptr(o), _ptr(_c(z, np.float64)), _ptr(_c(w, np.float64)), float(eps), _ptr(y))
    return y


def l2norm(x, eps=1e-6, scale=1.0):
    lib = _load()
    x = _c(x, np.float64).copy()
    lib.oracle_l2norm(x.size, _ptr(x), float(eps), float(scale))
    return x


def chunked_rule(S0, Q, K, V, g, beta, chunk):
    """Chunked (WY/UT) form of the recurrence for one head; returns (S, O)."""
    lib = _load()
    S = _c(S0, np.float64).copy()
    dv, dk = S.shape
    L = Q.shape[0]
    O = np.empty((L, dv), np.float64)
    lib.oracle_chunked_rule(dv, dk, L, chunk, _ptr(S), _ptr(_c(Q, np.float64)), _ptr(_c(K, np.float64)),
                            _ptr(_c(V, np.float64)), _ptr(_c(g, np.float64)), _ptr(_c(beta, np.float64)), _ptr(O))
    return S, O


# ---- one stream's rows through the layer ----------------------------------

def gdn_rows(dims: Dims, w: dict, state0, tail0, mixed, z, a, b, parent=None, *,
             record=True, final=False, extras=False, heads=None, threads=1):
    """Run one stream's rows (a chain, or a tree when ``parent`` is given).

    ``w`` holds ``conv_w`` [CH, 4] (uint16 bf16 bits), ``A_log`` [Hv] and
    ``dt_bias`` [Hv] (float32), ``norm_w`` [dv] (uint16).  ``state0`` is the
    committed fp32 state [Hv, dv, dk]; ``tail0`` the committed bf16 tail
    [3, CH]; ``mixed`` [n, CH], ``z`` [n, Hv, dv], ``a``/``b`` [n, Hv] bf16
    bits.  Returns a dict with ``y`` [n, Hv, dv] (float64, unrounded) and,
    as requested, ``rec_state`` [n, Hv, dv, dk], ``rec_tail`` [n, 3, CH],
    ``final_state`` / ``final_tail`` (chains), and the per-row ``q``, ``k``,
    ``v``, ``decay``, ``beta`` (``extras``).  ``threads`` > 1 splits the value
    heads across host threads (heads are independent).
    """
    lib = _load()
    Hv, dk, dv, CH = dims.n_v_heads, dims.d_k, dims.d_v, dims.channels
    n = int(mixed.shape[0])
    h0, h1 = heads if heads is not None else (0, Hv)
    par = None if parent is None else _c(parent, np.int32)
    if par is not None:
        record = True
    arrs = dict(conv_w=_c(w["conv_w"], np.uint16), A_log=_c(w["A_log"], np.float32),
                dt_bias=_c(w["dt_bias"], np.float32), norm_w=_c(w["norm_w"], np.uint16),
                state0=_c(state0, np.float32), tail0=_c(tail0, np.uint16), mixed=_c(mixed, np.uint16),
                z=_c(z, np.uint16), a=_c(a, np.uint16), b=_c(b, np.uint16))
    out = {"y": np.zeros((n, Hv, dv), np.float64)}
    if record:
        out["rec_state"] = np.zeros((n, Hv, dv, dk), np.float64)
        out["rec_tail"] = np.zeros((n, 3, CH), np.uint16)
    if final and par is None:
        out["final_state"] = np.zeros((Hv, dv, dk), np.float64)
        out["final_tail"] = np.zeros((3, CH), np.uint16)
    if extras:
        out.update(q=np.zeros((n, Hv, dk)), k=np.zeros((n, Hv, dk)), v=np.zeros((n, Hv, dv)),
                   decay=np.zeros((n, Hv)), beta=np.zeros((n, Hv)))
    dc = dims._c()

    def run(lo, hi):
        rc = lib.oracle_gdn_rows(ctypes.byref(dc), _ptr(arrs["conv_w"]), _ptr(arrs["A_log"]),
                                 _ptr(arrs["dt_bias"]), _ptr(arrs["norm_w"]), n, _ptr(par),
                                 _ptr(arrs["state0"]), _ptr(arrs["tail0"]), _ptr(arrs["mixed"]),
                                 _ptr(arrs["z"]), _ptr(arrs["a"]), _ptr(arrs["b"]), lo, hi,
                                 _ptr(out["y"]), _ptr(out.get("rec_state")),
                                 _ptr(out.get("rec_tail")) if lo == h0 else None,
                                 _ptr(out.get("final_state")),
                                 _ptr(out.get("final_tail")) if lo == h0 else None,
                                 _ptr(out.get("q")), _ptr(out.get("k")), _ptr(out.get("v")),
                                 _ptr(out.get("decay")), _ptr(out.get("beta")))
        if rc != 0:
            raise ValueError("oracle_gdn_rows rejected its arguments")

    if threads <= 1 or h1 - h0 <= 1:
        run(h0, h1)
    else:
        nt = min(threads, h1 - h0)
        cuts = [h0 + (h1 - h0) * i // nt for i in range(nt + 1)]
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(lambda i: run(cuts[i], cuts[i + 1]), range(nt)))
    return out


def commit(rec_state, rec_tail, keep_row, state, tail):
    """Commit of the accepted path for one stream: returns (state, tail).

    ``keep_row`` >= 0 takes that window row's recorded state and tail;
    -1 leaves the committed state and tail as they are.
    """
    if keep_row < 0:
        return state, tail
    return np.array(rec_state[keep_row], copy=True), np.array(rec_tail[keep_row], copy=True)


def bf16_to_f64(bits):
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
