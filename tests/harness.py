"""Shared helpers of the parity tests: seeded inputs on both sides, oracle
runs per stream, and the comparison rules.

Tolerances (the layer's stated bar, with our reading of it):
  * y (bf16): |y_gpu - y_ref| <= 2e-3 + 1/2 ulp_bf16(|y_ref|), where y_ref is
    the oracle's unrounded double result: the half ulp is the output's own
    bf16 rounding, 2e-3 the arithmetic budget.
  * fp32 states: per (row or slot, value head) tile,
    max |S_gpu - S_ref| <= 1e-4 * max |S_ref|  (normwise relative; an
    elementwise relative bound is meaningless where entries cross zero).
  * conv tails are copies of bf16 inputs: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_deltanet_speculative_gb300 import synth

Y_ABS = 2e-3
STATE_REL = 1e-4


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def dev(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def check_y(y_gpu_bits: np.ndarray, y_ref: np.ndarray, what="y"):
    y = synth.bf16_bits_to_f32(y_gpu_bits).astype(np.float64)
    assert np.all(np.isfinite(y)), f"{what}: non-finite GPU output (unwritten element?)"
    bound = Y_ABS + 0.5 * bf16_ulp(np.abs(y_ref) + Y_ABS)
    err = np.abs(y - y_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside 2e-3 + ulp/2; "
                           f"worst {err.max():.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def check_state(S_gpu: np.ndarray, S_ref: np.ndarray, what="state"):
    """Tiles are the last two axes."""
    S_gpu = np.asarray(S_gpu, np.float64)
    assert np.all(np.isfinite(S_gpu)), f"{what}: non-finite GPU state (unwritten element?)"
    lead = S_ref.shape[:-2]
    d = np.abs(S_gpu - S_ref).reshape(*lead, -1).max(-1)
    m = np.abs(S_ref).reshape(*lead, -1).max(-1)
    rel = d / np.maximum(m, 1e-30)
    assert rel.max() <= STATE_REL, f"{what}: normwise relative error {rel.max():.3e} > {STATE_REL}"
    return float(rel.max())


class Case:
    """Seeded inputs of one call: a layer, a slot cache and packed rows."""

    def __init__(self, g: synth.Geometry, lengths, seed: int, n_slots=None, tree=False, slots=None,
                 zero_state=False):
        self.g = g
        self.lengths = list(lengths)
        self.S = len(self.lengths)
        self.R = int(sum(self.lengths))
        rng = np.random.default_rng([seed, 9])
        self.n_slots = n_slots or self.S
        self.slots = (np.asarray(slots, np.int32) if slots is not None
                      else rng.permutation(self.n_slots)[: self.S].astype(np.int32))
        self.w = synth.layer_weights(g, seed)
        self.cache = synth.slot_cache(g, self.n_slots, seed, zero=zero_state)
        self.rows = synth.row_inputs(g, max(self.R, 1), seed)
        self.row_ptr = synth.row_ptr(self.lengths)
        self.parent = None
        if tree:
            self.parent = np.concatenate([synth.random_tree(n, rng) for n in self.lengths]).astype(np.int32) \
                if self.R else np.zeros(0, np.int32)

    def dims_oracle(self):
        g = self.g
        return oracle.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)

    def dims_gpu(self):
        from gated_deltanet_speculative_gb300 import Dims
        g = self.g
        return Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)

    def stream_rows(self, s):
        lo, hi = int(self.row_ptr[s]), int(self.row_ptr[s + 1])
        return lo, hi

    def oracle_stream(self, s, threads=8, record=True):
        lo, hi = self.stream_rows(s)
        sl = int(self.slots[s])
        par = None if self.parent is None else self.parent[lo:hi]
        r = self.rows
        return oracle.gdn_rows(self.dims_oracle(), self.w, self.cache["state"][sl], self.cache["tail"][sl],
                               r["mixed"][lo:hi], r["z"][lo:hi], r["a"][lo:hi], r["b"][lo:hi], parent=par,
                               record=record, threads=threads)

    # ---- device copies ----
    def dev_weights(self):
        return {"conv_w": dev_bf16(self.w["conv_w"]), "A_log": dev(self.w["A_log"]),
                "dt_bias": dev(self.w["dt_bias"]), "norm_w": dev_bf16(self.w["norm_w"])}

    def dev_cache(self):
        return {"state": dev(self.cache["state"]), "tail": dev_bf16(self.cache["tail"])}

    def dev_rows(self, poison=True):
        R = max(self.R, 1)
        g = self.g
        y = torch.full((R, g.n_v_heads, g.d_v), float("nan") if poison else 0.0, dtype=torch.bfloat16,
                       device="cuda")
        return {"mixed": dev_bf16(self.rows["mixed"]), "z": dev_bf16(self.rows["z"]), "a": dev_bf16(self.rows["a"]),
                "b": dev_bf16(self.rows["b"]), "y": y}

    def dev_records(self, poison=True):
        R = max(self.R, 1)
        g = self.g
        rs = torch.full((R, g.n_v_heads, g.d_v, g.d_k), float("nan") if poison else 0.0, dtype=torch.float32,
                        device="cuda")
        rt = torch.full((R, 3, g.channels), float("nan") if poison else 0.0, dtype=torch.bfloat16, device="cuda")
        return rs, rt
