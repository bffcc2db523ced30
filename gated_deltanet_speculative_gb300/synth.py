"""Seeded synthetic inputs for the GDN verify path.

This module only draws numbers: it holds none of the layer's arithmetic, so
the CUDA path and the CPU oracle can both be fed from it.  Everything is
drawn with numpy's PCG64 generator (platform-independent), in float32, and
bf16 tensors are returned as their raw ``uint16`` bit patterns (round to
nearest even), fp32 tensors as ``float32``, indices as ``int32``.

Distributions (the workloads' stated shapes; readings where they are silent):
  activations mixed / z / a / b   ~ N(0, 1)          bf16
  A_log                           ~ U(0, 2)          fp32  [Hv]
  dt_bias                         ~ N(0, 0.1)        fp32  [Hv]
  committed state S0              ~ N(0, 0.05)       fp32  [slots, Hv, dv, dk]
    (0.05 read as the standard deviation)
  committed conv tail             ~ N(0, 1)          bf16  [slots, 3, CH]
  conv weight                     ~ N(0, 0.5)        bf16  [CH, 4]
  norm weight                     1 + N(0, 0.1)      bf16  [dv]
  tree parents                    parent[0] = -1, parent[i] ~ U{0..i-1}
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def to_bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Geometry:
    """Head geometry of one GDN layer."""
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int

    @property
    def channels(self) -> int:
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    @property
    def group(self) -> int:
        return self.n_v_heads // self.n_k_heads


# Named head shapes of the workloads.
TINY = Geometry(2, 4, 32, 32)            # 1 stream, window of 4
LIKE_2B = Geometry(16, 16, 128, 128)     # decode step, 24 layers
LIKE_27B = Geometry(16, 48, 128, 128)    # verify rounds, trees, prefill


def layer_weights(g: Geometry, seed: int) -> dict:
    rng = np.random.default_rng([seed, 1])
    return {
        "conv_w": to_bf16_bits(rng.normal(0.0, 0.5, size=(g.channels, 4)).astype(np.float32)),
        "A_log": rng.uniform(0.0, 2.0, size=g.n_v_heads).astype(np.float32),
        "dt_bias": rng.normal(0.0, 0.1, size=g.n_v_heads).astype(np.float32),
        "norm_w": to_bf16_bits((1.0 + rng.normal(0.0, 0.1, size=g.d_v)).astype(np.float32)),
    }


def slot_cache(g: Geometry, n_slots: int, seed: int, zero: bool = False) -> dict:
    rng = np.random.default_rng([seed, 2])
    if zero:
        state = np.zeros((n_slots, g.n_v_heads, g.d_v, g.d_k), np.float32)
        tail = np.zeros((n_slots, 3, g.channels), np.uint16)
    else:
        state = rng.normal(0.0, 0.05, size=(n_slots, g.n_v_heads, g.d_v, g.d_k)).astype(np.float32)
        tail = to_bf16_bits(rng.normal(0.0, 1.0, size=(n_slots, 3, g.channels)).astype(np.float32))
    return {"state": state, "tail": tail}


def row_inputs(g: Geometry, n_rows: int, seed: int) -> dict:
    rng = np.random.default_rng([seed, 3])
    f = lambda *shape: to_bf16_bits(rng.normal(0.0, 1.0, size=shape).astype(np.float32))
    return {
        "mixed": f(n_rows, g.channels),
        "z": f(n_rows, g.n_v_heads, g.d_v),
        "a": f(n_rows, g.n_v_heads),
        "b": f(n_rows, g.n_v_heads),
    }


def row_ptr(lengths) -> np.ndarray:
    """Packed-row offsets [S+1] of streams with the given window lengths."""
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def random_tree(n: int, rng: np.random.Generator) -> np.ndarray:
    """Window-local parents of an n-node tree: node 0 hangs off the committed
    slot (-1); node i's parent is uniform in [0, i)."""
    p = np.empty(n, np.int32)
    if n:
        p[0] = -1
    for i in range(1, n):
        p[i] = rng.integers(0, i)
    return p


def random_leaf(parent: np.ndarray, rng: np.random.Generator) -> int:
    """A uniformly chosen leaf (a node no other node points to)."""
    n = len(parent)
    has_child = np.zeros(n, bool)
    for i in range(n):
        if parent[i] >= 0:
            has_child[parent[i]] = True
    leaves = np.flatnonzero(~has_child)
    return int(rng.choice(leaves))


def accepted_lengths(n_streams: int, max_len: int, rng: np.random.Generator) -> np.ndarray:
    """Accepted window lengths, uniform in {0..max_len} per stream."""
    return rng.integers(0, max_len + 1, size=n_streams).astype(np.int32)
