"""Seeded synthetic inputs for the FAD-KV per-token KV encoding path.

This module only draws random data: dictionaries, inactive-atom sets and the
key/value head-vectors to encode. It holds none of the method's arithmetic
(no screening, selection, refit or replacement), so both the CUDA path's tests
and the CPU oracle's tests may use it.

Every draw goes through numpy's PCG64 generator seeded from a tuple of
integers, so a (workload, dictionary, step) triple always yields the same
arrays on every machine.

Shapes follow the workloads described for FAD-KV in "FAD-KV: Adaptive
Dictionary KV Caching for Efficient Reasoning Decoding" (Table 5 hyper-
parameters: N = 4096 / 8192 atoms, s = 8 / 16, n = 256 / 512; head dimension
128 for the Llama-3.2-3B / Llama-3.1-8B KV heads).  No model KV data is
available, so:

* atoms are i.i.d. Gaussian vectors scaled to unit norm, then stored in the
  dictionary precision (binary16, or binary32 for the tiny check);
* an input is a sparse mixture of ``k`` distinct source atoms with
  heavy-tailed (Student-t, nu = 3) coefficients plus an off-dictionary
  Gaussian component whose norm is ``off_frac`` times the mixture's norm
  (or, for the tiny check, N(0,1) coefficients plus N(0, sigma^2) noise).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "generator",
    "make_dictionary",
    "make_usage",
    "make_sparse_inputs",
    "make_tiny_inputs",
    "DriftingSources",
]


def generator(*seed: int) -> np.random.Generator:
    """PCG64 generator for an integer seed tuple (order matters)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(s) for s in seed])))


def _store(a: np.ndarray, dtype) -> np.ndarray:
    """Round a float64 array once to the storage precision (RNE)."""
    return np.ascontiguousarray(a.astype(dtype))


def make_dictionary(N: int, d: int, dtype=np.float16, *seed: int) -> np.ndarray:
    """[N][d] atoms: i.i.d. N(0,1) entries, each row scaled to unit norm
    in float64, then rounded once to ``dtype``."""
    g = generator(*seed)
    a = g.standard_normal((N, d))
    a /= np.linalg.norm(a, axis=1, keepdims=True)
    return _store(a, dtype)


def make_usage(N: int, n_inactive: int, *seed: int) -> np.ndarray:
    """int32[N] usage counts: ``n_inactive`` atoms chosen by a seeded
    permutation start at 0, every other atom starts at 1."""
    g = generator(*seed)
    usage = np.ones(N, dtype=np.int32)
    if n_inactive > 0:
        usage[g.permutation(N)[:n_inactive]] = 0
    return usage


def _distinct_rows(g: np.random.Generator, M: int, V: int, k: int) -> np.ndarray:
    """[V][k] row ids, distinct within each row, uniform over [0, M).

    Draws with replacement, then redraws any row holding a repeat until it
    has none (deterministic for a given generator state)."""
    if k > M:
        raise ValueError("need at least k source atoms")
    rows = g.integers(0, M, size=(V, k))
    srt = np.sort(rows, axis=1)
    bad = np.nonzero((srt[:, 1:] == srt[:, :-1]).any(axis=1))[0] if k > 1 else []
    for v in bad:
        rows[v] = g.choice(M, size=k, replace=False)
    return rows


def make_sparse_inputs(sources: np.ndarray, V: int, k: int, *seed: int,
                       off_frac: float = 0.05, dtype=np.float16) -> np.ndarray:
    """[V][d] vectors x = sum_i b_i s_i + off_frac * ||sum_i b_i s_i|| * g/||g||.

    ``sources`` is a [M][d] array of candidate atoms (any precision); each
    vector mixes ``k`` distinct rows drawn uniformly, with b_i ~ Student-t(3),
    and g ~ N(0, I).  Built in float64, rounded once to ``dtype``.
    """
    g = generator(*seed)
    src = np.asarray(sources, dtype=np.float64)
    M, d = src.shape
    rows = _distinct_rows(g, M, V, k)
    b = g.standard_t(3.0, size=(V, k))
    noise = g.standard_normal((V, d))
    mix = np.einsum("vk,vkd->vd", b, src[rows])
    mn = np.linalg.norm(mix, axis=1, keepdims=True)
    nn = np.linalg.norm(noise, axis=1, keepdims=True)
    x = mix + off_frac * mn * noise / np.where(nn > 0, nn, 1.0)
    return _store(x, dtype)


def make_tiny_inputs(atoms: np.ndarray, V: int, k: int, *seed: int,
                     sigma: float = 0.01, dtype=np.float32) -> np.ndarray:
    """[V][d] vectors: an exact k-sparse combination of random atoms with
    N(0,1) coefficients plus N(0, sigma^2) noise in every coordinate."""
    g = generator(*seed)
    src = np.asarray(atoms, dtype=np.float64)
    M, d = src.shape
    rows = _distinct_rows(g, M, V, k)
    b = g.standard_normal((V, k))
    x = np.einsum("vk,vkd->vd", b, src[rows]) + sigma * g.standard_normal((V, d))
    return _store(x, dtype)


class DriftingSources:
    """Generating subspace that drifts during decoding.

    Starts as a given set of source atoms; every ``period`` steps a fraction
    ``frac`` of the sources is replaced by fresh random unit vectors (drawn
    from the seed tuple and the epoch number).
    """

    def __init__(self, initial: np.ndarray, period: int = 128, frac: float = 0.10, *seed: int):
        self.period = int(period)
        self.frac = float(frac)
        self.seed = tuple(int(s) for s in seed)
        self._epoch = 0
        self._src = np.array(initial, dtype=np.float64, copy=True)

    def sources_at(self, step: int) -> np.ndarray:
        epoch = step // self.period
        while self._epoch < epoch:
            self._epoch += 1
            g = generator(*self.seed, self._epoch)
            M, d = self._src.shape
            m = max(1, int(round(self.frac * M)))
            rows = g.choice(M, size=m, replace=False)
            fresh = g.standard_normal((m, d))
            fresh /= np.linalg.norm(fresh, axis=1, keepdims=True)
            self._src[rows] = fresh
        return self._src


# ---------------------------------------------------------------------------
# Named workloads: shapes and input recipes of the FAD-KV decode / prefill
# settings (Table 5 shapes; Llama-3.2-3B: 28 layers, Llama-3.1-8B: 32 layers,
# 8 KV heads, head dimension 128).  Dictionary g = 2*layer + {0: key, 1: value}.
# ---------------------------------------------------------------------------

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    G: int                 # dictionaries (layers x {K, V})
    N: int
    d: int
    n: int
    s: int
    V: int                 # vectors per dictionary per step
    steps: int
    dtype: type = np.float16
    inactive: float = 0.30           # initial inactive fraction (or count if >= 1)
    kind: str = "mixture"            # "mixture" (Student-t + off-dictionary part) or "tiny"
    off_frac: float = 0.05
    sigma: float = 0.01
    drift_period: int = 0            # >0: sources drift every drift_period steps
    drift_frac: float = 0.10
    seed: int = 0
    deltas: tuple = field(default=())

    def delta(self, g: int) -> float:
        if self.deltas:
            return self.deltas[g]
        return 0.50 if g % 2 == 0 else 0.70   # Table 5: key 0.50, value 0.70

    @property
    def n_inactive(self) -> int:
        return int(self.inactive) if self.inactive >= 1 else int(round(self.inactive * self.N))


WORKLOADS = {
    # d=64, N=512 fp32, n=32, s=4, 256 vectors, 16 inactive atoms, delta 0.5
    "tiny": Workload("tiny", 1, 512, 64, 32, 4, 256, 1, np.float32, inactive=16, kind="tiny",
                     deltas=(0.5,)),
    # Llama-3.2-3B decode step: 28 layers x {K,V}, 8 KV heads x 16 sequences
    "decode_3b": Workload("decode_3b", 56, 4096, 128, 256, 8, 128, 1024, seed=2),
    # Llama-3.2-3B prefill at 16K context: 16384 tokens x 8 heads per dictionary
    "prefill_3b_16k": Workload("prefill_3b_16k", 2, 4096, 128, 256, 8, 131072, 1, seed=3),
    # Llama-3.1-8B decode step: 32 layers x {K,V}, 8 KV heads x 64 sequences
    "decode_8b": Workload("decode_8b", 64, 8192, 128, 512, 16, 512, 1024, seed=4),
    # adaptation stress: one K and one V dictionary, 8 heads x 32 sequences,
    # generating subspace drifts every 128 steps (10% of sources replaced)
    "adapt_stress": Workload("adapt_stress", 2, 4096, 128, 256, 8, 256, 2048, seed=5,
                             drift_period=128, drift_frac=0.10),
}


class WorkloadData:
    """Initial dictionaries, usage counts and per-step inputs of a workload,
    restricted to a subset of its dictionaries if asked."""

    def __init__(self, w: Workload, dicts=None):
        self.w = w
        self.dicts = list(range(w.G)) if dicts is None else list(dicts)
        self.atoms = np.stack([make_dictionary(w.N, w.d, w.dtype, w.seed, 1, g) for g in self.dicts])
        self.usage = np.stack([make_usage(w.N, w.n_inactive, w.seed, 2, g) for g in self.dicts])
        if w.kind == "tiny":
            self._sources = [self.atoms[i] for i in range(len(self.dicts))]
        else:
            self._sources = [self.atoms[i][self.usage[i] > 0] for i in range(len(self.dicts))]
        self._drift = None
        if w.drift_period > 0:
            self._drift = [DriftingSources(self._sources[i], w.drift_period, w.drift_frac, w.seed, 3, g)
                           for i, g in enumerate(self.dicts)]

    def deltas(self):
        return [self.w.delta(g) for g in self.dicts]

    def inputs(self, step: int, V: int | None = None) -> np.ndarray:
        """[len(dicts)][V][d] inputs of decode step ``step``."""
        w = self.w
        V = w.V if V is None else V
        out = []
        for i, g in enumerate(self.dicts):
            src = self._drift[i].sources_at(step) if self._drift else self._sources[i]
            if w.kind == "tiny":
                out.append(make_tiny_inputs(src, V, w.s, w.seed, 4, g, step, sigma=w.sigma, dtype=w.dtype))
            else:
                out.append(make_sparse_inputs(src, V, w.s, w.seed, 4, g, step, off_frac=w.off_frac,
                                              dtype=w.dtype))
        return np.ascontiguousarray(np.stack(out))
