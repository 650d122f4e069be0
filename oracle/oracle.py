"""ctypes front end of the CPU oracle (TEST INFRASTRUCTURE ONLY).

The oracle is the plain C file ``fadkv_oracle.c`` in this directory: double
precision, plain loops, no code shared with the CUDA library.  Only the tests,
the smoke check and the benchmark's CPU-baseline leg may import this module.

``build()`` compiles the C file with the host C compiler into
``oracle/_build/liboracle.so``; every other function here only marshals
numpy arrays into and out of the C entry points.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fadkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

F16 = 0
F32 = 1


class _Params(C.Structure):
    _fields_ = [
        ("N", C.c_int32),
        ("d", C.c_int32),
        ("n", C.c_int32),
        ("s", C.c_int32),
        ("lambda_abs", C.c_double),
        ("lambda_rel", C.c_double),
        ("dtype", C.c_int32),
    ]


@dataclass(frozen=True)
class Params:
    N: int
    d: int
    n: int
    s: int
    lambda_abs: float = 1e-4
    lambda_rel: float = 0.20
    dtype: int = F16

    def c(self) -> _Params:
        return _Params(self.N, self.d, self.n, self.s, self.lambda_abs, self.lambda_rel, self.dtype)

    @property
    def np_dtype(self):
        return np.float16 if self.dtype == F16 else np.float32


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (idempotent)."""
    return compile_source(_SRC, _LIB_PATH, force)


def compile_source(src: str, out: str, force: bool = False) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".{os.getpid()}.tmp"
    cc = os.environ.get("CC", "cc")
    subprocess.run([cc, "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def load(path: str):
    """Load an oracle shared library and declare its entry points."""
    L = C.CDLL(path)
    P = C.POINTER
    L.oracle_encode.argtypes = [P(_Params), C.c_void_p, C.c_void_p, C.c_int32,
                                C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32]
    L.oracle_encode.restype = C.c_int
    L.oracle_adapt.argtypes = [P(_Params), C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32,
                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_double,
                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    L.oracle_adapt.restype = C.c_int
    L.oracle_adapt_append.argtypes = L.oracle_adapt.argtypes
    L.oracle_adapt_append.restype = C.c_int
    L.oracle_reconstruct.argtypes = [P(_Params), C.c_void_p, C.c_int32, C.c_void_p,
                                     C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    L.oracle_reconstruct.restype = C.c_int
    L.oracle_greedy_on_pool.argtypes = [P(_Params), C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p,
                                        C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    L.oracle_greedy_on_pool.restype = C.c_int
    L.oracle_encode_pl.argtypes = [P(_Params), C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p,
                                   C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    L.oracle_encode_pl.restype = C.c_int
    L.oracle_pack_word.argtypes = [C.c_double, C.c_int32]
    L.oracle_pack_word.restype = C.c_uint32
    L.oracle_word_coef.argtypes = [C.c_uint32]
    L.oracle_word_coef.restype = C.c_double
    L.oracle_word_id.argtypes = [C.c_uint32]
    L.oracle_word_id.restype = C.c_int32
    L.oracle_attend.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                C.c_int32, C.c_double, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_void_p, C.c_void_p, C.c_void_p]
    L.oracle_attend.restype = C.c_int
    L.oracle_half_to_double.argtypes = [C.c_uint16]
    L.oracle_half_to_double.restype = C.c_double
    L.oracle_double_to_half.argtypes = [C.c_double]
    L.oracle_double_to_half.restype = C.c_uint16
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


class Variant:
    """The same front end bound to another build of the oracle source (used
    by the tests that plant mistakes in a copy of the oracle)."""

    F16, F32 = F16, F32

    def __init__(self, path: str):
        self._L = load(path)
        import types
        mod = globals()
        for name in ("encode", "adapt", "reconstruct", "half_to_double", "double_to_half",
                     "encode_threaded", "greedy_on_pool", "encode_pl", "pack_codes", "pack_word", "word_coef", "word_id",
                     "attend"):
            fn = mod[name]
            setattr(self, name, types.FunctionType(fn.__code__, dict(mod, lib=lambda: self._L),
                                                   fn.__name__, fn.__defaults__, fn.__closure__))
        self.Params = Params


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check_store(a, p: Params, name):
    if a.dtype != p.np_dtype or not a.flags.c_contiguous:
        raise TypeError(f"{name} must be a C-contiguous {np.dtype(p.np_dtype).name} array")


@dataclass
class EncodeResult:
    idx: np.ndarray        # int32 [V][s], pick order
    coef: np.ndarray       # float64 [V][s]
    relres: np.ndarray     # float64 [V]
    pool: np.ndarray       # int32 [V][n] in (-|r|, j) order
    cut_gap: np.ndarray    # float64 [V]
    pick_gap: np.ndarray   # float64 [V][s]
    macs: int


def encode(p: Params, atoms: np.ndarray, x: np.ndarray, full_omp: bool = False) -> EncodeResult:
    """Encode the rows of ``x`` (storage precision) against ``atoms``."""
    _check_store(atoms, p, "atoms")
    _check_store(x, p, "x")
    V = x.shape[0]
    n = p.N if full_omp else p.n
    idx = np.empty((V, p.s), np.int32)
    coef = np.empty((V, p.s), np.float64)
    rel = np.empty(V, np.float64)
    pool = np.empty((V, n), np.int32)
    cut = np.empty(V, np.float64)
    gap = np.empty((V, p.s), np.float64)
    macs = C.c_int64(0)
    pc = p.c()
    rc = lib().oracle_encode(C.byref(pc), _ptr(atoms), _ptr(x), V, _ptr(idx), _ptr(coef),
                             _ptr(rel), _ptr(pool), _ptr(cut), _ptr(gap), C.addressof(macs),
                             1 if full_omp else 0)
    if rc != 0:
        raise RuntimeError(f"oracle_encode failed: {rc}")
    return EncodeResult(idx, coef, rel, pool, cut, gap, int(macs.value))


def greedy_on_pool(p: Params, atoms: np.ndarray, x: np.ndarray, pool: np.ndarray) -> EncodeResult:
    """Greedy selection + refit of each row of ``x`` over the given pool
    ([V][n] atom ids).  pool/cut_gap of the result are the inputs / NaN."""
    _check_store(atoms, p, "atoms")
    _check_store(x, p, "x")
    V = x.shape[0]
    pool = np.ascontiguousarray(pool, np.int32)
    if pool.shape != (V, p.n):
        raise ValueError("pool must be [V][n]")
    idx = np.empty((V, p.s), np.int32)
    coef = np.empty((V, p.s), np.float64)
    rel = np.empty(V, np.float64)
    gap = np.empty((V, p.s), np.float64)
    pc = p.c()
    rc = lib().oracle_greedy_on_pool(C.byref(pc), _ptr(atoms), _ptr(x), V, _ptr(pool), _ptr(idx),
                                     _ptr(coef), _ptr(rel), _ptr(gap))
    if rc != 0:
        raise RuntimeError(f"oracle_greedy_on_pool failed: {rc}")
    return EncodeResult(idx, coef, rel, pool, np.full(V, np.nan), gap, 0)


def encode_pl(p: Params, atoms: np.ndarray, x: np.ndarray) -> EncodeResult:
    """PL encode of the rows of ``x``: the s atoms of largest |r| (ties to
    the lower index), in ascending atom order, and one ridge fit over them.
    ``cut_gap`` is the relative margin of the Top-s cut; pool and pick_gap
    of the result are empty."""
    _check_store(atoms, p, "atoms")
    _check_store(x, p, "x")
    V = x.shape[0]
    idx = np.empty((V, p.s), np.int32)
    coef = np.empty((V, p.s), np.float64)
    rel = np.empty(V, np.float64)
    cut = np.empty(V, np.float64)
    macs = C.c_int64(0)
    pc = p.c()
    rc = lib().oracle_encode_pl(C.byref(pc), _ptr(atoms), _ptr(x), V, _ptr(idx), _ptr(coef),
                                _ptr(rel), _ptr(cut), C.addressof(macs))
    if rc != 0:
        raise RuntimeError(f"oracle_encode_pl failed: {rc}")
    return EncodeResult(idx, coef, rel, np.empty((V, 0), np.int32), cut,
                        np.empty((V, 0), np.float64), int(macs.value))


def encode_threaded(p: Params, atoms: np.ndarray, x: np.ndarray, threads: int,
                    coder: str = "gm") -> EncodeResult:
    """The same encode (coder "gm": greedy in the pool; "pl": encode_pl),
    with the rows of ``x`` split across host threads (ctypes releases the
    GIL during each C call)."""
    fn = encode_pl if coder == "pl" else encode
    V = x.shape[0]
    threads = max(1, min(threads, V))
    bounds = np.linspace(0, V, threads + 1).astype(int)
    parts = [None] * threads

    def run(i):
        parts[i] = fn(p, atoms, np.ascontiguousarray(x[bounds[i]:bounds[i + 1]]))

    ts = [threading.Thread(target=run, args=(i,)) for i in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return EncodeResult(
        np.concatenate([r.idx for r in parts]), np.concatenate([r.coef for r in parts]),
        np.concatenate([r.relres for r in parts]), np.concatenate([r.pool for r in parts]),
        np.concatenate([r.cut_gap for r in parts]), np.concatenate([r.pick_gap for r in parts]),
        sum(r.macs for r in parts))


@dataclass
class AdaptResult:
    repl_id: np.ndarray    # int32 [V]
    repl_coef: np.ndarray  # float64 [V]
    replaced: int
    overflow: int


def adapt(p: Params, atoms: np.ndarray, usage: np.ndarray, x: np.ndarray, idx: np.ndarray,
          coef: np.ndarray, relres: np.ndarray, delta: float, append: bool = False) -> AdaptResult:
    """Fixed-size adaptation (or, with ``append``, append-only growth into the
    free slots, usage < 0); mutates ``atoms`` and ``usage`` in place."""
    _check_store(atoms, p, "atoms")
    _check_store(x, p, "x")
    if usage.dtype != np.int32 or not usage.flags.c_contiguous:
        raise TypeError("usage must be C-contiguous int32")
    V = x.shape[0]
    idx = np.ascontiguousarray(idx, np.int32)
    coef = np.ascontiguousarray(coef, np.float64)
    relres = np.ascontiguousarray(relres, np.float64)
    rid = np.empty(V, np.int32)
    rcoef = np.empty(V, np.float64)
    rep = C.c_int64(0)
    ovf = C.c_int64(0)
    pc = p.c()
    fn = lib().oracle_adapt_append if append else lib().oracle_adapt
    rc = fn(C.byref(pc), _ptr(atoms), _ptr(usage), _ptr(x), V, _ptr(idx),
            _ptr(coef), _ptr(relres), float(delta), _ptr(rid), _ptr(rcoef),
            C.addressof(rep), C.addressof(ovf))
    if rc != 0:
        raise RuntimeError(f"oracle_adapt failed: {rc}")
    return AdaptResult(rid, rcoef, int(rep.value), int(ovf.value))


def reconstruct(p: Params, atoms: np.ndarray, idx: np.ndarray, coef: np.ndarray,
                repl_id: np.ndarray | None = None, repl_coef: np.ndarray | None = None) -> np.ndarray:
    _check_store(atoms, p, "atoms")
    idx = np.ascontiguousarray(idx, np.int32)
    coef = np.ascontiguousarray(coef, np.float64)
    V = idx.shape[0]
    if repl_id is not None:
        repl_id = np.ascontiguousarray(repl_id, np.int32)
        repl_coef = np.ascontiguousarray(repl_coef, np.float64)
    out = np.empty((V, p.d), np.float64)
    pc = p.c()
    rc = lib().oracle_reconstruct(C.byref(pc), _ptr(atoms), V, _ptr(idx), _ptr(coef),
                                  _ptr(repl_id), _ptr(repl_coef), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"oracle_reconstruct failed: {rc}")
    return out


def pack_codes(idx: np.ndarray, coef: np.ndarray, repl_id: np.ndarray | None = None,
               repl_coef: np.ndarray | None = None) -> np.ndarray:
    """[..., s] codes (+ optional [...] replacement terms) -> [..., s+1]
    packed uint32 words (coefficient rounded to 11 significant bits, id in
    the low 13 bits)."""
    idx = np.asarray(idx)
    coef = np.asarray(coef, np.float64)
    lead = idx.shape[:-1]
    s = idx.shape[-1]
    out = np.zeros(lead + (s + 1,), np.uint32)
    L = lib()
    for pos in np.ndindex(*lead):
        for k in range(s):
            out[pos + (k,)] = L.oracle_pack_word(float(coef[pos + (k,)]), int(idx[pos + (k,)]))
        if repl_id is not None:
            out[pos + (s,)] = L.oracle_pack_word(float(repl_coef[pos]), int(repl_id[pos]))
    return out


def pack_word(coef: float, idx: int) -> int:
    """One packed word (see pack_codes)."""
    return lib().oracle_pack_word(float(coef), int(idx))


def word_coef(w: int) -> float:
    return lib().oracle_word_coef(int(w))


def word_id(w: int) -> int:
    return lib().oracle_word_id(int(w))


def attend(dict_k: np.ndarray, dict_v: np.ndarray, cache_k: np.ndarray, cache_v: np.ndarray,
           lengths: np.ndarray, q: np.ndarray, scale: float | None = None) -> np.ndarray:
    """Decode attention of one layer over packed caches [B][Hkv][Tmax][s+1];
    q [B][Hq][d]; returns [B][Hq][d] float64."""
    N, d = dict_k.shape
    B, Hkv, Tmax, W = cache_k.shape
    Hq = q.shape[1]
    dtype = F16 if dict_k.dtype == np.float16 else F32
    dict_k = np.ascontiguousarray(dict_k)
    dict_v = np.ascontiguousarray(dict_v, dict_k.dtype)
    cache_k = np.ascontiguousarray(cache_k, np.uint32)
    cache_v = np.ascontiguousarray(cache_v, np.uint32)
    lengths = np.ascontiguousarray(lengths, np.int32)
    q = np.ascontiguousarray(q, np.float64)
    out = np.empty((B, Hq, d), np.float64)
    sc = 1.0 / np.sqrt(d) if scale is None else scale
    rc = lib().oracle_attend(B, Hq, Hkv, d, W - 1, N, Tmax, dtype, float(sc), _ptr(dict_k), _ptr(dict_v),
                             _ptr(cache_k), _ptr(cache_v), _ptr(lengths), _ptr(q), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"oracle_attend failed: {rc}")
    return out


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(bits)


def double_to_half(v: float) -> int:
    return lib().oracle_double_to_half(v)
