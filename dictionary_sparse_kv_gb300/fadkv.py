"""Thin Python binding of the FAD-KV C ABI (include/fadkv.h).

Only marshals arguments: every step of encode / adapt / reconstruct runs in
the CUDA library ``_build/libfadkv.so``.  There is no fallback: if the library
is missing, importing the functions raises ``FadkvLibraryMissing``.

Functions carry the C names without the ``fadkv_`` prefix.  Device arrays are
passed as torch CUDA tensors (their ``data_ptr()``) or raw integer addresses;
the stream defaults to torch's current stream on the tensors' device.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libfadkv.so")

F16 = 0
F32 = 1
STATS_FIELDS = 8
STATS_NAMES = ("encoded", "replaced", "flagged", "overflow", "nonfinite", "topn_slow_path", "status", "reserved")
DEV_NONFINITE_INPUT = 0x1
DEV_NOT_SPD = 0x2
MAX_DICTS = 256

STATUS = {0: "FADKV_OK", 1: "FADKV_ERR_INVALID_ARG", 2: "FADKV_ERR_UNSUPPORTED", 3: "FADKV_ERR_SEQUENCE",
          4: "FADKV_ERR_CUDA", 5: "FADKV_ERR_WORKSPACE"}


class FadkvLibraryMissing(RuntimeError):
    pass


class FadkvError(RuntimeError):
    def __init__(self, func: str, status: int, detail: str = ""):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{func} -> {self.name}" + (f": {detail}" if detail else ""))


class Params(C.Structure):
    _fields_ = [
        ("num_dicts", C.c_int32),
        ("N", C.c_int32),
        ("d", C.c_int32),
        ("n", C.c_int32),
        ("s", C.c_int32),
        ("lambda_abs", C.c_float),
        ("lambda_rel", C.c_float),
        ("dtype", C.c_int32),
        ("max_batch", C.c_int32),
    ]


class AttnParams(C.Structure):
    _fields_ = [
        ("layers", C.c_int32),
        ("B", C.c_int32),
        ("Hq", C.c_int32),
        ("Hkv", C.c_int32),
        ("d", C.c_int32),
        ("N", C.c_int32),
        ("s", C.c_int32),
        ("Tmax", C.c_int32),
        ("dtype", C.c_int32),
        ("scale", C.c_float),
        ("dict_stride", C.c_int64),
        ("cache_stride", C.c_int64),
    ]


def params(num_dicts, N, d, n, s, dtype=F16, max_batch=1, lambda_abs=1e-4, lambda_rel=0.20) -> Params:
    """Handle parameters; the ridge defaults are Table 5's 1e-4 + 0.20 diag(G)."""
    return Params(num_dicts, N, d, n, s, lambda_abs, lambda_rel, dtype, max_batch)


_lib = None
_lock = threading.Lock()

_SIGS = {
    "fadkv_abi_version": ([], C.c_int32),
    "fadkv_status_string": ([C.c_int], C.c_char_p),
    "fadkv_last_error": ([], C.c_char_p),
    "fadkv_workspace_bytes": ([C.POINTER(Params), C.POINTER(C.c_size_t)], C.c_int),
    "fadkv_dict_create": ([C.POINTER(Params), C.c_void_p, C.c_void_p, C.POINTER(C.c_float), C.c_void_p,
                           C.c_size_t, C.POINTER(C.c_void_p)], C.c_int),
    "fadkv_dict_destroy": ([C.c_void_p], C.c_int),
    "fadkv_dict_refresh": ([C.c_void_p, C.c_void_p], C.c_int),
    "fadkv_encode": ([C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p],
                     C.c_int),
    "fadkv_encode_pl": ([C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p],
                        C.c_int),
    "fadkv_adapt": ([C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                     C.c_void_p, C.c_void_p], C.c_int),
    "fadkv_adapt_append": ([C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                            C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "fadkv_adapt_noalloc": ([C.POINTER(Params), C.c_void_p, C.c_void_p, C.POINTER(C.c_float), C.c_void_p,
                             C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                             C.c_void_p], C.c_int),
    "fadkv_reconstruct": ([C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                           C.c_void_p], C.c_int),
    "fadkv_dict_stats": ([C.c_void_p, C.POINTER(C.c_int64), C.c_void_p], C.c_int),
    "fadkv_debug_pool": ([C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "fadkv_debug_scores": ([C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p], C.c_int),
    "fadkv_debug_wait_limit": ([C.c_void_p, C.c_uint64], C.c_int),
    "fadkv_debug_wait_probe": ([C.c_void_p, C.c_uint64, C.c_void_p], C.c_int),
    "fadkv_store_codes": ([C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                           C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p], C.c_int),
    "fadkv_attend": ([C.POINTER(AttnParams), C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                      C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "fadkv_attend_workspace_bytes": ([C.POINTER(AttnParams), C.POINTER(C.c_size_t)], C.c_int),
    "fadkv_profile_enable": ([C.c_void_p, C.c_int32], C.c_int),
    "fadkv_profile_select": ([C.c_void_p, C.c_uint32], C.c_int),
    "fadkv_profile_read": ([C.c_void_p, C.POINTER(C.c_int64), C.POINTER(C.c_double), C.c_int32], C.c_int),
}

PROFILE_KERNELS = 8
KERNEL_NAMES = ("screen", "topn", "greedy", "adapt", "reconstruct", "gram", "k6", "k7")


def lib():
    """The loaded CUDA library (raises FadkvLibraryMissing if not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise FadkvLibraryMissing(
                    f"{LIB_PATH} is not built; run `python -m dictionary_sparse_kv_gb300.build`")
            L = C.CDLL(LIB_PATH)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _addr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, *tensors):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    dev = next((t.device for t in tensors if hasattr(t, "device") and t.device.type == "cuda"), None)
    return torch.cuda.current_stream(dev).cuda_stream


def _check(func, rc):
    if rc != 0:
        raise FadkvError(func, rc, lib().fadkv_last_error().decode() if rc == 4 else "")


def abi_version() -> int:
    return lib().fadkv_abi_version()


def status_string(status: int) -> str:
    return lib().fadkv_status_string(status).decode()


def last_error() -> str:
    return lib().fadkv_last_error().decode()


def workspace_bytes(p: Params) -> int:
    out = C.c_size_t(0)
    _check("fadkv_workspace_bytes", lib().fadkv_workspace_bytes(C.byref(p), C.byref(out)))
    return out.value


def dict_create(p: Params, atoms, usage, delta, workspace, workspace_bytes_: int) -> int:
    arr = (C.c_float * len(delta))(*[float(v) for v in delta])
    h = C.c_void_p(0)
    _check("fadkv_dict_create", lib().fadkv_dict_create(C.byref(p), _addr(atoms), _addr(usage), arr,
                                                         _addr(workspace), workspace_bytes_, C.byref(h)))
    return h.value


def dict_destroy(h: int) -> None:
    _check("fadkv_dict_destroy", lib().fadkv_dict_destroy(h))


def dict_refresh(h: int, stream=None) -> None:
    """Rebuild the handle's Gram matrices after atoms changed outside its adapt calls."""
    _check("fadkv_dict_refresh", lib().fadkv_dict_refresh(h, stream if isinstance(stream, int) else
                                                           (stream.cuda_stream if stream is not None
                                                            else _default_stream())))


def _default_stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def encode(h: int, x, V: int, idx, coef, relres, stream=None) -> None:
    st = _stream(stream, x, idx)
    _check("fadkv_encode", lib().fadkv_encode(h, _addr(x), V, _addr(idx), _addr(coef), _addr(relres), st))


def encode_pl(h: int, x, V: int, idx, coef, relres, stream=None) -> None:
    """PL encode: Top-s atoms (ascending ids) and one ridge fit."""
    st = _stream(stream, x, idx)
    _check("fadkv_encode_pl", lib().fadkv_encode_pl(h, _addr(x), V, _addr(idx), _addr(coef), _addr(relres), st))


def adapt(h: int, x, V: int, idx, coef, relres, repl_id, repl_coef, stream=None) -> None:
    st = _stream(stream, x, idx)
    _check("fadkv_adapt", lib().fadkv_adapt(h, _addr(x), V, _addr(idx), _addr(coef), _addr(relres),
                                            _addr(repl_id), _addr(repl_coef), st))


def adapt_append(h: int, x, V: int, idx, coef, relres, repl_id, repl_coef, stream=None) -> None:
    """Append-only growth into the free slots (usage < 0)."""
    st = _stream(stream, x, idx)
    _check("fadkv_adapt_append", lib().fadkv_adapt_append(h, _addr(x), V, _addr(idx), _addr(coef), _addr(relres),
                                                          _addr(repl_id), _addr(repl_coef), st))


def adapt_noalloc(p: Params, atoms, usage, delta, x, V: int, idx, coef, relres, repl_id, repl_coef,
                  stream=None) -> None:
    """Handle-free adaptation on the library's static scratch (no allocation)."""
    arr = (C.c_float * len(delta))(*[float(v) for v in delta])
    st = _stream(stream, atoms, x)
    rc = lib().fadkv_adapt_noalloc(C.byref(p), _addr(atoms), _addr(usage), arr, _addr(x), V, _addr(idx),
                                   _addr(coef), _addr(relres), _addr(repl_id), _addr(repl_coef), st)
    if rc != 0:
        raise FadkvError("fadkv_adapt_noalloc", rc, last_error())


def store_codes(G: int, B: int, H: int, s: int, N: int, idx, coef, repl_id, repl_coef, pos, cache, Tmax: int,
                stream=None) -> None:
    """Packed words of one step's codes into caches [G][B][H][Tmax][s+1] at pos[b]."""
    st = _stream(stream, idx, cache)
    _check("fadkv_store_codes", lib().fadkv_store_codes(G, B, H, s, N, _addr(idx), _addr(coef), _addr(repl_id),
                                                        _addr(repl_coef), _addr(pos), _addr(cache), Tmax, st))


def attend_workspace_bytes(p: AttnParams) -> int:
    out = C.c_size_t(0)
    _check("fadkv_attend_workspace_bytes", lib().fadkv_attend_workspace_bytes(C.byref(p), C.byref(out)))
    return out.value


def attend(p: AttnParams, dict_k, dict_v, cache_k, cache_v, lengths, q, out, workspace=None,
           stream=None) -> None:
    """Decode attention over packed K/V codes (see fadkv_attend).  Without
    a workspace one is allocated here (a torch tensor on q's device)."""
    need = attend_workspace_bytes(p)
    if workspace is None and need > 0:
        import torch
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    nbytes = 0 if workspace is None else (workspace.numel() * workspace.element_size()
                                          if hasattr(workspace, "numel") else need)
    st = _stream(stream, q, out)
    _check("fadkv_attend", lib().fadkv_attend(C.byref(p), _addr(dict_k), _addr(dict_v), _addr(cache_k),
                                              _addr(cache_v), _addr(lengths), _addr(q), _addr(out),
                                              _addr(workspace), nbytes, st))


def reconstruct(h: int, V: int, idx, coef, repl_id, repl_coef, xhat, stream=None) -> None:
    st = _stream(stream, idx, xhat)
    _check("fadkv_reconstruct", lib().fadkv_reconstruct(h, V, _addr(idx), _addr(coef), _addr(repl_id),
                                                        _addr(repl_coef), _addr(xhat), st))


def dict_stats(h: int, num_dicts: int, stream=None):
    buf = (C.c_int64 * (num_dicts * STATS_FIELDS))()
    st = stream if isinstance(stream, int) else (stream.cuda_stream if stream is not None else None)
    if st is None:
        import torch
        st = torch.cuda.current_stream().cuda_stream
    _check("fadkv_dict_stats", lib().fadkv_dict_stats(h, buf, st))
    return [dict(zip(STATS_NAMES, buf[g * STATS_FIELDS:(g + 1) * STATS_FIELDS])) for g in range(num_dicts)]


def debug_pool(h: int, x, V: int, pool, pool_r=None, stream=None) -> None:
    st = _stream(stream, x, pool)
    _check("fadkv_debug_pool", lib().fadkv_debug_pool(h, _addr(x), V, _addr(pool), _addr(pool_r), st))


def debug_scores(h: int, x, V: int, scores, stream=None) -> None:
    st = _stream(stream, x, scores)
    _check("fadkv_debug_scores", lib().fadkv_debug_scores(h, _addr(x), V, _addr(scores), st))


def debug_wait_limit(h: int, limit_ns: int) -> None:
    """Test hook: limit of the screening pipeline's waits (0 = default)."""
    _check("fadkv_debug_wait_limit", lib().fadkv_debug_wait_limit(h, int(limit_ns)))


def debug_wait_probe(h: int, limit_ns: int, stream=None) -> None:
    """Test hook: a wait that nothing completes, limited to limit_ns."""
    st = stream if isinstance(stream, int) else (stream.cuda_stream if stream is not None else _default_stream())
    _check("fadkv_debug_wait_probe", lib().fadkv_debug_wait_probe(h, int(limit_ns), st))


def profile_enable(h: int, enable: bool = True) -> None:
    _check("fadkv_profile_enable", lib().fadkv_profile_enable(h, 1 if enable else 0))


def profile_select(h: int, classes=None) -> None:
    """Kernel classes bracketed with events while profiling (names from
    KERNEL_NAMES or class numbers); None selects all."""
    if classes is None:
        mask = 0xFFFFFFFF
    else:
        mask = 0
        for c in classes:
            mask |= 1 << (KERNEL_NAMES.index(c) if isinstance(c, str) else int(c))
    _check("fadkv_profile_select", lib().fadkv_profile_select(h, C.c_uint32(mask)))


def profile_read(h: int, reset: bool = False):
    """{kernel class: (launches, device ms)} since the last reset."""
    n = (C.c_int64 * PROFILE_KERNELS)()
    ms = (C.c_double * PROFILE_KERNELS)()
    _check("fadkv_profile_read", lib().fadkv_profile_read(h, n, ms, 1 if reset else 0))
    return {KERNEL_NAMES[i]: (int(n[i]), float(ms[i])) for i in range(PROFILE_KERNELS) if n[i] or ms[i]}


# ---------------------------------------------------------------------------
# Convenience owner of the device memory of one handle (torch allocates it).
# ---------------------------------------------------------------------------

@dataclass
class Codes:
    idx: "object"       # int32 [G][V][s]
    coef: "object"      # float32 [G][V][s]
    relres: "object"    # float32 [G][V]
    repl_id: "object"   # int32 [G][V]
    repl_coef: "object"  # float32 [G][V]
    buf: "object" = None  # int32 words holding all five back to back (one copy moves every code)


class Dictionary:
    """G dictionaries of one shape plus their usage counts and workspace,
    allocated with torch on one CUDA device, behind one C-ABI handle."""

    def __init__(self, atoms, usage, delta, n: int, s: int, max_batch: int,
                 lambda_abs: float = 1e-4, lambda_rel: float = 0.20):
        import torch
        if atoms.dim() != 3 or usage.dim() != 2:
            raise ValueError("atoms must be [G][N][d] and usage [G][N]")
        self.atoms = atoms.contiguous()
        self.usage = usage.contiguous()
        G, N, d = self.atoms.shape
        dt = F16 if self.atoms.dtype == torch.float16 else F32
        self.p = params(G, N, d, n, s, dt, max_batch, lambda_abs, lambda_rel)
        self.G, self.N, self.d, self.n, self.s = G, N, d, n, s
        self.max_batch = max_batch
        nbytes = workspace_bytes(self.p)
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=self.atoms.device)
        self.delta = [float(v) for v in delta]
        self.h = dict_create(self.p, self.atoms, self.usage, self.delta, self.workspace, nbytes)

    def close(self):
        if getattr(self, "h", None):
            dict_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_codes(self, V: int) -> Codes:
        import torch
        dev = self.atoms.device
        G, s = self.G, self.s
        # the five arrays as slices of one buffer, each starting on a
        # 256-byte boundary
        sizes = [G * V * s, G * V * s, G * V, G * V, G * V]
        offs, o = [], 0
        for n_ in sizes:
            offs.append(o)
            o += (n_ + 63) // 64 * 64
        buf = torch.empty(max(o, 1), dtype=torch.int32, device=dev)
        part = lambda i, shape: buf[offs[i]:offs[i] + sizes[i]].view(shape)
        return Codes(part(0, (G, V, s)), part(1, (G, V, s)).view(torch.float32), part(2, (G, V)).view(torch.float32),
                     part(3, (G, V)), part(4, (G, V)).view(torch.float32), buf)

    def refresh(self, stream=None):
        """Rebuild the Gram matrices (after changing self.atoms in place)."""
        dict_refresh(self.h, stream if stream is not None else _stream(None, self.atoms))

    def encode(self, x, codes: Codes, stream=None):
        V = x.shape[1]
        encode(self.h, x, V, codes.idx, codes.coef, codes.relres, stream)

    def encode_pl(self, x, codes: Codes, stream=None):
        V = x.shape[1]
        encode_pl(self.h, x, V, codes.idx, codes.coef, codes.relres, stream)

    def adapt(self, x, codes: Codes, stream=None):
        V = x.shape[1]
        adapt(self.h, x, V, codes.idx, codes.coef, codes.relres, codes.repl_id, codes.repl_coef, stream)

    def adapt_append(self, x, codes: Codes, stream=None):
        V = x.shape[1]
        adapt_append(self.h, x, V, codes.idx, codes.coef, codes.relres, codes.repl_id, codes.repl_coef, stream)

    def reconstruct(self, codes: Codes, xhat, with_replacement: bool = True, stream=None):
        V = codes.idx.shape[1]
        reconstruct(self.h, V, codes.idx, codes.coef, codes.repl_id if with_replacement else None,
                    codes.repl_coef if with_replacement else None, xhat, stream)

    def step(self, x, codes: Codes, xhat=None, stream=None, coder: str = "gm"):
        """One decode step: encode (coder "gm": greedy in the pool, "pl":
        Top-s and one fit), adapt and (optionally) reconstruct."""
        if coder == "pl":
            self.encode_pl(x, codes, stream)
        elif coder == "gm":
            self.encode(x, codes, stream)
        else:
            raise ValueError(f"unknown coder {coder!r}")
        self.adapt(x, codes, stream)
        if xhat is not None:
            self.reconstruct(codes, xhat, True, stream)

    def stats(self, stream=None):
        return dict_stats(self.h, self.G, stream)

    def scores(self, x, stream=None):
        import torch
        V = x.shape[1]
        out = torch.empty((self.G, V, self.N), dtype=torch.float32, device=x.device)
        debug_scores(self.h, x, V, out, stream)
        return out

    def pool(self, x, stream=None):
        import torch
        V = x.shape[1]
        pool = torch.empty((self.G, V, self.n), dtype=torch.int32, device=x.device)
        pr = torch.empty((self.G, V, self.n), dtype=torch.float32, device=x.device)
        debug_pool(self.h, x, V, pool, pr, stream)
        return pool, pr
