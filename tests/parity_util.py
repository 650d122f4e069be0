"""Comparison of the CUDA library with the CPU oracle on the same inputs.

Tolerances (the spec of this library):
  * pool ids, selected ids and replacement ids are compared exactly, except
    for vectors the oracle itself shows to sit on a near tie: the relative
    gap at the Top-n cut, (|r|_(n) - |r|_(n+1)) / |r|_(n), below 1e-5, or a
    greedy step whose best and runner-up correlations differ by less than
    1e-5 relative.  fp32 accumulation cannot order such pairs reliably;
  * coefficients: ||c_gpu - c_oracle|| <= 1e-3 ||c_oracle|| per vector, and
    element by element |c_gpu,i - c_oracle,i| <= 1e-3 |c_oracle,i| for every
    coefficient with |c_oracle,i| >= 1e-2 ||c_oracle|| (smaller ones carry
    the conditioning of the refit and are held by the norm-wise bound);
  * relres: |rho_gpu - rho_oracle| <= 1e-3 rho_oracle;
  * replaced atoms: every element within one binary16 (or binary32) ulp of
    the oracle's rounding (the GPU rounds an fp32 value, the oracle a double);
  * reconstruction: ||xhat_gpu - xhat_oracle|| <= 1e-5 ||xhat_oracle|| + 1e-6.
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import numpy as np

from oracle import oracle as O

CUT_GAP = 1e-5
PICK_GAP = 1e-5
COEF_TOL = 1e-3
RELRES_TOL = 1e-3
XHAT_TOL = 1e-5
COEF_FLOOR = 1e-2       # element-wise check for |c_i| >= COEF_FLOOR * ||c||
MAX_EXEMPT_FRAC = 0.05  # vectors on a near tie left unchecked, at most (or 2)
THREADS = max(1, min(16, os.cpu_count() or 1))


def oparams(w, dtype=None):
    dt = w.dtype if dtype is None else dtype
    return O.Params(w.N, w.d, w.n, w.s, 1e-4, 0.20, O.F16 if dt == np.float16 else O.F32)


@dataclass
class EncodeReport:
    checked: int
    exempt: int
    mismatched_idx: list
    worst_coef: float
    worst_relres: float
    worst_coef_elem: float = 0.0    # worst |dc_i|/|c_i| over |c_i| >= COEF_FLOOR ||c||
    worst_coef_elem_any: float = 0.0   # the same over every nonzero c_i (reported only)


def exempt_mask(res: O.EncodeResult) -> np.ndarray:
    return (res.cut_gap < CUT_GAP) | (res.pick_gap.min(axis=1) < PICK_GAP)


def check_cut_tie(p, atoms, x, res, gpu_pool, v):
    """A vector on a near tie at the Top-n cut: the GPU pool may differ from
    the oracle's only by atoms inside the tie band (|r| within CUT_GAP of
    the cut value), and the oracle's greedy run on the GPU's pool is then the
    unique answer.  Returns the oracle result on the GPU pool (or None if
    that run itself sits on a greedy near tie)."""
    r = np.abs(atoms.astype(np.float64) @ x[v].astype(np.float64))
    cut = r[res.pool[v][-1]]
    diff = set(gpu_pool[v].tolist()) ^ set(res.pool[v].tolist())
    for j in diff:
        assert abs(r[j] - cut) <= 2 * CUT_GAP * cut, f"pool atom {j} outside the tie band"
    alt = O.greedy_on_pool(p, atoms, np.ascontiguousarray(x[v:v + 1]), gpu_pool[v:v + 1])
    if alt.pick_gap.min() < PICK_GAP:
        return None
    return alt


def compare_encode(res: O.EncodeResult, idx, coef, relres, gpu_pool=None, p=None, atoms=None,
                   x=None) -> EncodeReport:
    """res: oracle result for V vectors; idx/coef/relres: GPU arrays [V]...
    With gpu_pool/p/atoms/x given, vectors on a near tie at the Top-n cut are
    checked against the oracle's greedy run on the GPU's pool instead of
    being skipped.  Vectors off any near tie are compared all at once."""
    ex = exempt_mask(res)
    idx = np.asarray(idx)
    coef = np.asarray(coef).astype(np.float64)
    relres = np.asarray(relres).astype(np.float64)
    worst_c = worst_r = worst_e = worst_a = 0.0
    # vectors on no near tie: ids exact, then the tolerances
    ok = ~ex
    same = np.all(idx == res.idx, axis=1)
    bad = [int(v) for v in np.nonzero(ok & ~same)[0]]
    nonfinite = ok & same & (res.idx[:, 0] < 0)
    assert np.all(np.isnan(relres[nonfinite])), "a non-finite input must give relres = NaN"
    chk = ok & same & (res.idx[:, 0] >= 0)
    if chk.any():
        co = res.coef[chk]
        cn = np.linalg.norm(co, axis=1)
        dcv = np.abs(coef[chk] - co)
        dc = np.linalg.norm(dcv, axis=1)
        worst_c = float(np.max(np.where(cn > 0, dc / np.where(cn > 0, cn, 1.0), dc)))
        big = (np.abs(co) >= COEF_FLOOR * cn[:, None]) & (cn[:, None] > 0)
        if big.any():
            worst_e = float(np.max(dcv[big] / np.abs(co[big])))
        nz = co != 0
        if nz.any():
            worst_a = float(np.max(dcv[nz] / np.abs(co[nz])))
        ro = res.relres[chk]
        dr = np.abs(relres[chk] - ro)
        worst_r = float(np.max(np.where(ro > 0, dr / np.where(ro > 0, ro, 1.0), dr)))
    # vectors on a near tie at the cut: checked on the GPU's pool
    for v in np.nonzero(ex)[0]:
        if gpu_pool is None or res.pick_gap[v].min() < PICK_GAP or res.idx[v][0] < 0:
            continue
        alt = check_cut_tie(p, atoms, x, res, gpu_pool, v)
        if alt is None:
            continue
        one = O.EncodeResult(alt.idx, alt.coef, alt.relres, alt.pool, np.full(1, np.inf), alt.pick_gap, 0)
        sub = compare_encode(one, idx[v:v + 1], coef[v:v + 1], relres[v:v + 1])
        bad += [int(v)] if sub.mismatched_idx else []
        worst_c = max(worst_c, sub.worst_coef)
        worst_r = max(worst_r, sub.worst_relres)
        worst_e = max(worst_e, sub.worst_coef_elem)
        worst_a = max(worst_a, sub.worst_coef_elem_any)
        ex[v] = False
    return EncodeReport(len(ex) - int(ex.sum()), int(ex.sum()), sorted(bad), worst_c, worst_r, worst_e, worst_a)


def assert_encode_ok(rep: EncodeReport, max_exempt_frac=MAX_EXEMPT_FRAC):
    assert not rep.mismatched_idx, f"selected ids differ on vectors {rep.mismatched_idx[:10]}"
    assert rep.worst_coef <= COEF_TOL, rep.worst_coef
    assert rep.worst_coef_elem <= COEF_TOL, rep.worst_coef_elem
    assert rep.worst_relres <= RELRES_TOL, rep.worst_relres
    total = rep.checked + rep.exempt
    assert rep.exempt <= max(2, max_exempt_frac * total), f"{rep.exempt} of {total} vectors exempt"


def ulp(a: np.ndarray) -> np.ndarray:
    """Spacing of the storage type at |a| (binary16 or binary32)."""
    return np.spacing(np.abs(a).astype(a.dtype)).astype(np.float64)


def compare_atoms(gpu: np.ndarray, orc: np.ndarray, rows, bound=None) -> float:
    """Max deviation over the given rows, in units of the allowed error:
    one ulp of the storage type plus, if given, bound[j] (an [d] array of the
    fp32 arithmetic's error bound for that row).  <= 1 passes."""
    worst = 0.0
    for j in rows:
        g = gpu[j].astype(np.float64)
        o = orc[j].astype(np.float64)
        u = np.maximum(ulp(orc[j]), ulp(gpu[j]))
        if bound is not None:
            u = u + bound[j]
        worst = max(worst, float(np.max(np.abs(g - o) / u)))
    return worst


def replacement_bounds(atoms_before, x, idx, coef, repl_id, s):
    """Per replaced atom j = repl_id[v]: an elementwise bound on the fp32
    error of e/||e|| with e = x - sum_k c_k d_k formed by s fused
    multiply-adds (unit roundoff 2^-24 each, plus the division):
    (s + 3) * 2^-24 * (|x_t| + sum_k |c_k d_kt|) / ||e||."""
    u = 2.0 ** -24
    out = {}
    for v, j in enumerate(repl_id):
        if j < 0:
            continue
        A = atoms_before[idx[v]].astype(np.float64)
        c = coef[v].astype(np.float64)
        xv = x[v].astype(np.float64)
        e = xv - c @ A
        mag = np.abs(xv) + np.abs(c) @ np.abs(A)
        out[int(j)] = (s + 3) * u * mag / np.linalg.norm(e) + 2 * u * np.abs(e) / np.linalg.norm(e)
    return out
