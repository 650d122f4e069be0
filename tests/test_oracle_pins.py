"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test pins one part of the oracle to something other than the oracle's
own formulas: the pages' printed values (Table 4 cost, Table 5 defaults), a
closed form, a theorem's special case, an exhaustive search on tiny inputs,
or a library routine applied to a case that reduces to it.  A plausible slip
in the oracle (a dropped ridge term, a wrong sign in the residual, a wrong
index in the tie rule, a transposed Gram matrix) fails at least one of them.

Source: "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning
Decoding" (abstract; Fig. 1 and Fig. 2 captions; Table 4; Table 5).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from dictionary_sparse_kv_gb300 import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LA, LR = 1e-4, 0.20


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _ridge_closed_form(D, S_ids, x, la=LA, lr=LR):
    """Normal equations of the ridge refit, solved by numpy (LAPACK)."""
    DS = D[S_ids].astype(np.float64)
    G = DS @ DS.T
    A = G + np.diag(la + lr * np.diag(G))
    return np.linalg.solve(A, DS @ x.astype(np.float64))


# --------------------------------------------------------------------------
# binary16 codec: against numpy's float16 conversion (exhaustive decode)
# --------------------------------------------------------------------------

def test_half_decode_exhaustive(oracle_lib):
    O = oracle_lib
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([O.half_to_double(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_half_encode_rounding(oracle_lib):
    O = oracle_lib
    g = np.random.default_rng(7)
    b = np.arange(0, 0x7bff, 3, dtype=np.uint16)
    mid = (b.view(np.float16).astype(np.float64) + (b + 1).view(np.float16).astype(np.float64)) / 2
    vals = np.concatenate([
        g.standard_normal(20000) * 10.0 ** g.integers(-9, 6, 20000),
        # exact midpoints between neighbouring finite halves (ties to even), both signs
        mid, -mid,
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e9, 2.0**-24, 2.0**-25,
         3 * 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25, np.inf, -np.inf],
    ])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([O.double_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert (got == ref).all()


# --------------------------------------------------------------------------
# Table 5 defaults and Table 4 cost
# --------------------------------------------------------------------------

def test_table4_cost_reproduced_by_operation_count(oracle_lib):
    """Table 4 prints Cost 0.19 for GM relative to OMP over the whole
    dictionary (1.00).  Counting the oracle's multiply-accumulates at the 3B
    shape (N=4096, d=128, n=256, s=8) must reproduce that to two decimals."""
    O = oracle_lib
    g = _golden("table4_cost.json")
    sh = g["shape"]
    p = O.Params(sh["N"], sh["d"], sh["n"], sh["s"])
    D = S.make_dictionary(sh["N"], sh["d"], np.float16, 11)
    x = S.make_sparse_inputs(D, 3, sh["s"], 12)
    gm = O.encode(p, D, x)
    omp = O.encode(p, D, x, full_omp=True)
    cost = gm.macs / omp.macs
    assert round(cost, 2) == g["GM"]
    # the count has a closed form: screening N d; at step k, correlations over
    # the n - k unpicked pool atoms, the (k+1)(k+2)/2 Gram entries and k+1
    # right-hand-side products of the refit, and the k+1 residual terms
    N, d, n, s = sh["N"], sh["d"], sh["n"], sh["s"]
    per_vec = N * d + sum(((n - k) + (k + 1) * (k + 2) // 2 + 2 * (k + 1)) * d for k in range(s))
    assert gm.macs == 3 * per_vec
    assert omp.macs == 3 * sum(((N - k) + (k + 1) * (k + 2) // 2 + 2 * (k + 1)) * d for k in range(s))


def test_table5_defaults_file():
    g = _golden("table5_defaults.json")
    assert g["ridge_lambda_abs"] == LA and g["ridge_lambda_rel"] == LR
    assert (g["delta_key"], g["delta_value"]) == (0.5, 0.7)


# --------------------------------------------------------------------------
# screening + Top-n against a full stable sort
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,d,n,dt", [(512, 64, 32, np.float32), (4096, 128, 256, np.float16)])
def test_topn_matches_full_sort(oracle_lib, N, d, n, dt):
    O = oracle_lib
    p = O.Params(N, d, n, 4, dtype=O.F32 if dt == np.float32 else O.F16)
    D = S.make_dictionary(N, d, dt, 21, N)
    x = S.make_sparse_inputs(D, 40, 4, 22, N, dtype=dt)
    r = O.encode(p, D, x)
    R = x.astype(np.float64) @ D.astype(np.float64).T
    for v in range(x.shape[0]):
        mag = np.abs(R[v])
        order = np.lexsort((np.arange(N), -mag))      # key (-|r|, j), stable
        if r.cut_gap[v] < 1e-9:
            continue
        assert list(r.pool[v]) == list(order[:n])


def test_topn_tie_rule_on_exact_zeros(oracle_lib):
    """Signed permutation dictionary (N = d): a 4-sparse x leaves N-4 scores
    exactly zero, so the pool is the 4 support atoms by |coefficient|, then
    the lowest remaining ids in ascending order."""
    O = oracle_lib
    d = N = 64
    g = np.random.default_rng(3)
    perm = g.permutation(N)
    D = np.zeros((N, d), np.float32)
    D[np.arange(N), perm] = g.choice([-1.0, 1.0], N)
    supp = np.array([40, 7, 55, 13])
    b = np.array([-3.0, 2.5, 2.0, -1.0])
    x = (b @ D[supp]).astype(np.float32)[None]
    p = O.Params(N, d, 10, 3, dtype=O.F32)
    r = O.encode(p, D, x)
    rest = [j for j in range(N) if j not in supp][:6]
    assert list(r.pool[0]) == list(supp) + rest
    assert r.cut_gap[0] == 0.0


# --------------------------------------------------------------------------
# ridge refit
# --------------------------------------------------------------------------

def test_ridge_matches_normal_equations(oracle_lib):
    O = oracle_lib
    p = O.Params(512, 64, 32, 4, dtype=O.F32)
    D = S.make_dictionary(512, 64, np.float32, 0)
    x = S.make_tiny_inputs(D, 64, 4, 1)
    r = O.encode(p, D, x)
    for v in range(64):
        c = _ridge_closed_form(D, r.idx[v], x[v])
        assert np.allclose(r.coef[v], c, rtol=1e-10, atol=1e-12)


def test_orthogonal_closed_form(oracle_lib):
    """Orthogonal atoms of norms w_j: G is diagonal, so
    c_i = b_i w_i^2 / (w_i^2 (1 + lambda_rel) + lambda_abs), picks go by
    |b_i| w_i^2 (ties to the lower id), and the residual is known exactly."""
    O = oracle_lib
    d = N = 32
    w = np.array([0.5, 1.0, 2.0, 1.5] * 8)
    D = (np.diag(w)).astype(np.float32)            # atom j = w_j e_j
    supp = np.array([2, 5, 9, 20, 30])
    b = np.array([0.75, -2.0, 1.0, -0.5, 0.25])    # |b| w^2 = 3, 2, 0.25, 4, 0.5625... see below
    x = np.zeros(d)
    x[supp] = b * w[supp]
    x32 = x.astype(np.float32)[None]
    s = 5
    p = O.Params(N, d, 8, s, dtype=O.F32)
    r = O.encode(p, D, x32)
    score = np.abs(b) * w[supp] ** 2
    order = supp[np.lexsort((supp, -score))]
    assert list(r.idx[0]) == list(order)
    w2 = w ** 2
    c_expect = {j: b[i] * w2[j] / (w2[j] * (1 + LR) + LA) for i, j in enumerate(supp)}
    for k, j in enumerate(r.idx[0]):
        assert r.coef[0, k] == pytest.approx(c_expect[j], rel=1e-13)
    e = x.copy()
    for k, j in enumerate(r.idx[0]):
        e[j] -= r.coef[0, k] * w[j]
    assert r.relres[0] == pytest.approx(np.linalg.norm(e) / np.linalg.norm(x), rel=1e-13)


def test_unit_orthonormal_relres_constant(oracle_lib):
    """Unit-norm orthonormal atoms and a noise-free s-sparse x: c = b/1.2001
    and relres = 0.2001/1.2001 whatever b is."""
    O = oracle_lib
    d = N = 64
    D = np.eye(N, dtype=np.float32)[::-1].copy()
    g = np.random.default_rng(5)
    for trial in range(5):
        supp = g.choice(N, 6, replace=False)
        b = g.choice([-1, 1], 6) * (1 + g.integers(0, 64, 6) / 16.0)
        x = (b @ D[supp]).astype(np.float32)[None]
        r = O.encode(O.Params(N, d, 12, 6, dtype=O.F32), D, x)
        assert sorted(r.idx[0]) == sorted(supp)
        for k, j in enumerate(r.idx[0]):
            assert r.coef[0, k] == pytest.approx(b[list(supp).index(j)] / 1.2001, rel=1e-14)
        assert r.relres[0] == pytest.approx(0.2001 / 1.2001, rel=1e-13)


# --------------------------------------------------------------------------
# greedy selection: exact recovery (Tropp's condition) and brute force
# --------------------------------------------------------------------------

def _sylvester(m):
    H = np.array([[1.0]])
    while H.shape[0] < m:
        H = np.block([[H, H], [H, -H]])
    return H


@pytest.mark.parametrize("ridge", [False, True])
def test_exact_recovery_incoherent(oracle_lib, ridge):
    """D = [I | H/sqrt(d)] at d = 64 has coherence 1/8; s = 4 < (1 + 8)/2,
    so OMP recovers every noise-free 4-sparse x exactly (Tropp 2004).  Here
    the pool is the whole dictionary.  The same recovery is checked with the
    ridge refit of Table 5."""
    O = oracle_lib
    d = 64
    D = np.vstack([np.eye(d), _sylvester(d) / 8.0]).astype(np.float32)
    N = D.shape[0]
    g = np.random.default_rng(9)
    p = O.Params(N, d, N, 4, lambda_abs=LA if ridge else 0.0,
                 lambda_rel=LR if ridge else 0.0, dtype=O.F32)
    fails = 0
    for trial in range(200):
        supp = g.choice(N, 4, replace=False)
        b = g.choice([-1, 1], 4) * (1 + g.integers(0, 9, 4) / 8.0)   # |b| in [1, 2]
        x = (b @ D[supp].astype(np.float64)).astype(np.float32)[None]
        r = O.encode(p, D, x)
        fails += sorted(r.idx[0]) != sorted(supp)
        if not ridge:
            assert np.allclose(sorted(zip(r.idx[0], r.coef[0])), sorted(zip(supp, b)), atol=1e-6)
    assert fails == 0


def test_greedy_steps_brute_force(oracle_lib):
    """Tiny inputs (d=16, N=32, n=8): at every step k the pick must be the
    argmax over P \\ S_k of |<d_j, e_k>| (ties to the lower id), where e_k is
    rebuilt by numpy from the oracle's own k-atom encode, and the final
    support's objective must equal the best over its own coefficients."""
    O = oracle_lib
    d, N, n = 16, 32, 8
    D = S.make_dictionary(N, d, np.float32, 31)
    x = S.make_tiny_inputs(D, 30, 3, 32, sigma=0.05)
    D64 = D.astype(np.float64)
    for s in (2, 3):
        full = O.encode(O.Params(N, d, n, s, dtype=O.F32), D, x)
        for v in range(x.shape[0]):
            P = list(full.pool[v])
            for k in range(s):
                if k == 0:
                    e = x[v].astype(np.float64)
                else:
                    part = O.encode(O.Params(N, d, n, k, dtype=O.F32), D, x[v:v + 1])
                    assert list(part.idx[0]) == list(full.idx[v][:k])
                    e = x[v] - part.coef[0] @ D64[part.idx[0]]
                cand = [j for j in P if j not in full.idx[v][:k]]
                a = np.abs(D64[cand] @ e)
                best = min(cand[i] for i in range(len(cand)) if a[i] == a.max())
                if full.pick_gap[v, k] > 1e-9:
                    assert full.idx[v][k] == best


def test_brute_force_subset_objective(oracle_lib):
    """Exhaustive search over every s-subset of the pool of the ridge
    objective ||x - D_T c||^2 + sum_i (lambda_abs + lambda_rel G_ii) c_i^2.
    The greedy support's objective, evaluated at the oracle's c, equals the
    closed-form minimum for that support and is >= the global minimum; on
    noise-free inputs over orthogonal atoms greedy attains the minimum."""
    O = oracle_lib

    def objective(D, T, c, x):
        DT = D[list(T)].astype(np.float64)
        G = DT @ DT.T
        lam = LA + LR * np.diag(G)
        e = x - c @ DT
        return e @ e + lam @ (c * c)

    d, N, n = 16, 32, 8
    D = S.make_dictionary(N, d, np.float32, 41)
    x = S.make_tiny_inputs(D, 20, 3, 42, sigma=0.1).astype(np.float64)
    for s in (2, 3):
        r = O.encode(O.Params(N, d, n, s, dtype=O.F32), D, x.astype(np.float32))
        for v in range(x.shape[0]):
            xv = x[v].astype(np.float32).astype(np.float64)
            f_g = objective(D, r.idx[v], r.coef[v], xv)
            f_cf = objective(D, r.idx[v], _ridge_closed_form(D, r.idx[v], xv), xv)
            assert f_g == pytest.approx(f_cf, rel=1e-12)
            best = min(objective(D, T, _ridge_closed_form(D, list(T), xv), xv)
                       for T in itertools.combinations(r.pool[v], s))
            assert f_g >= best * (1 - 1e-12)
    # orthogonal atoms, noise-free: greedy == exhaustive argmin
    Q = np.eye(d, dtype=np.float32)
    Dq = np.vstack([Q, Q[::-1] * 0.5]).astype(np.float32)   # N = 32, pairs of parallel atoms
    g = np.random.default_rng(4)
    for trial in range(20):
        supp = g.choice(d, 3, replace=False)
        b = g.choice([-1, 1], 3) * (1 + g.integers(0, 16, 3) / 8.0)
        xv = (b @ Dq[supp]).astype(np.float32)
        r = O.encode(O.Params(32, d, 8, 3, dtype=O.F32), Dq, xv[None])
        vals = {T: objective(Dq, T, _ridge_closed_form(Dq, list(T), xv.astype(np.float64)),
                             xv.astype(np.float64))
                for T in itertools.combinations(sorted(r.pool[0]), 3)}
        assert objective(Dq, r.idx[0], r.coef[0], xv.astype(np.float64)) == pytest.approx(
            min(vals.values()), rel=1e-12)


# --------------------------------------------------------------------------
# greedy selection on a given pool (steps 3-4 without the screening)
# --------------------------------------------------------------------------

def test_greedy_on_pool_restricted_closed_form(oracle_lib):
    """Unit orthonormal atoms, noise-free 6-sparse x on support T, and a
    given pool P holding only some of T: the picks must come from P alone.
    With G = I the ridge gives c_j = <d_j, x>/1.2001, so the atoms of T in P
    come first (by |b|, then id), then pool atoms of zero correlation in id
    order with c = 0, and relres is known exactly:
    ||e||^2 = sum_{T in P} (0.2001 b_j / 1.2001)^2 + sum_{T not in P} b_j^2.
    Every vector has its own pool, whose first entry is its largest in-pool
    support atom (so a pool read from the wrong row, or shifted, fails)."""
    O = oracle_lib
    d = N = 64
    D = np.eye(N, dtype=np.float32)[::-1].copy()          # atom j = e_{63-j}
    g = np.random.default_rng(12)
    n, s, V = 10, 6, 8
    pools, xs, expect = [], [], []
    for v in range(V):
        T = g.choice(N, 6, replace=False)
        b = g.choice([-1, 1], 6) * (1 + g.permutation(6) / 4.0)   # distinct |b|
        inP = T[:3]                                        # three support atoms in the pool
        others = [j for j in g.permutation(N) if j not in T][:n - 3]
        lead = inP[np.argmax(np.abs(b[:3]))]
        P = [int(lead)] + [int(j) for j in inP if j != lead] + [int(j) for j in others]
        pools.append(P)
        xs.append((b @ D[T].astype(np.float64)).astype(np.float32))
        order = [int(j) for j in inP[np.lexsort((inP, -np.abs(b[:3])))]]
        zero = sorted(others)[:s - 3]
        ce = {int(T[i]): b[i] / 1.2001 for i in range(3)}
        e2 = sum((0.2001 * b[i] / 1.2001) ** 2 for i in range(3)) + sum(b[i] ** 2 for i in range(3, 6))
        expect.append((order + zero, ce, math.sqrt(e2) / np.linalg.norm(b)))
    r = O.greedy_on_pool(O.Params(N, d, n, s, dtype=O.F32), D, np.stack(xs), np.array(pools, np.int32))
    for v in range(V):
        ids, ce, rel = expect[v]
        assert list(r.idx[v]) == ids, v
        for k, j in enumerate(ids):
            assert r.coef[v, k] == pytest.approx(ce.get(j, 0.0), rel=1e-14, abs=1e-15)
        assert r.relres[v] == pytest.approx(rel, rel=1e-13)


def test_greedy_on_pool_matches_encode_and_ignores_order(oracle_lib):
    """Given the oracle's own Top-n pools, greedy_on_pool reproduces
    encode bit for bit; given the same pools shuffled, it returns the same
    ids, coefficients and relres (the pool is a set: ties go by atom id,
    never by position)."""
    O = oracle_lib
    w = S.WORKLOADS["tiny"]
    D = S.make_dictionary(w.N, w.d, np.float32, 0)
    x = S.make_tiny_inputs(D, 24, w.s, 1)
    p = O.Params(w.N, w.d, w.n, w.s, dtype=O.F32)
    full = O.encode(p, D, x)
    same = O.greedy_on_pool(p, D, x, full.pool)
    for a, b in ((same.idx, full.idx), (same.coef, full.coef), (same.relres, full.relres),
                 (same.pick_gap, full.pick_gap)):
        assert np.array_equal(a, b)
    g = np.random.default_rng(13)
    shuffled = np.stack([g.permutation(row) for row in full.pool]).astype(np.int32)
    sh = O.greedy_on_pool(p, D, x, shuffled)
    assert np.array_equal(sh.idx, full.idx)
    assert np.array_equal(sh.coef, full.coef) and np.array_equal(sh.relres, full.relres)


# --------------------------------------------------------------------------
# special inputs
# --------------------------------------------------------------------------

def test_zero_and_nonfinite_inputs(oracle_lib):
    O = oracle_lib
    p = O.Params(512, 64, 32, 4, dtype=O.F32)
    D = S.make_dictionary(512, 64, np.float32, 0)
    x = np.zeros((3, 64), np.float32)
    x[1, 5] = np.nan
    x[2, 9] = np.inf
    r = O.encode(p, D, x)
    assert list(r.idx[0]) == [0, 1, 2, 3] and (r.coef[0] == 0).all() and r.relres[0] == 0
    assert list(r.pool[0]) == list(range(32))
    for v in (1, 2):
        assert (r.idx[v] == -1).all() and math.isnan(r.relres[v])


# --------------------------------------------------------------------------
# PL encode: screening + one ridge fit (the PL rows of Tables 1-4)
# --------------------------------------------------------------------------

def test_table4_pl_cost_reproduced_by_operation_count(oracle_lib):
    """Table 4 prints Cost 0.13 for PL.  Screening (N d) plus one fit over
    s atoms (s(s+1)/2 Gram entries, s right-hand sides, s residual terms,
    each d long), against the oracle's count for OMP over the whole
    dictionary, must give that to two decimals."""
    O = oracle_lib
    g = _golden("table4_cost.json")
    sh = g["shape"]
    N, d, n, s = sh["N"], sh["d"], sh["n"], sh["s"]
    p = O.Params(N, d, n, s)
    D = S.make_dictionary(N, d, np.float16, 11)
    x = S.make_sparse_inputs(D, 3, s, 12)
    pl = O.encode_pl(p, D, x)
    omp = O.encode(p, D, x, full_omp=True)
    assert round(pl.macs / omp.macs, 2) == g["PL"]
    assert pl.macs == 3 * (N * d + (s * (s + 1) // 2 + 2 * s) * d)


def test_pl_weighted_orthogonal_closed_form(oracle_lib):
    """Orthogonal atoms w_j e_j: r_j = w_j x_j, the fit decouples into
    c_j = r_j / (w_j^2 (1 + lambda_rel) + lambda_abs), and the residual is
    known exactly.  The support holds a tie in |r| at the Top-s cut (atoms
    11 and 27, |r| = 2 each), which the lower id must win; idx comes out in
    ascending atom order."""
    O = oracle_lib
    d = N = 32
    w = np.array([0.5, 1.0, 2.0, 1.5] * 8)
    D = np.diag(w).astype(np.float32)
    # |r_j| = |x_j| w_j: 3 (atom 6), 2 (atoms 11, 27), 4.5 (atom 15),
    # 1.5 (atom 20), 1 (atom 2), 6 (atom 30)
    x = np.zeros(d)
    for j, r in [(6, -3.0), (11, 2.0), (27, -2.0), (15, 4.5), (20, -1.5), (2, 1.0), (30, 6.0)]:
        x[j] = r / w[j]
    x32 = x.astype(np.float32)[None]
    x = x32[0].astype(np.float64)                  # the stored values, exactly
    s = 4
    r = O.encode_pl(O.Params(N, d, 8, s, dtype=O.F32), D, x32)
    assert list(r.idx[0]) == [6, 11, 15, 30]
    e = x.copy()
    for k, j in enumerate(r.idx[0]):
        rj = w[j] * x[j]
        assert r.coef[0, k] == pytest.approx(rj / (w[j] ** 2 * (1 + LR) + LA), rel=1e-13)
        e[j] -= r.coef[0, k] * w[j]
    assert r.relres[0] == pytest.approx(np.linalg.norm(e) / np.linalg.norm(x), rel=1e-13)
    assert r.cut_gap[0] == 0.0                     # |r|_(4) = |r|_(5) = 2


@pytest.mark.parametrize("dt", [np.float16, np.float32])
def test_pl_with_one_atom_is_the_first_greedy_pick(oracle_lib, dt):
    """With s = 1 the greedy coder's only pick is the atom of largest |r|
    and its refit is the same one-atom fit: PL and GM agree bit for bit."""
    O = oracle_lib
    N, d = 512, 64
    kind = O.F16 if dt == np.float16 else O.F32
    D = S.make_dictionary(N, d, dt, 31)
    x = S.make_sparse_inputs(D, 40, 3, 32, dtype=dt)
    p = O.Params(N, d, 16, 1, dtype=kind)
    pl = O.encode_pl(p, D, x)
    gm = O.encode(p, D, x)
    assert (pl.idx == gm.idx).all()
    assert (pl.coef == gm.coef).all() and (pl.relres == gm.relres).all()


def test_pl_is_greedy_over_a_pool_of_s(oracle_lib):
    """A greedy coder whose pool holds exactly s atoms picks all of them, and
    its last refit is the ridge fit over that pool: PL gives the same set,
    the same coefficients per atom and the same relres (up to rounding
    order)."""
    O = oracle_lib
    N, d, s = 1024, 128, 8
    D = S.make_dictionary(N, d, np.float16, 41)
    x = S.make_sparse_inputs(D, 30, s, 42)
    p = O.Params(N, d, s, s)
    pl = O.encode_pl(p, D, x)
    gm = O.encode(p, D, x)
    for v in range(x.shape[0]):
        assert list(pl.idx[v]) == sorted(gm.idx[v])
        order = np.argsort(gm.idx[v])
        np.testing.assert_allclose(pl.coef[v], gm.coef[v][order], rtol=1e-11, atol=1e-13)
        assert pl.relres[v] == pytest.approx(gm.relres[v], rel=1e-11)
        # the cut is the one the greedy coder's pool was cut at
        assert pl.cut_gap[v] == gm.cut_gap[v]


def test_pl_fit_matches_normal_equations(oracle_lib):
    """The fit on the Top-s set against numpy's solve of the same normal
    equations, with the Top-s set from a full stable sort."""
    O = oracle_lib
    N, d, s = 512, 64, 6
    D = S.make_dictionary(N, d, np.float32, 51)
    x = S.make_sparse_inputs(D, 25, 4, 52, dtype=np.float32)
    r = O.encode_pl(O.Params(N, d, 32, s, dtype=O.F32), D, x)
    R = x.astype(np.float64) @ D.astype(np.float64).T
    for v in range(x.shape[0]):
        top = np.sort(np.lexsort((np.arange(N), -np.abs(R[v])))[:s])
        assert list(r.idx[v]) == list(top)
        c = _ridge_closed_form(D, top, x[v])
        np.testing.assert_allclose(r.coef[v], c, rtol=1e-9, atol=1e-12)
        e = x[v].astype(np.float64) - c @ D[top].astype(np.float64)
        xn = np.linalg.norm(x[v].astype(np.float64))
        assert r.relres[v] == pytest.approx(np.linalg.norm(e) / xn, rel=1e-9)


def test_pl_zero_and_nonfinite_inputs(oracle_lib):
    O = oracle_lib
    p = O.Params(512, 64, 32, 4, dtype=O.F32)
    D = S.make_dictionary(512, 64, np.float32, 0)
    x = np.zeros((3, 64), np.float32)
    x[1, 5] = np.nan
    x[2, 9] = -np.inf
    r = O.encode_pl(p, D, x)
    assert list(r.idx[0]) == [0, 1, 2, 3] and (r.coef[0] == 0).all() and r.relres[0] == 0
    for v in (1, 2):
        assert (r.idx[v] == -1).all() and (r.coef[v] == 0).all() and math.isnan(r.relres[v])


# --------------------------------------------------------------------------
# compressed store: packed words, and attention over packed codes
# --------------------------------------------------------------------------

def test_pack_word_matches_binary16_rounding(oracle_lib):
    """Inside binary16's normal range [2^-14, 65504] a value rounded to 11
    significant bits (ties to even) is exactly what numpy's binary16
    conversion gives, so that routine pins the rounding: random values,
    exact midpoints between neighbouring binary16 numbers, both signs."""
    O = oracle_lib
    g = np.random.default_rng(17)
    vals = np.exp(g.uniform(np.log(2.0 ** -14), np.log(65000.0), 3000))
    b = np.arange(0x0400, 0x7bff, 37, dtype=np.uint16)
    mids = (b.view(np.float16).astype(np.float64) + (b + 1).view(np.float16).astype(np.float64)) / 2
    for v in np.concatenate([vals, mids]):
        for sgn in (1.0, -1.0):
            w = O.pack_word(sgn * v, 4321)
            assert O.word_id(w) == 4321
            assert O.word_coef(w) == float(np.float16(sgn * v)), (sgn * v)


def test_pack_word_layout(oracle_lib):
    """Bits 31..13 are the top 19 bits of the binary32 encoding of the
    rounded coefficient; bits 12..0 the id.  Zero coefficients and skipped
    terms are word 0; magnitudes below 2^-126 keep only the id; outside
    binary16's range the rounding still keeps 11 significant bits with an
    error of at most half a unit in the last place."""
    O = oracle_lib
    g = np.random.default_rng(18)
    for c in np.concatenate([g.standard_normal(500) * 10.0 ** g.integers(-30, 30, 500), [1e-20, -3e25]]):
        j = int(g.integers(0, 8192))
        w = O.pack_word(float(c), j)
        r = O.word_coef(w)
        assert (w & 0x1FFF) == j
        assert (w >> 13) == (int(np.float32(r).view(np.uint32)) >> 13)
        m, e = np.frexp(abs(r))
        assert float(np.ldexp(m, 11)).is_integer()                     # 11 significant bits
        assert abs(r - c) <= np.ldexp(1.0, int(np.frexp(abs(c))[1]) - 12) * (1 + 1e-12)
    assert O.pack_word(0.0, 5) == 0 and O.pack_word(1.5, -1) == 0
    assert O.pack_word(1e-39, 5) == 5


def _identity_case(N=64, Tmax=8):
    D = np.eye(N, dtype=np.float32)
    return D, D.copy()


def test_attend_single_token_is_its_value(oracle_lib):
    """One cached token: softmax over one score is 1, the output is v_0."""
    O = oracle_lib
    N = d = 64
    g = np.random.default_rng(19)
    Dk = S.make_dictionary(N, d, np.float32, 5)
    Dv = S.make_dictionary(N, d, np.float32, 6)
    ck = O.pack_codes(np.array([[[[3, 9, 40]]]]), np.array([[[[0.5, -1.25, 2.0]]]]))
    cv = O.pack_codes(np.array([[[[7, 8, 60]]]]), np.array([[[[1.5, 0.75, -0.5]]]]))
    q = g.standard_normal((1, 1, d))
    out = O.attend(Dk, Dv, ck, cv, np.array([1]), q)
    Dv64 = Dv.astype(np.float64)
    v0 = 1.5 * Dv64[7] + 0.75 * Dv64[8] - 0.5 * Dv64[60]
    np.testing.assert_allclose(out[0, 0], v0, rtol=1e-14, atol=1e-15)


def test_attend_two_tokens_closed_form(oracle_lib):
    """Identity dictionaries (atom j = e_j): k_0 = 1.5 e_3 (+ a replacement
    term 0.5 e_3), k_1 = -0.75 e_10, so the scores are (2 q_3, -0.75 q_10) /
    sqrt(d); v_0 = 2 e_5,
    v_1 = -0.5 e_6 (+ a replacement term 0.25 e_5 on token 1); the output
    is p_0 v_0 + p_1 v_1 with p the softmax of the two scores."""
    O = oracle_lib
    D, _ = _identity_case()
    d = 64
    q = np.zeros((1, 1, d))
    q[0, 0, 3], q[0, 0, 10] = 2.0, -2.0
    ck = O.pack_codes(np.array([[[[3], [10]]]]), np.array([[[[1.5], [-0.75]]]]),
                      np.array([[[3, -1]]]), np.array([[[0.5, 0.0]]]))
    cv = O.pack_codes(np.array([[[[5], [6]]]]), np.array([[[[2.0], [-0.5]]]]),
                      np.array([[[-1, 5]]]), np.array([[[0.0, 0.25]]]))
    out = O.attend(D, D, ck, cv, np.array([2]), q)
    s0, s1 = (1.5 + 0.5) * 2.0 / 8.0, -0.75 * -2.0 / 8.0
    p0 = math.exp(s0) / (math.exp(s0) + math.exp(s1))
    p1 = 1.0 - p0
    want = np.zeros(d)
    want[5] = 2.0 * p0 + 0.25 * p1
    want[6] = -0.5 * p1
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-14, atol=1e-15)


def test_attend_grouped_heads_and_lengths(oracle_lib):
    """Four query heads over two KV heads: heads 0, 1 read KV head 0 and
    heads 2, 3 KV head 1.  Every value token of KV head k is c_k e_(20+k),
    so the output is that vector whatever the weights; tokens at or past a
    sequence's length hold codes of another atom and must not count; an
    empty sequence gives 0."""
    O = oracle_lib
    D, _ = _identity_case()
    d, Tmax = 64, 6
    g = np.random.default_rng(20)
    B, Hkv, Hq = 3, 2, 4
    lengths = np.array([6, 2, 0])
    kid = g.integers(0, 64, (B, Hkv, Tmax, 2))
    kco = g.standard_normal((B, Hkv, Tmax, 2))
    vid = np.zeros((B, Hkv, Tmax, 2), np.int64)
    vco = np.zeros((B, Hkv, Tmax, 2))
    for b in range(B):
        for k in range(Hkv):
            for t in range(Tmax):
                inside = t < lengths[b]
                vid[b, k, t] = [20 + k, 40] if inside else [50, 51]
                vco[b, k, t] = [1.0 + k, 0.0] if inside else [9.0, 9.0]
    ck = O.pack_codes(kid, kco)
    cv = O.pack_codes(vid, vco)
    q = g.standard_normal((B, Hq, d))
    out = O.attend(D, D, ck, cv, lengths, q)
    for b in range(B):
        for h in range(Hq):
            want = np.zeros(d)
            if lengths[b] > 0:
                want[20 + h // 2] = 1.0 + h // 2
            np.testing.assert_allclose(out[b, h], want, rtol=1e-13, atol=1e-14)


def test_attend_identical_keys_average_values(oracle_lib):
    """All keys equal: every token gets weight 1/T and the output is the
    mean of the value vectors."""
    O = oracle_lib
    N = d = 64
    T = 5
    g = np.random.default_rng(21)
    Dk = S.make_dictionary(N, d, np.float32, 7)
    Dv = S.make_dictionary(N, d, np.float32, 8)
    kid = np.broadcast_to(np.array([2, 11]), (1, 1, T, 2))
    kco = np.broadcast_to(np.array([0.5, -1.0]), (1, 1, T, 2))
    vid = g.integers(0, N, (1, 1, T, 2))
    vco = np.round(g.standard_normal((1, 1, T, 2)) * 64) / 64     # exact in 11 bits
    out = O.attend(Dk, Dv, O.pack_codes(kid, kco), O.pack_codes(vid, vco), np.array([T]),
                   g.standard_normal((1, 2, d)))
    Dv64 = Dv.astype(np.float64)
    mean = sum(vco[0, 0, t, i] * Dv64[vid[0, 0, t, i]] for t in range(T) for i in range(2)) / T
    for h in range(2):
        np.testing.assert_allclose(out[0, h], mean, rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------
# adapt: hand-derived cases and invariants
# --------------------------------------------------------------------------

def test_adapt_golden_cases(oracle_lib):
    O = oracle_lib
    g = _golden("adapt_cases.json")
    for case in g["cases"]:
        atoms = np.array(g["atoms"], np.float32)
        before = atoms.copy()
        usage = np.array(case["usage"], np.int32)
        x = np.array(case["x"], np.float32)
        idx = np.array(case["idx"], np.int32)
        coef = np.array(case["coef"], np.float64)
        rel = np.array([float(v) for v in case["relres"]], np.float64)
        p = O.Params(atoms.shape[0], atoms.shape[1], 2, idx.shape[1], dtype=O.F32)
        res = O.adapt(p, atoms, usage, x, idx, coef, rel, case["delta"], append=case.get("mode") == "append")
        assert list(usage) == case["expect_usage"], case["name"]
        assert list(res.repl_id) == case["expect_repl_id"], case["name"]
        assert np.allclose(res.repl_coef, case["expect_repl_coef"], rtol=0, atol=1e-12)
        assert (res.replaced, res.overflow) == (case["expect_replaced"], case["expect_overflow"])
        changed = {int(k): v for k, v in case["expect_atoms_changed"].items()}
        for j in range(atoms.shape[0]):
            want = changed.get(j, before[j])
            assert np.array_equal(atoms[j], np.array(want, np.float32)), (case["name"], j)


def test_append_growth_against_fixed_size(oracle_lib):
    """The contrast the pages draw (abstract; Fig. 2 caption; Fig. 3a): over a
    run of decode steps the append-only dictionary grows by one atom per
    flagged vector until its capacity is used up, and never rewrites an
    atom; the fixed-size dictionary never changes size (every row stays an
    atom) and only rewrites atoms that were inactive."""
    O = oracle_lib
    from dataclasses import replace
    w = replace(S.WORKLOADS["tiny"], off_frac=0.0, sigma=0.3)   # large residuals: many flagged vectors
    data = S.WorkloadData(w)
    N0 = 448                                   # atoms at the start; 64 free slots in append mode
    p = O.Params(w.N, w.d, w.n, w.s, dtype=O.F32)
    at_f, us_f = data.atoms[0].copy(), data.usage[0].copy()
    at_a, us_a = data.atoms[0].copy(), data.usage[0].copy()
    at_a[N0:] = 0
    us_a[N0:] = -1
    size = N0
    for step in range(4):
        x = data.inputs(step, 48)[0]
        for at, us, app in ((at_f, us_f, False), (at_a, us_a, True)):
            before, ub = at.copy(), us.copy()
            r = O.encode(p, at, x)
            a = O.adapt(p, at, us, x, r.idx, r.coef, r.relres, 0.5, append=app)
            flagged = int((r.relres > 0.5).sum())
            rows = set(np.nonzero((at != before).any(axis=1))[0].tolist())
            assert rows <= set(a.repl_id[a.repl_id >= 0].tolist())
            if app:
                assert a.replaced == min(flagged, w.N - size) and a.overflow == flagged - a.replaced
                assert sorted(a.repl_id[a.repl_id >= 0]) == list(range(size, size + a.replaced))
                size += a.replaced
                assert int((us >= 0).sum()) == size
            else:
                assert int((us < 0).sum()) == 0
                assert all(ub[j] == 0 for j in a.repl_id[a.repl_id >= 0])
    assert size > N0


def test_adapt_invariants_random(oracle_lib):
    """Row count fixed at N; usage never decreases and is conserved
    (sum after = sum before + s * #encoded + #replaced); only atoms inactive
    after the increments are overwritten, in ascending order, by unit-norm
    rows (within d * 2^-11 for binary16)."""
    O = oracle_lib
    N, d, n, s = 4096, 128, 256, 8
    p = O.Params(N, d, n, s)
    D = S.make_dictionary(N, d, np.float16, 51)
    usage = S.make_usage(N, int(0.3 * N), 52)
    src = D[usage > 0]
    x = S.make_sparse_inputs(src, 96, s, 53, off_frac=0.9)   # large residuals: many flags
    r = O.encode(p, D, x)
    before_D, before_u = D.copy(), usage.copy()
    res = O.adapt(p, D, usage, x, r.idx, r.coef, r.relres, 0.5)
    assert D.shape == (N, d)
    inc = np.zeros(N, np.int64)
    np.add.at(inc, r.idx.ravel(), 1)
    after_inc = before_u + inc
    L = np.nonzero(after_inc == 0)[0]
    F = np.nonzero(r.relres > 0.5)[0]
    m = min(len(L), len(F))
    assert res.replaced == m and res.overflow == len(F) - m
    assert m > 0
    assert list(res.repl_id[F[:m]]) == list(L[:m])
    assert (res.repl_id[np.setdiff1d(np.arange(len(x)), F[:m])] == -1).all()
    assert usage.sum() == before_u.sum() + s * len(x) + m
    assert (usage >= before_u).all()
    changed = np.nonzero((D != before_D).any(axis=1))[0]
    assert set(changed) <= set(L[:m])
    norms = np.linalg.norm(D[L[:m]].astype(np.float64), axis=1)
    assert np.all(np.abs(norms - 1) <= d * 2.0 ** -11)
    # each new atom is the normalised ridge residual of its vector
    for v, j in zip(F[:m], L[:m]):
        e = x[v].astype(np.float64) - r.coef[v] @ before_D[r.idx[v]].astype(np.float64)
        assert res.repl_coef[v] == pytest.approx(np.linalg.norm(e), rel=1e-12)
        assert np.array_equal(D[j], (e / np.linalg.norm(e)).astype(np.float16))


# --------------------------------------------------------------------------
# reconstruct
# --------------------------------------------------------------------------

def test_reconstruct_consistency(oracle_lib):
    """reconstruct(encode(x)) = x - e_s, so ||x - xhat|| / ||x|| = relres;
    after a replacement, xhat = x up to the binary16 rounding of the new atom."""
    O = oracle_lib
    N, d, n, s = 4096, 128, 256, 8
    p = O.Params(N, d, n, s)
    D = S.make_dictionary(N, d, np.float16, 61)
    usage = S.make_usage(N, 400, 62)
    x = S.make_sparse_inputs(D[usage > 0], 32, s, 63, off_frac=0.9)
    r = O.encode(p, D, x)
    xh = O.reconstruct(p, D, r.idx, r.coef)
    x64 = x.astype(np.float64)
    rel = np.linalg.norm(x64 - xh, axis=1) / np.linalg.norm(x64, axis=1)
    assert np.allclose(rel, r.relres, rtol=1e-10)
    res = O.adapt(p, D, usage, x, r.idx, r.coef, r.relres, 0.5)
    xh2 = O.reconstruct(p, D, r.idx, r.coef, res.repl_id, res.repl_coef)
    rep = res.repl_id >= 0
    assert rep.any()
    err = np.linalg.norm(xh2[rep] - x64[rep], axis=1)
    bound = res.repl_coef[rep] * np.sqrt(d) * 2.0 ** -11
    assert (err <= bound).all()
