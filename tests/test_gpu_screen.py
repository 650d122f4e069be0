"""Screening kernels on the GPU: tensor-core scores and the candidate filter.

* Raw scores of the tensor-core kernel (binary16 dictionaries) and of the
  FP32 kernel against the exact products in float64, within the fp32
  accumulation bound d * 2^-24 * sum_t |x_t d_jt| per score.
* Encodes through the two screening paths agree with each other and with
  the oracle.
* The exact slow path: a candidate list shorter than n (x is a basis vector
  of a dictionary made of repeated signed bases, so only a few scores pass
  the threshold) and a list that overflows (x = 0: every score passes).
"""
import numpy as np
import pytest

from dictionary_sparse_kv_gb300 import synthetic as S
from oracle import oracle as O
from tests import parity_util as PU

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dictionary_sparse_kv_gb300 import build as B
    B.build()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _dict(atoms, usage, deltas, n, s, max_batch):
    from dictionary_sparse_kv_gb300 import fadkv as F
    return F.Dictionary(_t(atoms), _t(usage), deltas, n, s, max_batch)


@pytest.mark.parametrize("path", ["tc", "ffma"])
@pytest.mark.parametrize("N,d,G,V", [(4096, 128, 3, 200), (8192, 128, 2, 128), (1024, 64, 2, 300)])
def test_scores_against_float64(monkeypatch, path, N, d, G, V):
    if path == "ffma":
        monkeypatch.setenv("FADKV_SCREEN", "ffma")
    atoms = np.stack([S.make_dictionary(N, d, np.float16, 7, g) for g in range(G)])
    x = np.stack([S.make_sparse_inputs(atoms[g], V, 8, 8, g) for g in range(G)])
    D = _dict(atoms, np.ones((G, N), np.int32), [0.5] * G, 64, 8, V)
    sc = D.scores(_t(x)).cpu().numpy().astype(np.float64)
    for g in range(G):
        A = atoms[g].astype(np.float64)
        X = x[g].astype(np.float64)
        exact = X @ A.T
        bound = d * 2.0 ** -24 * (np.abs(X) @ np.abs(A).T) + 1e-30
        err = np.abs(sc[g] - exact)
        assert np.all(err <= bound), float(np.max(err / bound))


def test_two_screening_paths_agree(monkeypatch):
    from dataclasses import replace
    w = replace(S.WORKLOADS["decode_3b"], G=3)
    data = S.WorkloadData(w)
    x = data.inputs(0, 160)
    outs = {}
    for path in ("tc", "ffma"):
        if path == "ffma":
            monkeypatch.setenv("FADKV_SCREEN", "ffma")
        D = _dict(data.atoms, data.usage, data.deltas(), w.n, w.s, 160)
        c = D.new_codes(160)
        D.encode(_t(x), c)
        torch.cuda.synchronize()
        pool = D.pool(_t(x))[0].cpu().numpy()
        outs[path] = (c.idx.cpu().numpy(), c.coef.cpu().numpy(), np.sort(pool, axis=2))
    p = PU.oparams(w)
    for g in range(w.G):
        res = O.encode_threaded(p, data.atoms[g], x[g], PU.THREADS)
        ok = ~PU.exempt_mask(res)
        for path in ("tc", "ffma"):
            idx, coef, pool = outs[path]
            assert np.array_equal(idx[g][ok], res.idx[ok])
            assert np.array_equal(pool[g][ok], np.sort(res.pool[ok], axis=1))
        assert np.array_equal(outs["tc"][0][g][ok], outs["ffma"][0][g][ok])


def test_slow_path_short_and_overflowing_lists():
    d, N, n, s = 128, 4096, 256, 8
    g = np.random.default_rng(11)
    # 32 signed copies of the standard basis: x = e_t has exactly 32 nonzero
    # scores (|r| = 1), far fewer than n, all others exactly 0
    A = np.zeros((N, d), np.float16)
    A[np.arange(N), np.arange(N) % d] = g.choice([-1.0, 1.0], N)
    x = np.zeros((1, 4, d), np.float16)
    x[0, 0, 5] = 1.0                     # short list
    x[0, 1] = 0.0                        # x = 0: every score passes, list overflows
    x[0, 2, 17] = -2.0
    x[0, 2, 99] = 0.5
    x[0, 3] = S.make_sparse_inputs(A, 1, 8, 3)[0]
    D = _dict(A[None], np.ones((1, N), np.int32), [0.5], n, s, 4)
    pool = D.pool(_t(x))[0].cpu().numpy()[0]
    c = D.new_codes(4)
    D.encode(_t(x), c)
    torch.cuda.synchronize()
    st = D.stats()[0]
    assert st["topn_slow_path"] >= 3 * 2          # pool() and encode() both took it
    p = O.Params(N, d, n, s)
    res = O.encode(p, A, x[0])
    for v in range(4):
        assert np.array_equal(np.sort(pool[v]), np.sort(res.pool[v])), v
    # every tie here is exact (equal |r| or |a| in both precisions), so the
    # index rule decides it identically on both sides: no exemption
    idx, coef, rel = (t.cpu().numpy()[0] for t in (c.idx, c.coef, c.relres))
    assert np.array_equal(idx, res.idx)
    for v in range(4):
        cn = np.linalg.norm(res.coef[v])
        assert np.linalg.norm(coef[v] - res.coef[v]) <= PU.COEF_TOL * cn + 1e-7
        assert abs(rel[v] - res.relres[v]) <= PU.RELRES_TOL * res.relres[v] + 1e-7


def test_overflowing_record_scores_recomputed():
    """Forty atoms of the first 128-atom chunk are near-copies of x's
    direction, so x keeps more scores in that chunk than a record holds
    (27): the record keeps its masks, and the selection recomputes the kept
    atoms' scores on the FP32 pipe instead of redoing the whole vector.  The
    next vector of the tile (whose record the overflow ran into) takes the
    same path.  Neither vector needs the slow path, and pools and codes
    match the oracle."""
    d, N, n, s = 128, 4096, 256, 8
    g = np.random.default_rng(21)
    A = g.standard_normal((N, d))
    u = g.standard_normal(d)
    u /= np.linalg.norm(u)
    A[:40] = u + 0.5 * g.standard_normal((40, d)) / np.sqrt(d)
    A = (A / np.linalg.norm(A, axis=1, keepdims=True)).astype(np.float16)
    x = np.empty((1, 3, d), np.float16)
    x[0, 0] = (3.0 * u + 0.3 * g.standard_normal(d) / np.sqrt(d)).astype(np.float16)
    x[0, 1] = S.make_sparse_inputs(A[100:], 1, s, 5)[0]
    x[0, 2] = S.make_sparse_inputs(A[100:], 1, s, 6)[0]
    D = _dict(A[None], np.ones((1, N), np.int32), [0.5], n, s, 3)
    pool = D.pool(_t(x))[0].cpu().numpy()[0]
    c = D.new_codes(3)
    D.encode(_t(x), c)
    torch.cuda.synchronize()
    assert D.stats()[0]["topn_slow_path"] == 0
    p = O.Params(N, d, n, s)
    res = O.encode(p, A, x[0])
    assert len(set(range(40)) & set(res.pool[0].tolist())) == 40      # the chunk's 40 atoms are all kept
    ok = ~PU.exempt_mask(res)
    for v in range(3):
        if ok[v]:
            assert np.array_equal(np.sort(pool[v]), np.sort(res.pool[v])), v
    idx, coef, rel = (t.cpu().numpy()[0] for t in (c.idx, c.coef, c.relres))
    PU.assert_encode_ok(PU.compare_encode(res, idx, coef, rel, pool, p, A, x[0]))


def test_more_candidates_than_the_selection_holds():
    """A vector with far more candidates than the selection kernel's 2n-key
    buffer, none of its 128-atom records overflowing (512 near-copies of x's
    direction, one in every 8 atoms): the selection hands it to the exact
    slow path, and pool and code match the oracle."""
    d, N, n, s = 128, 4096, 128, 8
    g = np.random.default_rng(13)
    A = g.standard_normal((N, d))
    u = g.standard_normal(d)
    u /= np.linalg.norm(u)
    near = np.arange(0, N, 8)
    A[near] = u + g.standard_normal((near.size, d)) / np.sqrt(d)
    A = (A / np.linalg.norm(A, axis=1, keepdims=True)).astype(np.float16)
    x = np.empty((1, 2, d), np.float16)
    x[0, 0] = (3.0 * u).astype(np.float16)
    x[0, 1] = S.make_sparse_inputs(A, 1, s, 7)[0]      # an ordinary vector beside it
    D = _dict(A[None], np.ones((1, N), np.int32), [0.5], n, s, 2)
    pool = D.pool(_t(x))[0].cpu().numpy()[0]
    c = D.new_codes(2)
    D.encode(_t(x), c)
    torch.cuda.synchronize()
    assert D.stats()[0]["topn_slow_path"] >= 2            # pool() and encode(): vector 0
    p = O.Params(N, d, n, s)
    res = O.encode(p, A, x[0])
    ok = ~PU.exempt_mask(res)                              # no near tie at the Top-n cut
    for v in range(2):
        if ok[v]:
            assert np.array_equal(np.sort(pool[v]), np.sort(res.pool[v])), v
    idx, coef, rel = (t.cpu().numpy()[0] for t in (c.idx, c.coef, c.relres))
    PU.assert_encode_ok(PU.compare_encode(res, idx, coef, rel, pool, p, A, x[0]))


def test_scores_far_above_the_threshold_are_kept_exactly():
    """A dictionary with one atom 300 times longer than the others: the
    vector along it scores hundreds of times its threshold, and the vector
    beside it (a sparse mixture) scores well above it on the long atom too.
    The screening records hold every kept score as an exact binary32 value,
    so neither vector needs the slow path, and pools and codes match the
    oracle."""
    d, N, n, s = 128, 4096, 256, 8
    g = np.random.default_rng(14)
    A = g.standard_normal((N, d))
    A /= np.linalg.norm(A, axis=1, keepdims=True)
    A[777] *= 300.0
    A = A.astype(np.float16)
    x = np.empty((1, 2, d), np.float16)
    x[0, 0] = (A[777].astype(np.float64) / 300.0 + 0.05 * g.standard_normal(d) / np.sqrt(d)).astype(np.float16)
    x[0, 1] = S.make_sparse_inputs(A[:700], 1, s, 8)[0]
    D = _dict(A[None], np.ones((1, N), np.int32), [0.5], n, s, 2)
    pool = D.pool(_t(x))[0].cpu().numpy()[0]
    c = D.new_codes(2)
    D.encode(_t(x), c)
    torch.cuda.synchronize()
    assert D.stats()[0]["topn_slow_path"] == 0
    p = O.Params(N, d, n, s)
    res = O.encode(p, A, x[0])
    assert 777 in res.pool[0] and 777 in res.pool[1]
    ok = ~PU.exempt_mask(res)
    for v in range(2):
        if ok[v]:
            assert np.array_equal(np.sort(pool[v]), np.sort(res.pool[v])), v
    idx, coef, rel = (t.cpu().numpy()[0] for t in (c.idx, c.coef, c.relres))
    PU.assert_encode_ok(PU.compare_encode(res, idx, coef, rel, pool, p, A, x[0]))


@pytest.mark.parametrize("name,G,V", [("decode_3b", 3, 200), ("decode_8b", 2, 64)])
def test_greedy_kernels_agree(monkeypatch, name, G, V):
    """Both greedy kernels match the oracle on coefficients and residuals as
    well as ids: the batch-OMP kernel over the Gram matrices (behind the
    tensor-core screening, the default) and the FP32-pipe kernel (behind the
    FP32 screening, FADKV_SCREEN=ffma)."""
    from dataclasses import replace
    w = replace(S.WORKLOADS[name], G=G)
    data = S.WorkloadData(w)
    x = data.inputs(0, V)
    outs = {}
    paths = ("gram", "ffma")
    for path in paths:
        if path == "ffma":
            monkeypatch.setenv("FADKV_SCREEN", "ffma")
        D = _dict(data.atoms, data.usage, data.deltas(), w.n, w.s, V)
        c = D.new_codes(V)
        D.encode(_t(x), c)
        torch.cuda.synchronize()
        outs[path] = tuple(t.cpu().numpy() for t in (c.idx, c.coef, c.relres))
    p = PU.oparams(w)
    for g in range(w.G):
        res = O.encode_threaded(p, data.atoms[g], x[g], PU.THREADS)
        for path in paths:
            idx, coef, rel = outs[path]
            PU.assert_encode_ok(PU.compare_encode(res, idx[g], coef[g], rel[g]))


@pytest.mark.parametrize("case", ["crowded_tie", "rank_tie", "whole_bucket"])
def test_select_exact_ties(case):
    """Top-n selection with exact ties at the cut (32 signed copies of each
    basis vector, x a combination of basis vectors): the pool must be the
    oracle's -- all atoms above the cut plus the lowest-index tied ones --
    whichever branch of the selection kernel decides the boundary."""
    d, N, s = 128, 4096, 8
    g = np.random.default_rng(12)
    A = np.zeros((N, d), np.float16)
    A[np.arange(N), np.arange(N) % d] = g.choice([-1.0, 1.0], N)
    x = np.zeros((1, 1, d), np.float32)
    if case == "crowded_tie":      # 512 atoms tie at |r| = 1; n = 256 of them
        n = 256
        x[0, 0, :16] = 1.0
    elif case == "rank_tie":       # 224 above the cut, 32 tied at the cut, 16 taken
        n = 240
        x[0, 0, :7] = 2.0
        x[0, 0, 7] = 1.0
        x[0, 0, 8] = 0.9
    else:                          # the boundary bucket is taken whole
        n = 256
        x[0, 0, :7] = 2.0
        x[0, 0, 7] = 1.0
        x[0, 0, 8] = 0.9
    x = x.astype(np.float16)
    D = _dict(A[None], np.ones((1, N), np.int32), [0.5], n, s, 1)
    pool = D.pool(_t(x))[0].cpu().numpy()[0, 0]
    assert D.stats()[0]["topn_slow_path"] == 0      # decided by the selection kernel
    res = O.encode(O.Params(N, d, n, s), A, x[0])
    assert sorted(pool) == sorted(res.pool[0])



@pytest.mark.parametrize("N,d,G,V", [(4096, 128, 3, 1), (4096, 128, 2, 7), (8192, 128, 2, 16), (1024, 64, 2, 12)])
def test_small_batch_scores_against_float64(N, d, G, V):
    """A few vectors per dictionary fill a small part of the 128-row tile
    (the rest of the epilogue's warps skip their units): raw scores within
    the fp32 accumulation bound."""
    atoms = np.stack([S.make_dictionary(N, d, np.float16, 9, g) for g in range(G)])
    x = np.stack([S.make_sparse_inputs(atoms[g], V, 8, 8, 100 + g) for g in range(G)])
    D = _dict(atoms, np.ones((G, N), np.int32), [0.5] * G, 64, 8, V)
    sc = D.scores(_t(x)).cpu().numpy().astype(np.float64)
    for g in range(G):
        A = atoms[g].astype(np.float64)
        X = x[g].astype(np.float64)
        exact = X @ A.T
        bound = d * 2.0 ** -24 * (np.abs(X) @ np.abs(A).T) + 1e-30
        err = np.abs(sc[g] - exact)
        assert np.all(err <= bound), float(np.max(err / bound))


@pytest.mark.parametrize("name,V", [("decode_3b", 1), ("decode_3b", 8), ("decode_3b", 16), ("decode_3b", 33),
                                    ("decode_3b", 100), ("decode_8b", 33)])
def test_small_batch_encode_matches_oracle(name, V):
    """Encodes of small and ragged batches (1, 8, 16, 33 and 100 vectors: one,
    two or four of the epilogue's lane groups hold rows; and the 8B shape's
    n = 512, s = 16) match the oracle: pools off near ties, coefficients and
    residuals within the parity bar."""
    from dataclasses import replace
    w = replace(S.WORKLOADS[name], G=2 if name == "decode_8b" else 3, V=V)
    data = S.WorkloadData(w)
    D = _dict(data.atoms, data.usage, data.deltas(), w.n, w.s, V)
    x = data.inputs(0, V)
    c = D.new_codes(V)
    D.encode(_t(x), c)
    assert sum(st["topn_slow_path"] for st in D.stats()) == 0
    idx, coef, rel = c.idx.cpu().numpy(), c.coef.cpu().numpy(), c.relres.cpu().numpy()
    p = O.Params(w.N, w.d, w.n, w.s)
    for g in range(w.G):
        res = O.encode_threaded(p, data.atoms[g], x[g], PU.THREADS)
        PU.assert_encode_ok(PU.compare_encode(res, idx[g], coef[g], rel[g]))
