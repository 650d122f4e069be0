"""PL encode (screening + one ridge fit over the Top-s atoms) against the
CPU oracle, through the C ABI (needs a GPU).

Tolerances as for the greedy coder (tests/parity_util.py): the selected set
exactly, except for vectors the oracle shows on a near tie at the Top-s cut
(relative gap below 1e-5), where the GPU's set may differ only inside the
tie band; coefficients norm-wise within 1e-3, relres within 1e-3 relative.
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


def _small(name, **kw):
    from dataclasses import replace
    return replace(S.WORKLOADS[name], **kw)


def _dict(w, data, max_batch):
    from dictionary_sparse_kv_gb300 import fadkv as F
    return F.Dictionary(_t(data.atoms), _t(data.usage), data.deltas(), w.n, w.s, max_batch)


def _encode_pl(D, x):
    codes = D.new_codes(x.shape[1])
    D.encode_pl(_t(x), codes)
    torch.cuda.synchronize()
    return codes


def _compare(w, atoms, x, res, idx, coef, rel, vs=None):
    """Checks the vectors vs (all by default); returns the number on a tie."""
    ties = 0
    for v in (range(x.shape[0]) if vs is None else vs):
        if res.idx[v][0] < 0:
            assert np.all(idx[v] == -1) and np.isnan(rel[v])
            continue
        assert np.all(np.diff(idx[v]) > 0), f"ids not ascending at {v}"
        if res.cut_gap[v] < PU.CUT_GAP:
            ties += 1
            r = np.abs(atoms.astype(np.float64) @ x[v].astype(np.float64))
            cut = np.sort(r)[::-1][w.s - 1]
            for j in set(idx[v].tolist()) ^ set(res.idx[v].tolist()):
                assert abs(r[j] - cut) <= 2 * PU.CUT_GAP * cut, (v, j)
            continue
        assert np.array_equal(idx[v], res.idx[v]), (v, idx[v], res.idx[v])
        cn = np.linalg.norm(res.coef[v])
        dc = np.linalg.norm(coef[v].astype(np.float64) - res.coef[v])
        assert dc <= PU.COEF_TOL * cn + 1e-12, (v, dc, cn)
        ro = res.relres[v]
        assert abs(float(rel[v]) - ro) <= PU.RELRES_TOL * ro + 1e-7, (v, rel[v], ro)
    return ties


CASES = [
    ("tiny", dict(), None),                         # binary32, FP32 screening + radix Top-s
    ("decode_3b", dict(G=3), 200),                  # tensor-core screening, ragged tail
    ("decode_8b", dict(G=2), 70),                   # s = 16, N = 8192
    ("adapt_stress", dict(), 96),
    ("decode_3b", dict(G=2, N=1984), 50),           # binary16, N not a multiple of 128: FP32 screening
    ("decode_3b", dict(G=1, s=1), 64),
    ("decode_3b", dict(G=1, s=32, n=64), 64),       # the largest s
    ("decode_3b", dict(G=2), 1),                    # one vector a dictionary: one live epilogue warp
    ("decode_3b", dict(G=2, d=64, N=2048, n=128, s=4), 40),   # binary16, d = 64 tiles
]


@pytest.mark.parametrize("name,over,V", CASES, ids=[f"{c[0]}-{i}" for i, c in enumerate(CASES)])
def test_pl_matches_oracle(name, over, V):
    w = _small(name, **over)
    data = S.WorkloadData(w)
    V = w.V if V is None else V
    x = data.inputs(0, V)
    D = _dict(w, data, V)
    c = _encode_pl(D, x)
    idx, coef, rel = (t.cpu().numpy() for t in (c.idx, c.coef, c.relres))
    p = PU.oparams(w)
    ties = 0
    for g in range(w.G):
        res = O.encode_pl(p, data.atoms[g], x[g])
        ties += _compare(w, data.atoms[g], x[g], res, idx[g], coef[g], rel[g])
    assert ties <= max(2, 0.02 * w.G * V)


def test_pl_special_inputs():
    """Zero vector (ids 0..s-1, c = 0, relres 0), non-finite vectors (ids -1,
    relres NaN, counted, status bit) and an input equal to an atom."""
    w = _small("decode_3b", G=1)
    data = S.WorkloadData(w)
    x = data.inputs(0, 6)
    x[0, 0] = 0
    x[0, 1, 3] = np.nan
    x[0, 2, 7] = -np.inf
    x[0, 3] = data.atoms[0, 1234]
    D = _dict(w, data, 6)
    c = _encode_pl(D, x)
    idx, coef, rel = (t.cpu().numpy()[0] for t in (c.idx, c.coef, c.relres))
    assert list(idx[0]) == list(range(w.s)) and np.all(coef[0] == 0) and rel[0] == 0
    for v in (1, 2):
        assert np.all(idx[v] == -1) and np.all(coef[v] == 0) and np.isnan(rel[v])
    assert 1234 in idx[3]
    st = D.stats()[0]
    assert st["nonfinite"] == 2 and (st["status"] & 1)
    res = O.encode_pl(PU.oparams(w), data.atoms[0], x[0])
    _compare(w, data.atoms[0], x[0], res, idx, coef, rel, vs=[0, 3, 4, 5])


def test_pl_sequence_adapt_and_reconstruct():
    """A PL batch is an encode: a second encode before adapt is refused;
    adapt and reconstruct on PL codes match the oracle's adapt and
    reconstruct of the same codes."""
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = _small("adapt_stress", off_frac=0.8)
    data = S.WorkloadData(w)
    V = 128
    x = data.inputs(0, V)
    D = _dict(w, data, V)
    atoms0 = D.atoms.cpu().numpy().copy()
    usage0 = D.usage.cpu().numpy().copy()
    c = _encode_pl(D, x)
    with pytest.raises(F.FadkvError) as e:
        D.encode_pl(_t(x), c)
    assert e.value.status == 3
    with pytest.raises(F.FadkvError):
        D.encode(_t(x), c)
    D.adapt(_t(x), c)
    xh = torch.empty((w.G, V, w.d), dtype=torch.float32, device=DEV)
    D.reconstruct(c, xh, True)
    torch.cuda.synchronize()
    idx = c.idx.cpu().numpy()
    coef = c.coef.cpu().numpy().astype(np.float64)
    rel = c.relres.cpu().numpy().astype(np.float64)
    gid, gco = c.repl_id.cpu().numpy(), c.repl_coef.cpu().numpy()
    gat, gus, gx = D.atoms.cpu().numpy(), D.usage.cpu().numpy(), xh.cpu().numpy()
    p = PU.oparams(w)
    total = 0
    for g in range(w.G):
        oat, ous = atoms0[g].copy(), usage0[g].copy()
        r = O.adapt(p, oat, ous, x[g], idx[g], coef[g], rel[g], data.deltas()[g])
        assert np.array_equal(gus[g], ous) and np.array_equal(gid[g], r.repl_id)
        rep = r.repl_id >= 0
        assert np.allclose(gco[g][rep], r.repl_coef[rep], rtol=1e-5)
        bnd = PU.replacement_bounds(atoms0[g], x[g], idx[g], coef[g], r.repl_id, w.s)
        assert PU.compare_atoms(gat[g], oat, r.repl_id[rep], bnd) <= 1.0
        ox = O.reconstruct(p, gat[g], idx[g], coef[g], gid[g], gco[g].astype(np.float64))
        err = np.linalg.norm(gx[g] - ox, axis=1)
        assert np.all(err <= PU.XHAT_TOL * np.linalg.norm(ox, axis=1) + 1e-6)
        total += r.replaced
    assert total > 0


def test_pl_full_size_sampled():
    """decode_3b at full size (56 dictionaries x 128 vectors, one call):
    sampled vectors against the oracle, and the set property on every vector
    (s distinct ascending ids in range)."""
    w = S.WORKLOADS["decode_3b"]
    data = S.WorkloadData(w)
    x = data.inputs(0)
    D = _dict(w, data, w.V)
    c = _encode_pl(D, x)
    idx, coef, rel = (t.cpu().numpy() for t in (c.idx, c.coef, c.relres))
    assert np.all(np.diff(idx, axis=2) > 0) and idx.min() >= 0 and idx.max() < w.N
    assert np.all(np.isfinite(rel)) and np.all(rel >= 0)
    p = PU.oparams(w)
    rng = np.random.default_rng(77)
    for g in rng.choice(w.G, 8, replace=False):
        vs = rng.choice(w.V, 8, replace=False)
        res = O.encode_pl(p, data.atoms[g], np.ascontiguousarray(x[g][vs]))
        _compare(w, data.atoms[g], np.ascontiguousarray(x[g][vs]), res, idx[g][vs], coef[g][vs], rel[g][vs])
