"""Append-only growth (fadkv_adapt_append) against the CPU oracle, through the
C ABI (needs a GPU), next to the fixed-size adaptation it is contrasted
with.

A dictionary with capacity N starts with N0 atoms; the other rows are free
slots (zero rows, usage -1).  The GPU's usage counts and appended ids must
equal the oracle's exactly, appended atoms within one storage ulp plus the
fp32 bound of forming e/||e|| (tests/parity_util.py), and the dictionary
size (rows with usage >= 0) must grow by one per flagged vector until the
free slots run out, while the fixed-size dictionary never grows.
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


def _with_free_slots(data, n_free):
    """Atoms and usage of `data` with the last n_free rows turned into free
    slots (zero rows, usage -1)."""
    atoms = data.atoms.copy()
    usage = data.usage.copy()
    atoms[:, -n_free:] = 0
    usage[:, -n_free:] = -1
    return atoms, usage


def _check_adapt(w, data, x, c, atoms0, usage0, gat, gus, append):
    idx = c.idx.cpu().numpy()
    coef = c.coef.cpu().numpy().astype(np.float64)
    rel = c.relres.cpu().numpy().astype(np.float64)
    gid, gco = c.repl_id.cpu().numpy(), c.repl_coef.cpu().numpy()
    p = PU.oparams(w)
    out = []
    for g in range(w.G):
        oat, ous = atoms0[g].copy(), usage0[g].copy()
        r = O.adapt(p, oat, ous, x[g], idx[g], coef[g], rel[g], data.deltas()[g], append=append)
        assert np.array_equal(gus[g], ous), g
        assert np.array_equal(gid[g], r.repl_id), g
        rep = r.repl_id >= 0
        assert np.allclose(gco[g][rep], r.repl_coef[rep], rtol=1e-5)
        same = np.setdiff1d(np.arange(w.N), r.repl_id[rep])
        assert np.array_equal(gat[g][same], atoms0[g][same])
        bnd = PU.replacement_bounds(atoms0[g], x[g], idx[g], coef[g], r.repl_id, w.s)
        assert PU.compare_atoms(gat[g], oat, r.repl_id[rep], bnd) <= 1.0
        out.append(r)
    return out


@pytest.mark.parametrize("n_free", [512, 7])      # plenty of room / capacity runs out
def test_append_matches_oracle(n_free):
    from dataclasses import replace
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = replace(S.WORKLOADS["adapt_stress"], off_frac=1.2, deltas=(0.5, 0.6))   # most vectors flagged
    data = S.WorkloadData(w)
    atoms0, usage0 = _with_free_slots(data, n_free)
    V = 128
    x = data.inputs(0, V)
    D = F.Dictionary(_t(atoms0), _t(usage0), data.deltas(), w.n, w.s, V)
    c = D.new_codes(V)
    D.encode(_t(x), c)
    D.adapt_append(_t(x), c)
    torch.cuda.synchronize()
    gat, gus = D.atoms.cpu().numpy(), D.usage.cpu().numpy()
    res = _check_adapt(w, data, x, c, atoms0, usage0, gat, gus, True)
    st = D.stats()
    for g, r in enumerate(res):
        assert st[g]["replaced"] == r.replaced and st[g]["overflow"] == r.overflow
        appended = r.repl_id[r.repl_id >= 0]
        assert np.all(appended >= w.N - n_free)          # only free slots are written
        assert int((gus[g] >= 0).sum()) == w.N - n_free + r.replaced
    if n_free == 7:
        assert all(r.overflow > 0 for r in res)


def test_append_grows_fixed_size_does_not():
    """Several decode steps side by side on the same inputs: the append-only
    dictionary grows by the number of appended atoms each step (checked
    against the oracle's adaptation of the GPU's codes every step), the
    fixed-size one keeps N atoms; reconstruction of the last step's codes
    matches the oracle in both."""
    from dataclasses import replace
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = replace(S.WORKLOADS["adapt_stress"], off_frac=1.2, deltas=(0.5, 0.6))
    data = S.WorkloadData(w)
    n_free = 1024
    at_a, us_a = _with_free_slots(data, n_free)
    V = 64
    Da = F.Dictionary(_t(at_a), _t(us_a), data.deltas(), w.n, w.s, V)
    Df = F.Dictionary(_t(data.atoms), _t(data.usage), data.deltas(), w.n, w.s, V)
    sizes = [np.full(w.G, w.N - n_free)]
    for step in range(3):
        x = data.inputs(step, V)
        for D, app in ((Da, True), (Df, False)):
            a0, u0 = D.atoms.cpu().numpy().copy(), D.usage.cpu().numpy().copy()
            c = D.new_codes(V)
            D.encode(_t(x), c)
            (D.adapt_append if app else D.adapt)(_t(x), c)
            torch.cuda.synchronize()
            gat, gus = D.atoms.cpu().numpy(), D.usage.cpu().numpy()
            res = _check_adapt(w, data, x, c, a0, u0, gat, gus, app)
            if app:
                sizes.append((gus >= 0).sum(axis=1))
                assert np.array_equal(sizes[-1], sizes[-2] + np.array([r.replaced for r in res]))
            else:
                assert int((gus < 0).sum()) == 0
            xh = torch.empty((w.G, V, w.d), dtype=torch.float32, device=DEV)
            D.reconstruct(c, xh, True)
            torch.cuda.synchronize()
            gx = xh.cpu().numpy()
            p = PU.oparams(w)
            for g in range(w.G):
                ox = O.reconstruct(p, gat[g], c.idx.cpu().numpy()[g], c.coef.cpu().numpy()[g].astype(np.float64),
                                   c.repl_id.cpu().numpy()[g], c.repl_coef.cpu().numpy()[g].astype(np.float64))
                err = np.linalg.norm(gx[g] - ox, axis=1)
                assert np.all(err <= PU.XHAT_TOL * np.linalg.norm(ox, axis=1) + 1e-6)
    assert np.all(sizes[-1] > sizes[0])


def test_append_sequence_contract():
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = S.WORKLOADS["tiny"]
    data = S.WorkloadData(w)
    D = F.Dictionary(_t(data.atoms), _t(data.usage), data.deltas(), w.n, w.s, 16)
    x = _t(data.inputs(0, 16))
    c = D.new_codes(16)
    with pytest.raises(F.FadkvError) as e:
        D.adapt_append(x, c)
    assert e.value.status == 3
    D.encode(x, c)
    D.adapt_append(x, c)
    with pytest.raises(F.FadkvError):
        D.adapt(x, c)
