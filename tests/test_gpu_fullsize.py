"""The CUDA path at the workloads' full sizes, in the launch configuration the
benchmark uses, against the CPU oracle on sampled outputs.

Every shape runs whole on the GPU through the C ABI (one call covering every
dictionary; the prefill shape in the library's vector chunks).  The oracle
then recomputes a seeded sample of the vectors one by one; the sampled codes
must match with the parity tolerances and near-tie rules of
tests/parity_util.py.  For the 3B decode step the adaptation of two whole
dictionaries is replayed by the oracle as well, and the reconstruction of the
sampled vectors is checked against the oracle's.
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


def _run_step(w, x):
    """One full step on the GPU: encode, adapt, reconstruct."""
    from dictionary_sparse_kv_gb300 import fadkv as F
    data = S.WorkloadData(w)
    atoms0, usage0 = data.atoms.copy(), data.usage.copy()
    D = F.Dictionary(_t(atoms0), _t(usage0), data.deltas(), w.n, w.s, x.shape[1])
    c = D.new_codes(x.shape[1])
    xh = torch.empty((w.G, x.shape[1], w.d), dtype=torch.float32, device=DEV)
    D.step(_t(x), c, xh)
    torch.cuda.synchronize()
    out = {k: getattr(c, k).cpu().numpy() for k in ("idx", "coef", "relres", "repl_id", "repl_coef")}
    out["xhat"] = xh.cpu().numpy()
    out["atoms"] = D.atoms.cpu().numpy()
    out["usage"] = D.usage.cpu().numpy()
    out["stats"] = D.stats()
    return data, atoms0, usage0, out


def _check_sample(w, atoms0, x, out, pairs):
    """Oracle encode of each sampled (g, v) against the GPU codes."""
    p = PU.oparams(w)
    exempt = checked = 0
    for g, v in pairs:
        res = O.encode(p, atoms0[g], np.ascontiguousarray(x[g, v:v + 1]))
        rep = PU.compare_encode(res, out["idx"][g, v:v + 1], out["coef"][g, v:v + 1], out["relres"][g, v:v + 1])
        assert not rep.mismatched_idx, (g, v, out["idx"][g, v], res.idx[0])
        assert rep.worst_coef <= PU.COEF_TOL, (g, v, rep.worst_coef)
        assert rep.worst_relres <= PU.RELRES_TOL, (g, v, rep.worst_relres)
        exempt += rep.exempt
        checked += rep.checked
    assert exempt <= max(2, 0.05 * len(pairs)), f"{exempt} of {len(pairs)} sampled vectors exempt"
    return checked


def _pairs(w, V, count, seed):
    g = np.random.default_rng(seed)
    return [(int(a), int(b)) for a, b in zip(g.integers(0, w.G, count), g.integers(0, V, count))]


def test_decode_3b_full_step():
    w = S.WORKLOADS["decode_3b"]                       # 56 dictionaries x 128 vectors: the benchmark's step
    data = S.WorkloadData(w)
    x = data.inputs(0)
    data, atoms0, usage0, out = _run_step(w, x)
    pairs = _pairs(w, w.V, 64, 31)
    assert _check_sample(w, atoms0, x, out, pairs) >= 60
    # the adaptation of two whole dictionaries, replayed by the oracle on the
    # GPU's codes
    p = PU.oparams(w)
    for g in (0, w.G - 1):
        oat, ous = atoms0[g].copy(), usage0[g].copy()
        r = O.adapt(p, oat, ous, x[g], out["idx"][g], out["coef"][g].astype(np.float64),
                    out["relres"][g].astype(np.float64), data.deltas()[g])
        assert np.array_equal(out["usage"][g], ous), g
        assert np.array_equal(out["repl_id"][g], r.repl_id), g
        assert out["stats"][g]["replaced"] == r.replaced and out["stats"][g]["overflow"] == r.overflow
    # reconstruction of the sampled vectors from the GPU's codes
    for g, v in pairs[:16]:
        ox = O.reconstruct(p, out["atoms"][g], out["idx"][g, v:v + 1], out["coef"][g, v:v + 1].astype(np.float64),
                           out["repl_id"][g, v:v + 1], out["repl_coef"][g, v:v + 1].astype(np.float64))[0]
        assert np.linalg.norm(out["xhat"][g, v] - ox) <= PU.XHAT_TOL * np.linalg.norm(ox) + 1e-6


def test_decode_8b_full_step():
    w = S.WORKLOADS["decode_8b"]                       # 64 dictionaries x 512 vectors, N=8192, n=512, s=16
    data = S.WorkloadData(w)
    x = data.inputs(0)
    _, atoms0, _, out = _run_step(w, x)
    assert _check_sample(w, atoms0, x, out, _pairs(w, w.V, 32, 41)) >= 28


def test_prefill_3b_16k_full():
    w = S.WORKLOADS["prefill_3b_16k"]                  # 2 dictionaries x 131072 vectors, in vector chunks
    data = S.WorkloadData(w)
    x = data.inputs(0)
    data, atoms0, usage0, out = _run_step(w, x)
    assert np.all(out["idx"] >= 0)
    assert _check_sample(w, atoms0, x, out, _pairs(w, w.V, 48, 51)) >= 44
    # the adaptation of both dictionaries (1M usage increments each), replayed
    # by the oracle on the GPU's codes
    p = PU.oparams(w)
    for g in range(w.G):
        oat, ous = atoms0[g].copy(), usage0[g].copy()
        r = O.adapt(p, oat, ous, x[g], out["idx"][g], out["coef"][g].astype(np.float64),
                    out["relres"][g].astype(np.float64), data.deltas()[g])
        assert np.array_equal(out["usage"][g], ous), g
        assert np.array_equal(out["repl_id"][g], r.repl_id), g
        assert out["stats"][g]["replaced"] == r.replaced and out["stats"][g]["overflow"] == r.overflow
