"""CUDA path against the CPU oracle, through the C ABI (needs a GPU).

Every test feeds the same seeded synthetic inputs to the library (via the
Python binding of include/fadkv.h) and to the oracle, and compares with the
tolerances of tests/parity_util.py.
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


def make_dict(w, data, max_batch, lambda_abs=1e-4, lambda_rel=0.20):
    from dictionary_sparse_kv_gb300 import fadkv as F
    return F.Dictionary(_t(data.atoms), _t(data.usage), data.deltas(), w.n, w.s, max_batch,
                        lambda_abs, lambda_rel)


def small(w, **kw):
    from dataclasses import replace
    return replace(w, **kw)


def gpu_encode(D, x):
    codes = D.new_codes(x.shape[1])
    D.encode(_t(x), codes)
    torch.cuda.synchronize()
    return codes


# ---------------------------------------------------------------------------
# Top-n pool
# ---------------------------------------------------------------------------

CASES = [
    ("tiny", dict(), None),
    ("decode_3b", dict(G=3), 200),          # ragged: 200 vectors per dictionary
    ("decode_8b", dict(G=2), 70),
    ("adapt_stress", dict(), 96),
]


@pytest.mark.parametrize("name,over,V", CASES, ids=[c[0] for c in CASES])
def test_pool_matches_oracle(name, over, V):
    w = small(S.WORKLOADS[name], **over)
    data = S.WorkloadData(w)
    V = w.V if V is None else V
    x = data.inputs(0, V)
    D = make_dict(w, data, V)
    pool, _ = D.pool(_t(x))
    pool = pool.cpu().numpy()
    p = PU.oparams(w)
    ties = 0
    for g in range(w.G):
        res = O.encode_threaded(p, data.atoms[g], x[g], PU.THREADS)
        for v in range(V):
            if res.cut_gap[v] < PU.CUT_GAP:
                # near tie at the cut: the pools may differ only inside the band
                ties += 1
                PU.check_cut_tie(p, data.atoms[g], x[g], res, pool[g], v)
                continue
            assert np.array_equal(np.sort(pool[g, v]), np.sort(res.pool[v])), (g, v)
    assert ties <= max(3, 0.10 * w.G * V)


def test_pool_tie_rule_exact_zeros():
    """Signed-permutation atoms: all but 4 scores are exactly 0, so the pool is
    the support plus the lowest-index atoms (exact, no tolerance)."""
    N = d = 64
    g = np.random.default_rng(3)
    A = np.zeros((N, d), np.float16)
    A[np.arange(N), g.permutation(N)] = g.choice([-1.0, 1.0], N)
    supp = [40, 7, 55, 13]
    x = (np.array([-3.0, 2.5, 2.0, -1.0]) @ A[supp].astype(np.float64)).astype(np.float16)
    from dictionary_sparse_kv_gb300 import fadkv as F
    D = F.Dictionary(_t(A[None]), _t(np.ones((1, N), np.int32)), [0.5], 10, 3, 1)
    pool, _ = D.pool(_t(x[None, None]))
    rest = [j for j in range(N) if j not in supp][:6]
    assert sorted(pool.cpu().numpy()[0, 0]) == sorted(supp + rest)


# ---------------------------------------------------------------------------
# Encode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,over,V", CASES, ids=[c[0] for c in CASES])
def test_encode_matches_oracle(name, over, V):
    w = small(S.WORKLOADS[name], **over)
    data = S.WorkloadData(w)
    V = w.V if V is None else V
    x = data.inputs(0, V)
    D = make_dict(w, data, V)
    gpool = D.pool(_t(x))[0].cpu().numpy()
    c = gpu_encode(D, x)
    idx, coef, rel = (t.cpu().numpy() for t in (c.idx, c.coef, c.relres))
    p = PU.oparams(w)
    for g in range(w.G):
        res = O.encode_threaded(p, data.atoms[g], x[g], PU.THREADS)
        rep = PU.compare_encode(res, idx[g], coef[g], rel[g], gpool[g], p, data.atoms[g], x[g])
        PU.assert_encode_ok(rep, max_exempt_frac=0.02)


def test_encode_special_inputs():
    """Zero vector (picks 0..s-1, c = 0, relres 0), non-finite vectors
    (idx -1, relres NaN, status bit), an input equal to an atom, and the
    same input twice in a batch (identical codes)."""
    w = small(S.WORKLOADS["decode_3b"], G=1)
    data = S.WorkloadData(w)
    x = data.inputs(0, 8)
    x[0, 0] = 0
    x[0, 1, 3] = np.nan
    x[0, 2, 7] = np.inf
    x[0, 3] = data.atoms[0, 1234]
    x[0, 5] = x[0, 4]
    D = make_dict(w, data, 8)
    c = gpu_encode(D, x)
    idx, coef, rel = (t.cpu().numpy()[0] for t in (c.idx, c.coef, c.relres))
    assert list(idx[0]) == list(range(w.s)) and np.all(coef[0] == 0) and rel[0] == 0
    for v in (1, 2):
        assert np.all(idx[v] == -1) and np.isnan(rel[v])
    assert idx[3][0] == 1234
    assert np.array_equal(idx[4], idx[5]) and np.array_equal(coef[4], coef[5]) and rel[4] == rel[5]
    st = D.stats()[0]
    assert st["nonfinite"] == 2 and (st["status"] & 1)
    res = O.encode(PU.oparams(w), data.atoms[0], x[0])
    keep = [0, 3, 4, 5, 6, 7]
    PU.assert_encode_ok(PU.compare_encode(
        O.EncodeResult(res.idx[keep], res.coef[keep], res.relres[keep], res.pool[keep], res.cut_gap[keep],
                       res.pick_gap[keep], 0), idx[keep], coef[keep], rel[keep]))


def test_encode_empty_and_single():
    w = small(S.WORKLOADS["decode_3b"], G=2)
    data = S.WorkloadData(w)
    D = make_dict(w, data, 4)
    x0 = np.zeros((2, 0, w.d), np.float16)
    c = D.new_codes(0)
    D.encode(_t(x0), c)
    D.adapt(_t(x0), c)
    x1 = data.inputs(0, 1)
    c1 = gpu_encode(D, x1)
    res = O.encode(PU.oparams(w), data.atoms[1], x1[1])
    PU.assert_encode_ok(PU.compare_encode(res, c1.idx.cpu().numpy()[1], c1.coef.cpu().numpy()[1],
                                          c1.relres.cpu().numpy()[1]))


def test_encode_deterministic():
    w = small(S.WORKLOADS["decode_3b"], G=4)
    data = S.WorkloadData(w)
    x = data.inputs(0)
    outs = []
    for _ in range(2):
        D = make_dict(w, data, w.V)
        c = gpu_encode(D, x)
        outs.append([t.cpu().numpy().tobytes() for t in (c.idx, c.coef, c.relres)])
    assert outs[0] == outs[1]


# ---------------------------------------------------------------------------
# Adapt and reconstruct
# ---------------------------------------------------------------------------

def _adapt_case(w, V, step=0):
    data = S.WorkloadData(w)
    x = data.inputs(step, V)
    D = make_dict(w, data, V)
    c = gpu_encode(D, x)
    atoms0 = D.atoms.cpu().numpy().copy()
    usage0 = D.usage.cpu().numpy().copy()
    D.adapt(_t(x), c)
    torch.cuda.synchronize()
    return data, x, D, c, atoms0, usage0


@pytest.mark.parametrize("name,over,V", [
    ("tiny", dict(), None),
    ("adapt_stress", dict(off_frac=0.8), 256),        # large residuals: many replacements
    ("decode_3b", dict(G=2, off_frac=1.2), 128),
    ("decode_3b", dict(G=2, inactive=5, off_frac=1.5), 128),   # inactive list runs out
    ("adapt_stress", dict(off_frac=0.8), 4096),       # a batch whose usage increments run over the grid
    ("decode_8b", dict(G=2, deltas=(0.25, 0.25)), 64),   # N = 8192: replacements and their Gram rows
])
def test_adapt_matches_oracle(name, over, V):
    w = small(S.WORKLOADS[name], **over)
    V = w.V if V is None else V
    data, x, D, c, atoms0, usage0 = _adapt_case(w, V)
    idx = c.idx.cpu().numpy()
    coef = c.coef.cpu().numpy().astype(np.float64)
    rel = c.relres.cpu().numpy().astype(np.float64)
    gid = c.repl_id.cpu().numpy()
    gco = c.repl_coef.cpu().numpy()
    gat = D.atoms.cpu().numpy()
    gus = D.usage.cpu().numpy()
    st = D.stats()
    p = PU.oparams(w)
    total_rep = 0
    for g in range(w.G):
        oat = atoms0[g].copy()
        ous = usage0[g].copy()
        r = O.adapt(p, oat, ous, x[g], idx[g], coef[g], rel[g], data.deltas()[g])
        assert np.array_equal(gus[g], ous), g
        assert np.array_equal(gid[g], r.repl_id), g
        rep = r.repl_id >= 0
        assert np.allclose(gco[g][rep], r.repl_coef[rep], rtol=1e-5)
        assert np.all(gco[g][~rep] == 0)
        changed = r.repl_id[rep]
        same = np.setdiff1d(np.arange(w.N), changed)
        assert np.array_equal(gat[g][same], atoms0[g][same])
        bnd = PU.replacement_bounds(atoms0[g], x[g], idx[g], coef[g], r.repl_id, w.s)
        assert PU.compare_atoms(gat[g], oat, changed, bnd) <= 1.0
        assert st[g]["replaced"] == r.replaced and st[g]["overflow"] == r.overflow
        total_rep += r.replaced
    if name != "tiny":
        assert total_rep > 0


def test_reconstruct_matches_oracle():
    w = small(S.WORKLOADS["adapt_stress"], off_frac=0.8)
    data, x, D, c, atoms0, usage0 = _adapt_case(w, 128)
    xh = torch.empty((w.G, 128, w.d), dtype=torch.float32, device=DEV)
    for with_repl in (False, True):
        D.reconstruct(c, xh, with_repl)
        torch.cuda.synchronize()
        gx = xh.cpu().numpy()
        at = D.atoms.cpu().numpy()
        p = PU.oparams(w)
        for g in range(w.G):
            ox = O.reconstruct(p, at[g], c.idx.cpu().numpy()[g], c.coef.cpu().numpy()[g].astype(np.float64),
                               c.repl_id.cpu().numpy()[g] if with_repl else None,
                               c.repl_coef.cpu().numpy()[g].astype(np.float64) if with_repl else None)
            err = np.linalg.norm(gx[g] - ox, axis=1)
            assert np.all(err <= PU.XHAT_TOL * np.linalg.norm(ox, axis=1) + 1e-6)


def test_sequence_contract_on_gpu():
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = small(S.WORKLOADS["tiny"])
    data = S.WorkloadData(w)
    D = make_dict(w, data, 16)
    x = _t(data.inputs(0, 16))
    c = D.new_codes(16)
    D.encode(x, c)
    with pytest.raises(F.FadkvError) as e:
        D.encode(x, c)
    assert e.value.status == 3
    D.adapt(x, c)
    with pytest.raises(F.FadkvError):
        D.adapt(x, c)


# ---------------------------------------------------------------------------
# Multi-step runs: GPU state against the oracle's state, step by step
# ---------------------------------------------------------------------------

def _run_steps(w, steps, V, resync=True):
    """Run `steps` encode+adapt steps on the GPU; at every step check the
    encode against the oracle on the GPU's current state and the adapt
    against the oracle's adapt of the GPU's codes (state resynced from the
    GPU each step, so an exempt near-tie cannot make the two drift)."""
    data = S.WorkloadData(w)
    D = make_dict(w, data, V)
    p = PU.oparams(w)
    exempt = checked = reps = 0
    for t in range(steps):
        x = data.inputs(t, V)
        atoms0 = D.atoms.cpu().numpy().copy()
        usage0 = D.usage.cpu().numpy().copy()
        gpool = D.pool(_t(x))[0].cpu().numpy()        # the pools this step's encode uses
        c = gpu_encode(D, x)
        D.adapt(_t(x), c)
        torch.cuda.synchronize()
        idx, coef, rel = (a.cpu().numpy() for a in (c.idx, c.coef, c.relres))
        for g in range(w.G):
            res = O.encode_threaded(p, atoms0[g], x[g], PU.THREADS)
            rep = PU.compare_encode(res, idx[g], coef[g], rel[g], gpool[g], p, atoms0[g], x[g])
            PU.assert_encode_ok(rep)
            exempt += rep.exempt
            checked += rep.checked
            oat, ous = atoms0[g].copy(), usage0[g].copy()
            r = O.adapt(p, oat, ous, x[g], idx[g], coef[g].astype(np.float64), rel[g].astype(np.float64),
                        data.deltas()[g])
            assert np.array_equal(D.usage.cpu().numpy()[g], ous)
            assert np.array_equal(c.repl_id.cpu().numpy()[g], r.repl_id)
            bnd = PU.replacement_bounds(atoms0[g], x[g], idx[g], coef[g], r.repl_id, w.s)
            assert PU.compare_atoms(D.atoms.cpu().numpy()[g], oat, r.repl_id[r.repl_id >= 0], bnd) <= 1.0
            reps += r.replaced
    return exempt, checked, reps, D


def test_multistep_tiny_batch_and_sequential():
    """Tiny check: one batch of 256, and 32 one-vector steps (sequential
    per-token semantics are the V = 1 case of batch semantics)."""
    w = S.WORKLOADS["tiny"]
    _run_steps(w, 2, 256)
    _run_steps(w, 32, 1)


def test_multistep_adaptation_stress():
    """Drifting sources: replacements happen, N stays fixed, usage conserved."""
    from dataclasses import replace
    w = replace(S.WORKLOADS["adapt_stress"], drift_period=2, drift_frac=0.5)
    ex, ch, reps, D = _run_steps(w, 6, 64)
    assert reps > 0
    assert D.atoms.shape == (2, w.N, w.d)


@pytest.mark.parametrize("s,n,V", [(4, 128, 150), (8, 64, 33)], ids=["s4_n128_V150", "s8_n64_V33"])
def test_multistep_binary16_d64(s, n, V):
    """Binary16 dictionaries of d = 64 through the whole tensor-core path
    (screening with 64-wide tiles, the selection, the Gram greedy with fewer
    picks than its compile-time maximum, adapt and the Gram update): three
    steps, each against the oracle on the GPU's state."""
    from dataclasses import replace
    w = replace(S.WORKLOADS["decode_3b"], G=2, d=64, N=2048, n=n, s=s, off_frac=0.3)
    ex, ch, reps, D = _run_steps(w, 3, V)
    assert ch > 0
    assert D.atoms.shape == (2, w.N, w.d)


def test_multistep_8b_shape_with_replacements():
    """The 8B shape (N = 8192, n = 512, s = 16) over three steps with a low
    threshold: atoms are replaced every step, so every later encode reads
    Gram rows and columns the update rewrote; each step against the oracle
    on the GPU's state."""
    from dataclasses import replace
    w = replace(S.WORKLOADS["decode_8b"], G=2, deltas=(0.25, 0.25))
    ex, ch, reps, D = _run_steps(w, 3, 48)
    assert reps > 0 and ch > 0
