"""Parity over the workloads' stated lengths (needs a GPU; the slowest GPU tests).

The encode and adaptation of the CUDA library are compared with the oracle
at every step of long runs, each step on the GPU's own state (the oracle
takes the GPU's dictionary and usage counts at the start of the step, so a
near tie cannot make the two drift apart):

* Llama-3.2-3B decode: dictionaries 0, 1 (layer 0, K and V) and 54, 55 (the
  last layer) over all 1024 steps, and all 56 dictionaries over the first 8;
* Llama-3.1-8B decode: dictionaries 0, 1, 62, 63 over 256 of the 1024 steps;
* adaptation stress: both dictionaries, 256 vectors a step, 2048 steps, 10%
  of the generating sources redrawn every 128 steps; and 64 steps of it with
  a threshold low enough that atoms are replaced in every early step.

At every step: selected ids bit-exact (near ties checked on the GPU's pool),
coefficients and relres within 1e-3, the usage counts and replacement ids
equal to the oracle's adaptation of the GPU's codes, replaced atoms within
one storage ulp plus the fp32 bound, the dictionary size fixed at N and the
usage total conserved (before + s V + replaced).  Each run prints its
checked / exempt counts and replacements.

Workloads: "FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning
Decoding", Table 5 (N, n, s, delta; 1024 new tokens); Fig. 2 caption and
Fig. 3 caption (a dictionary adapted over a long decode).
"""
import numpy as np
import pytest

from dictionary_sparse_kv_gb300 import synthetic as S
from oracle import oracle as O
from tests import parity_util as PU

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dictionary_sparse_kv_gb300 import build as B
    B.build()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


class Totals:
    def __init__(self):
        self.checked = self.exempt = self.replaced = self.flagged = self.overflow = 0
        self.worst_c = self.worst_e = self.worst_r = 0.0


def check_step(w, p, deltas, t, x, atoms0, usage0, gpool, idx, coef, rel, rid, atoms1, usage1, tot):
    """Everything the oracle says about one step, on the GPU's state at its start."""
    G = atoms0.shape[0]
    assert atoms1.shape == (G, w.N, w.d) and usage1.shape == (G, w.N)
    for g in range(G):
        res = O.encode_threaded(p, atoms0[g], x[g], PU.THREADS)
        rep = PU.compare_encode(res, idx[g], coef[g], rel[g], gpool[g], p, atoms0[g], x[g])
        PU.assert_encode_ok(rep)
        tot.checked += rep.checked
        tot.exempt += rep.exempt
        tot.worst_c = max(tot.worst_c, rep.worst_coef)
        tot.worst_e = max(tot.worst_e, rep.worst_coef_elem)
        tot.worst_r = max(tot.worst_r, rep.worst_relres)
        oat, ous = atoms0[g].copy(), usage0[g].copy()
        r = O.adapt(p, oat, ous, x[g], idx[g], coef[g].astype(np.float64), rel[g].astype(np.float64), deltas[g])
        assert np.array_equal(usage1[g], ous), (t, g)
        assert np.array_equal(rid[g], r.repl_id), (t, g)
        changed = r.repl_id[r.repl_id >= 0]
        bnd = PU.replacement_bounds(atoms0[g], x[g], idx[g], coef[g], r.repl_id, w.s)
        assert PU.compare_atoms(atoms1[g], oat, changed, bnd) <= 1.0, (t, g)
        same = np.setdiff1d(np.arange(w.N), changed)
        assert np.array_equal(atoms1[g][same], atoms0[g][same]), (t, g)
        valid = int((idx[g] >= 0).sum())
        assert int(usage1[g].sum()) == int(usage0[g].sum()) + valid + r.replaced, (t, g)
        tot.replaced += r.replaced
        tot.overflow += r.overflow
        tot.flagged += int((rel[g].astype(np.float64) > deltas[g]).sum())


def run_long(w, dicts, steps, V=None):
    """Run `steps` steps of workload w on the given dictionaries, comparing
    every step with the oracle (the comparison of step t runs on the host
    while the GPU runs step t + 1); returns the totals."""
    from concurrent.futures import ThreadPoolExecutor
    from dictionary_sparse_kv_gb300 import fadkv as F
    data = S.WorkloadData(w, dicts)
    V = w.V if V is None else V
    D = F.Dictionary(_t(data.atoms), _t(data.usage), data.deltas(), w.n, w.s, V)
    p = PU.oparams(w)
    deltas = data.deltas()
    tot = Totals()
    pending = None
    with ThreadPoolExecutor(max_workers=1) as pool:
        for t in range(steps):
            x = data.inputs(t, V)
            atoms0 = D.atoms.cpu().numpy()
            usage0 = D.usage.cpu().numpy()
            xd = _t(x)
            gpool = D.pool(xd)[0].cpu().numpy()
            c = D.new_codes(V)
            D.encode(xd, c)
            D.adapt(xd, c)
            torch.cuda.synchronize()
            outs = [a.cpu().numpy() for a in (c.idx, c.coef, c.relres, c.repl_id)]
            atoms1 = D.atoms.cpu().numpy()
            usage1 = D.usage.cpu().numpy()
            if pending is not None:
                pending.result()
            pending = pool.submit(check_step, w, p, deltas, t, x, atoms0, usage0, gpool, *outs, atoms1, usage1, tot)
        pending.result()
    print(f"{w.name} dictionaries {list(dicts)}, {steps} steps x {V} vectors: {tot.checked} vectors checked, "
          f"{tot.exempt} exempt (near ties), {tot.flagged} flagged, {tot.replaced} atoms replaced, "
          f"{tot.overflow} overflow; worst coef {tot.worst_c:.2e} (element-wise {tot.worst_e:.2e}), "
          f"worst relres {tot.worst_r:.2e}")
    return tot


def test_decode_3b_every_dictionary_first_8_steps():
    w = S.WORKLOADS["decode_3b"]
    run_long(w, list(range(w.G)), 8)


def test_decode_3b_first_and_last_layer_1024_steps():
    w = S.WORKLOADS["decode_3b"]
    run_long(w, [0, 1, 54, 55], w.steps)


def test_decode_8b_first_and_last_layer_256_steps():
    w = S.WORKLOADS["decode_8b"]
    run_long(w, [0, 1, 62, 63], 256)


def test_adaptation_stress_2048_steps():
    """As specified.  The usage counts never decrease, and the greedy's last
    picks land on inactive atoms as well, so the initial inactive atoms are
    all in use within the first few dozen steps; the vectors flagged after
    each drift of the sources then overflow (no atom is free to take), which
    the oracle's adaptation of the same codes shows too."""
    w = S.WORKLOADS["adapt_stress"]
    tot = run_long(w, list(range(w.G)), w.steps)
    assert tot.flagged > 0 and tot.overflow == tot.flagged - tot.replaced


def test_adaptation_stress_low_threshold_replaces():
    """The same workload with delta = 0.25 for both dictionaries: vectors are
    flagged from the first step, so atoms are replaced while inactive ones
    remain, and every later encode reads the Gram rows the replacements
    rewrote; 64 steps."""
    from dataclasses import replace
    w = replace(S.WORKLOADS["adapt_stress"], deltas=(0.25, 0.25))
    tot = run_long(w, list(range(w.G)), 64)
    assert tot.replaced > 500
