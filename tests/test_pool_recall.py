"""Pool recall: the share of full-OMP atoms that the Top-n screened pool
contains, on synthetic data (CPU, oracle only).

"FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
Fig. 1 (b): on decode-time KV vectors a small Top-n screened pool recalls
most of the atoms OMP over the whole dictionary picks, which is what makes
screening before the greedy selection cheap.  This is the same diagnostic on
the synthetic inputs of this repository (the model's KV vectors are not
available), at the 3B decode shape.  Run with -s to see the table.
"""
import numpy as np
import pytest

from dictionary_sparse_kv_gb300 import synthetic as S

POOLS = (8, 16, 32, 64, 128, 256, 512)


def _recall(omp_idx, pool, n):
    """Mean over vectors of |top-n pool ∩ OMP support| / s."""
    s = omp_idx.shape[1]
    hits = [len(set(omp_idx[v].tolist()) & set(pool[v, :n].tolist())) for v in range(omp_idx.shape[0])]
    return float(np.mean(hits)) / s


def test_greedy_with_the_whole_dictionary_as_pool_is_omp(oracle_lib):
    """With n = N the pool is every atom and the greedy coder is plain OMP
    with the same refit: same picks, coefficients and relres, bit for bit."""
    O = oracle_lib
    w = S.WORKLOADS["tiny"]
    data = S.WorkloadData(w)
    x = data.inputs(0, 24)[0]
    p = O.Params(w.N, w.d, w.N, w.s, dtype=O.F32)
    gm = O.encode(p, data.atoms[0], x)
    omp = O.encode(p, data.atoms[0], x, full_omp=True)
    assert (gm.idx == omp.idx).all() and (gm.coef == omp.coef).all() and (gm.relres == omp.relres).all()


@pytest.mark.parametrize("off_frac", [0.05, 0.5])
def test_pool_recall_of_full_omp_atoms(oracle_lib, off_frac):
    """At N=4096, d=128, s=8: recall grows with n (pools are nested, so it
    cannot drop), and the default n = 256 holds most of the atoms OMP picks
    (the claim of Fig. 1 (b); on these inputs about 0.84-0.85 -- the atoms
    it misses carry the small Student-t coefficients, which OMP finds only
    after the large ones are removed)."""
    from dataclasses import replace
    O = oracle_lib
    w = replace(S.WORKLOADS["decode_3b"], off_frac=off_frac)
    data = S.WorkloadData(w, dicts=[0])
    x = data.inputs(0, 24)[0]
    p = O.Params(w.N, w.d, max(POOLS), w.s)
    ranked = O.encode(p, data.atoms[0], x)          # its pool: the 512 best atoms in (-|r|, j) order
    omp = O.encode(p, data.atoms[0], x, full_omp=True)
    rec = [_recall(omp.idx, ranked.pool, n) for n in POOLS]
    print(f"\noff_frac={off_frac}: recall of full-OMP atoms by the Top-n pool: "
          + ", ".join(f"n={n}: {r:.3f}" for n, r in zip(POOLS, rec)))
    assert all(b >= a for a, b in zip(rec, rec[1:]))
    assert rec[POOLS.index(256)] > 0.5
