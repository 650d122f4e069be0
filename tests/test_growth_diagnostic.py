"""Dictionary size and reconstruction error during decoding, fixed-size
adaptation against append-only growth, on synthetic data (CPU, oracle only).

"FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
Fig. 3 (a) and (b): the normalised dictionary size stays at 1 with FAD-KV's
fixed-size adaptation while append-only updates grow it, at a comparable
reconstruction error.  Here: one dictionary (N = 1024, d = 128, n = 128,
s = 8) whose generating sources drift every 5 steps; 30% of the rows start
as inactive atoms (fixed size) or as free slots (append-only).  Run with -s
to see the per-step table.
"""
import numpy as np

from dictionary_sparse_kv_gb300 import synthetic as S


def test_fixed_size_stays_put_append_only_grows(oracle_lib):
    from dataclasses import replace
    O = oracle_lib
    w = replace(S.WORKLOADS["adapt_stress"], N=1024, n=128, off_frac=0.3, drift_period=5, drift_frac=0.3)
    data = S.WorkloadData(w, dicts=[0])
    p = O.Params(w.N, w.d, w.n, w.s)
    delta = 0.5
    free = data.usage[0] == 0                          # the rows that start unused
    at_f, us_f = data.atoms[0].copy(), data.usage[0].copy()
    at_a, us_a = data.atoms[0].copy(), data.usage[0].copy()
    at_a[free] = 0
    us_a[free] = -1
    n0 = int((us_a >= 0).sum())
    rows = []
    for step in range(24):
        x = data.inputs(step, 32)[0]
        rf = O.encode(p, at_f, x)
        O.adapt(p, at_f, us_f, x, rf.idx, rf.coef, rf.relres, delta)
        ra = O.encode(p, at_a, x)
        O.adapt(p, at_a, us_a, x, ra.idx, ra.coef, ra.relres, delta, append=True)
        rows.append((step, w.N / w.N, int((us_a >= 0).sum()) / n0,
                     float(np.mean(rf.relres)), float(np.mean(ra.relres))))
        assert int((us_f < 0).sum()) == 0               # every row of the fixed-size dictionary is an atom
    print("\nstep  size(fixed)  size(append)  relres(fixed)  relres(append)")
    for r in rows:
        print(f"{r[0]:4d}  {r[1]:11.3f}  {r[2]:12.3f}  {r[3]:13.3f}  {r[4]:14.3f}")
    sizes = [r[2] for r in rows]
    assert all(b >= a for a, b in zip(sizes, sizes[1:]))
    assert sizes[-1] > 1.0
    # both policies keep the error in the same range (neither breaks down)
    assert abs(np.mean([r[3] for r in rows]) - np.mean([r[4] for r in rows])) < 0.1
