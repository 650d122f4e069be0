"""Pool recall on the pools the CUDA library actually builds (needs a GPU).

"FAD-KV: Adaptive Dictionary KV Caching for Efficient Reasoning Decoding",
Fig. 1 (b): a small Top-n screened pool recalls most of the atoms that OMP
over the whole dictionary picks.  Here the pools come from the library's
screening and selection (fadkv_debug_pool, the same kernels encode runs),
the full-OMP supports from the oracle's greedy with the whole dictionary as
its pool, at the Llama-3.2-3B decode shape (N = 4096, d = 128, s = 8).  For
every vector not on a near tie at the Top-n cut the GPU's pool equals the
oracle's, so its recall does too; the table is printed (run with -s).
"""
import numpy as np
import pytest

from dictionary_sparse_kv_gb300 import synthetic as S
from oracle import oracle as O
from tests import parity_util as PU

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
POOLS = (32, 128, 256, 512)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dictionary_sparse_kv_gb300 import build as B
    B.build()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("off_frac", [0.05, 0.5])
def test_gpu_pool_recall_of_full_omp_atoms(off_frac):
    from dataclasses import replace
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = replace(S.WORKLOADS["decode_3b"], off_frac=off_frac)
    data = S.WorkloadData(w, dicts=[0, 1])
    V = 48
    x = data.inputs(0, V)
    lines = []
    for g in range(2):
        omp = O.encode(O.Params(w.N, w.d, w.n, w.s), data.atoms[g], x[g], full_omp=True)
        supp = [set(r.tolist()) for r in omp.idx]
        for n in POOLS:
            D = F.Dictionary(_t(data.atoms[g:g + 1]), _t(data.usage[g:g + 1]), data.deltas()[g:g + 1], n, w.s, V)
            gpool = D.pool(_t(x[g:g + 1]))[0].cpu().numpy()[0]
            res = O.encode(O.Params(w.N, w.d, n, w.s), data.atoms[g], x[g])
            ok = res.cut_gap >= PU.CUT_GAP
            assert ok.sum() >= V - 2
            hits_gpu = [len(supp[v] & set(gpool[v].tolist())) for v in range(V) if ok[v]]
            hits_orc = [len(supp[v] & set(res.pool[v].tolist())) for v in range(V) if ok[v]]
            for v in np.nonzero(ok)[0]:
                assert set(gpool[v].tolist()) == set(res.pool[v].tolist()), (g, n, v)
            assert hits_gpu == hits_orc
            rec_all = float(np.mean([len(supp[v] & set(res.pool[v].tolist())) for v in range(V)])) / w.s
            lines.append((g, n, float(np.mean(hits_gpu)) / w.s, int(ok.sum()), rec_all))
            D.close()
    print(f"\noff_frac={off_frac}: recall of full-OMP atoms by the GPU's Top-n pools "
          + "; ".join(f"dict {g} n={n}: {r:.3f} ({c} vectors)" for g, n, r, c, _ in lines))
    for g in range(2):
        rec = [ra for gg, n, r, c, ra in lines if gg == g]
        assert all(b >= a for a, b in zip(rec, rec[1:]))   # nested pools: recall cannot drop
