"""A decode step captured in a CUDA graph and replayed (needs a GPU).

One encode + adapt + reconstruct step of several dictionaries is captured
once and replayed on fresh inputs copied into the captured input buffer;
the codes, the dictionary and the usage counts after every replay must be
bit-identical to the same steps run directly on a twin dictionary (every
kernel of the step is deterministic).
"""
import numpy as np
import pytest

from dictionary_sparse_kv_gb300 import synthetic as S

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


@pytest.mark.parametrize("coder", ["gm", "pl"])
def test_captured_step_replays_like_direct_steps(coder):
    from dataclasses import replace
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = replace(S.WORKLOADS["adapt_stress"], off_frac=1.0)     # replacements happen every step
    data = S.WorkloadData(w)
    V, steps = 64, 4
    xs = [data.inputs(t, V) for t in range(steps + 1)]
    Dg = F.Dictionary(_t(data.atoms), _t(data.usage), data.deltas(), w.n, w.s, V)
    Dd = F.Dictionary(_t(data.atoms), _t(data.usage), data.deltas(), w.n, w.s, V)
    cg, cd = Dg.new_codes(V), Dd.new_codes(V)
    xg = torch.empty((w.G, V, w.d), dtype=torch.float16, device=DEV)
    hg = torch.empty((w.G, V, w.d), dtype=torch.float32, device=DEV)
    hd = torch.empty_like(hg)
    # step 0 directly on both (first-use set-up happens outside the capture)
    xg.copy_(_t(xs[0]))
    Dg.step(xg, cg, hg, coder=coder)
    Dd.step(_t(xs[0]), cd, hd, coder=coder)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    xg.copy_(_t(xs[1]))
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        Dg.step(xg, cg, hg, coder=coder)
    # capturing ran nothing: replay step 1, then the others
    for t in range(1, steps + 1):
        xg.copy_(_t(xs[t]))
        graph.replay()
        Dd.step(_t(xs[t]), cd, hd, coder=coder)
        torch.cuda.synchronize()
        for a, b in ((cg.idx, cd.idx), (cg.coef, cd.coef), (cg.relres, cd.relres), (cg.repl_id, cd.repl_id),
                     (cg.repl_coef, cd.repl_coef), (hg, hd), (Dg.atoms, Dd.atoms), (Dg.usage, Dd.usage)):
            assert torch.equal(a, b), t
    assert int((cd.repl_id >= 0).sum()) > 0
