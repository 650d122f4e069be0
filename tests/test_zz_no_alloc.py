"""fadkv_adapt_noalloc against fadkv_adapt, through the C ABI.

The handle-free adaptation runs the same kernel on the library's static
scratch instead of a caller workspace, so two decode steps in a row must give
the same replacements, the same dictionary bytes and the same usage counts as
the handle path.  The size check runs on the host before any CUDA call.
This file is collected last so that the static scratch is exercised both in a
fresh process and after every other GPU test has run.
"""
import numpy as np
import pytest

from dictionary_sparse_kv_gb300 import build as B
from dictionary_sparse_kv_gb300 import fadkv as F
from dictionary_sparse_kv_gb300 import synthetic as S

DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    B.build()
    return F.lib()


def test_noalloc_rejects_oversized_scratch(lib):
    # 256 dictionaries of 8192 atoms need 8 MiB of inactive lists alone
    p = F.params(256, 8192, 128, 512, 16, F.F16, 1)
    fake = 1 << 20   # never dereferenced: the size check comes first
    with pytest.raises(F.FadkvError) as e:
        F.adapt_noalloc(p, fake, fake, [0.5] * 256, fake, 4, fake, fake, fake, fake, fake, stream=0)
    assert e.value.status == 5
    assert "static scratch holds 4194304" in str(e.value)
    with pytest.raises(F.FadkvError) as e:
        F.adapt_noalloc(p, fake, fake, [0.5] * 256, fake, -1, fake, fake, fake, fake, fake, stream=0)
    assert e.value.status == 1


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["adapt_stress", "tiny"])
def test_noalloc_matches_adapt_two_steps(lib, name):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = S.WORKLOADS[name]
    data = S.WorkloadData(w)
    V = w.V

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)

    # threshold 0 flags every vector with a nonzero residual, so both steps
    # replace atoms until the inactive ones run out
    deltas = [0.0] * w.G
    D = F.Dictionary(t(data.atoms), t(data.usage), deltas, w.n, w.s, V)
    atoms2 = D.atoms.clone()
    usage2 = D.usage.clone()
    replaced = 0
    for step in range(2):
        x = t(data.inputs(step, V))
        codes = D.new_codes(V)
        D.encode(x, codes)
        idx, coef, rel = codes.idx.clone(), codes.coef.clone(), codes.relres.clone()
        D.adapt(x, codes)
        rid = torch.full((w.G, V), -7, dtype=torch.int32, device=DEV)
        rco = torch.full((w.G, V), -7.0, dtype=torch.float32, device=DEV)
        F.adapt_noalloc(D.p, atoms2, usage2, D.delta, x, V, idx, coef, rel, rid, rco)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(rid.cpu().numpy(), codes.repl_id.cpu().numpy())
        np.testing.assert_allclose(rco.cpu().numpy(), codes.repl_coef.cpu().numpy(), rtol=1e-6, atol=0)
        # the dictionary and usage counts must stay bit-identical for the
        # next step's encode (run on the handle) to serve both paths
        bits = torch.int16 if atoms2.dtype == torch.float16 else torch.int32
        assert torch.equal(atoms2.view(bits), D.atoms.view(bits))
        assert torch.equal(usage2, D.usage)
        replaced += int((rid >= 0).sum())
    assert replaced > 0
