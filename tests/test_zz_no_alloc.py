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


SCRATCH = 4 << 20      # the static scratch's size, as the header states


def _round256(v):
    return (v + 255) // 256 * 256


def largest_v(G, N):
    """The largest V whose scratch (256-rounded inactive list [G][N] and
    flagged list [G][V], then [G][8] int64 counters) fits in the scratch."""
    V = (SCRATCH - _round256(4 * G * N) - 64 * G) // (4 * G)
    while V > 0 and _round256(4 * G * N) + _round256(4 * G * V) + 64 * G > SCRATCH:
        V -= 1
    return V


def test_noalloc_limit_at_the_decode_shape(lib):
    """56 dictionaries of 4096 atoms: the largest V that fits is accepted by
    the size check and one more is refused, before any CUDA call."""
    G, N = 56, 4096
    V = largest_v(G, N)
    assert V == 14612
    p = F.params(G, N, 128, 256, 8, F.F16, 1)
    fake = 1 << 20
    with pytest.raises(F.FadkvError) as e:
        F.adapt_noalloc(p, fake, fake, [0.5] * G, fake, V + 1, fake, fake, fake, fake, fake, stream=0)
    assert e.value.status == 5


@pytest.mark.gpu
@pytest.mark.parametrize("name,over", [("adapt_stress", {}), ("tiny", {}), ("decode_3b", {"V": 14612})],
                         ids=["adapt_stress", "tiny", "decode_3b_at_limit"])
def test_noalloc_matches_adapt_two_steps(lib, name, over):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dataclasses import replace
    w = replace(S.WORKLOADS[name], **over)
    data = S.WorkloadData(w)
    V = w.V
    if name == "decode_3b":
        assert V == largest_v(w.G, w.N)      # the scratch filled to its limit

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
