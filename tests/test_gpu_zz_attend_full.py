"""Decode attention over packed codes at the benchmark's full shape, against
the CPU oracle on sampled outputs, through the C ABI (needs a GPU).  Same
tolerance as tests/test_gpu_attend.py."""
import numpy as np
import pytest

from dictionary_sparse_kv_gb300 import synthetic as S
from oracle import oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ATT_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dictionary_sparse_kv_gb300 import build as B
    B.build()


def test_attend_full_size_sampled():
    """The benchmark's shape (Llama-3.2-3B decode: 28 layers x 16 sequences x
    24 query / 8 KV heads, N = 4096, s = 8, 4096 cached tokens), one call;
    the oracle recomputes every query head of four sampled (layer, sequence)
    pairs over the words the GPU read."""
    from dictionary_sparse_kv_gb300 import fadkv as F
    L, Bs, Hq, Hkv, d, N, s, T = 28, 16, 24, 8, 128, 4096, 8, 4096
    gen = torch.Generator(device=DEV)
    gen.manual_seed(70)
    atoms = torch.from_numpy(np.stack([S.make_dictionary(N, d, np.float16, 71, i) for i in range(2 * L)])).to(DEV)
    words = (L, 2, Bs, Hkv, T, s + 1)
    coefs = torch.randn(words, device=DEV, dtype=torch.float32, generator=gen).mul_(0.3)
    ids = torch.randint(0, N, words, device=DEV, dtype=torch.int32, generator=gen)
    cache = (coefs.view(torch.int32) & -8192) | ids
    del coefs, ids
    lengths = torch.full((Bs,), T, dtype=torch.int32, device=DEV)
    lengths[3] = 1000                                           # one shorter sequence
    q = torch.randn((L, Bs, Hq, d), device=DEV, dtype=torch.float32, generator=gen)
    out = torch.empty_like(q)
    p = F.AttnParams(L, Bs, Hq, Hkv, d, N, s, T, F.F16, 1.0 / np.sqrt(d), 2 * N * d, 2 * Bs * Hkv * T * (s + 1))
    F.attend(p, atoms[0], atoms[1], cache[:, 0], cache[:, 1], lengths, q, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    at = atoms.cpu().numpy()
    ln = lengths.cpu().numpy()
    for l, b in ((0, 0), (13, 3), (27, 15), (20, 7)):
        ck = cache[l, 0, b:b + 1].cpu().numpy().view(np.uint32)
        cv = cache[l, 1, b:b + 1].cpu().numpy().view(np.uint32)
        want = O.attend(at[2 * l], at[2 * l + 1], ck, cv, ln[b:b + 1], q[l, b:b + 1].cpu().numpy().astype(np.float64))
        for h in range(Hq):
            err = np.linalg.norm(got[l, b, h] - want[0, h])
            assert err <= ATT_TOL * np.linalg.norm(want[0, h]) + 1e-5, (l, b, h, err)
