"""The compressed store (fadkv_store_codes) and decode attention over packed
codes (fadkv_attend) against the CPU oracle, through the C ABI (needs a GPU).
Binary16 dictionaries take the three-kernel path (per-layer tensor-core
GEMMs around the token pass), binary32 the fused kernel.

Packed words: bit-exact.  Attention outputs: per (layer, sequence, query
head) ||o_gpu - o_oracle|| <= 1e-4 ||o_oracle|| + 1e-5 (FP32 products and
sums, exp, and a scatter whose order varies between runs, against double).
"""
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


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _random_words(g, shape, N, zero_frac=0.05, scale=0.3):
    """Seeded random packed words: a random binary32 coefficient with its low
    13 bits cleared, OR a random atom id; a share of empty (0) words."""
    c = (g.standard_normal(shape) * scale).astype(np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
    w = c | g.integers(0, N, shape).astype(np.uint32)
    w[g.random(shape) < zero_frac] = 0
    return w


def test_store_codes_matches_oracle_words():
    from dictionary_sparse_kv_gb300 import fadkv as F
    g = np.random.default_rng(30)
    G, B, H, s, N, Tmax = 2, 3, 2, 4, 1000, 10
    idx = g.integers(-1, N, (G, B * H, s)).astype(np.int32)
    coef = (g.standard_normal((G, B * H, s)) * 10.0 ** g.integers(-8, 8, (G, B * H, s))).astype(np.float32)
    coef[0, 0, 0] = 0.0
    coef[0, 1, 1] = 1e-40                               # below 2^-126
    coef[1, 2, 2] = -np.float32(1.0 + 2.0 ** -11)       # exactly between two 11-bit values: ties to even
    coef[1, 3, 3] = np.float32(1.0 + 3 * 2.0 ** -11)    # the other tie direction
    rid = g.integers(-1, N, (G, B * H)).astype(np.int32)
    rco = g.standard_normal((G, B * H)).astype(np.float32)
    for pos, with_repl in (([3, 0, 9], True), ([5, -1, 10], False)):
        cache = torch.full((G, B, H, Tmax, s + 1), 0xDEADBEEF & 0x7FFFFFFF, dtype=torch.int32, device=DEV)
        before = cache.cpu().numpy().view(np.uint32).copy()
        F.store_codes(G, B, H, s, N, _t(idx), _t(coef), _t(rid) if with_repl else None,
                      _t(rco) if with_repl else None, _t(np.array(pos, np.int32)), cache, Tmax)
        torch.cuda.synchronize()
        got = cache.cpu().numpy().view(np.uint32)
        want = O.pack_codes(idx.reshape(G, B, H, s), coef.reshape(G, B, H, s).astype(np.float64),
                            rid.reshape(G, B, H) if with_repl else None,
                            rco.reshape(G, B, H).astype(np.float64) if with_repl else None)
        exp = before.copy()
        for b, p in enumerate(pos):
            if 0 <= p < Tmax:
                exp[:, b, :, p, :] = want[:, b, :, :]
        assert np.array_equal(got, exp)


CASES = [
    # dtype, N, d, s, L, B, Hq, Hkv, Tmax, lengths
    (np.float16, 4096, 128, 8, 2, 3, 6, 2, 3000, [1, 2500, 0]),      # two softmax chunks, an empty sequence
    (np.float16, 8192, 128, 16, 1, 2, 8, 2, 700, [700, 333]),        # 4 heads per KV head in 2 passes
    (np.float32, 512, 64, 4, 1, 2, 2, 2, 100, [100, 37]),
    (np.float32, 999, 64, 4, 1, 2, 3, 1, 50, [50, 7]),               # odd N, 3 heads per KV head
    (np.float16, 1000, 64, 4, 2, 3, 4, 2, 40, [40, 3, 0]),           # N not a multiple of 16, d = 64
]


@pytest.mark.parametrize("dt,N,d,s,L,B,Hq,Hkv,Tmax,lengths", CASES)
def test_attend_matches_oracle(dt, N, d, s, L, B, Hq, Hkv, Tmax, lengths):
    from dictionary_sparse_kv_gb300 import fadkv as F
    g = np.random.default_rng(31 + N)
    dk = np.stack([S.make_dictionary(N, d, dt, 40, l, 0) for l in range(L)])
    dv = np.stack([S.make_dictionary(N, d, dt, 40, l, 1) for l in range(L)])
    ck = _random_words(g, (L, B, Hkv, Tmax, s + 1), N)
    cv = _random_words(g, (L, B, Hkv, Tmax, s + 1), N)
    q = g.standard_normal((L, B, Hq, d)).astype(np.float32)
    out = torch.empty((L, B, Hq, d), dtype=torch.float32, device=DEV)
    p = F.AttnParams(L, B, Hq, Hkv, d, N, s, Tmax, F.F16 if dt == np.float16 else F.F32, 1.0 / np.sqrt(d),
                     N * d, B * Hkv * Tmax * (s + 1))
    F.attend(p, _t(dk), _t(dv), _t(ck.view(np.int32)), _t(cv.view(np.int32)), _t(np.array(lengths, np.int32)),
             _t(q), out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for l in range(L):
        want = O.attend(dk[l], dv[l], ck[l], cv[l], np.array(lengths), q[l].astype(np.float64))
        for b in range(B):
            for h in range(Hq):
                err = np.linalg.norm(got[l, b, h] - want[b, h])
                assert err <= ATT_TOL * np.linalg.norm(want[b, h]) + 1e-5, (l, b, h, err)
                if lengths[b] == 0:
                    assert np.all(got[l, b, h] == 0)


def test_encode_store_attend_end_to_end():
    """Four decode steps of one layer (K and V dictionaries, 4 sequences x 8
    KV heads): encode, adapt and store every step's codes on the GPU, then
    attend with 24 query heads; the oracle attends over the cache the GPU
    wrote, and the attention over the uncompressed vectors is reported."""
    from dataclasses import replace
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = replace(S.WORKLOADS["decode_3b"], G=2)
    data = S.WorkloadData(w)
    Bs, H, steps, Hq = 4, 8, 4, 24
    V = Bs * H
    D = F.Dictionary(_t(data.atoms), _t(data.usage), data.deltas(), w.n, w.s, V)
    Tmax = 8
    cache = torch.zeros((2, Bs, H, Tmax, w.s + 1), dtype=torch.int32, device=DEV)
    xs = []
    for t in range(steps):
        x = data.inputs(t, V)
        xs.append(x)
        c = D.new_codes(V)
        D.step(_t(x), c)
        F.store_codes(2, Bs, H, w.s, w.N, c.idx, c.coef, c.repl_id, c.repl_coef,
                      _t(np.full(Bs, t, np.int32)), cache, Tmax)
    lengths = np.array([4, 3, 1, 0], np.int32)
    g = np.random.default_rng(32)
    q = g.standard_normal((1, Bs, Hq, w.d)).astype(np.float32)
    out = torch.empty((1, Bs, Hq, w.d), dtype=torch.float32, device=DEV)
    p = F.AttnParams(1, Bs, Hq, H, w.d, w.N, w.s, Tmax, F.F16, 1.0 / np.sqrt(w.d), 2 * w.N * w.d,
                     2 * Bs * H * Tmax * (w.s + 1))
    atoms = D.atoms
    F.attend(p, atoms[0], atoms[1], cache[0], cache[1], _t(lengths), _t(q), out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()[0]
    at = atoms.cpu().numpy()
    cw = cache.cpu().numpy().view(np.uint32)
    want = O.attend(at[0], at[1], cw[0], cw[1], lengths, q[0].astype(np.float64))
    for b in range(Bs):
        for h in range(Hq):
            err = np.linalg.norm(got[b, h] - want[b, h])
            assert err <= ATT_TOL * np.linalg.norm(want[b, h]) + 1e-5, (b, h, err)
    # the same attention over the uncompressed vectors (a quality figure, not a parity bound)
    rel = []
    for b in range(Bs):
        if lengths[b] == 0:
            continue
        K = np.stack([xs[t][0, b * H:(b + 1) * H] for t in range(lengths[b])]).astype(np.float64)
        Vv = np.stack([xs[t][1, b * H:(b + 1) * H] for t in range(lengths[b])]).astype(np.float64)
        for h in range(Hq):
            sc = K[:, h // 3] @ q[0, b, h] / np.sqrt(w.d)
            pr = np.exp(sc - sc.max())
            pr /= pr.sum()
            dense = pr @ Vv[:, h // 3]
            rel.append(np.linalg.norm(got[b, h] - dense) / np.linalg.norm(dense))
    print(f"\nattention over codes vs over the uncompressed vectors: median relative difference "
          f"{np.median(rel):.3f}")
    assert np.all(np.isfinite(rel))
