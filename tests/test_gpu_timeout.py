"""The bounded waits of the tensor-core kernels, made to run out (needs a GPU).

Every wait inside the screening pipeline gives up after a wall-clock limit,
sets FADKV_DEV_TIMEOUT in the dictionary's status word and lets the kernel
drain what it issued and return, so the CUDA context stays usable and the
host learns of it from fadkv_dict_stats.  Here the limit is made to expire
on purpose, with the library's two test hooks:

* fadkv_debug_wait_probe: one thread waits on a barrier nothing arrives on;
* fadkv_debug_wait_limit: the screening kernel's pipeline waits limited to
  one nanosecond, so waits give up while copies and MMAs are in flight (the
  kernel's drain still waits for those, with the full limit).

After either, the same handle must encode the next batch exactly as the
oracle does.
"""
import time

import numpy as np
import pytest

from dictionary_sparse_kv_gb300 import synthetic as S
from oracle import oracle as O
from tests import parity_util as PU

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TIMEOUT_BIT = 0x4          # FADKV_DEV_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dictionary_sparse_kv_gb300 import build as B
    B.build()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _dict(w, data, V):
    from dictionary_sparse_kv_gb300 import fadkv as F
    return F.Dictionary(_t(data.atoms), _t(data.usage), data.deltas(), w.n, w.s, V)


def _encode_matches_oracle(D, w, x):
    """Encode x on D and compare with the oracle on D's current state."""
    atoms = D.atoms.cpu().numpy()
    gpool = D.pool(_t(x))[0].cpu().numpy()
    c = D.new_codes(x.shape[1])
    D.encode(_t(x), c)
    D.adapt(_t(x), c)
    torch.cuda.synchronize()
    p = PU.oparams(w)
    idx, coef, rel = (a.cpu().numpy() for a in (c.idx, c.coef, c.relres))
    for g in range(w.G):
        res = O.encode_threaded(p, atoms[g], x[g], PU.THREADS)
        PU.assert_encode_ok(PU.compare_encode(res, idx[g], coef[g], rel[g], gpool[g], p, atoms[g], x[g]))


def test_wait_probe_runs_out_and_sets_the_status_bit():
    from dataclasses import replace
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = replace(S.WORKLOADS["decode_3b"], G=2)
    data = S.WorkloadData(w)
    D = _dict(w, data, 64)
    limit = 2_000_000                                   # 2 ms
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    F.debug_wait_probe(D.h, limit)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    st = D.stats()
    assert st[0]["status"] & TIMEOUT_BIT
    assert not st[1]["status"] & TIMEOUT_BIT
    assert waited >= 0.9 * limit * 1e-9, waited        # it did wait out its limit
    _encode_matches_oracle(D, w, data.inputs(0, 64))


def test_screening_waits_run_out_drain_and_the_handle_recovers():
    from dataclasses import replace
    from dictionary_sparse_kv_gb300 import fadkv as F
    w = replace(S.WORKLOADS["decode_3b"], G=8)
    data = S.WorkloadData(w)
    D = _dict(w, data, 128)
    F.debug_wait_limit(D.h, 1)                           # every pipeline wait gives up at once
    for step in range(2):
        x = _t(data.inputs(step, 128))
        c = D.new_codes(128)
        D.encode(x, c)                                   # no CUDA error: the kernel drained and returned
        D.adapt(x, c)
    torch.cuda.synchronize()
    idx = c.idx.cpu().numpy()
    assert ((idx >= 0) & (idx < w.N)).all()              # incomplete candidates, still valid atom ids
    timed_out = sum(bool(s["status"] & TIMEOUT_BIT) for s in D.stats())
    print(f"dictionaries whose screening waits ran out: {timed_out} of {w.G}")
    F.debug_wait_limit(D.h, 0)
    _encode_matches_oracle(D, w, data.inputs(2, 128))
