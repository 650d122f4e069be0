"""C-ABI library: loads without a GPU, exports every declared symbol, and its
host-side logic (argument checks, sequence contract, workspace sizing, fault
injection) behaves as include/fadkv.h documents.  No call here launches work."""
import ctypes as C
import os
import re

import pytest

from dictionary_sparse_kv_gb300 import build as B
from dictionary_sparse_kv_gb300 import fadkv as F

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fadkv.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return F.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fadkv_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 11
    for name in names:
        assert hasattr(L, name), name
    raw = C.CDLL(F.LIB_PATH)
    for name in names:
        C.cast(getattr(raw, name), C.c_void_p)


def test_version_and_strings(L):
    assert F.abi_version() == 1
    assert F.status_string(0) == "ok"
    assert F.status_string(3) == "encode/adapt called out of order"


def test_param_validation(L):
    ok = F.params(56, 4096, 128, 256, 8, F.F16, 128)
    assert F.workspace_bytes(ok) > 0
    bad = [
        F.params(0, 4096, 128, 256, 8),            # no dictionaries
        F.params(1, 4096, 128, 4, 8),              # s > n
        F.params(1, 128, 128, 256, 8),             # n > N
        F.params(1, 4096, 128, 256, 8, dtype=7),
        F.params(1, 4096, 128, 256, 8, lambda_abs=-1.0),
    ]
    for p in bad:
        with pytest.raises(F.FadkvError) as e:
            F.workspace_bytes(p)
        assert e.value.status == 1
    unsupported = [
        F.params(1, 4096, 96, 256, 8),             # d not 64/128
        F.params(1, 4096, 128, 256, 33),           # s above the maximum
        F.params(1, 4096, 128, 2048, 8),           # n above the maximum
        F.params(1, 4000, 128, 256, 8),            # N not a multiple of 64
        F.params(300, 4096, 128, 256, 8),          # too many dictionaries
    ]
    for p in unsupported:
        with pytest.raises(F.FadkvError) as e:
            F.workspace_bytes(p)
        assert e.value.status == 2


def test_workspace_grows_with_batch(L):
    a = F.workspace_bytes(F.params(2, 4096, 128, 256, 8, F.F16, 128))
    b = F.workspace_bytes(F.params(2, 4096, 128, 256, 8, F.F16, 4096))
    assert b > a


def test_create_checks_without_gpu(L):
    p = F.params(2, 512, 64, 32, 4, F.F32, 16)
    ws = F.workspace_bytes(p)
    fake = 0x10000   # never dereferenced: create makes no CUDA call
    h = F.dict_create(p, fake, fake, [0.5, 0.7], fake, ws)
    try:
        # workspace too small
        with pytest.raises(F.FadkvError) as e:
            F.dict_create(p, fake, fake, [0.5, 0.7], fake, ws - 1)
        assert e.value.status == 5
        # misaligned dictionary / workspace
        with pytest.raises(F.FadkvError):
            F.dict_create(p, fake + 4, fake, [0.5, 0.7], fake, ws)
        with pytest.raises(F.FadkvError):
            F.dict_create(p, fake, fake, [0.5, 0.7], fake + 16, ws)
        # negative threshold
        with pytest.raises(F.FadkvError):
            F.dict_create(p, fake, fake, [0.5, -0.1], fake, ws)
        # sequence: adapt before any encode
        with pytest.raises(F.FadkvError) as e:
            F.adapt(h, fake, 4, fake, fake, fake, fake, fake, stream=0)
        assert e.value.status == 3
        # batch above max_batch
        with pytest.raises(F.FadkvError) as e:
            F.encode(h, fake, 17, fake, fake, fake, stream=0)
        assert e.value.status == 1
        # repl_id without repl_coef
        with pytest.raises(F.FadkvError) as e:
            F.reconstruct(h, 4, fake, fake, fake, None, fake, stream=0)
        assert e.value.status == 1
    finally:
        F.dict_destroy(h)


def test_profile_controls_without_gpu(L):
    p = F.params(1, 512, 64, 32, 4, F.F32, 16)
    ws = F.workspace_bytes(p)
    fake = 0x10000
    h = F.dict_create(p, fake, fake, [0.5], fake, ws)
    try:
        F.profile_select(h, ["greedy"])
        F.profile_select(h, [0, "adapt"])
        F.profile_select(h, None)
        F.profile_enable(h, True)
        F.profile_enable(h, False)
        # nothing traced, nothing launched: all zero
        assert F.profile_read(h, reset=True) == {}
        with pytest.raises(ValueError):
            F.profile_select(h, ["no_such_kernel"])
    finally:
        F.dict_destroy(h)
    with pytest.raises(F.FadkvError) as e:
        F.profile_select(0, None)
    assert e.value.status == 1


def test_fault_injection_leaves_state(L, monkeypatch):
    p = F.params(1, 512, 64, 32, 4, F.F32, 16)
    ws = F.workspace_bytes(p)
    fake = 0x10000
    h = F.dict_create(p, fake, fake, [0.5], fake, ws)
    try:
        monkeypatch.setenv("FADKV_FAULT", "cuda")
        with pytest.raises(F.FadkvError) as e:
            F.encode(h, fake, 4, fake, fake, fake, stream=0)
        assert e.value.status == 4
        assert "fadkv_encode" in F.last_error()
        # the failed encode did not advance the sequence: adapt still refused
        with pytest.raises(F.FadkvError) as e:
            F.adapt(h, fake, 4, fake, fake, fake, fake, fake, stream=0)
        assert e.value.status == 3
    finally:
        F.dict_destroy(h)


def test_pl_and_append_entry_points_without_gpu(L, monkeypatch):
    """fadkv_encode_pl and fadkv_adapt_append share the sequence contract and
    the argument checks of fadkv_encode / fadkv_adapt."""
    p = F.params(1, 512, 64, 32, 4, F.F32, 16)
    ws = F.workspace_bytes(p)
    fake = 0x10000
    h = F.dict_create(p, fake, fake, [0.5], fake, ws)
    try:
        with pytest.raises(F.FadkvError) as e:
            F.adapt_append(h, fake, 4, fake, fake, fake, fake, fake, stream=0)
        assert e.value.status == 3
        with pytest.raises(F.FadkvError) as e:
            F.encode_pl(h, fake, 17, fake, fake, fake, stream=0)
        assert e.value.status == 1
        with pytest.raises(F.FadkvError) as e:
            F.encode_pl(h, fake + 4, 4, fake, fake, fake, stream=0)      # x not 16-byte aligned
        assert e.value.status == 1
        monkeypatch.setenv("FADKV_FAULT", "cuda")
        with pytest.raises(F.FadkvError) as e:
            F.encode_pl(h, fake, 4, fake, fake, fake, stream=0)
        assert e.value.status == 4 and "fadkv_encode_pl" in F.last_error()
        with pytest.raises(F.FadkvError) as e:
            F.adapt_append(h, fake, 4, fake, fake, fake, fake, fake, stream=0)
        assert e.value.status == 3
    finally:
        F.dict_destroy(h)


def test_store_codes_checks_without_gpu(L):
    fake = 0x10000
    # no vectors: nothing to launch, OK
    F.store_codes(0, 4, 8, 8, 4096, fake, fake, fake, fake, fake, fake, 16, stream=0)
    cases = [
        ((1, 4, 8, 8, 8193), 2),        # N beyond the 13-bit id
        ((1, 4, 8, 33, 4096), 2),       # s above the maximum
        ((1, 4, 0, 8, 4096), 1),        # no heads
        ((1, -1, 8, 8, 4096), 1),
    ]
    for (G, B, H, s, N), status in cases:
        with pytest.raises(F.FadkvError) as e:
            F.store_codes(G, B, H, s, N, fake, fake, fake, fake, fake, fake, 16, stream=0)
        assert e.value.status == status, (G, B, H, s, N)
    with pytest.raises(F.FadkvError) as e:      # repl_id without repl_coef
        F.store_codes(1, 4, 8, 8, 4096, fake, fake, fake, None, fake, fake, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(F.FadkvError) as e:      # misaligned cache
        F.store_codes(1, 4, 8, 8, 4096, fake, fake, fake, fake, fake, fake + 2, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(F.FadkvError) as e:      # Tmax 0
        F.store_codes(1, 4, 8, 8, 4096, fake, fake, fake, fake, fake, fake, 0, stream=0)
    assert e.value.status == 1


def test_attend_workspace_and_checks_without_gpu(L):
    def prm(layers=28, B=16, Hq=24, Hkv=8, d=128, N=4096, s=8, Tmax=4096, dtype=F.F16):
        return F.AttnParams(layers, B, Hq, Hkv, d, N, s, Tmax, dtype, 0.125, 2 * N * d, 2 * B * Hkv * Tmax * (s + 1))

    def up(x):
        return (x + 255) // 256 * 256

    p = prm()
    rows, Np = 28 * 16 * 24, 4096
    assert F.attend_workspace_bytes(p) == up(rows * Np * 4) + 2 * up(rows * Np * 2) + up(rows * 4)
    p_odd = prm(N=1000, d=64)
    assert F.attend_workspace_bytes(p_odd) == up(rows * 1008 * 4) + 2 * up(rows * 1008 * 2) + up(rows * 4)
    assert F.attend_workspace_bytes(prm(dtype=F.F32)) == 0
    for bad, status in ((prm(Hq=20), 1), (prm(d=96), 2), (prm(N=9000), 2), (prm(s=40), 2), (prm(B=-1), 1)):
        with pytest.raises(F.FadkvError) as e:
            F.attend_workspace_bytes(bad)
        assert e.value.status == status
    fake = 0x10000
    need = F.attend_workspace_bytes(p)
    rc = L.fadkv_attend(C.byref(p), fake, fake, fake, fake, fake, fake, fake, fake, need - 1, None)
    assert rc == 5                                        # workspace too small
    rc = L.fadkv_attend(C.byref(p), fake, fake, fake, fake, fake, fake, fake, fake + 16, need, None)
    assert rc == 1                                        # workspace not 256-byte aligned
    rc = L.fadkv_attend(C.byref(p), fake + 8, fake, fake, fake, fake, fake, fake, fake, need, None)
    assert rc == 1                                        # dictionary not 16-byte aligned
    assert L.fadkv_attend(C.byref(prm(layers=0)), fake, fake, fake, fake, fake, fake, fake, fake, 0, None) == 0
    rc = L.fadkv_attend(C.byref(p), fake, fake, fake, fake, fake, fake + 8, fake, fake, need, None)
    assert rc == 1                                        # queries not 16-byte aligned
