"""The boundary is plain C: include/fadkv.h compiles as C99 with warnings as
errors, and a C program linked against the built library can make the
host-only calls (version, status strings, workspace sizes, handle
create/destroy with placeholder pointers, argument errors).  No GPU."""
import os
import shutil
import subprocess
import tempfile

import pytest

from dictionary_sparse_kv_gb300 import build as B
from dictionary_sparse_kv_gb300 import fadkv as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fadkv.h"

#define CHECK(c) do { if (!(c)) { printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #c); return 1; } } while (0)

int main(void)
{
    CHECK(fadkv_abi_version() == FADKV_ABI_VERSION);
    CHECK(strcmp(fadkv_status_string(FADKV_OK), "ok") == 0);

    fadkv_params p;
    memset(&p, 0, sizeof p);
    p.num_dicts = 56; p.N = 4096; p.d = 128; p.n = 256; p.s = 8;
    p.lambda_abs = 1e-4f; p.lambda_rel = 0.20f; p.dtype = FADKV_F16; p.max_batch = 128;
    size_t ws = 0;
    CHECK(fadkv_workspace_bytes(&p, &ws) == FADKV_OK && ws > 0);
    p.s = 300;
    CHECK(fadkv_workspace_bytes(&p, &ws) != FADKV_OK);
    p.s = 8;

    /* a handle over placeholder device pointers: create makes no CUDA call */
    void* fake = (void*)0x10000;
    float delta[56];
    for (int i = 0; i < 56; ++i) delta[i] = (i % 2) ? 0.70f : 0.50f;
    fadkv_dict h = NULL;
    CHECK(fadkv_dict_create(&p, fake, (int32_t*)fake, delta, fake, ws, &h) == FADKV_OK && h != NULL);
    CHECK(fadkv_adapt(h, fake, 4, fake, fake, fake, fake, fake, NULL) == FADKV_ERR_SEQUENCE);
    CHECK(fadkv_encode(h, fake, 129, fake, fake, fake, NULL) == FADKV_ERR_INVALID_ARG);
    CHECK(fadkv_dict_destroy(h) == FADKV_OK);

    fadkv_attn_params a;
    memset(&a, 0, sizeof a);
    a.layers = 28; a.B = 16; a.Hq = 24; a.Hkv = 8; a.d = 128; a.N = 4096; a.s = 8; a.Tmax = 4096;
    a.dtype = FADKV_F16; a.scale = 0.0883883f;
    a.dict_stride = 2LL * 4096 * 128; a.cache_stride = 2LL * 16 * 8 * 4096 * 9;
    size_t aw = 0;
    CHECK(fadkv_attend_workspace_bytes(&a, &aw) == FADKV_OK && aw > 0);
    CHECK(fadkv_store_codes(1, 16, 8, 8, 9000, fake, fake, NULL, NULL, fake, fake, 16, NULL) == FADKV_ERR_UNSUPPORTED);
    printf("OK %zu %zu\n", ws, aw);
    return 0;
}
"""


def test_header_is_c99_and_the_library_links_from_c():
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    B.build()
    tmp = tempfile.mkdtemp(prefix="fadkv_c_")
    try:
        src = os.path.join(tmp, "abi_check.c")
        exe = os.path.join(tmp, "abi_check")
        with open(src, "w") as f:
            f.write(PROGRAM)
        libdir = os.path.dirname(F.LIB_PATH)
        subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        src, "-o", exe, "-L", libdir, "-lfadkv", f"-Wl,-rpath,{libdir}"], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
        assert out.returncode == 0, out.stdout + out.stderr
        assert out.stdout.startswith("OK ")
        ws, aw = (int(v) for v in out.stdout.split()[1:3])
        p = F.params(56, 4096, 128, 256, 8, F.F16, 128)
        assert ws == F.workspace_bytes(p)
        assert aw == F.attend_workspace_bytes(F.AttnParams(28, 16, 24, 8, 128, 4096, 8, 4096, F.F16, 0.0883883,
                                                           2 * 4096 * 128, 2 * 16 * 8 * 4096 * 9))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
