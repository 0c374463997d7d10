"""The C ABI without a GPU: the library loads, exports every entry point include/csa.h declares,
and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

import long_context_sparse_19_b300 as L
from long_context_sparse_19_b300.binding import CsaCache, CsaConfig

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "csa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z_]+)\s*\(", src)))


def test_every_declared_function_is_exported():
    lib = L.load()
    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert getattr(lib, n, None) is not None, n
    assert sorted(L.EXPORTS) == names


def test_status_strings():
    assert L.csa_status_string(0) == "ok"
    assert L.csa_status_string(4) == "workspace too small"
    assert L.csa_status_string(8) == "a device-side wait ran out"
    assert L.csa_status_string(99) == "unknown status"


def _cfg(**kw):
    c = L.Config(**kw).c()
    return c


def test_workspace_bytes():
    lib = L.load()
    c = _cfg()
    n = lib.csa_workspace_bytes(ctypes.byref(c), 32, 1, 16384)
    # at least the indexer scores and the selection of 32 requests
    assert n >= 32 * 16384 * 4 + 32 * 512 * 4
    bad = _cfg(d=256)
    assert lib.csa_workspace_bytes(ctypes.byref(bad), 32, 1, 16384) == 0
    hca = _cfg(top_k=0, ratio=128)
    assert lib.csa_workspace_bytes(ctypes.byref(hca), 16, 1, 2048) > 0


def test_cache_bytes_match_the_format():
    """csa_cache_bytes: plain arrays for f32 / bf16; for fp4 the stride of the oracle's own description
    of the three-plane layout (written independently of the library)."""
    from oracle import cache_lowp as Q
    for n in (1, 7, 8, 2048, 16385):
        assert L.csa_cache_bytes(L.Config(storage="bf16"), 0, n) == n * 512 * 2
        assert L.csa_cache_bytes(L.Config(storage="f32"), 1, n) == n * 128 * 4
        fp4 = L.Config(storage="fp4")
        assert L.csa_cache_bytes(fp4, 0, n) == Q.cache_layout(512, n)["stride"]
        assert L.csa_cache_bytes(fp4, 1, n) == Q.cache_layout(128, n)["stride"]
    assert L.csa_cache_bytes(L.Config(storage="fp4"), 2, 16) == 0
    assert L.csa_cache_bytes(L.Config(d=256), 0, 16) == 0
    # the low-precision caches need the bf16 copies in the workspace where no fused kernel reads them
    assert L.csa_workspace_bytes(L.Config(storage="fp4"), 1, 2, 4096) >= \
        L.csa_workspace_bytes(L.Config(storage="bf16"), 1, 2, 4096) + 4096 * (512 + 128) * 2


FAKE = 1 << 20          # a 16-byte aligned address that is never dereferenced


def _cache(**kw):
    k = CsaCache()
    for f in ("kv", "gate", "gate_bias", "idx_k", "idx_gate", "idx_bias", "ckv", "cidx"):
        setattr(k, f, FAKE)
    k.N, k.n_cap = 4096, 1024
    for f, v in kw.items():
        setattr(k, f, v)
    return k


@pytest.mark.parametrize("cfg_kw,cache_kw,first,n,status", [
    (dict(d=256), {}, 0, 4, 2),
    (dict(H=65), {}, 0, 4, 2),
    (dict(top_k=4096), {}, 0, 4, 2),
    (dict(storage="f32", ratio=0), {}, 0, 4, 2),
    ({}, dict(kv=None), 0, 4, 1),
    ({}, dict(kv=FAKE + 8), 0, 4, 1),
    ({}, {}, 1000, 100, 2),            # entries beyond n_cap
    ({}, dict(N=100), 0, 26, 2),       # entries need more raw tokens than N
    ({}, {}, -1, 4, 1),
])
def test_compress_argument_errors(cfg_kw, cache_kw, first, n, status):
    lib = L.load()
    c = L.Config(**cfg_kw).c()
    k = _cache(**cache_kw)
    assert lib.csa_compress(ctypes.byref(c), 2, ctypes.byref(k), first, n, None) == status
    assert lib.csa_last_error()


def test_null_config_and_dtype():
    lib = L.load()
    k = _cache()
    assert lib.csa_compress(None, 1, ctypes.byref(k), 0, 1, None) == 1
    c = L.Config().c()
    c.storage = 7
    assert lib.csa_compress(ctypes.byref(c), 1, ctypes.byref(k), 0, 1, None) == 3


def test_decode_workspace_too_small_and_hca_indexer():
    lib = L.load()
    c = L.Config().c()
    k = _cache()
    st = lib.csa_decode(ctypes.byref(c), 4, FAKE, ctypes.byref(k), FAKE, FAKE, FAKE, FAKE, FAKE, None,
                        FAKE, 16, None)
    assert st == 4 and b"workspace" in lib.csa_last_error()
    h = L.Config(top_k=0, ratio=128).c()
    st = lib.csa_index_topk(ctypes.byref(h), 1, 1, FAKE, FAKE, FAKE, FAKE, 16, FAKE, None, FAKE, 1 << 30, None)
    assert st == 1


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "long_context_sparse_19_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
