"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
symbol include/dsa.h declares, and rejects bad arguments on the host (before
any device work) with the documented status codes."""
import ctypes
import os
import re

import pytest
import torch

from sparse_mla_attention_page_gb300 import binding
from sparse_mla_attention_page_gb300 import build as build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dsa.h")


def declared_functions():
    with open(HEADER) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
    assert sorted(binding.EXPORTS) == sorted(names)


def test_status_strings_and_row_bytes(L):
    for code in range(11):
        assert binding.status_string(code).startswith("DSA_")
    assert L.dsa_kv_row_bytes(0) == 512
    assert L.dsa_kv_row_bytes(1) == 528
    assert L.dsa_kv_row_bytes(7) == 0


FAKE = 0x10000          # 16-byte aligned non-null address that is never dereferenced


def decode(L, **kw):
    a = dict(q=FAKE, T=4, H=16, D=512, pool=FAKE, rows=4096, layout=0, kvd=512, pt=None, B=1,
             mp=64, ps=64, ts=None, topk=FAKE, K=128, sc=0.1, o=FAKE, lse=FAKE, ws=None, wsb=0,
             err=None)
    a.update(kw)
    return L.dsa_sparse_attn_decode(a["q"], a["T"], a["H"], a["D"], a["pool"], a["rows"],
                                    a["layout"], a["kvd"], a["pt"], a["B"], a["mp"], a["ps"],
                                    a["ts"], a["topk"], a["K"], a["sc"], a["o"], a["lse"],
                                    a["ws"], a["wsb"], a["err"], None)


def prefill(L, **kw):
    a = dict(q=FAKE, qs=FAKE, T=4, H=16, D=512, pool=FAKE, rows=4096, layout=0, kvd=512, pt=None,
             B=1, mp=64, ps=64, ts=None, topk=FAKE, K=128, sc=0.1, o=FAKE, lse=FAKE, ws=None,
             wsb=0, err=None)
    a.update(kw)
    return L.dsa_sparse_attn_prefill_q8(a["q"], a["qs"], a["T"], a["H"], a["D"], a["pool"], a["rows"],
                                        a["layout"], a["kvd"], a["pt"], a["B"], a["mp"], a["ps"],
                                        a["ts"], a["topk"], a["K"], a["sc"], a["o"], a["lse"],
                                        a["ws"], a["wsb"], a["err"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=576), 4), (dict(kvd=528), 4), (dict(layout=3), 3), (dict(layout=2), 4),
    (dict(layout=2, D=576, kvd=576, H=24), 6), (dict(K=0), 5), (dict(K=2000), 5),
    (dict(H=12), 6), (dict(H=256), 6), (dict(T=-1), 2), (dict(q=None), 1), (dict(pool=None), 1),
    (dict(topk=None), 1), (dict(o=None), 1), (dict(lse=None), 1), (dict(rows=0), 2),
    (dict(pt=FAKE, B=0), 2), (dict(pt=FAKE, ps=0), 2), (dict(q=FAKE + 8), 10), (dict(o=FAKE + 4), 10),
    (dict(pool=FAKE + 1), 10), (dict(T=0), 0),
])
def test_decode_host_validation(L, kw, code):
    assert decode(L, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(layout=2, D=576, kvd=576), 3), (dict(layout=3), 3), (dict(layout=-1), 3), (dict(qs=None), 1), (dict(D=1024), 4), (dict(K=64), 5), (dict(H=7), 6),
])
def test_prefill_host_validation(L, kw, code):
    assert prefill(L, **kw) == code


def gather(L, **kw):
    a = dict(pool=FAKE, rows=4096, layout=0, pt=None, B=1, mp=64, ps=64, ts=None, topk=FAKE, T=4, K=100,
             out=FAKE, ob=1 << 30, idx=FAKE, err=None)
    a.update(kw)
    return L.dsa_gather_dequant(a["pool"], a["rows"], a["layout"], a["pt"], a["B"], a["mp"], a["ps"], a["ts"],
                                a["topk"], a["T"], a["K"], a["out"], a["ob"], a["idx"], a["err"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), 2), (dict(K=0), 2), (dict(layout=5), 3), (dict(T=0), 0), (dict(pool=None), 1),
    (dict(topk=None), 1), (dict(out=None), 1), (dict(idx=None), 1), (dict(rows=0), 2),
    (dict(T=1 << 20, K=4096), 2), (dict(pt=FAKE, B=0), 2), (dict(pool=FAKE + 4), 10),
    (dict(out=FAKE + 8), 10), (dict(topk=FAKE + 2), 10),
    (dict(ob=400 * 1024 - 1), 7), (dict(layout=2, ob=400 * 1152 - 2), 7),
    (dict(T=64, K=2048, rows=131072, ob=131072 * 1024 - 1), 7),
])
def test_gather_host_validation(L, kw, code):
    assert gather(L, **kw) == code


def test_gather_workspace_bytes(L):
    """min(pool rows, selected entries) rows of 1024 bytes (1152 for 656-byte rows)."""
    f = L.dsa_gather_dequant_workspace_bytes
    assert f(4, 100, 4096, 0) == 400 * 1024
    assert f(4, 100, 4096, 1) == 400 * 1024
    assert f(4, 100, 4096, 2) == 400 * 1152
    assert f(64, 2048, 131072, 0) == 131072 * 1024          # T*K == pool rows: the full pool
    assert f(128, 2048, 131072, 1) == 131072 * 1024
    assert f(4096, 2048, 16384, 0) == 16384 * 1024
    assert f(1, 1, 10, 7) == 0 and f(-1, 4, 10, 0) == 0


def test_writer_host_validation(L):
    assert L.dsa_kv_write_raw(None, 0, None, None, 10, None, None) == 0          # empty: no-op
    assert L.dsa_kv_write_raw(None, 4, None, None, 10, None, None) == 1
    assert L.dsa_kv_write_scaled(FAKE, -1, FAKE, FAKE, 10, None, None) == 2
    assert L.dsa_kv_write_raw(FAKE + 2, 4, FAKE, FAKE, 10, None, None) == 10
    assert L.dsa_quantize_q8(None, 3, None, None, None) == 1
    assert L.dsa_quantize_q8(FAKE, -3, FAKE, FAKE, None) == 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_reports_device(L):
    assert decode(L) == 8
    assert L.dsa_kv_write_raw(FAKE, 4, FAKE, FAKE, 10, None, None) == 8
    assert binding.dsa_sparse_attn_workspace_bytes(64, 16, 2048) > 0


def test_binding_refuses_cpu_tensors(L):
    x = torch.zeros(4, 512, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        binding.dsa_kv_write_raw(x, torch.zeros(4, dtype=torch.int64), torch.zeros(8, 512, dtype=torch.uint8))
