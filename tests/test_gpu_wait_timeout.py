"""The attention kernel's bounded waits, made to run out on purpose.

With the wait limit set to 0 ns, the first wait on a phase that has not yet
completed gives up at once: the kernel must then stop, drain its own copies
and tensor-core work, release its tensor memory, return, and report
DSA_DEV_ERR_TIMEOUT in the caller's flag.  The CUDA context stays usable:
a call made right after, with the default limit restored, matches the oracle.
No GPU fault or hang is involved; the limit is a plain host-side setting
passed to the kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attn_close, bf16_dev, dev, pool_dev
from sparse_mla_attention_page_gb300 import binding
from sparse_mla_attention_page_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _decode(w, pool_d, err):
    T, H, K = w["T"], w["H"], w["K"]
    o = torch.zeros(T, H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(T, H, dtype=torch.float32, device="cuda")
    binding.dsa_sparse_attn_decode(bf16_dev(w["q_bf16"]), pool_d, w["layout"], dev(w["topk"]), w["sm_scale"],
                                   o, lse, binding.workspace_for(T, H, K), page_table=dev(w["page_table"]),
                                   page_size=w["page_size"], err_flag=err)
    return o, lse


@pytest.mark.parametrize("layout", ["raw512", "scaled528"])
def test_wait_runs_out_then_context_recovers(layout):
    if layout == "raw512":
        w = W.decode_raw512(seed=400, T=32, H=16, K=2048, pool_rows=32768)
    else:
        w = W.decode_scaled528(seed=401, T=32, H=32, K=2048, pool_rows=32768)
    pool = oracle.fill_pool(w)
    pool_d = pool_dev(pool)
    old = binding.dsa_set_wait_limit_ns(0)
    try:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        _decode(w, pool_d, err)
        torch.cuda.synchronize()                     # returns: nothing hangs
        assert int(err.item()) & binding.DSA_DEV_ERR_TIMEOUT
    finally:
        assert binding.dsa_set_wait_limit_ns(old) == 0
    assert old == 1_000_000_000
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = _decode(w, pool_d, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    tok = np.array([0, 2, 5, 17, 31])
    Or, Lr, _ = oracle.sparse_attn(pool, layout, w["topk"], w["sm_scale"], q_bf16=w["q_bf16"],
                                   page_table=w["page_table"], page_size=w["page_size"], tokens=tok)
    O = o.float().cpu().numpy().astype(np.float64)[tok]
    L = lse.cpu().numpy().astype(np.float64)[tok]
    assert_attn_close(O, L, Or, Lr, f"after a timed-out call ({layout})")
