"""The bounded waits inside the kernels, made to run out on purpose.

pkv_test_hold_first_load makes CTA 0 arm the barrier of its first K/V tile
without issuing the copy, and pkv_set_wait_limit shortens the bound on every
wait, so the waits on that tile give up: the kernel records PKV_DEV_TIMEOUT,
drains its copies in flight, frees its tensor memory and returns. Nothing
faults. The same context must then compute correct results again.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_15_gb300 import binding as B
from paged_kv_cache_15_gb300.runner import DeviceBatch
from paged_kv_cache_15_gb300.workloads import preset
from tests._pipeline import oracle_reference

pytestmark = pytest.mark.gpu

LIMIT_NS = 200_000  # 0.2 ms: far above any wait of a working kernel at these sizes


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_15_gb300 import build
    build.build()
    oracle.build()


def _close(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both = np.isneginf(got) & np.isneginf(ref)
    err = np.where(both, 0.0, np.abs(got - ref))
    assert (err <= 1e-2 + 1e-2 * np.abs(np.where(both, 0.0, ref))).all()


@pytest.mark.parametrize("case", ["decode", "extend", "extend_fp8", "verify_decode_path"])
def test_wait_runs_out_then_context_recovers(case):
    spec = B.PKV_SPEC_PREFILL
    if case == "decode":
        W = preset("llama3_8b_decode", bs=6, len_scale=0.1)
    elif case == "extend":
        W = preset("prefix_extend", bs=2, len_scale=0.1)
    elif case == "extend_fp8":
        W = preset("prefix_extend_fp8", bs=2, len_scale=0.1)
    else:  # the tcgen05 tile kernel over the decode path's plan
        W = preset("spec_verify", bs=4, len_scale=0.05)
        spec = B.PKV_SPEC_DECODE
    d = DeviceBatch(W)
    B.pkv_set_wait_limit(d.ctx, LIMIT_NS)
    B.pkv_test_hold_first_load(d.ctx, True)
    d.step(spec)
    torch.cuda.synchronize()
    assert d.device_error() == B.PKV_DEV_TIMEOUT
    # the same context, default bound, loads issued: correct results
    B.pkv_test_hold_first_load(d.ctx, False)
    B.pkv_set_wait_limit(d.ctx, 0)
    d.out.zero_()
    d.step(spec)
    torch.cuda.synchronize()
    assert d.device_error() == 0
    ref_o, ref_lse = oracle_reference(W)
    _close(d.out.double().cpu().numpy(), ref_o)
    _close(d.lse.double().cpu().numpy(), ref_lse)
