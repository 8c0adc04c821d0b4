"""pkv_forward_decode_static: decode for callers that cannot allocate device memory.

A caller embedded in another framework's caching allocator, or a latency-bound
loop that must not call cudaMalloc (which can synchronise the device), has no
workspace to hand to pkv_create. This entry point keeps its scratch in a fixed
array inside the library instead. These tests check, through the C ABI, on two
calls in a row (the second call reuses the array the first one left behind):
that it returns bit for bit what pkv_build_metadata + pkv_forward_decode
return (the same kernels on the same plan), and that both are within the
attention tolerance of the fp64 oracle; and that a configuration too large
for the array is refused before anything launches. This file is collected
last so a failure here never hides another test.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_15_gb300 import binding as B
from paged_kv_cache_15_gb300.runner import DeviceBatch, config_for
from paged_kv_cache_15_gb300.workloads import make_workload, preset
from tests._pipeline import oracle_reference

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


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
    assert (err <= ATOL + RTOL * np.abs(np.where(both, 0.0, ref))).all()


def _check(d: DeviceBatch, got, ref):
    """got (static entry) == ref (context decode) bit for bit, and both close to the oracle."""
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    o, lse = oracle_reference(d.W)
    _close(got[0].double().cpu().numpy(), o)
    _close(got[1].double().cpu().numpy(), lse)


def _static_call(d: DeviceBatch):
    W = d.W
    out = torch.full_like(d.out, 3.0)
    lse = torch.full_like(d.lse, 3.0)
    err = torch.full((1,), -1, dtype=torch.int32, device=d.out.device)
    B.pkv_forward_decode_static(d.cfg, W.bs, d.seq_lens, d.page_table, d.q, d.k_pool, d.v_pool, W.sm_scale, out,
                                lse, err, W.k_scale, W.v_scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, lse


def _reference(d: DeviceBatch):
    d.set_kv_buffer()
    d.build_metadata()
    d.forward()
    torch.cuda.synchronize()
    assert d.device_error() == 0
    return d.out.clone(), d.lse.clone()


@pytest.mark.parametrize("second", ["same", "other"])
def test_static_decode_matches_context_decode_twice(second):
    d1 = DeviceBatch(preset("llama3_8b_decode", bs=12, len_scale=0.2))
    ref1 = _reference(d1)
    got1 = _static_call(d1)
    _check(d1, got1, ref1)
    if second == "same":
        d2 = d1
    else:  # shorter batch, other head counts: the array still holds the first call's metadata
        d2 = DeviceBatch(make_workload("s2", "decode", 5, 8, 2, 64, [3, 400, 17, 0, 1000], np.ones(5)))
    ref2 = _reference(d2)
    got2 = _static_call(d2)
    _check(d2, got2, ref2)


def test_static_decode_fp8_pool():
    d = DeviceBatch(preset("long_fp8_decode", bs=3, len_scale=1 / 32))
    ref = _reference(d)
    got = _static_call(d)
    _check(d, got, ref)


def test_static_decode_rejects_configs_beyond_the_array():
    W = preset("tiny_decode")
    cfg = config_for(W, max_q_tokens=1 << 16)  # partial-output scratch far beyond the fixed array
    d = DeviceBatch(W)
    with pytest.raises(B.PkvError) as ei:
        B.pkv_forward_decode_static(cfg, W.bs, d.seq_lens, d.page_table, d.q, d.k_pool, d.v_pool, W.sm_scale,
                                    d.out)
    assert ei.value.status == B.PKV_ERR_CAPACITY
