"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Metadata and KV scatter must be bit-exact. Attention outputs (bf16) and LSE
(fp32) must satisfy |got - ref| <= 1e-2 + 1e-2 |ref| element by element: bf16
output rounding (2^-9 relative) and fp32 accumulation with bf16 (FP8 pools:
f16) MMA operands stay well inside that bound.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_15_gb300 import binding as B
from paged_kv_cache_15_gb300.runner import DeviceBatch, config_for
from paged_kv_cache_15_gb300.workloads import (chain_tree_masks, make_workload, pool_bits, preset, random_sinks,
                                               random_tree_masks)
from tests._pipeline import oracle_meta, oracle_pools, oracle_reference

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="session", autouse=True)
def _built():
    from paged_kv_cache_15_gb300 import build
    build.build()
    oracle.build()


def check_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_ninf = np.isneginf(got) & np.isneginf(ref)
    err = np.where(both_ninf, 0.0, np.abs(got - ref))
    tol = ATOL + RTOL * np.abs(np.where(both_ninf, 0.0, ref))
    bad = ~(err <= tol)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {idx}: "
                             f"got {got[idx]} ref {ref[idx]}")


def run_path(W, spec_mode=B.PKV_SPEC_PREFILL, cfg=None):
    d = DeviceBatch(W, cfg=cfg)
    d.step(spec_mode)
    torch.cuda.synchronize()
    assert d.device_error() == 0
    return d


def full_check(W, spec_mode=B.PKV_SPEC_PREFILL):
    d = run_path(W, spec_mode)
    ref_o, ref_lse = oracle_reference(W)
    check_close(d.out.double().cpu().numpy(), ref_o, "o")
    check_close(d.lse.double().cpu().numpy(), ref_lse, "lse")
    return d


def workspace_ints(d: DeviceBatch, ptr: int, n: int) -> np.ndarray:
    """int32 view of n values at a device address inside the context's workspace."""
    ws = d.attn.workspace
    off = ptr - ws.data_ptr()
    assert 0 <= off and off + 4 * n <= ws.numel()
    return ws[off:off + 4 * n].view(torch.int32).cpu().numpy()


# ------------------------------------------------------------------ metadata
def _meta_case(name):
    if name == "tiny_decode":
        return preset("tiny_decode")
    if name == "decode_ragged":
        return make_workload("r", "decode", 37, 8, 2, 64, np.arange(37) * 29 % 700, np.ones(37))
    if name == "extend":
        return preset("prefix_extend", bs=5, len_scale=0.25)
    if name == "verify":
        return preset("spec_verify", bs=6, len_scale=0.1)
    if name == "many_requests":
        rng = np.random.default_rng(3)
        return make_workload("m", "extend", 300, 4, 2, 64, rng.integers(0, 90, 300), rng.integers(1, 20, 300))
    raise KeyError(name)


@pytest.mark.parametrize("name", ["tiny_decode", "decode_ragged", "extend", "verify", "many_requests"])
def test_metadata_bit_exact(name):
    W = _meta_case(name)
    d = DeviceBatch(W)
    d.build_metadata()
    torch.cuda.synchronize()
    assert d.device_error() == 0
    ref = oracle_meta(W)
    p_indptr, p_indices, p_last, p_qo = B.pkv_get_metadata(d.ctx)
    bs = W.bs
    n_pages = int(ref["kv_indptr"][-1])
    assert np.array_equal(workspace_ints(d, p_indptr, bs + 1), ref["kv_indptr"])
    assert np.array_equal(workspace_ints(d, p_indices, n_pages), ref["kv_indices"])
    assert np.array_equal(workspace_ints(d, p_last, bs), ref["kv_last_page_len"])
    assert np.array_equal(workspace_ints(d, p_qo, bs + 1), ref["qo_indptr"])


# ------------------------------------------------------------------ set_kv_buffer
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_set_kv_buffer_bit_exact(kv_dtype):
    W = make_workload("s", "extend", 6, 16, 8, 128, [0, 40, 7, 100, 3, 64], [37, 16, 1, 200, 90, 5],
                      kv_dtype=kv_dtype)
    d = DeviceBatch(W)
    d.set_kv_buffer()
    torch.cuda.synchronize()
    assert d.device_error() == 0
    kp, vp = oracle_pools(W)
    assert np.array_equal(pool_bits(d.k_pool.cpu()), kp)
    assert np.array_equal(pool_bits(d.v_pool.cpu()), vp)


def test_set_kv_buffer_fp8_saturates_like_oracle():
    W = make_workload("sat", "extend", 1, 8, 8, 128, [0], [64], kv_dtype="fp8_e4m3")
    W.k_new.mul_(300.0)  # many values beyond +-448 after scaling
    d = DeviceBatch(W)
    d.set_kv_buffer()
    torch.cuda.synchronize()
    kp, _ = oracle_pools(W)
    assert np.array_equal(pool_bits(d.k_pool.cpu()), kp)


def test_set_kv_buffer_bad_slot_recorded_and_skipped():
    W = make_workload("bad", "extend", 1, 8, 8, 128, [0], [4])
    W.loc[2] = W.num_slots + 10
    d = DeviceBatch(W)
    before = pool_bits(d.k_pool.cpu()).copy()
    d.set_kv_buffer()
    assert d.device_error() == B.PKV_DEV_BAD_SLOT
    after = pool_bits(d.k_pool.cpu())
    assert np.array_equal(np.delete(after, W.loc[[0, 1, 3]], axis=0), np.delete(before, W.loc[[0, 1, 3]], axis=0))


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("case", ["tiny", "llama_small", "fp8_small", "ragged_short", "single_key"])
def test_decode_parity(case):
    if case == "tiny":
        W = preset("tiny_decode")
    elif case == "llama_small":
        W = preset("llama3_8b_decode", bs=8, len_scale=0.25)
    elif case == "fp8_small":
        W = preset("long_fp8_decode", bs=4, len_scale=1 / 16)
    elif case == "ragged_short":
        rng = np.random.default_rng(9)
        W = make_workload("rs", "decode", 21, 32, 8, 128, rng.integers(0, 300, 21), np.ones(21))
    elif case == "single_key":
        W = make_workload("one", "decode", 3, 8, 2, 64, [0, 0, 0], [1, 1, 1])
    full_check(W)


@pytest.mark.parametrize("case", ["g16", "g16_fp8", "g12_d64", "g3", "mha_d64", "g8_fp8", "verify_q2", "verify_q4"])
def test_decode_tile_shapes(case):
    """Decode-path units of 1 to 16 query rows: one 8-row key-major tile for
    up to 8 rows, two for 9 to 16 (groups of 12 and 16, four drafts of a group
    of 4), bf16 and FP8 pools, head_dim 64 and 128; the verify cases put
    several tokens with different causal limits into one tile."""
    rng = np.random.default_rng(31)
    lens = lambda n: rng.integers(0, 900, n)
    if case == "g16":
        W = make_workload("t_g16", "decode", 5, 32, 2, 128, lens(5), np.ones(5))
    elif case == "g16_fp8":
        W = make_workload("t_g16f", "decode", 4, 32, 2, 128, lens(4), np.ones(4), kv_dtype="fp8_e4m3")
    elif case == "g12_d64":
        W = make_workload("t_g12", "decode", 5, 24, 2, 64, lens(5), np.ones(5))
    elif case == "g3":
        W = make_workload("t_g3", "decode", 6, 24, 8, 128, lens(6), np.ones(6))
    elif case == "mha_d64":
        W = make_workload("t_mha", "decode", 4, 8, 8, 64, lens(4), np.ones(4))
    elif case == "g8_fp8":
        W = make_workload("t_g8f", "decode", 3, 32, 4, 128, lens(3), np.ones(3), kv_dtype="fp8_e4m3")
    elif case == "verify_q2":
        W = make_workload("t_vq2", "verify", 4, 16, 4, 128, lens(4), [2, 1, 2, 2])
    else:
        W = make_workload("t_vq4", "verify", 4, 16, 4, 128, lens(4), [4, 3, 4, 1])
    full_check(W, spec_mode=B.PKV_SPEC_DECODE)


def test_decode_padding_requests_give_zero_and_neg_inf():
    W = make_workload("pad", "decode", 4, 8, 2, 64, [50, 0, 17, 0], [1, 0, 1, 0])
    W_dec = make_workload("pad", "decode", 4, 8, 2, 64, [50, 0, 17, 0], [1, 0, 1, 0])
    # two padding requests with seq_len 0 but one query row each, as a padded graph batch has
    W_dec.seq_lens[:] = [51, 0, 18, 0]
    W_dec.qo_lens[:] = 1
    q = torch.zeros((4, 8, 64), dtype=torch.bfloat16)
    q[[0, 2]] = W.q
    W_dec.q = q
    d = run_path(W_dec)
    out = d.out.float().cpu().numpy()
    lse = d.lse.cpu().numpy()
    assert np.all(out[[1, 3]] == 0) and np.all(np.isneginf(lse[[1, 3]]))
    ref_o, ref_lse = oracle.attention(
        np.ascontiguousarray(q.view(torch.int16).numpy().view(np.uint16)), *oracle_pools(W_dec),
        oracle.build_metadata(W_dec.seq_lens, W_dec.page_table, 16), 8, 2, 16, W_dec.sm_scale)
    check_close(out, ref_o, "o")
    check_close(lse, ref_lse, "lse")


def test_decode_nan_unused_slots_never_read():
    # workloads fill every slot that holds no token with NaN; a read of one shows up as NaN
    W = preset("llama3_8b_decode", bs=16, len_scale=0.05)
    d = run_path(W)
    assert torch.isfinite(d.out.float()).all() and torch.isfinite(d.lse).all()


def test_idle_and_empty_batch_are_no_ops():
    W = preset("tiny_decode")
    d = DeviceBatch(W)
    d.out.fill_(7.0)
    B.pkv_build_metadata(d.ctx, B.PKV_MODE_IDLE, 0, None, None, None)
    B.pkv_forward(d.ctx, B.PKV_MODE_IDLE, B.PKV_SPEC_PREFILL, d.q, d.k_pool, d.v_pool, 1.0, d.out, d.lse)
    torch.cuda.synchronize()
    assert torch.all(d.out.float() == 7.0)


# ------------------------------------------------------------------ verify on the decode path
@pytest.mark.parametrize("bs,len_scale", [(8, 0.1), (3, 0.02)])
def test_verify_decode_path_parity(bs, len_scale):
    W = preset("spec_verify", bs=bs, len_scale=len_scale)
    full_check(W, spec_mode=B.PKV_SPEC_DECODE)


@pytest.mark.parametrize("case", ["rows128_g8", "one_token_rows", "ragged_tiles", "d64_g16"])
def test_verify_decode_path_tensor_core_tiles(case):
    """The decode path's verify shapes run on 128-row tcgen05 tiles over the
    decode plan's split items: a full tile (16 drafts x group 8), one-token
    requests on a configuration sized for drafts (16 valid rows of 128),
    lengths that end anywhere inside a 128-key tile and splits of many
    lengths, and head_dim 64."""
    cfg = None
    if case == "rows128_g8":
        W = make_workload("vt128", "verify", 4, 32, 4, 128, [3000, 17, 900, 6100], [16, 16, 9, 16])
    elif case == "one_token_rows":
        W = make_workload("vt1", "verify", 6, 64, 4, 128, [5000, 300, 0, 2047, 129, 12000], np.ones(6))
        cfg = config_for(W, max_qo_len=8)
    elif case == "ragged_tiles":
        W = make_workload("vtr", "verify", 5, 64, 4, 128, [2045, 126, 16380, 3999, 257], [4, 8, 5, 7, 6])
    else:
        W = make_workload("vt64", "verify", 4, 32, 2, 64, [700, 4000, 33, 9000], [8, 3, 8, 5])
    d = DeviceBatch(W, cfg=cfg)
    d.step(B.PKV_SPEC_DECODE)
    torch.cuda.synchronize()
    assert d.device_error() == 0
    assert "tcgen05" in B.pkv_describe(d.ctx).split("| decode:")[1].split("|")[0]
    ref_o, ref_lse = oracle_reference(W)
    check_close(d.out.double().cpu().numpy(), ref_o, "o")
    check_close(d.lse.double().cpu().numpy(), ref_lse, "lse")


def test_verify_decode_path_fp8():
    W = make_workload("vf8", "verify", 5, 32, 8, 128, [100, 2000, 517, 33, 4096], [4, 8, 5, 7, 6],
                      kv_dtype="fp8_e4m3")
    full_check(W, spec_mode=B.PKV_SPEC_DECODE)


# ------------------------------------------------------------------ full sizes, every row
FULL_PRESETS = ["tiny_decode", "llama3_8b_decode", "prefix_extend", "prefix_extend_fp8", "spec_verify",
                "long_fp8_decode"]


@pytest.mark.parametrize("name", FULL_PRESETS)
def test_full_size_metadata_and_pools_bit_exact(name):
    """Every named case at its full size: the pools after set_kv_buffer (every
    byte, untouched NaN slots included) and the metadata, bit for bit."""
    W = preset(name)
    d = DeviceBatch(W)
    d.set_kv_buffer()
    d.build_metadata()
    torch.cuda.synchronize()
    assert d.device_error() == 0
    kp, vp = oracle_pools(W)
    assert np.array_equal(pool_bits(d.k_pool.cpu()), kp)
    assert np.array_equal(pool_bits(d.v_pool.cpu()), vp)
    del kp, vp
    ref = oracle_meta(W)
    p_indptr, p_indices, p_last, p_qo = B.pkv_get_metadata(d.ctx)
    n_pages = int(ref["kv_indptr"][-1])
    assert np.array_equal(workspace_ints(d, p_indptr, W.bs + 1), ref["kv_indptr"])
    assert np.array_equal(workspace_ints(d, p_indices, n_pages), ref["kv_indices"])
    assert np.array_equal(workspace_ints(d, p_last, W.bs), ref["kv_last_page_len"])
    assert np.array_equal(workspace_ints(d, p_qo, W.bs + 1), ref["qo_indptr"])


@pytest.mark.parametrize("name", ["llama3_8b_decode", "long_fp8_decode"])
def test_full_size_decode_every_row(name):
    full_check(preset(name))


def test_full_size_verify_decode_path_every_row():
    full_check(preset("spec_verify"), spec_mode=B.PKV_SPEC_DECODE)


# ------------------------------------------------------------------ 128-token pages
@pytest.mark.parametrize("name", FULL_PRESETS)
def test_page_size_128_metadata_and_pools_bit_exact(name):
    """Every named case at full size in 128-token pages: kv_indptr /
    kv_indices / kv_last_page_len count 128-token pages, bit for bit against
    the oracle; the pools after set_kv_buffer likewise."""
    W = preset(name, page_size=128)
    d = DeviceBatch(W)
    d.set_kv_buffer()
    d.build_metadata()
    torch.cuda.synchronize()
    assert d.device_error() == 0
    kp, vp = oracle_pools(W)
    assert np.array_equal(pool_bits(d.k_pool.cpu()), kp)
    assert np.array_equal(pool_bits(d.v_pool.cpu()), vp)
    del kp, vp
    ref = oracle_meta(W)
    p_indptr, p_indices, p_last, p_qo = B.pkv_get_metadata(d.ctx)
    n_pages = int(ref["kv_indptr"][-1])
    assert np.array_equal(workspace_ints(d, p_indptr, W.bs + 1), ref["kv_indptr"])
    assert np.array_equal(workspace_ints(d, p_indices, n_pages), ref["kv_indices"])
    assert np.array_equal(workspace_ints(d, p_last, W.bs), ref["kv_last_page_len"])
    assert np.array_equal(workspace_ints(d, p_qo, W.bs + 1), ref["qo_indptr"])


@pytest.mark.parametrize("name", ["llama3_8b_decode", "prefix_extend"])
def test_page_size_128_full_size_every_row(name):
    """The Llama-3-8B-shaped decode and the prefix-cached extend at full size
    in 128-token pages, every row against the oracle."""
    full_check(preset(name, page_size=128))


@pytest.mark.parametrize("case", ["tiny", "fp8_decode", "verify_decode", "verify_prefill", "fp8_extend", "tree",
                                  "mixed_extend", "d64"])
def test_page_size_128_parity(case):
    """128-token pages on every path: decode (bf16 and E4M3), verify on both
    paths, extend on E4M3 pools, draft trees with sinks, mixed extend batches
    whose lengths end anywhere inside a page, head_dim 64."""
    spec = B.PKV_SPEC_PREFILL
    if case == "tiny":
        W = preset("tiny_decode", page_size=128)
    elif case == "fp8_decode":
        W = preset("long_fp8_decode", bs=4, len_scale=1 / 16, page_size=128)
    elif case == "verify_decode":
        W = preset("spec_verify", bs=8, len_scale=0.1, page_size=128)
        spec = B.PKV_SPEC_DECODE
    elif case == "verify_prefill":
        W = preset("spec_verify", bs=8, len_scale=0.1, page_size=128)
    elif case == "fp8_extend":
        W = preset("prefix_extend_fp8", bs=3, len_scale=0.2, page_size=128)
    elif case == "tree":
        rng = np.random.default_rng(51)
        W = make_workload("t128", "verify", 5, 32, 4, 128, rng.integers(0, 3000, 5), rng.integers(1, 17, 5),
                          page_size=128)
        W.tree_mask = random_tree_masks(W.qo_lens, seed=51)
        W.sinks = random_sinks(W.num_q_heads, seed=52)
    elif case == "mixed_extend":
        W = make_workload("m128", "extend", 6, 32, 8, 128, [0, 127, 128, 129, 1000, 4095], [1, 1, 300, 2, 129, 64],
                          page_size=128)
    else:
        W = make_workload("d128", "extend", 4, 8, 2, 64, [5, 0, 300, 129], [200, 33, 7, 128], page_size=128)
    full_check(W, spec_mode=spec)


def test_page_size_128_row_shorter_than_a_request_recorded():
    """The page-table row holds 128-token pages: a request of 300 tokens needs
    3 entries, so a stride of 2 makes it a bad length (recorded, empty)."""
    W = make_workload("s128", "decode", 3, 8, 2, 64, [99, 299, 200], np.ones(3), page_size=128)
    d = DeviceBatch(W)
    table = torch.zeros((W.bs + 2, 2), dtype=torch.int32, device=d.page_table.device)
    table[:W.bs] = d.page_table[:, :2]
    d.page_table = table[:W.bs]
    d.step()
    torch.cuda.synchronize()
    assert d.device_error() == B.PKV_DEV_BAD_LENGTH
    out = d.out.double().cpu().numpy()
    lse = d.lse.double().cpu().numpy()
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    W.seq_lens = np.array([W.seq_lens[0], 0, W.seq_lens[2]], dtype=W.seq_lens.dtype)
    ref_o, ref_lse = oracle_reference(W)
    check_close(out, ref_o, "o")
    check_close(lse, ref_lse, "lse")


# ------------------------------------------------------------------ device-side data errors
def test_bad_page_id_recorded_without_fault():
    W = preset("tiny_decode")
    W.page_table[1, 2] = W.num_pages + 3
    d = DeviceBatch(W)
    d.set_kv_buffer()
    d.build_metadata()
    d.forward()
    assert d.device_error() == B.PKV_DEV_BAD_PAGE
    assert d.device_error() == 0  # reading clears the word


def test_page_table_row_shorter_than_a_request_recorded():
    """A request with more pages than one page-table row holds is recorded as
    a bad length and treated as empty, and its gather never runs past its row.
    Two spare rows follow the batch's rows, so a gather that ignored the
    stride would still read inside this allocation (pages that hold other
    requests' keys, or the NaN sentinel page) and show up in the output."""
    W = preset("tiny_decode")  # 3, 7, 14 and 19 pages
    stride = 10
    d = DeviceBatch(W)
    table = torch.zeros((W.bs + 2, stride), dtype=torch.int32, device=d.page_table.device)
    table[:W.bs] = d.page_table[:, :stride]
    table[W.bs:] = d.page_table[:2, :stride]
    d.page_table = table[:W.bs]
    d.step()
    torch.cuda.synchronize()
    assert d.device_error() == B.PKV_DEV_BAD_LENGTH
    out = d.out.double().cpu().numpy()
    lse = d.lse.double().cpu().numpy()
    assert np.all(out[2:] == 0) and np.all(np.isneginf(lse[2:]))
    W.seq_lens = np.array([W.seq_lens[0], W.seq_lens[1], 0, 0], dtype=W.seq_lens.dtype)
    ref_o, ref_lse = oracle_reference(W)
    check_close(out, ref_o, "o")
    check_close(lse, ref_lse, "lse")


def test_capacity_overflow_recorded():
    W = preset("tiny_decode")
    cfg = config_for(W, max_pages_total=10)
    d = DeviceBatch(W, cfg=cfg)
    d.build_metadata()
    assert d.device_error() == B.PKV_DEV_CAPACITY


# ------------------------------------------------------------------ CUDA graph capture / replay
def test_graph_replay_with_new_lengths():
    """Capture save_kv_cache + metadata + decode once, replay with other lengths."""
    shape = dict(bs=6, num_q_heads=32, num_kv_heads=8, head_dim=128)
    pages = 700
    W1 = make_workload("g1", "decode", 6, 32, 8, 128, [1500, 30, 700, 2047, 5, 999], np.ones(6), num_pages=pages)
    W2 = make_workload("g2", "decode", 6, 32, 8, 128, [100, 2500, 16, 1, 1300, 444], np.ones(6), num_pages=pages)
    width = max(W1.page_table.shape[1], W2.page_table.shape[1])
    cfg = config_for(W1, max_pages_total=pages - 1)
    d = DeviceBatch(W1, cfg=cfg)
    d.page_table = torch.zeros((6, width), dtype=torch.int32, device="cuda")
    d.page_table[:, :W1.page_table.shape[1]] = torch.from_numpy(W1.page_table)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d.step()  # warm-up outside the graph
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d.step()
    for W in (W1, W2):
        d.q.copy_(W.q)
        d.k_pool.copy_(W.k_pool)
        d.v_pool.copy_(W.v_pool)
        d.k_new.copy_(W.k_new)
        d.v_new.copy_(W.v_new)
        d.loc.copy_(torch.from_numpy(W.loc))
        d.seq_lens.copy_(torch.from_numpy(W.seq_lens))
        d.page_table.zero_()
        d.page_table[:, :W.page_table.shape[1]] = torch.from_numpy(W.page_table)
        g.replay()
        torch.cuda.synchronize()
        assert d.device_error() == 0
        ref_o, ref_lse = oracle_reference(W)
        check_close(d.out.double().cpu().numpy(), ref_o, f"o ({W.name})")
        check_close(d.lse.double().cpu().numpy(), ref_lse, f"lse ({W.name})")


# ------------------------------------------------------------------ extend (tcgen05) and verify on the prefill path
@pytest.mark.parametrize("case", ["small", "ragged", "d64", "mha", "prefix_zero", "long_new", "g3", "g6_d64"])
def test_extend_parity(case):
    if case == "small":
        W = make_workload("e", "extend", 3, 8, 2, 128, [0, 37, 200], [130, 9, 61])
    elif case == "ragged":
        rng = np.random.default_rng(21)
        W = make_workload("er", "extend", 9, 32, 8, 128, rng.integers(0, 700, 9), rng.integers(1, 300, 9))
    elif case == "d64":
        W = make_workload("e64", "extend", 4, 8, 2, 64, [5, 0, 300, 129], [200, 33, 7, 128])
    elif case == "mha":
        W = make_workload("emha", "extend", 2, 4, 4, 128, [100, 17], [150, 260])
    elif case == "prefix_zero":
        W = make_workload("ez", "extend", 2, 16, 4, 128, [0, 0], [1, 383])
    elif case == "long_new":
        W = preset("prefix_extend", bs=2, len_scale=0.3)
    elif case == "g3":  # group size that does not divide the 128-row tile
        W = make_workload("e3", "extend", 3, 12, 4, 128, [20, 300, 0], [77, 140, 33])
    elif case == "g6_d64":
        W = make_workload("e6", "extend", 2, 6, 1, 64, [100, 7], [90, 200])
    full_check(W)


def _shift_scores(W, q_scale=1.0, heads=None, bias=0.0):
    """Moves the scores far outside the N(0,1) range of the presets: Q (or only
    the given query heads) is multiplied by q_scale, and bias is added to the
    first component of every Q row and subtracted from that of every K row,
    which shifts q.k by about -bias^2. The oracle sees the same bf16 values."""
    q = W.q.float()
    sel = slice(None) if heads is None else list(heads)
    q[:, sel] = q[:, sel] * q_scale
    if bias:
        q[:, :, 0] += bias
        for name in ("k_pool", "k_new"):
            t = getattr(W, name).float()
            t[..., 0] -= bias
            setattr(W, name, t.bfloat16())
    W.q = q.bfloat16()
    return W


@pytest.mark.parametrize("case", ["large_scores", "mixed_heads", "far_below"])
@pytest.mark.parametrize("mode", ["extend", "decode"])
def test_scores_far_from_reference(mode, case):
    """Scores of magnitude ~2^5 to ~2^7 in the exponent: the softmax reference
    has to move up for every row (large_scores), for some rows of a warp only
    (mixed_heads: two query heads scaled), or down for rows whose scores all
    sit far below zero (far_below: without a move every p would flush to 0)."""
    if mode == "extend":
        W = make_workload("sx_" + case, "extend", 3, 8, 2, 128, [40, 0, 300], [150, 70, 9])
    else:
        W = make_workload("sd_" + case, "decode", 4, 8, 2, 128, [37, 100, 211, 1300], [1, 1, 1, 1])
    if case == "large_scores":
        _shift_scores(W, q_scale=12.0)
    elif case == "mixed_heads":
        _shift_scores(W, q_scale=12.0, heads=[1, 6])
    else:
        _shift_scores(W, bias=34.0)
    full_check(W)


def test_extend_rows_exceeding_group_tiles():
    # group 16: a 128-row tile holds 8 tokens
    W = make_workload("g16", "extend", 3, 64, 4, 128, [10, 500, 0], [20, 9, 130])
    full_check(W)


@pytest.mark.parametrize("case", ["d64_g8", "g3"])
@pytest.mark.parametrize("spec", ["prefill", "decode"])
def test_verify_other_shapes_both_paths(case, spec):
    """Verify batches outside the preset's shape: head_dim 64 with a group of
    8, and a group of 3 (Q tiles copied by the softmax warps, not by TMA),
    both with contexts long enough to be split along KV."""
    if case == "d64_g8":
        W = make_workload("v64", "verify", 4, 16, 2, 64, [900, 3000, 40, 12000], [5, 8, 3, 6])
    else:
        W = make_workload("vg3", "verify", 3, 12, 4, 128, [7000, 150, 2600], [4, 7, 5])
    full_check(W, spec_mode=B.PKV_SPEC_PREFILL if spec == "prefill" else B.PKV_SPEC_DECODE)


@pytest.mark.parametrize("bs,len_scale", [(8, 0.1), (3, 0.02)])
def test_verify_prefill_path_parity(bs, len_scale):
    W = preset("spec_verify", bs=bs, len_scale=len_scale)
    full_check(W, spec_mode=B.PKV_SPEC_PREFILL)


def test_verify_paths_agree():
    """target_verify through the decode path and through the prefill path."""
    W = preset("spec_verify", bs=6, len_scale=0.05)
    d1 = run_path(W, spec_mode=B.PKV_SPEC_DECODE)
    o1, l1 = d1.out.double().cpu().numpy(), d1.lse.double().cpu().numpy()
    d2 = run_path(W, spec_mode=B.PKV_SPEC_PREFILL)
    o2, l2 = d2.out.double().cpu().numpy(), d2.lse.double().cpu().numpy()
    check_close(o1, o2, "decode-path vs prefill-path output")
    check_close(l1, l2, "decode-path vs prefill-path lse")


def test_extend_nan_unused_slots_never_read():
    W = preset("prefix_extend", bs=4, len_scale=0.05)
    d = run_path(W)
    assert torch.isfinite(d.out.float()).all() and torch.isfinite(d.lse).all()


@pytest.mark.parametrize("case", ["small", "g16", "long_prefix", "verify_prefill", "with_sinks"])
def test_extend_fp8_pool(case):
    """E4M3 pools on the extend path: the producer warps widen each tile's
    codes to f16 in shared memory (no copy of the pool), k_scale goes into
    the score scale and v_scale into the output; every row against the
    oracle's exact E4M3 decoding."""
    spec = B.PKV_SPEC_PREFILL
    if case == "small":
        W = make_workload("e8", "extend", 3, 8, 2, 128, [10, 0, 300], [20, 130, 7], kv_dtype="fp8_e4m3")
    elif case == "g16":
        W = make_workload("e8g", "extend", 3, 32, 2, 128, [500, 33, 0], [64, 1, 200], kv_dtype="fp8_e4m3")
    elif case == "long_prefix":
        W = make_workload("e8l", "extend", 2, 32, 8, 128, [6000, 2500], [300, 45], kv_dtype="fp8_e4m3")
    elif case == "verify_prefill":
        rng = np.random.default_rng(48)
        W = make_workload("e8v", "verify", 6, 64, 4, 128, rng.integers(100, 3000, 6), rng.integers(4, 9, 6),
                          kv_dtype="fp8_e4m3")
    else:
        W = make_workload("e8s", "extend", 3, 16, 4, 128, [700, 0, 90], [50, 300, 1], kv_dtype="fp8_e4m3")
        W.sinks = random_sinks(W.num_q_heads, seed=14)
    full_check(W, spec_mode=spec)


@pytest.mark.parametrize("name", ["prefix_extend", "prefix_extend_fp8"])
def test_full_size_extend_every_row(name):
    """The prefix-cached extend case at full size (about 296k rows), bf16 and
    E4M3 pools (the new tokens quantised by set_kv_buffer), every row against
    the oracle."""
    full_check(preset(name))


def test_full_size_verify_prefill_path_every_row():
    full_check(preset("spec_verify"), spec_mode=B.PKV_SPEC_PREFILL)


def test_extend_graph_replay():
    W = make_workload("eg", "extend", 3, 32, 8, 128, [64, 1000, 3], [200, 50, 317])
    d = DeviceBatch(W)
    d.step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d.step()
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        d.step()
    d.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle_reference(W)
    check_close(d.out.double().cpu().numpy(), ref_o, "o (graph)")
    check_close(d.lse.double().cpu().numpy(), ref_lse, "lse (graph)")


@pytest.mark.parametrize("spec", ["prefill", "decode"])
def test_draft_extend_mode_both_paths(spec):
    """DRAFT_EXTEND is routed like TARGET_VERIFY (by the speculative attention
    mode) and computes the same bottom-right causal attention over the drafts."""
    W = make_workload("dx", "verify", 5, 16, 4, 128, [700, 0, 2100, 33, 1500], [3, 1, 4, 2, 4])
    sm = B.PKV_SPEC_PREFILL if spec == "prefill" else B.PKV_SPEC_DECODE
    assert B.pkv_select_backend(B.PKV_MODE_DRAFT_EXTEND, sm) == (B.PKV_PATH_EXTEND if spec == "prefill" else B.PKV_PATH_DECODE)
    d = DeviceBatch(W)
    d.set_kv_buffer()
    d.build_metadata(mode=B.PKV_MODE_DRAFT_EXTEND)
    d.forward(sm, mode=B.PKV_MODE_DRAFT_EXTEND)
    torch.cuda.synchronize()
    assert d.device_error() == 0
    ref_o, ref_lse = oracle_reference(W)
    check_close(d.out.double().cpu().numpy(), ref_o, "o")
    check_close(d.lse.double().cpu().numpy(), ref_lse, "lse")


def test_prefill_chunks_and_decode_rows_in_one_extend_call():
    """A mixed batch on the extend path: prefill chunks of hundreds of tokens
    next to one-token (decode) requests and short chunks, with and without a
    cached prefix."""
    W = make_workload("mix", "extend", 7, 32, 8, 128, [0, 900, 3000, 40, 0, 1200, 5000], [300, 1, 1, 77, 1, 2, 1])
    full_check(W)


# ------------------------------------------------------------------ draft trees
def _tree_verify(name, bs, hq, hkv, d, max_drafts, seed, kv_dtype="bf16"):
    rng = np.random.default_rng(seed)
    W = make_workload(name, "verify", bs, hq, hkv, d, rng.integers(0, 1500, bs),
                      rng.integers(1, max_drafts + 1, bs), kv_dtype=kv_dtype)
    W.tree_mask = random_tree_masks(W.qo_lens, seed=seed)
    return W


@pytest.mark.parametrize("case", ["g16", "g4_d64", "g4_32_drafts", "g8_fp8"])
@pytest.mark.parametrize("spec", ["prefill", "decode"])
def test_tree_verify_parity(case, spec):
    """Target verify with random draft trees (each draft sees the cached
    prefix, its ancestors and itself) on both paths."""
    if case == "g16":
        W = _tree_verify("tv16", 6, 32, 2, 128, 8, 41)
    elif case == "g4_d64":
        W = _tree_verify("tv4", 5, 16, 4, 64, 8, 42)
    elif case == "g4_32_drafts":
        W = _tree_verify("tv32", 4, 16, 4, 128, 32, 43)
    else:
        W = _tree_verify("tv8f", 4, 32, 4, 128, 16, 44, kv_dtype="fp8_e4m3")
    full_check(W, spec_mode=B.PKV_SPEC_PREFILL if spec == "prefill" else B.PKV_SPEC_DECODE)


@pytest.mark.parametrize("spec", ["prefill", "decode"])
def test_chain_tree_matches_no_tree(spec):
    """A chain-shaped tree gives the causal result of a batch without a mask."""
    W = _tree_verify("tvc", 5, 32, 2, 128, 8, 45)
    W.tree_mask = None
    sm = B.PKV_SPEC_PREFILL if spec == "prefill" else B.PKV_SPEC_DECODE
    plain = run_path(W, sm)
    W.tree_mask = chain_tree_masks(W.qo_lens)
    chain = run_path(W, sm)
    assert torch.equal(plain.out, chain.out)
    assert torch.equal(plain.lse, chain.lse)


def test_tree_mask_ignored_by_extend_batches():
    """The mask applies to verify batches only: an EXTEND batch stays causal."""
    W = make_workload("tve", "extend", 3, 16, 4, 128, [300, 0, 1000], [40, 9, 3])
    W.tree_mask = random_tree_masks(W.qo_lens, seed=46)
    d = run_path(W)
    W.tree_mask = None
    ref_o, ref_lse = oracle_reference(W)
    check_close(d.out.double().cpu().numpy(), ref_o, "o")
    check_close(d.lse.double().cpu().numpy(), ref_lse, "lse")


def test_tree_of_more_than_64_drafts_recorded():
    W = make_workload("tv65", "verify", 2, 8, 2, 128, [100, 50], [65, 3])
    W.tree_mask = np.concatenate([np.full(65, np.uint64(0xFFFFFFFFFFFFFFFF)), chain_tree_masks([3])])
    d = DeviceBatch(W)
    d.step(B.PKV_SPEC_PREFILL)
    torch.cuda.synchronize()
    assert d.device_error() == B.PKV_DEV_TREE_TOO_LONG
    assert torch.isfinite(d.out.float()).all()


def test_non_positive_scales_rejected():
    W = preset("tiny_decode")
    d = DeviceBatch(W)
    d.set_kv_buffer()
    d.build_metadata()
    for bad in (0.0, -0.125, float("nan"), float("inf")):
        with pytest.raises(B.PkvError) as e:
            B.pkv_forward(d.ctx, d.mode, B.PKV_SPEC_PREFILL, d.q, d.k_pool, d.v_pool, bad, d.out, d.lse)
        assert e.value.status == B.PKV_ERR_INVALID_ARG
    Wf = preset("long_fp8_decode", bs=2, len_scale=1 / 64)
    df = DeviceBatch(Wf)
    df.set_kv_buffer()
    df.build_metadata()
    with pytest.raises(B.PkvError):
        B.pkv_forward(df.ctx, df.mode, B.PKV_SPEC_PREFILL, df.q, df.k_pool, df.v_pool, Wf.sm_scale, df.out,
                      df.lse, 0.0, Wf.v_scale)


# ------------------------------------------------------------------ attention sinks
@pytest.mark.parametrize("case", ["decode", "decode_fp8", "decode_g16", "extend", "verify_prefill", "verify_decode",
                                  "tree_verify"])
def test_attention_sinks_parity(case):
    """Each query head's sink logit joins its softmax as a zero-value key, on
    single-split rows (the attention kernels apply it) and split rows (the
    merge applies it)."""
    spec = B.PKV_SPEC_PREFILL
    if case == "decode":
        W = preset("llama3_8b_decode", bs=8, len_scale=0.25)
    elif case == "decode_fp8":
        W = preset("long_fp8_decode", bs=3, len_scale=1 / 32)
    elif case == "decode_g16":
        W = make_workload("sk16", "decode", 5, 32, 2, 128, [0, 40, 700, 3000, 9], np.ones(5))
    elif case == "extend":
        W = make_workload("skx", "extend", 4, 16, 4, 128, [0, 300, 1200, 5], [200, 70, 1, 400])
    elif case == "verify_prefill":
        W = preset("spec_verify", bs=6, len_scale=0.1)
    elif case == "verify_decode":
        W = preset("spec_verify", bs=6, len_scale=0.1)
        spec = B.PKV_SPEC_DECODE
    else:
        W = _tree_verify("sktv", 5, 32, 2, 128, 8, 47)
    W.sinks = random_sinks(W.num_q_heads, seed=12)
    full_check(W, spec_mode=spec)


def test_sinks_on_padding_rows_and_minus_inf_sinks():
    """A request without keys reports o = 0 and lse = the sink; -inf sinks
    give bit for bit the result without sinks."""
    W = make_workload("skp", "decode", 4, 8, 2, 64, [0, 37, 0, 211], np.ones(4))
    W.seq_lens = np.array([0, 38, 0, 212], dtype=W.seq_lens.dtype)
    W.sinks = random_sinks(W.num_q_heads, seed=13)
    d = full_check(W)
    assert torch.equal(d.lse[0].cpu(), torch.from_numpy(W.sinks))
    W2 = preset("llama3_8b_decode", bs=6, len_scale=0.2)
    plain = run_path(W2)
    W2.sinks = np.full(W2.num_q_heads, -np.inf, dtype=np.float32)
    neg = run_path(W2)
    assert torch.equal(plain.out, neg.out) and torch.equal(plain.lse, neg.lse)


def test_extend_mixed_split_and_unsplit_requests():
    """Requests whose rows fit one 256-row unit are split along their KV range
    (partials + merge); long query blocks are not. Both in one batch."""
    W = make_workload("mix", "extend", 5, 32, 8, 128, [6000, 0, 3000, 9000, 17],
                      [3, 700, 64, 1, 40])
    full_check(W)


def test_extend_output_buffer_only_16_byte_aligned():
    """The API asks for 16-byte aligned buffers; the extend epilogue's 32-byte
    stores are used only when the output is 32-byte aligned."""
    W = make_workload("a16", "extend", 3, 8, 2, 128, [0, 37, 200], [130, 9, 61])
    d = DeviceBatch(W)
    big = torch.empty(d.out.numel() + 8, dtype=d.out.dtype, device=d.out.device)
    d.out = big[8:].view_as(d.q)  # 16 bytes past a 256-byte aligned allocation
    assert d.out.data_ptr() % 32 == 16
    d.step()
    torch.cuda.synchronize()
    assert d.device_error() == 0
    ref_o, ref_lse = oracle_reference(W)
    check_close(d.out.double().cpu().numpy(), ref_o, "o")
    check_close(d.lse.double().cpu().numpy(), ref_lse, "lse")


@pytest.mark.parametrize("mode", ["decode", "verify"])
def test_merge_at_the_split_cap(mode):
    """One 100k-token request alone in the batch: the plan would cut its KV
    range into hundreds of splits but stops at the cap of 64 per request (the
    merge reads two splits per lane), and the merge combines all of them,
    more than one lane's worth included."""
    if mode == "decode":
        W = make_workload("m32d", "decode", 1, 8, 1, 128, [100000], [1])
        d = full_check(W)
    else:
        W = make_workload("m32v", "verify", 1, 16, 1, 128, [100000], [5])
        d = full_check(W, spec_mode=B.PKV_SPEC_PREFILL)
    # the plan words open the workspace; word 5 counts the (request, split) items
    plan = workspace_ints(d, d.attn.workspace.data_ptr(), 16)
    assert 32 < plan[5] <= 64


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_lone_long_request_spreads_over_the_grid(kv_dtype):
    """A batch of one 131k-token request with eight KV heads: 24 splits would
    give 192 units for a grid of two CTAs per SM, so the plan cuts it into
    more than 32 (up to 64) and the merge's second split per lane is used;
    sinks ride along. Every row against the oracle."""
    W = make_workload("lone", "decode", 1, 32, 8, 128, [131071], [1], kv_dtype=kv_dtype)
    W.sinks = random_sinks(W.num_q_heads, seed=15)
    d = full_check(W)
    plan = workspace_ints(d, d.attn.workspace.data_ptr(), 16)
    assert 32 < plan[5] <= 64


def test_verify_prefill_path_long_context_split():
    W = make_workload("vlong", "verify", 4, 64, 4, 128, [20000, 300, 12000, 5000], [8, 4, 6, 7])
    full_check(W, spec_mode=B.PKV_SPEC_PREFILL)


# ------------------------------------------------------------------ K and V heads of different widths
# Q/K heads 192 wide, V heads (and output rows) 128 wide: the shape that
# "--attention-backend", section "How SGLang picks a default", routes to a
# dedicated backend on SM100/SM103.
W192 = (192, 128)


def _widths_case(case):
    rng = np.random.default_rng(60)
    if case == "decode_g4":  # one 8-row key-major tile
        return preset("llama3_8b_decode", bs=12, len_scale=0.2, head_dims=W192), B.PKV_SPEC_PREFILL
    if case == "decode_g16_ragged":  # two 8-row tiles; empty, one-key and page-tail lengths
        return make_workload("w16", "decode", 7, 32, 2, 192, [0, 0, 15, 16, 1000, 3333, 77], np.ones(7),
                             head_dim_v=128), B.PKV_SPEC_PREFILL
    if case == "extend":
        return preset("prefix_extend", bs=3, len_scale=0.25, head_dims=W192), B.PKV_SPEC_PREFILL
    if case == "extend_g16_q_tma":  # Q tiles by TMA (the group divides 128), three column blocks
        return make_workload("we16", "extend", 3, 32, 2, 192, [3000, 17, 0], [300, 129, 1],
                             head_dim_v=128), B.PKV_SPEC_PREFILL
    if case == "extend_g6_q_copied":  # the softmax warps copy Q rows (group 6)
        return make_workload("we6", "extend", 3, 12, 2, 192, [500, 0, 64], [77, 200, 5],
                             head_dim_v=128), B.PKV_SPEC_PREFILL
    if case in ("verify_decode", "verify_prefill"):
        W = preset("spec_verify", bs=6, len_scale=0.1, head_dims=W192)
        return W, B.PKV_SPEC_DECODE if case == "verify_decode" else B.PKV_SPEC_PREFILL
    if case == "page_size_128":
        return preset("prefix_extend", bs=3, len_scale=0.25, page_size=128, head_dims=W192), B.PKV_SPEC_PREFILL
    if case in ("tree_sinks_decode", "tree_sinks_prefill"):
        W = make_workload("wt", "verify", 5, 32, 4, 192, rng.integers(50, 900, 5), rng.integers(2, 16, 5),
                          head_dim_v=128)
        W.tree_mask = random_tree_masks(W.qo_lens, seed=61)
        W.sinks = random_sinks(W.num_q_heads, seed=62)
        return W, B.PKV_SPEC_DECODE if case == "tree_sinks_decode" else B.PKV_SPEC_PREFILL
    raise KeyError(case)


@pytest.mark.parametrize("case", ["decode_g4", "decode_g16_ragged", "extend", "extend_g16_q_tma",
                                  "extend_g6_q_copied", "verify_decode", "verify_prefill", "page_size_128",
                                  "tree_sinks_decode", "tree_sinks_prefill"])
def test_head_widths_192_128_parity(case):
    """Every row against the oracle with 192-wide Q/K heads and 128-wide V
    heads, on both paths: scores over 192 columns, outputs of 128."""
    W, spec = _widths_case(case)
    d = full_check(W, spec_mode=spec)
    assert d.out.shape[-1] == 128


def test_head_widths_192_128_pools_bit_exact():
    """set_kv_buffer writes 192-wide K rows and 128-wide V rows, bit for bit,
    every other slot untouched."""
    W = make_workload("wp", "extend", 5, 16, 8, 192, [0, 40, 7, 100, 3], [37, 16, 1, 200, 90], head_dim_v=128)
    d = DeviceBatch(W)
    d.set_kv_buffer()
    torch.cuda.synchronize()
    assert d.device_error() == 0
    kp, vp = oracle_pools(W)
    assert np.array_equal(pool_bits(d.k_pool.cpu()), kp)
    assert np.array_equal(pool_bits(d.v_pool.cpu()), vp)


def test_head_widths_192_128_full_size_decode_every_row():
    """The Llama-3-8B-shaped decode batch at full size with 192/128 heads."""
    full_check(preset("llama3_8b_decode", head_dims=W192))


def test_fp8_workspace_holds_no_copy_of_the_pool():
    """The E4M3 extend path widens codes in shared memory: an E4M3 context
    needs exactly the workspace of the same configuration with bf16 pools,
    however many pages it may touch."""
    W = preset("long_fp8_decode", bs=2, len_scale=1 / 16)
    cfg8 = config_for(W, max_pages_total=1 << 20)
    cfg16 = config_for(W, max_pages_total=1 << 20)
    cfg16.kv_dtype = B.PKV_KV_BF16
    assert B.pkv_workspace_bytes(cfg8) == B.pkv_workspace_bytes(cfg16)
