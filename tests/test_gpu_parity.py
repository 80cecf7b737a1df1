"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Pass bars: kv_write bit-exact over the whole pool; fp32 storage max |err| <=
1e-5; bf16 storage (fp32 accumulation) max |err| <= 2e-2 and mean |err| <= 2e-3.
Inputs are the seeded synthetic workloads of paged_kv_cache_loc_gb300.workloads.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_loc_gb300 as pkv
from paged_kv_cache_loc_gb300 import _lib, build
from paged_kv_cache_loc_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_F32_MAX = 1e-5
TOL_BF16_MAX = 2e-2
TOL_BF16_MEAN = 2e-3


@pytest.fixture(scope="session", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _lib.load()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def f64(t):
    return oracle.to_f64(W.host_of(t))


def assert_close(got, ref, dtype, what=""):
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    if dtype == "f32":
        assert err.max() <= TOL_F32_MAX, f"{what}: max err {err.max():.3g}"
    else:
        assert err.max() <= TOL_BF16_MAX, f"{what}: max err {err.max():.3g}"
        assert err.mean() <= TOL_BF16_MEAN, f"{what}: mean err {err.mean():.3g}"


def no_device_error():
    st, detail = pkv.last_device_error()
    assert st == _lib.PKV_OK, f"device error word set (detail {detail})"


def prepare(case):
    """Upload the pre-write pool, write the new rows on the GPU, and apply the
    oracle's write to the host copy (which then holds the expected pool)."""
    cache, q, kn, vn = W.upload(case)
    pkv.kv_write(cache, case.layer_id, kn, vn)
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    return cache, q


def ws_for(case, splits=1024):
    return pkv.Workspace(max(case.batch, 1), case.n_heads, case.head_dim, splits)


def oracle_decode(case, **kw):
    return oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.seq_lens, case.q, case.layer_id, kv_indptr=case.kv_indptr, **kw)


def check_pool_bit_exact(cache, case):
    assert np.array_equal(W.host_of(cache.k_buffer), case.k_buffer)
    assert np.array_equal(W.host_of(cache.v_buffer), case.v_buffer)


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

def test_tiny_decode_fp32_all_split_sizes():
    case = W.tiny_decode()
    cache, q = prepare(case)
    check_pool_bit_exact(cache, case)
    ref = oracle_decode(case)
    ws = ws_for(case)
    outs = {}
    for chunk in (0, 32, 64, 96, 256):
        o = pkv.paged_decode(cache, case.layer_id, q, workspace=ws, chunk=chunk)
        no_device_error()
        outs[chunk] = f64(o)
        assert_close(outs[chunk], ref, "f32", f"chunk {chunk}")
    # split count changes only the fp32 summation order
    for chunk, o in outs.items():
        assert np.abs(o - outs[256]).max() <= 1e-6


@pytest.fixture(scope="module")
def batched():
    case = W.batched_decode()
    cache, q = prepare(case)
    return case, cache, q


def test_batched_decode_kv_write_bit_exact(batched):
    case, cache, _ = batched
    check_pool_bit_exact(cache, case)


def test_batched_decode_full(batched):
    case, cache, q = batched
    ws = ws_for(case)
    # a batch of fewer than 1024 positions per SM runs on 12/13 of the SMs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert case.max_len * case.batch < 1024 * sms
    assert pkv.decode_plan(cache, case.n_heads, ws) == (0, sms * 12 // 13)
    o = pkv.paged_decode(cache, case.layer_id, q, workspace=ws)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", "batched decode")


@pytest.mark.parametrize("chunk", [32, 512, 2048])
def test_batched_decode_split_invariance(batched, chunk):
    case, cache, q = batched
    ws = ws_for(case)
    o = pkv.paged_decode(cache, case.layer_id, q, workspace=ws, chunk=chunk)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", f"chunk {chunk}")


@pytest.mark.parametrize("ctx", W.LONG_CONTEXTS)
def test_long_context_decode(ctx):
    case = W.long_decode(ctx)
    cache, q = prepare(case)
    ws = ws_for(case)
    # the balanced plan: ~32 tokens per CTA at least, one CTA per SM at most,
    # and 4/5 of the SMs for one request with 96 to 320 positions per SM
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cap = sms * 4 // 5 if 96 * sms <= ctx < 320 * sms else sms
    assert pkv.decode_plan(cache, case.n_heads, ws) == (0, min(-(-ctx // 32), cap))
    o = pkv.paged_decode(cache, case.layer_id, q, workspace=ws)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", f"ctx {ctx}")


def test_prefix_shared_decode():
    case = W.prefix_shared_decode()
    cache, q = prepare(case)
    check_pool_bit_exact(cache, case)
    o = pkv.paged_decode(cache, case.layer_id, q, workspace=ws_for(case))
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", "prefix-shared")


def run_prefill(case, causal=True):
    cache, q = prepare(case)
    o = pkv.paged_prefill(cache, case.layer_id, q, case.max_q_len, case.max_len, causal=causal)
    no_device_error()
    return cache, q, o


@pytest.mark.parametrize("causal,d", [(True, 128), (False, 128), (True, 64), (False, 64)])
def test_ragged_prefill_reduced_full_check(causal, d):
    case = W.ragged_prefill(batch=4, q_lo=1, q_hi=256, p_hi=512, size=8192, seed=2005, head_dim=d)
    _, _, o = run_prefill(case, causal)
    ref = oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.qo_indptr, case.kv_indptr, case.q, case.layer_id, causal=causal)
    assert_close(f64(o), ref, "bf16", "reduced prefill")


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_with_a_workspace_takes_entries_longest_first(causal):
    """With a workspace a planning kernel orders the entries by decreasing
    kv_len and the prefill takes them in that order: the same bits as batch
    order, equal to the oracle, also replayed from a CUDA graph."""
    case = W.ragged_prefill(batch=12, q_lo=1, q_hi=300, p_hi=700, size=16384, seed=2011)
    cache, q = prepare(case)
    o0 = pkv.paged_prefill(cache, case.layer_id, q, case.max_q_len, case.max_len, causal=causal)
    ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1)
    o1 = pkv.paged_prefill(cache, case.layer_id, q, case.max_q_len, case.max_len, causal=causal,
                           workspace=ws)
    no_device_error()
    assert torch.equal(o0, o1)
    ref = oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.qo_indptr, case.kv_indptr, case.q, case.layer_id, causal=causal)
    assert_close(f64(o1), ref, "bf16", "prefill with a workspace")
    o2 = torch.full_like(q, float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        pkv.paged_prefill(cache, case.layer_id, q, case.max_q_len, case.max_len, causal=causal, o=o2,
                          workspace=ws, stream=side)
    g.replay()
    torch.cuda.synchronize()
    no_device_error()
    assert torch.equal(o0, o2)


@pytest.mark.parametrize("with_ws", [False, True])
def test_prefill_entry_with_a_bad_request_row_leaves_the_others_exact(with_ws):
    """One entry's request row lies outside req_to_token: it is recorded, its
    rows of o are not written, and every other entry still matches the
    oracle, in batch order and in the planned order."""
    case = W.ragged_prefill(batch=6, q_lo=1, q_hi=200, p_hi=400, size=8192, seed=2013)
    cache, q = prepare(case)
    ref = oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.qo_indptr, case.kv_indptr, case.q, case.layer_id)
    rpi = case.req_pool_indices.copy()
    rpi[2] = case.num_reqs + 5
    cache.req_pool_indices = torch.from_numpy(rpi).cuda()
    o = torch.full_like(q, 7.0)
    ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1) if with_ws else None
    pkv.paged_prefill(cache, case.layer_id, q, case.max_q_len, case.max_len, o=o, workspace=ws)
    st, detail = pkv.last_device_error()
    assert st == _lib.PKV_ERR_INDEX and detail == case.num_reqs + 5
    got = f64(o)
    lo, hi = int(case.qo_indptr[2]), int(case.qo_indptr[3])
    assert np.all(got[lo:hi] == 7.0), "the bad entry's rows were written"
    keep = np.r_[0:lo, hi:got.shape[0]]
    assert_close(got[keep], ref[keep], "bf16", "the other entries")


@pytest.mark.parametrize("batch", [2, 256, 257, 300])
def test_prefill_with_a_workspace_at_the_planned_batch_limits(batch):
    """2 and 256 entries are ordered by the planning kernel, 257 and more run
    in batch order: all equal to the oracle, and the same bits as without a
    workspace."""
    rng = np.random.Generator(np.random.PCG64(12 + batch))
    q_lens = rng.integers(0, 4, batch)
    kv = q_lens + rng.integers(0, 40, batch)
    case = W.make_case("plan_big", mode="prefill", dtype="bf16", n_layers=1, layer_id=0, size=16384,
                       n_heads=8, n_kv_heads=2, head_dim=128, kv_lens=kv, q_lens=q_lens, seed=13)
    cache, q = prepare(case)
    ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1)
    o = pkv.paged_prefill(cache, 0, q, case.max_q_len, case.max_len, workspace=ws)
    no_device_error()
    ref = oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.qo_indptr, case.kv_indptr, case.q, 0)
    assert_close(f64(o), ref, "bf16", f"{batch} entries")
    assert torch.equal(o, pkv.paged_prefill(cache, 0, q, case.max_q_len, case.max_len))


def test_ragged_prefill_full_size_sampled():
    case = W.ragged_prefill()
    cache, q, o = run_prefill(case)
    check_pool_bit_exact(cache, case)
    rows = W.prefill_sample_rows(case, n_random=64)
    ref = oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.qo_indptr, case.kv_indptr, case.q, case.layer_id, rows=rows)
    assert_close(f64(o)[rows], ref, "bf16", "full prefill (sampled rows)")


# ---------------------------------------------------------------------------
# edge cases and variants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,heads,hk,d", [
    ("bf16", 8, 8, 128), ("bf16", 16, 8, 128), ("bf16", 32, 4, 128), ("bf16", 16, 4, 64),
    ("bf16", 64, 8, 64),
    ("f32", 32, 8, 128), ("f32", 8, 1, 64), ("f32", 4, 2, 64),
])
def test_decode_variants_and_ragged_lengths(dtype, heads, hk, d):
    kv = [0, 1, 31, 32, 33, 95, 300, 1000]
    case = W.make_case("edge", mode="decode", dtype=dtype, n_layers=3, layer_id=2, size=4096,
                       n_heads=heads, n_kv_heads=hk, head_dim=d, kv_lens=kv,
                       q_lens=[0 if n == 0 else 1 for n in kv], seed=77, num_reqs=11,
                       max_ctx_len=1000)
    # the empty context writes no token, but decode still has a query row for it
    extra = W._values(np.random.Generator(np.random.PCG64(5)), (1, heads, d), dtype)
    case.q = np.concatenate([extra, case.q])
    cache, qd = prepare(case)
    ref = oracle_decode(case)
    for chunk in (0, 32, 128, 1024):
        o = pkv.paged_decode(cache, case.layer_id, qd, workspace=ws_for(case), chunk=chunk)
        no_device_error()
        got = f64(o)
        assert np.all(got[0] == 0.0), "empty context must give 0"
        assert_close(got, ref, dtype, f"chunk {chunk}")


@pytest.mark.parametrize("heads,hk,d", [(8, 8, 128), (16, 8, 128), (64, 8, 128), (8, 8, 64), (16, 8, 64),
                                         (32, 8, 64), (64, 8, 64)])
def test_prefill_variants(heads, hk, d):
    q_lens = [0, 1, 5, 64, 65, 130]
    pre = [7, 0, 100, 0, 63, 1]
    kv = [a + b for a, b in zip(q_lens, pre)]
    case = W.make_case("pre_edge", mode="prefill", dtype="bf16", n_layers=2, layer_id=1,
                       size=4096, n_heads=heads, n_kv_heads=hk, head_dim=d, kv_lens=kv,
                       q_lens=q_lens, seed=88)
    _, _, o = run_prefill(case)
    ref = oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.qo_indptr, case.kv_indptr, case.q, case.layer_id)
    assert_close(f64(o), ref, "bf16", "prefill variants")


@pytest.mark.parametrize("dtype,heads,hk,d", [("bf16", 32, 16, 128), ("bf16", 32, 32, 64), ("bf16", 6, 3, 128),
                                               ("f32", 32, 32, 64), ("f32", 48, 12, 128)])
def test_decode_with_more_or_odd_kv_heads(dtype, heads, hk, d):
    """kv head counts outside {1, 2, 4, 8} (3, 12, 16, 32): the decode step,
    then the chunked plans, which also serve these counts when kv_indptr is
    given."""
    kv = [1, 33, 500, 2049, 130]
    case = W.make_case("kvh", mode="decode", dtype=dtype, n_layers=2, layer_id=1, size=8192,
                       n_heads=heads, n_kv_heads=hk, head_dim=d, kv_lens=kv, seed=515)
    cache, q, kn, vn = W.upload(case)
    ws = ws_for(case, splits=64)
    o = pkv.decode_step(cache, case.layer_id, kn, vn, q, workspace=ws)
    no_device_error()
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    check_pool_bit_exact(cache, case)
    ref = oracle_decode(case)
    assert_close(f64(o), ref, dtype, "decode step")
    for chunk in (0, 64, 2048):
        o = pkv.paged_decode(cache, case.layer_id, q, workspace=ws, chunk=chunk)
        no_device_error()
        assert_close(f64(o), ref, dtype, f"chunk {chunk}")


@pytest.mark.parametrize("heads,hk,d", [(32, 16, 128), (32, 32, 64), (6, 3, 128), (48, 12, 64)])
def test_prefill_with_more_or_odd_kv_heads(heads, hk, d):
    q_lens = [1, 65, 130, 300]
    pre = [0, 7, 100, 513]
    case = W.make_case("kvh_pre", mode="prefill", dtype="bf16", n_layers=2, layer_id=1, size=8192,
                       n_heads=heads, n_kv_heads=hk, head_dim=d,
                       kv_lens=[a + b for a, b in zip(q_lens, pre)], q_lens=q_lens, seed=516)
    _, _, o = run_prefill(case)
    ref = oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.qo_indptr, case.kv_indptr, case.q, case.layer_id)
    assert_close(f64(o), ref, "bf16", f"prefill hk={hk}")


def test_causal_prefill_row_matches_decode_kernel():
    """Prefill row i (prefix P) and decode at context P+i+1 agree on the GPU."""
    case = W.make_case("cross", mode="prefill", dtype="bf16", n_layers=2, layer_id=0, size=2048,
                       n_heads=32, n_kv_heads=8, head_dim=128, kv_lens=[300], q_lens=[100],
                       seed=99)
    cache, q, o = run_prefill(case)
    P = 200
    rows = [0, 37, 99]
    for i in rows:
        dc = pkv.KVCache(k_buffer=cache.k_buffer, v_buffer=cache.v_buffer,
                         req_to_token=cache.req_to_token, req_pool_indices=cache.req_pool_indices,
                         seq_lens=torch.tensor([P + i + 1], dtype=torch.int32, device="cuda"),
                         max_len=P + i + 1)
        od = pkv.paged_decode(dc, 0, q[i:i + 1].contiguous(), workspace=ws_for(case), chunk=64)
        assert_close(f64(od)[0], f64(o)[i], "bf16", f"row {i}")


@pytest.mark.parametrize("dtype,hq,hk,d", [("bf16", 8, 4, 128), ("bf16", 2, 1, 128), ("bf16", 6, 3, 64),
                                            ("f32", 6, 3, 64), ("f32", 10, 5, 128)])
def test_rope_kv_write(dtype, hq, hk, d):
    """The fused write takes kv heads two per pass: odd and single head
    counts leave a partial pass."""
    case = W.make_case("rope", mode="prefill", dtype=dtype, n_layers=2, layer_id=1, size=1024,
                       n_heads=hq, n_kv_heads=hk, head_dim=d, kv_lens=[40, 90], q_lens=[40, 60],
                       seed=123)
    rng = np.random.Generator(np.random.PCG64(5))
    max_pos = 256
    ang = rng.uniform(-math.pi, math.pi, (max_pos, d // 2)).astype(np.float32)
    fc = np.stack([np.cos(ang), np.sin(ang)], -1).astype(np.float32)
    pos = rng.integers(0, max_pos, case.out_cache_loc.size).astype(np.int32)
    cache, q, kn, vn = W.upload(case)
    pkv.rope_kv_write(cache, 1, kn, vn, torch.from_numpy(fc).cuda(), torch.from_numpy(pos).cuda())
    no_device_error()
    k_rot = oracle.rope(case.k_new, fc, pos)
    got_k = f64(cache.k_buffer)[1, case.out_cache_loc]
    if dtype == "bf16":
        # one bf16 rounding of an fp32 rotation: |err| <= 2^-8 |x| + tiny
        assert np.all(np.abs(got_k - k_rot) <= np.abs(k_rot) * 2.0 ** -8 + 1e-6)
    else:
        # an fp32 rotation: a few fp32 roundings of terms bounded by the
        # pair's norm, which the rotation preserves
        x = np.asarray(case.k_new, np.float64).reshape(*case.k_new.shape[:-1], d // 2, 2)
        norm = np.repeat(np.sqrt((x ** 2).sum(-1)), 2, axis=-1)
        assert np.all(np.abs(got_k - k_rot) <= norm * 2.0 ** -20 + 1e-30)
    assert np.array_equal(W.host_of(cache.v_buffer)[1, case.out_cache_loc], case.v_new)


def test_kv_write_duplicate_free_scatter_leaves_other_rows():
    case = W.make_case("kvw", mode="prefill", dtype="f32", n_layers=3, layer_id=0, size=3000,
                       n_heads=4, n_kv_heads=2, head_dim=64, kv_lens=[700, 5, 1200],
                       q_lens=[700, 5, 600], seed=9)
    cache, _ = prepare(case)
    no_device_error()
    check_pool_bit_exact(cache, case)


@pytest.mark.parametrize("hk,indptr", [(2, False), (2, True), (8, True)])
def test_device_data_errors_are_reported_not_faulted(hk, indptr):
    """Bad device data is recorded in the error word, never faulted, on the
    chunked plan and on the balanced plan (with 8 kv heads, its staged-slot
    pass)."""
    case = W.make_case("bad", mode="decode", dtype="bf16", n_layers=2, layer_id=1, size=512,
                       n_heads=8, n_kv_heads=hk, head_dim=128, kv_lens=[20, 40], seed=3)
    cache, q = prepare(case)
    no_device_error()
    ws = ws_for(case)
    kvi = cache.kv_indptr if indptr else None
    # a slot outside the pool in req_to_token
    r2t = case.req_to_token.copy()
    r2t[case.req_pool_indices[1], 7] = case.size + 5
    bad = pkv.KVCache(k_buffer=cache.k_buffer, v_buffer=cache.v_buffer,
                      req_to_token=torch.from_numpy(r2t).cuda(),
                      req_pool_indices=cache.req_pool_indices, seq_lens=cache.seq_lens,
                      kv_indptr=kvi, max_len=case.max_len)
    assert (pkv.decode_plan(bad, case.n_heads, ws)[0] == 0) == indptr
    pkv.paged_decode(bad, 1, q, workspace=ws)
    st, detail = pkv.last_device_error()
    assert st == _lib.PKV_ERR_INDEX and detail == case.size + 5
    # a request row outside req_to_token
    bad.req_to_token = cache.req_to_token
    bad.req_pool_indices = torch.tensor([0, 9], dtype=torch.int32, device="cuda")
    pkv.paged_decode(bad, 1, q, workspace=ws)
    assert pkv.last_device_error()[0] == _lib.PKV_ERR_INDEX
    if indptr:
        # kv_indptr that disagrees with seq_lens
        bad.req_pool_indices = cache.req_pool_indices
        bad.seq_lens = torch.tensor([20, 41], dtype=torch.int32, device="cuda")
        pkv.paged_decode(bad, 1, q, workspace=ws)
        assert pkv.last_device_error()[0] == _lib.PKV_ERR_INDEX
    # a write location outside the pool
    wr = pkv.KVCache(k_buffer=cache.k_buffer, v_buffer=cache.v_buffer,
                     req_to_token=cache.req_to_token, req_pool_indices=cache.req_pool_indices,
                     out_cache_loc=torch.tensor([3, -1], dtype=torch.int32, device="cuda"))
    k2 = torch.zeros(2, hk, 128, dtype=torch.bfloat16, device="cuda")
    pkv.kv_write(wr, 1, k2, k2)
    assert pkv.last_device_error() == (_lib.PKV_ERR_INDEX, -1)
    # the context is still healthy and the word was cleared
    o = pkv.paged_decode(cache, 1, q, workspace=ws)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", "after errors")


@pytest.mark.parametrize("d,with_ws", [(128, False), (64, False), (128, True)])
def test_prefill_rows_outside_q_are_reported_not_touched(d, with_ws):
    """A qo_indptr entry whose packed rows fall outside [0, qo_indptr[batch])
    is recorded and its rows are neither read nor written.  q and o are
    views into buffers padded by 64 rows on each side, so that even an
    unchecked access would stay inside the allocation."""
    case = W.make_case("bad_qo", mode="prefill", dtype="bf16", n_layers=2, layer_id=1, size=1024,
                       n_heads=8, n_kv_heads=4, head_dim=d, kv_lens=[30, 50], q_lens=[20, 40],
                       seed=21)
    cache, q = prepare(case)
    pad = 64
    qp = torch.zeros(pad + q.shape[0] + pad, *q.shape[1:], dtype=q.dtype, device="cuda")
    qp[pad:pad + q.shape[0]] = q
    op = torch.full_like(qp, 7.0)
    for qo in ([-20, 0, 40], [0, 30, 20]):
        # entry 0 starts before row 0, or entry 1 ends past qo_indptr[batch]
        bad = pkv.KVCache(k_buffer=cache.k_buffer, v_buffer=cache.v_buffer,
                          req_to_token=cache.req_to_token, req_pool_indices=cache.req_pool_indices,
                          kv_indptr=cache.kv_indptr, max_len=case.max_len,
                          qo_indptr=torch.tensor(qo, dtype=torch.int32, device="cuda"))
        ws = pkv.Workspace(case.batch, case.n_heads, d, 1) if with_ws else None
        pkv.paged_prefill(bad, case.layer_id, qp[pad:pad + q.shape[0]], 40, case.max_len,
                          o=op[pad:pad + q.shape[0]], workspace=ws)
        assert pkv.last_device_error()[0] == _lib.PKV_ERR_INDEX
        assert torch.all(op[:pad] == 7.0) and torch.all(op[-pad:] == 7.0), "padding was written"
    # the context is still healthy and the word was cleared
    _, _, o = run_prefill(case)
    ref = oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.qo_indptr, case.kv_indptr, case.q, case.layer_id)
    assert_close(f64(o), ref, "bf16", "prefill after errors")


def _short_lens(kind):
    rng = np.random.Generator(np.random.PCG64(len(kind)))
    if kind == "uniform_0_12":        # 300 entries, a few pieces per CTA, empty ones among them
        return rng.integers(0, 13, 300)
    if kind == "clustered_ones":      # 500 x 40 tokens, then 500 x 1: ~135 pieces per CTA there
        return np.array([40] * 500 + [1] * 500)
    return rng.integers(0, 4, 1100)   # more than 1024 entries


@pytest.mark.parametrize("kind", ["uniform_0_12", "clustered_ones", "over_1024"])
def test_balanced_decode_many_short_entries(kind):
    """Balanced plan over many short entries.  A CTA with at most 64 pieces
    (in a batch of at most 1024 entries) stages all its slots and streams
    across piece boundaries; the CTAs over the 1-token run of
    "clustered_ones" hold ~135 pieces and every CTA of "over_1024" sees more
    than 1024 entries, so those take the piece-by-piece pass.  Empty entries
    give 0."""
    kv = _short_lens(kind)
    n_entries = kv.size
    rng = np.random.Generator(np.random.PCG64(n_entries))
    case = W.make_case("short", mode="decode", dtype="bf16", n_layers=1, layer_id=0, size=32768,
                       n_heads=16, n_kv_heads=8, head_dim=128, kv_lens=kv,
                       q_lens=(kv > 0).astype(np.int64), seed=n_entries)
    case.q = W._values(rng, (n_entries, 16, 128), "bf16")
    cache, qd = prepare(case)
    ws = ws_for(case, splits=2)
    assert pkv.decode_plan(cache, case.n_heads, ws)[0] == 0      # balanced
    o = pkv.paged_decode(cache, case.layer_id, qd, workspace=ws)
    no_device_error()
    got = f64(o)
    assert np.all(got[kv == 0] == 0.0), "empty context must give 0"
    assert_close(got, oracle_decode(case), "bf16", kind)


def test_balanced_decode_long_ranges():
    """More than 2048 tokens per CTA (T > SMs * 2048): the slot indices of a
    CTA no longer fit at once, so its pieces stream one by one."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_entries = 40
    ctx = -(-sms * (2048 + 64) // n_entries)
    case = W.make_case("longr", mode="decode", dtype="bf16", n_layers=1, layer_id=0,
                       size=ctx * n_entries, n_heads=8, n_kv_heads=8, head_dim=64,
                       kv_lens=[ctx] * n_entries, seed=9)
    cache, q = prepare(case)
    ws = ws_for(case, splits=8)
    assert pkv.decode_plan(cache, case.n_heads, ws) == (0, sms)
    o = pkv.paged_decode(cache, case.layer_id, q, workspace=ws)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", "long ranges")


def test_single_context_of_half_a_million_positions():
    """B=1 at 524,295 positions (1 GB of bf16 K/V rows): the balanced plan
    gives every CTA more than 2048 positions, and the chunked plan (no
    kv_indptr) cuts the context into host-chosen chunks."""
    ctx = 524295
    case = W.make_case("b1_max", mode="decode", dtype="bf16", n_layers=1, layer_id=0, size=ctx,
                       n_heads=32, n_kv_heads=8, head_dim=128, kv_lens=[ctx], seed=77, max_ctx_len=ctx)
    cache, q = prepare(case)
    ref = oracle_decode(case)
    ws = ws_for(case, splits=1024)
    o = pkv.paged_decode(cache, case.layer_id, q, workspace=ws)
    no_device_error()
    assert_close(f64(o), ref, "bf16", "balanced")
    cache.kv_indptr = None
    o = pkv.paged_decode(cache, case.layer_id, q, workspace=ws)
    no_device_error()
    assert_close(f64(o), ref, "bf16", "chunked")


def test_workspace_too_small_is_rejected():
    case = W.make_case("ws", mode="decode", dtype="bf16", n_layers=1, layer_id=0, size=4096,
                       n_heads=8, n_kv_heads=2, head_dim=128, kv_lens=[3000], seed=4)
    cache, q = prepare(case)
    small = pkv.Workspace(1, 8, 128, 2)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode(cache, 0, q, workspace=small, chunk=32)
    assert e.value.status == _lib.PKV_ERR_WORKSPACE
    # the automatic plan respects the workspace: 2 splits of 1504 tokens
    assert pkv.decode_plan(cache, 8, small) == (1504, 2)
    o = pkv.paged_decode(cache, 0, q, workspace=small)
    assert_close(f64(o), oracle_decode(case), "bf16", "2-split plan")


def test_write_then_chunked_decode_replays_in_a_cuda_graph():
    """kv_write + decode (fixed 64-token splits) captured once, replayed with
    metadata updated in place."""
    case = W.batched_decode(batch=8, lo=100, hi=700, size=16384, seed=515)
    cache, q, kn, vn = W.upload(case)
    ws = ws_for(case, splits=64)
    o = torch.empty_like(q)
    chunk = 64
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkv.kv_write(cache, case.layer_id, kn, vn, stream=s)
        pkv.paged_decode(cache, case.layer_id, q, o, workspace=ws, chunk=chunk, stream=s)
    s.synchronize()
    eager = o.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.kv_write(cache, case.layer_id, kn, vn, stream=s)
        pkv.paged_decode(cache, case.layer_id, q, o, workspace=ws, chunk=chunk, stream=s)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, eager)
    # shorten every context in place and replay: matches the oracle on the new lengths
    new_lens = np.maximum(case.seq_lens - 50, 1).astype(np.int32)
    cache.seq_lens.copy_(torch.from_numpy(new_lens))
    g.replay()
    torch.cuda.synchronize()
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    ref = oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                        new_lens, case.q, case.layer_id)
    assert_close(f64(o), ref, "bf16", "graph replay with new lengths")
    no_device_error()


def test_balanced_decode_replays_in_a_cuda_graph():
    """The automatic (balanced over kv_indptr) plan, captured once and replayed
    after seq_lens and kv_indptr are updated in place."""
    case = W.batched_decode(batch=12, lo=50, hi=2500, size=32768, seed=616)
    cache, q, kn, vn = W.upload(case)
    ws = ws_for(case, splits=64)
    assert pkv.decode_plan(cache, case.n_heads, ws)[0] == 0      # balanced
    o = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkv.kv_write(cache, case.layer_id, kn, vn, stream=s)
        pkv.paged_decode(cache, case.layer_id, q, o, workspace=ws, stream=s)
    s.synchronize()
    eager = o.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.kv_write(cache, case.layer_id, kn, vn, stream=s)
        pkv.paged_decode(cache, case.layer_id, q, o, workspace=ws, stream=s)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, eager)
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    rng = np.random.Generator(np.random.PCG64(7))
    new_lens = np.maximum(case.seq_lens - rng.integers(0, 400, case.batch), 0).astype(np.int32)
    new_lens[3] = 0
    new_indptr = np.concatenate([[0], np.cumsum(new_lens)]).astype(np.int32)
    cache.seq_lens.copy_(torch.from_numpy(new_lens))
    cache.kv_indptr.copy_(torch.from_numpy(new_indptr))
    g.replay()
    torch.cuda.synchronize()
    no_device_error()
    ref = oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                        new_lens, case.q, case.layer_id, kv_indptr=new_indptr)
    assert_close(f64(o), ref, "bf16", "balanced graph replay")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_step_equals_write_then_decode(dtype):
    """pkv_decode_step (the write, then the decode launched as its
    programmatic dependent) leaves the pool the oracle's write gives and
    returns o equal to kv_write followed by paged_decode.  Every context ends
    with the token just written, so a decode that read K/V rows before the
    write finished would miss it."""
    if dtype == "bf16":
        case = W.batched_decode(batch=16, lo=200, hi=3000, size=65536, seed=717)
    else:
        case = W.tiny_decode()
    cache, q, kn, vn = W.upload(case)
    ws = ws_for(case, splits=64)
    o = pkv.decode_step(cache, case.layer_id, kn, vn, q, workspace=ws)
    no_device_error()
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    check_pool_bit_exact(cache, case)
    assert_close(f64(o), oracle_decode(case), dtype, "decode step")
    o2 = pkv.paged_decode(cache, case.layer_id, q, workspace=ws)
    assert torch.equal(o, o2)


def test_decode_step_new_rows_read_mid_context():
    """A step whose new rows include slots other entries read in the middle of
    their contexts (besides each entry's last position): the decode sees the
    new rows there too, bit-identical to kv_write followed by paged_decode,
    and the pool ends the same."""
    import dataclasses
    case = W.batched_decode(batch=16, lo=200, hi=3000, size=65536, seed=733)
    cache, q, kn, vn = W.upload(case)
    extra = []
    for b, frac in ((3, 0.5), (7, 0.25), (7, 0.75), (12, 0.1), (15, 0.0)):
        r, n = int(case.req_pool_indices[b]), int(case.seq_lens[b])
        extra.append(int(case.req_to_token[r, int((n - 1) * frac)]))
    rng = np.random.Generator(np.random.PCG64(12))
    shape = (len(extra),) + tuple(kn.shape[1:])
    bits = lambda: torch.from_numpy(W._values(rng, shape, "bf16").view(np.int16)).view(torch.bfloat16).cuda()
    kn2, vn2 = torch.cat([kn, bits()]), torch.cat([vn, bits()])
    loc = torch.cat([cache.out_cache_loc, torch.tensor(extra, dtype=torch.int32, device="cuda")])
    step = dataclasses.replace(cache, out_cache_loc=loc)
    ref = dataclasses.replace(cache, out_cache_loc=loc, k_buffer=cache.k_buffer.clone(),
                              v_buffer=cache.v_buffer.clone())
    o = pkv.decode_step(step, case.layer_id, kn2, vn2, q, workspace=ws_for(case, splits=64))
    pkv.kv_write(ref, case.layer_id, kn2, vn2)
    o_ref = pkv.paged_decode(ref, case.layer_id, q, workspace=ws_for(case, splits=64))
    torch.cuda.synchronize()
    no_device_error()
    assert torch.equal(o, o_ref)
    assert torch.equal(step.k_buffer, ref.k_buffer) and torch.equal(step.v_buffer, ref.v_buffer)


def test_decode_step_replays_in_a_cuda_graph():
    """The step captured once (its programmatic edge becomes a graph edge),
    replayed after new K/V rows are put in the step's input buffers: the
    decode sees the rows written in the same replay."""
    case = W.batched_decode(batch=12, lo=50, hi=2500, size=32768, seed=818)
    cache, q, kn, vn = W.upload(case)
    ws = ws_for(case, splits=64)
    o = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.decode_step(cache, case.layer_id, kn, vn, q, o, workspace=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    no_device_error()
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    assert_close(f64(o), oracle_decode(case), "bf16", "step graph replay")
    rng = np.random.Generator(np.random.PCG64(19))
    for name in ("k_new", "v_new"):
        bits = W._values(rng, getattr(case, name).shape, "bf16")
        setattr(case, name, bits)
        (kn if name == "k_new" else vn).copy_(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    no_device_error()
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    check_pool_bit_exact(cache, case)
    assert_close(f64(o), oracle_decode(case), "bf16", "step graph replay, new rows")


def page_table(case):
    """req_to_page of a case whose slots come in pages of page_size
    consecutive slots (checked against req_to_token)."""
    ps = case.page_size
    r2t = case.req_to_token
    n_cols = -(-r2t.shape[1] // ps)
    table = np.zeros((r2t.shape[0], n_cols), np.int32)
    table[:, :] = r2t[:, ::ps] // ps
    for b in range(case.batch):
        r, n = int(case.req_pool_indices[b]), int(case.seq_lens[b])
        j = np.arange(n)
        assert np.array_equal(r2t[r, :n], table[r, j // ps] * ps + j % ps)
    return table


def test_prefix_shared_decode_through_the_page_table():
    """The prefix-shared workload (page_size 16) through req_to_page: equal to
    the oracle, and bit-identical to the decode through req_to_token."""
    case = W.prefix_shared_decode()
    cache, q = prepare(case)
    ws = ws_for(case)
    table = torch.from_numpy(page_table(case)).cuda()
    o = pkv.paged_decode_pages(cache, case.layer_id, table, case.page_size, q, workspace=ws)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", "page table")
    assert torch.equal(o, pkv.paged_decode(cache, case.layer_id, q, workspace=ws))


@pytest.mark.parametrize("heads,hk,d,ps,indptr", [(16, 4, 128, 8, False), (8, 8, 64, 4, True),
                                                 (32, 8, 128, 32, False)])
def test_page_table_variants(heads, hk, d, ps, indptr):
    """Page sizes 4..32, kv heads 4 or 8, head_dim 64 or 128, the balanced and
    the chunked plans; ragged lengths that end inside a page."""
    kv = [1, 15, 16, 17, 130, 700, 1023]
    case = W.make_case("pages", mode="decode", dtype="bf16", n_layers=2, layer_id=1, size=8192,
                       n_heads=heads, n_kv_heads=hk, head_dim=d, kv_lens=kv, page_size=ps, seed=31)
    cache, q = prepare(case)
    if not indptr:
        cache.kv_indptr = None
    ws = ws_for(case, splits=64)
    table = torch.from_numpy(page_table(case)).cuda()
    o = pkv.paged_decode_pages(cache, case.layer_id, table, ps, q, workspace=ws)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", f"pages ps={ps}")


def test_page_index_outside_the_pool_is_reported():
    case = W.make_case("pbad", mode="decode", dtype="bf16", n_layers=1, layer_id=0, size=1024,
                       n_heads=8, n_kv_heads=8, head_dim=128, kv_lens=[40, 70], page_size=16, seed=5)
    cache, q = prepare(case)
    table = page_table(case)
    table[case.req_pool_indices[1], 2] = 1024 // 16 + 3
    pkv.paged_decode_pages(cache, 0, torch.from_numpy(table).cuda(), 16, q, workspace=ws_for(case))
    st, detail = pkv.last_device_error()
    assert st == _lib.PKV_ERR_INDEX and detail == 1024 // 16 + 3


def test_decode_on_slot_maps_from_the_page_pool():
    """req_to_token rows produced by the host allocator after churn (shared
    prefixes reused from the prefix cache, freed and evicted pages, decode
    growth) drive the decode; the oracle reads the same rows."""
    from paged_kv_cache_loc_gb300.pool import PagePool
    ps, n_pages, H, Hk, d = 16, 256, 16, 4, 128
    rng = np.random.Generator(np.random.PCG64(321))
    pool = PagePool(n_pages, ps)
    prefix = rng.integers(0, 1000, 64).tolist()
    live = {}
    for t in range(40):
        prompt = prefix + rng.integers(0, 1000, int(rng.integers(1, 90))).tolist()
        if pool.task_alloc(t, prompt)[0] != 0:
            continue
        pool.task_record_hashes(t, prompt)
        live[t] = len(prompt)
        if rng.random() < 0.5 and len(live) > 3:      # some tasks finish
            done = list(live)[int(rng.integers(0, len(live)))]
            pool.task_free(done)
            del live[done]
    for t in live:                                      # one decode step each
        assert pool.task_extend(t, live[t]) == 0
        live[t] += 1
    tids = sorted(live)
    B = len(tids)
    seq = np.array([live[t] for t in tids], np.int32)
    max_ctx = int(seq.max())
    r2t = np.zeros((B, max_ctx), np.int32)
    for b, t in enumerate(tids):
        r2t[b, :seq[b]] = pool.task_slots(t, int(seq[b]))
    size = n_pages * ps
    kb = W.to_bf16_bits(rng.standard_normal((2, size, Hk, d), dtype=np.float32))
    vb = W.to_bf16_bits(rng.standard_normal((2, size, Hk, d), dtype=np.float32))
    q = W.to_bf16_bits(rng.standard_normal((B, H, d), dtype=np.float32))
    rpi = np.arange(B, dtype=np.int32)
    kvi = np.concatenate([[0], np.cumsum(seq)]).astype(np.int32)
    dev = lambda a: (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
                     else torch.from_numpy(a)).cuda()
    cache = pkv.KVCache(k_buffer=dev(kb), v_buffer=dev(vb), req_to_token=dev(r2t),
                        req_pool_indices=dev(rpi), seq_lens=dev(seq), kv_indptr=dev(kvi),
                        max_len=max_ctx)
    o = pkv.paged_decode(cache, 1, dev(q), workspace=pkv.Workspace(B, H, d, 64))
    no_device_error()
    ref = oracle.decode(kb, vb, r2t, rpi, seq, q, 1, kv_indptr=kvi)
    assert_close(f64(o), ref, "bf16", "pool slot maps")


def shared_case(batch, heads, ps, shared, priv_hi, seed, d=128, hk=8):
    """A decode case whose rows share their first `shared` positions (whole
    pages), each with 1 + U[0, priv_hi] private positions."""
    rng = np.random.Generator(np.random.PCG64(seed))
    kv = shared + rng.integers(0, priv_hi, size=batch, endpoint=True) + 1
    pages = shared // ps + int(np.sum(-(-(kv - shared) // ps))) + 8
    size = -(-pages * ps // 1024) * 1024
    return W.make_case("shared", mode="decode", dtype="bf16", n_layers=2, layer_id=1, size=size,
                       n_heads=heads, n_kv_heads=hk, head_dim=d, kv_lens=kv, page_size=ps,
                       shared_prefix=shared, seed=seed, rng=rng)


def test_prefix_shared_decode_reads_the_shared_pages_once():
    """The prefix-shared workload with its 128 shared pages stated (read once
    per launch, on the tensor cores): equal to the oracle, and (another
    summation order) not bit-identical to the decode that reads every
    request's prefix."""
    case = W.prefix_shared_decode()
    cache, q = prepare(case)
    ws = ws_for(case)
    table = torch.from_numpy(page_table(case)).cuda()
    o = pkv.paged_decode_pages(cache, case.layer_id, table, case.page_size, q, workspace=ws,
                               shared_pages=case.shared_prefix // case.page_size)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", "shared pages")
    plain = pkv.paged_decode_pages(cache, case.layer_id, table, case.page_size, q, workspace=ws)
    assert not torch.equal(o, plain)


@pytest.mark.parametrize("batch,heads,ps,shared,priv_hi,d", [
    (37, 8, 16, 512, 300, 128),      # G = 1: groups of 16 requests, the last one partial
    (9, 16, 4, 256, 64, 128),        # G = 2: groups of 8, page_size 4
    (5, 64, 32, 1024, 2000, 128),    # G = 8: pairs, long private tails
    (3, 32, 1, 64, 10, 128),         # single-slot pages, the shortest shared prefix used
    (40, 32, 16, 4096, 50, 128),     # long prefix: four chunks of 1024 positions
    (70, 32, 16, 1008, 100, 128),    # 280 query rows: two row blocks; a partial last key tile
    (24, 16, 4, 1500, 80, 128),      # two chunks, the last one ragged
    (20, 32, 16, 1024, 200, 64),     # head_dim 64: the group role inside the split kernel
])
def test_shared_prefix_variants(batch, heads, ps, shared, priv_hi, d):
    case = shared_case(batch, heads, ps, shared, priv_hi, seed=batch * 7 + ps, d=d)
    cache, q = prepare(case)
    ws = ws_for(case)
    table = torch.from_numpy(page_table(case)).cuda()
    o = pkv.paged_decode_pages(cache, case.layer_id, table, ps, q, workspace=ws,
                               shared_pages=shared // ps)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", f"shared {shared} ps={ps} G={heads // 8}")
    plain = pkv.paged_decode_pages(cache, case.layer_id, table, ps, q, workspace=ws)
    assert not torch.equal(o, plain)   # the shared-prefix mode ran


def test_shared_prefix_with_empty_private_parts_replays_in_a_cuda_graph():
    """Entries whose context is exactly the shared prefix (no private
    positions), captured once and replayed after the lengths change."""
    case = shared_case(12, 32, 16, 768, 400, seed=41)
    cache, q = prepare(case)
    ws = ws_for(case)
    table = torch.from_numpy(page_table(case)).cuda()
    lens = case.seq_lens.copy()
    lens[[0, 5, 11]] = 768
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cache.seq_lens.copy_(torch.from_numpy(lens))
    cache.kv_indptr.copy_(torch.from_numpy(indptr))
    o = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    call = lambda: pkv.paged_decode_pages(cache, case.layer_id, table, 16, q, o, workspace=ws,
                                          stream=s, shared_pages=48)
    with torch.cuda.stream(s):
        call()
    s.synchronize()
    no_device_error()
    ref = oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                        lens, case.q, case.layer_id, kv_indptr=indptr)
    assert_close(f64(o), ref, "bf16", "empty private parts")
    eager = o.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, eager)
    lens2 = case.seq_lens.copy()
    lens2[[2, 3]] = 768
    lens2[7] -= 1
    indptr2 = np.concatenate([[0], np.cumsum(lens2)]).astype(np.int32)
    cache.seq_lens.copy_(torch.from_numpy(lens2))
    cache.kv_indptr.copy_(torch.from_numpy(indptr2))
    g.replay()
    torch.cuda.synchronize()
    no_device_error()
    ref2 = oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         lens2, case.q, case.layer_id, kv_indptr=indptr2)
    assert_close(f64(o), ref2, "bf16", "shared graph replay, new lengths")


def test_false_shared_prefix_claims_are_reported_not_faulted():
    """A row whose leading pages differ from its group's, or a context
    shorter than the stated prefix: the device error word is set and the
    call completes."""
    case = shared_case(10, 32, 16, 512, 100, seed=77)
    cache, q = prepare(case)
    ws = ws_for(case)
    table = page_table(case)
    bad = table.copy()
    r = int(case.req_pool_indices[6])
    bad[r, 3] = (bad[r, 3] + 1) % (case.k_buffer.shape[1] // 16)
    pkv.paged_decode_pages(cache, case.layer_id, torch.from_numpy(bad).cuda(), 16, q, workspace=ws,
                           shared_pages=32)
    st, detail = pkv.last_device_error()
    assert st == _lib.PKV_ERR_INDEX and detail == -100000 - 6
    lens = case.seq_lens.copy()
    lens[4] = 300   # below the 512 stated shared positions
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cache.seq_lens.copy_(torch.from_numpy(lens))
    cache.kv_indptr.copy_(torch.from_numpy(indptr))
    pkv.paged_decode_pages(cache, case.layer_id, torch.from_numpy(table).cuda(), 16, q,
                           workspace=ws, shared_pages=32)
    st, _ = pkv.last_device_error()
    assert st == _lib.PKV_ERR_INDEX


@pytest.mark.parametrize("hk,shared_pages,splits,batch,d", [
    (4, 32, 1024, 6, 128), (8, 3, 1024, 6, 128), (8, 32, 1024, 1, 128), (8, 32, 64, 6, 64)])
def test_shared_prefix_statement_ignored_where_it_does_not_apply(hk, shared_pages, splits, batch, d):
    """4 kv heads, fewer than 64 shared positions, a single entry, or (head_dim
    64) a workspace without room for the group partials: the decode runs as
    without the statement (bit-identical)."""
    case = shared_case(batch, 4 * hk, 16, 512, 100, seed=88, hk=hk, d=d)
    cache, q = prepare(case)
    ws = ws_for(case, splits=splits)
    table = torch.from_numpy(page_table(case)).cuda()
    o = pkv.paged_decode_pages(cache, case.layer_id, table, 16, q, workspace=ws,
                               shared_pages=shared_pages)
    no_device_error()
    assert torch.equal(o, pkv.paged_decode_pages(cache, case.layer_id, table, 16, q, workspace=ws))


@pytest.mark.parametrize("heads,shared,batch", [(32, 2048, 64), (16, 320, 11)])
def test_shared_prefix_through_req_to_token(heads, shared, batch):
    """The per-token path with the shared prefix stated (slots compared at
    every position): equal to the oracle, and not the plain decode's
    summation order."""
    case = shared_case(batch, heads, 16, shared, 500, seed=heads + shared)
    cache, q = prepare(case)
    ws = ws_for(case)
    o = pkv.paged_decode_shared(cache, case.layer_id, shared, q, workspace=ws)
    no_device_error()
    assert_close(f64(o), oracle_decode(case), "bf16", f"shared {shared} via req_to_token")
    assert not torch.equal(o, pkv.paged_decode(cache, case.layer_id, q, workspace=ws))


def test_shared_prefix_through_req_to_token_reports_a_differing_slot():
    case = shared_case(8, 32, 1, 256, 40, seed=5)
    cache, q = prepare(case)
    r2t = case.req_to_token.copy()
    r = int(case.req_pool_indices[5])
    r2t[r, 100] = r2t[r, 101]   # one shared position of entry 5 points elsewhere
    cache.req_to_token.copy_(torch.from_numpy(r2t))
    pkv.paged_decode_shared(cache, case.layer_id, 256, q, workspace=ws_for(case))
    st, detail = pkv.last_device_error()
    assert st == _lib.PKV_ERR_INDEX and detail == -100000 - 5


def _pinned(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if t.dtype == torch.int16:
        t = t.view(torch.bfloat16)
    return t.pin_memory()


def _host_step_case():
    case = W.batched_decode(batch=16, lo=200, hi=3000, size=65536, seed=919)
    cache, q, kn, vn = W.upload(case)
    host = {"q": _pinned(case.q.view(np.int16)), "k_new": _pinned(case.k_new.view(np.int16)),
            "v_new": _pinned(case.v_new.view(np.int16)), "seq_lens": _pinned(case.seq_lens),
            "req_pool_indices": _pinned(case.req_pool_indices),
            "out_cache_loc": _pinned(case.out_cache_loc), "kv_indptr": _pinned(case.kv_indptr)}
    hcache = pkv.KVCache(k_buffer=cache.k_buffer, v_buffer=cache.v_buffer,
                         req_to_token=cache.req_to_token, req_pool_indices=host["req_pool_indices"],
                         seq_lens=host["seq_lens"], out_cache_loc=host["out_cache_loc"],
                         kv_indptr=host["kv_indptr"], max_len=case.max_len)
    return case, cache, q, kn, vn, host, hcache


def test_decode_step_reads_and_writes_pinned_host_memory():
    """The step's inputs (q, the new rows, the metadata) and o in pinned host
    memory: the kernels use them in place (no copies) and the result is
    bit-identical to the step on device copies."""
    case, cache, q, kn, vn, host, hcache = _host_step_case()
    ws = ws_for(case, splits=64)
    o_dev = pkv.decode_step(cache, case.layer_id, kn, vn, q, workspace=ws)
    o_host = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    pkv.decode_step(hcache, case.layer_id, host["k_new"], host["v_new"], host["q"], o_host,
                    workspace=ws)
    torch.cuda.synchronize()
    no_device_error()
    assert torch.equal(o_host, o_dev.cpu())
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    check_pool_bit_exact(cache, case)


@pytest.mark.parametrize("hq,hk,d", [(8, 8, 128), (16, 8, 64), (64, 8, 128), (32, 8, 64),
                                     (32, 4, 128), (8, 2, 64)])
def test_decode_step_with_q_in_pinned_host_memory(hq, hk, d):
    """q alone in pinned host memory, for every group size and head_dim of the
    tensor-core split kernel (8 kv heads) and its piece-by-piece path (fewer kv
    heads): the step copies q into the workspace for the decode, and o is
    bit-identical to the step with q on the device."""
    rng = np.random.Generator(np.random.PCG64(hq * 1000 + hk * 10 + d))
    kv = rng.integers(1, 2500, size=12, endpoint=True)
    case = W.make_case("q_host", mode="decode", dtype="bf16", n_layers=2, layer_id=1, size=40000,
                       n_heads=hq, n_kv_heads=hk, head_dim=d, kv_lens=kv, seed=hq + d, rng=rng)
    cache, q, kn, vn = W.upload(case)
    ws = ws_for(case, splits=64)
    o_dev = pkv.decode_step(cache, case.layer_id, kn, vn, q, workspace=ws)
    q_host = _pinned(case.q.view(np.int16))
    o = torch.empty_like(o_dev)
    pkv.decode_step(cache, case.layer_id, kn, vn, q_host, o, workspace=ws)
    torch.cuda.synchronize()
    no_device_error()
    assert torch.equal(o, o_dev)
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    assert_close(f64(o), oracle_decode(case), "bf16", f"q host {hq}/{hk}/{d}")


def test_decode_step_graph_on_pinned_host_buffers():
    """A serving loop without copies: the step captured once on pinned host
    buffers; the host rewrites q in place between replays and reads o."""
    case, cache, q, kn, vn, host, hcache = _host_step_case()
    ws = ws_for(case, splits=64)
    o_host = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    call = lambda: pkv.decode_step(hcache, case.layer_id, host["k_new"], host["v_new"], host["q"],
                                   o_host, workspace=ws, stream=s)
    with torch.cuda.stream(s):
        call()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    rng = np.random.Generator(np.random.PCG64(3))
    for _ in range(2):
        bits = W._values(rng, case.q.shape, "bf16")
        host["q"].copy_(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        no_device_error()
        ref = pkv.decode_step(cache, case.layer_id, kn, vn, host["q"].cuda(), workspace=ws)
        assert torch.equal(o_host, ref.cpu())


def test_unregistered_host_memory_is_refused_before_launch():
    """A plain (unpinned) host address would fault the device: the C ABI
    refuses it with PKV_ERR_ARG and enqueues nothing."""
    import ctypes
    case = W.tiny_decode()
    cache, q = prepare(case)
    c = cache.c_struct()
    plain = np.zeros(q.numel() * 2, np.uint8)   # q-sized, 16-byte aligned by numpy
    assert plain.ctypes.data % 16 == 0
    o = torch.empty_like(q)
    rc = _lib.load().pkv_paged_decode(ctypes.byref(c), case.layer_id, ctypes.c_void_p(plain.ctypes.data),
                                      ctypes.c_void_p(o.data_ptr()), case.n_heads, 0.125, None, None)
    assert rc == _lib.PKV_ERR_ARG
    no_device_error()


def test_rope_kv_write_full_size():
    """The fused RoPE write at the size the bench times it: the ragged
    prefill's 17,418 new tokens, the standard rotary table, each token at its
    position.  K within one bf16 rounding of the fp64 rotation, V and every
    other pool row bit-exact."""
    case = W.ragged_prefill()
    d = case.head_dim
    max_pos = int(case.seq_lens.max())
    inv = 10000.0 ** (-np.arange(0, d, 2, dtype=np.float64) / d)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    fc = np.stack([np.cos(ang), np.sin(ang)], -1).astype(np.float32)
    pos = np.concatenate([np.arange(int(case.seq_lens[b] - case.q_lens[b]), int(case.seq_lens[b]))
                          for b in range(case.batch)]).astype(np.int32)
    cache, q, kn, vn = W.upload(case)
    pkv.rope_kv_write(cache, case.layer_id, kn, vn, torch.from_numpy(fc).cuda(), torch.from_numpy(pos).cuda())
    no_device_error()
    k_rot = oracle.rope(case.k_new, fc, pos)
    got_k = f64(cache.k_buffer)[case.layer_id, case.out_cache_loc]
    assert np.all(np.abs(got_k - k_rot) <= np.abs(k_rot) * 2.0 ** -8 + 1e-6)
    vb = W.host_of(cache.v_buffer)
    assert np.array_equal(vb[case.layer_id, case.out_cache_loc], case.v_new)
    # rows the write does not touch keep their contents
    kb = W.host_of(cache.k_buffer)
    mask = np.ones(case.k_buffer.shape[1], bool)
    mask[case.out_cache_loc] = False
    assert np.array_equal(kb[case.layer_id][mask], case.k_buffer[case.layer_id][mask])
    assert np.array_equal(vb[case.layer_id][mask], case.v_buffer[case.layer_id][mask])


def test_kv_write_and_prefill_on_pinned_host_memory():
    """The cache write from new rows and locations in pinned host memory, and
    the prefill reading q from and writing o to pinned host memory: the same
    bits as with device copies."""
    case = W.ragged_prefill(batch=3, q_hi=300, p_hi=500, size=8192, seed=77)
    cache_d, q, kn, vn = W.upload(case)
    pkv.kv_write(cache_d, case.layer_id, kn, vn)
    o_d = pkv.paged_prefill(cache_d, case.layer_id, q, case.max_q_len, case.max_len)
    cache_h, _, _, _ = W.upload(case)
    cache_h.out_cache_loc = cache_h.out_cache_loc.cpu().pin_memory()
    pkv.kv_write(cache_h, case.layer_id, kn.cpu().pin_memory(), vn.cpu().pin_memory())
    torch.cuda.synchronize()
    assert torch.equal(cache_h.k_buffer, cache_d.k_buffer) and torch.equal(cache_h.v_buffer, cache_d.v_buffer)
    o_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    pkv.paged_prefill(cache_h, case.layer_id, q.cpu().pin_memory(), case.max_q_len, case.max_len, o=o_h)
    torch.cuda.synchronize()
    no_device_error()
    assert torch.equal(o_h, o_d.cpu())
