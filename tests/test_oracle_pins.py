"""Pins for the fp64 oracle, against things other than the oracle itself.

* torch's float64 ``scaled_dot_product_attention`` (a library routine the
  oracle never calls) on contiguous-mode caches, where ``req_to_token`` is the
  linear map slot = req_idx * max_seq_len + pos (AstrAI docs/guides/inference.md,
  "KVCache System", contiguous mode);
* numpy fancy-index assignment for the cache write ``k_buffer[layer_id,
  out_cache_loc] = k`` (same page, "KVCache System");
* numpy complex multiplication for the rotary embedding ("Rotary Embedding
  Backend": complex multiply against freqs_cis [max_len, dim/2, 2]);
* hand-derived closed forms under ``tests/golden/``;
* invariants: slot permutation, length-1 context, equal keys, prefill row i ==
  decode at position P + i.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_loc_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def contiguous_case(batch, n_heads, n_kv_heads, head_dim, kv_lens, q_lens=None, dtype="f32",
                    seed=0, n_layers=2, layer_id=1):
    """Contiguous mode: request row r owns slots [r*max_len, (r+1)*max_len)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    max_len = int(max(kv_lens))
    size = batch * max_len
    shape = (n_layers, size, n_kv_heads, head_dim)
    kb = rng.standard_normal(shape, dtype=np.float32)
    vb = rng.standard_normal(shape, dtype=np.float32)
    q_lens = [1] * batch if q_lens is None else q_lens
    q = rng.standard_normal((int(sum(q_lens)), n_heads, head_dim), dtype=np.float32)
    if dtype == "bf16":
        kb, vb, q = W.to_bf16_bits(kb), W.to_bf16_bits(vb), W.to_bf16_bits(q)
    r2t = (np.arange(batch)[:, None] * max_len + np.arange(max_len)[None, :]).astype(np.int32)
    return kb, vb, r2t, np.arange(batch, dtype=np.int32), np.asarray(kv_lens, np.int32), q


def sdpa(q, k, v, mask=None, scale=None):
    """q [H, Lq, d], k/v [Hk, Lk, d] float64 torch -> [H, Lq, d]."""
    return F.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=mask,
                                          scale=scale, enable_gqa=True)[0]


@pytest.mark.parametrize("heads", [(8, 2), (4, 4), (8, 1), (6, 3)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_equals_sdpa_on_contiguous_cache(heads, dtype):
    H, Hk = heads
    d, kv = 16, [1, 7, 33, 64]
    kb, vb, r2t, rpi, sl, q = contiguous_case(4, H, Hk, d, kv, dtype=dtype, seed=H * 10 + Hk)
    o = oracle.decode(kb, vb, r2t, rpi, sl, q, layer_id=1)
    K, V, Q = (torch.from_numpy(oracle.to_f64(x)) for x in (kb[1], vb[1], q))
    for b, n in enumerate(kv):
        slots = r2t[b, :n]
        ref = sdpa(Q[b][:, None, :], K[slots].permute(1, 0, 2), V[slots].permute(1, 0, 2))
        np.testing.assert_allclose(o[b], ref[:, 0, :].numpy(), rtol=0, atol=1e-12)


def test_decode_explicit_scale_matches_sdpa():
    kb, vb, r2t, rpi, sl, q = contiguous_case(2, 4, 2, 8, [5, 9], seed=3)
    o = oracle.decode(kb, vb, r2t, rpi, sl, q, layer_id=1, sm_scale=0.3)
    K, V, Q = (torch.from_numpy(oracle.to_f64(x)) for x in (kb[1], vb[1], q))
    for b, n in enumerate([5, 9]):
        s = r2t[b, :n]
        ref = sdpa(Q[b][:, None], K[s].permute(1, 0, 2), V[s].permute(1, 0, 2), scale=0.3)
        np.testing.assert_allclose(o[b], ref[:, 0].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("heads", [(8, 2), (4, 4)])
def test_prefill_equals_sdpa_with_prefix(causal, heads):
    H, Hk = heads
    d = 16
    q_lens = [1, 5, 12, 3]
    kv_lens = [4, 5, 20, 3]          # prefixes 3, 0, 8, 0
    kb, vb, r2t, rpi, _, q = contiguous_case(4, H, Hk, d, kv_lens, q_lens=q_lens, seed=11)
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    kvi = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    o = oracle.prefill(kb, vb, r2t, rpi, qo, kvi, q, layer_id=1, causal=causal)
    K, V, Q = (torch.from_numpy(oracle.to_f64(x)) for x in (kb[1], vb[1], q))
    for b, (ql, kl) in enumerate(zip(q_lens, kv_lens)):
        s = r2t[b, :kl]
        P = kl - ql
        mask = None
        if causal:   # bottom-right aligned: row i sees j <= P + i
            mask = torch.arange(kl)[None, :] <= (P + torch.arange(ql))[:, None]
        qb = Q[qo[b]:qo[b + 1]].permute(1, 0, 2)
        ref = sdpa(qb, K[s].permute(1, 0, 2), V[s].permute(1, 0, 2), mask=mask)
        np.testing.assert_allclose(o[qo[b]:qo[b + 1]], ref.permute(1, 0, 2).numpy(), rtol=0,
                                   atol=1e-12)


def test_prefill_without_prefix_equals_sdpa_is_causal():
    """P = 0: the bottom-right and top-left alignments agree, use torch's own flag."""
    kb, vb, r2t, rpi, _, q = contiguous_case(1, 4, 2, 8, [9], q_lens=[9], seed=5)
    qo = np.array([0, 9], np.int32)
    o = oracle.prefill(kb, vb, r2t, rpi, qo, qo, q, layer_id=1, causal=True)
    K, V, Q = (torch.from_numpy(oracle.to_f64(x)) for x in (kb[1], vb[1], q))
    ref = F.scaled_dot_product_attention(Q.permute(1, 0, 2)[None], K[:9].permute(1, 0, 2)[None],
                                         V[:9].permute(1, 0, 2)[None], is_causal=True,
                                         enable_gqa=True)[0]
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def _pool_from_golden(g, n_layers=2, layer_id=1):
    d = g["head_dim"]
    size = g["pool_size"]
    kb = np.full((n_layers, size, 1, d), 99.0, np.float32)
    vb = np.full((n_layers, size, 1, d), -99.0, np.float32)
    for j, s in enumerate(g["slots"]):
        kb[layer_id, s, 0] = g["k"][j]
        vb[layer_id, s, 0] = g["v"][j]
    r2t = np.array([g["slots"]], np.int32)
    return kb, vb, r2t


def test_golden_two_token_closed_form():
    g = json.load(open(os.path.join(GOLDEN, "two_token_ln3.json")))
    kb, vb, r2t = _pool_from_golden(g)
    q = np.array([[g["q"]]], np.float32)
    o = oracle.decode(kb, vb, r2t, [0], [2], q, layer_id=1, sm_scale=g["sm_scale"])
    np.testing.assert_allclose(o[0, 0], g["expected_o"], rtol=0, atol=g["tol"])


def test_golden_prefill_prefix_causal():
    g = json.load(open(os.path.join(GOLDEN, "prefill_prefix_causal.json")))
    kb, vb, r2t = _pool_from_golden(g)
    q = np.array(g["q"], np.float32)[:, None, :]
    qo = np.array([0, 2], np.int32)
    kv = np.array([0, 3], np.int32)
    o = oracle.prefill(kb, vb, r2t, [0], qo, kv, q, layer_id=1, causal=True,
                       sm_scale=g["sm_scale"])
    np.testing.assert_allclose(o[:, 0], g["expected_o"], rtol=0, atol=g["tol"])
    o = oracle.prefill(kb, vb, r2t, [0], qo, kv, q, layer_id=1, causal=False,
                       sm_scale=g["sm_scale"], rows=[0])
    np.testing.assert_allclose(o[0, 0], g["expected_o_noncausal_row0"], rtol=0, atol=g["tol"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_slot_permutation_invariance_bit_exact(dtype):
    c = W.make_case("perm", mode="decode", dtype=dtype, n_layers=3, layer_id=1, size=512,
                    n_heads=8, n_kv_heads=2, head_dim=32, kv_lens=[3, 50, 130], seed=21,
                    num_reqs=5, max_ctx_len=160)
    o1 = oracle.decode(c.k_buffer, c.v_buffer, c.req_to_token, c.req_pool_indices, c.seq_lens,
                       c.q, c.layer_id)
    pi = np.random.Generator(np.random.PCG64(99)).permutation(c.size)
    kb2 = np.empty_like(c.k_buffer)
    vb2 = np.empty_like(c.v_buffer)
    kb2[:, pi] = c.k_buffer
    vb2[:, pi] = c.v_buffer
    r2t2 = pi[c.req_to_token].astype(np.int32)
    o2 = oracle.decode(kb2, vb2, r2t2, c.req_pool_indices, c.seq_lens, c.q, c.layer_id)
    assert np.array_equal(o1, o2)


def test_length_one_context_returns_v_exactly():
    c = W.make_case("len1", mode="decode", dtype="bf16", n_layers=2, layer_id=0, size=64,
                    n_heads=4, n_kv_heads=2, head_dim=16, kv_lens=[1, 1], seed=4)
    o = oracle.decode(c.k_buffer, c.v_buffer, c.req_to_token, c.req_pool_indices, c.seq_lens,
                      c.q, c.layer_id)
    V = oracle.to_f64(c.v_buffer[c.layer_id])
    for b in range(2):
        slot = c.slots_of(b)[0]
        for h in range(4):
            assert np.array_equal(o[b, h], V[slot, h // 2])


def test_equal_keys_return_mean_of_v():
    rng = np.random.Generator(np.random.PCG64(8))
    n, d = 37, 8
    kb = np.zeros((1, 64, 1, d), np.float32)
    kb[0, :, 0] = rng.standard_normal(d, dtype=np.float32)       # every slot: the same key
    vb = rng.standard_normal((1, 64, 1, d), dtype=np.float32)
    slots = rng.permutation(64)[:n].astype(np.int32)
    q = rng.standard_normal((1, 1, d), dtype=np.float32)
    o = oracle.decode(kb, vb, slots[None], [0], [n], q, 0)
    np.testing.assert_allclose(o[0, 0], vb[0, slots, 0].astype(np.float64).mean(0), rtol=0,
                               atol=1e-15)


def test_zero_scale_gives_uniform_weights():
    c = W.make_case("scale0", mode="decode", dtype="f32", n_layers=1, layer_id=0, size=256,
                    n_heads=2, n_kv_heads=1, head_dim=8, kv_lens=[40], seed=12)
    o = oracle.decode(c.k_buffer, c.v_buffer, c.req_to_token, c.req_pool_indices, c.seq_lens,
                      c.q, 0, sm_scale=0.0)
    mean = c.v_buffer[0, c.slots_of(0), 0].astype(np.float64).mean(0)
    np.testing.assert_allclose(o[0, 0], mean, rtol=0, atol=1e-14)


def test_empty_context_gives_zero():
    c = W.make_case("empty", mode="decode", dtype="f32", n_layers=1, layer_id=0, size=64,
                    n_heads=2, n_kv_heads=1, head_dim=8, kv_lens=[0, 3], q_lens=[0, 1], seed=2)
    q = np.ones((2, 2, 8), np.float32)
    o = oracle.decode(c.k_buffer, c.v_buffer, c.req_to_token, c.req_pool_indices, [0, 3], q, 0)
    assert np.all(o[0] == 0.0)


def test_causal_prefill_row_equals_decode_at_that_position():
    c = W.make_case("pre", mode="prefill", dtype="bf16", n_layers=2, layer_id=1, size=1024,
                    n_heads=8, n_kv_heads=2, head_dim=32, kv_lens=[40, 77], q_lens=[15, 77],
                    seed=31)
    kb, vb = c.k_buffer.copy(), c.v_buffer.copy()
    oracle.kv_write(kb, vb, c.layer_id, c.k_new, c.v_new, c.out_cache_loc)
    o = oracle.prefill(kb, vb, c.req_to_token, c.req_pool_indices, c.qo_indptr, c.kv_indptr,
                       c.q, c.layer_id, causal=True)
    for b in range(c.batch):
        P = int(c.seq_lens[b] - c.q_lens[b])
        for i in range(int(c.q_lens[b])):
            p = int(c.qo_indptr[b]) + i
            od = oracle.decode(kb, vb, c.req_to_token, c.req_pool_indices[b:b + 1], [P + i + 1],
                               c.q[p:p + 1], c.layer_id)
            assert np.array_equal(o[p], od[0])
    # Non-causal rows all equal decode over the whole context.
    onc = oracle.prefill(kb, vb, c.req_to_token, c.req_pool_indices, c.qo_indptr, c.kv_indptr,
                         c.q, c.layer_id, causal=False)
    for b in range(c.batch):
        for p in range(int(c.qo_indptr[b]), int(c.qo_indptr[b + 1])):
            od = oracle.decode(kb, vb, c.req_to_token, c.req_pool_indices[b:b + 1],
                               c.seq_lens[b:b + 1], c.q[p:p + 1], c.layer_id)
            assert np.array_equal(onc[p], od[0])


def test_prefill_row_subset_matches_full():
    c = W.make_case("rows", mode="prefill", dtype="f32", n_layers=1, layer_id=0, size=512,
                    n_heads=4, n_kv_heads=2, head_dim=8, kv_lens=[30, 50, 9], q_lens=[10, 50, 4],
                    seed=41)
    full = oracle.prefill(c.k_buffer, c.v_buffer, c.req_to_token, c.req_pool_indices,
                          c.qo_indptr, c.kv_indptr, c.q, 0)
    rows = np.array([63, 0, 10, 59, 5])
    sub = oracle.prefill(c.k_buffer, c.v_buffer, c.req_to_token, c.req_pool_indices,
                         c.qo_indptr, c.kv_indptr, c.q, 0, rows=rows)
    assert np.array_equal(sub, full[rows])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kv_write_equals_numpy_index_assignment(dtype):
    c = W.make_case("kvw", mode="prefill", dtype=dtype, n_layers=3, layer_id=2, size=777,
                    n_heads=4, n_kv_heads=2, head_dim=24, kv_lens=[10, 300, 31],
                    q_lens=[10, 120, 1], seed=51)
    kb, vb = c.k_buffer.copy(), c.v_buffer.copy()
    oracle.kv_write(kb, vb, c.layer_id, c.k_new, c.v_new, c.out_cache_loc)
    ek, ev = c.k_buffer.copy(), c.v_buffer.copy()
    ek[c.layer_id, c.out_cache_loc] = c.k_new
    ev[c.layer_id, c.out_cache_loc] = c.v_new
    assert np.array_equal(kb.view(np.uint8), ek.view(np.uint8))
    assert np.array_equal(vb.view(np.uint8), ev.view(np.uint8))
    untouched = np.ones(c.size, bool)
    untouched[c.out_cache_loc] = False
    assert np.array_equal(kb[:, untouched], c.k_buffer[:, untouched])
    assert np.array_equal(kb[:2], c.k_buffer[:2])


def test_kv_write_rejects_out_of_range_slot():
    kb = np.zeros((1, 8, 1, 4), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.kv_write(kb, kb.copy(), 0, np.ones((1, 1, 4), np.float32),
                        np.ones((1, 1, 4), np.float32), np.array([8], np.int32))


def test_decode_checks_kv_indptr_against_seq_lens():
    c = W.make_case("kvi", mode="decode", dtype="f32", n_layers=1, layer_id=0, size=64,
                    n_heads=2, n_kv_heads=1, head_dim=8, kv_lens=[3, 5], seed=6)
    oracle.decode(c.k_buffer, c.v_buffer, c.req_to_token, c.req_pool_indices, c.seq_lens, c.q,
                  0, kv_indptr=c.kv_indptr)
    with pytest.raises(oracle.OracleError):
        oracle.decode(c.k_buffer, c.v_buffer, c.req_to_token, c.req_pool_indices, c.seq_lens,
                      c.q, 0, kv_indptr=np.array([0, 3, 9], np.int32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rope_equals_complex_multiply(dtype):
    rng = np.random.Generator(np.random.PCG64(61))
    n, heads, d, max_pos = 9, 3, 16, 40
    ang = rng.uniform(-np.pi, np.pi, (max_pos, d // 2)).astype(np.float32)
    fc = np.stack([np.cos(ang), np.sin(ang)], -1).astype(np.float32)
    x = rng.standard_normal((n, heads, d), dtype=np.float32)
    if dtype == "bf16":
        x = W.to_bf16_bits(x)
    pos = rng.integers(0, max_pos, n).astype(np.int32)
    out = oracle.rope(x, fc, pos)
    xf = oracle.to_f64(x)
    z = xf[..., 0::2] + 1j * xf[..., 1::2]
    rot = fc[pos, :, 0].astype(np.float64) + 1j * fc[pos, :, 1].astype(np.float64)
    ref = z * rot[:, None, :]
    np.testing.assert_allclose(out[..., 0::2], ref.real, rtol=0, atol=1e-13)
    np.testing.assert_allclose(out[..., 1::2], ref.imag, rtol=0, atol=1e-13)
    # The identity table (cos 1, sin 0) leaves x unchanged.
    ident = np.zeros_like(fc)
    ident[..., 0] = 1.0
    assert np.array_equal(oracle.rope(x, ident, pos), xf)
