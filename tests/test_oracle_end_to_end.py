"""End-to-end pins of the oracle's layer step (CPU only)."""

import numpy as np
import torch
import torch.nn.functional as F

from learned_sparse_attention_gb300 import workloads as W
from oracle import qsa_oracle as O
from tests.oracle_io import OracleState


def _dense_reference(st: OracleState, row: int) -> np.ndarray:
    """Causal dense GQA of one row over tokens 0..p through torch SDPA, then
    the bf16 rounding and sigmoid gate."""
    s = st.spec
    req = int(st.token_to_req[row])
    p = int(st.logical_positions[row])
    toks = np.arange(p + 1)
    blocks = st.block_table[req][toks // s.page]
    kv = st.kv[blocks, :, toks % s.page]          # [L, Hkv, 2D]
    D = s.head_dim
    g = s.hq // s.hkv
    k = torch.from_numpy(kv[..., :D]).permute(1, 0, 2).repeat_interleave(g, 0)
    v = torch.from_numpy(kv[..., D:]).permute(1, 0, 2).repeat_interleave(g, 0)
    o = F.scaled_dot_product_attention(torch.from_numpy(st.q[row])[:, None, :], k, v)[:, 0].numpy()
    o = O.round_bf16(o)
    return O.round_bf16(o * (1.0 / (1.0 + np.exp(-st.gate[row]))))


def test_within_budget_step_equals_dense_attention():
    # every row has V(p) <= K_b = 16, so QSA must attend to the whole prefix
    spec = W.small_spec(contexts=(12, 40, 64, 3), rows_per_req=(1, 3, 2, 1))
    st = OracleState(W.make_workload(spec))
    q_idx, packed, out = st.step()
    for row in range(spec.rows):
        p = int(st.logical_positions[row])
        n = packed[row, -1]
        assert n == p + 1
        np.testing.assert_array_equal(np.sort(packed[row, :n]), np.arange(p + 1))
        np.testing.assert_allclose(out[row], _dense_reference(st, row), atol=1e-2, rtol=1e-2)


def test_tiny_workload_selection_invariants():
    spec = W.named_spec("tiny_bf16")
    st = OracleState(W.make_workload(spec))
    q_idx, packed, out = st.step()
    cfg = st.cfg
    for row in range(spec.rows):
        p = int(st.logical_positions[row])
        n = packed[row, -1]
        assert n == O.expected_count(cfg, p)
        toks = packed[row, :n]
        assert toks.max() <= p and toks.min() >= 0 and len(set(toks.tolist())) == n
        # the tail tokens of the open group are always kept
        V = O.visible_blocks(p, cfg.compress_ratio)
        assert set(range(V * cfg.compress_ratio, p + 1)) <= set(toks.tolist())
    assert np.isfinite(out).all()


def test_skip_topk_reuses_buffer_and_updates_caches():
    spec = W.small_spec(contexts=(101, 64), rows_per_req=(2, 1))
    wl = W.make_workload(spec)
    st = OracleState(wl)
    _, packed0, _ = st.step()
    ring_before = st.ring.copy()
    st.raw_keys = st.raw_keys + 1.0  # a new step's raw keys
    _, packed1, out1 = st.step(skip_topk=True, packed=packed0)
    np.testing.assert_array_equal(packed1, packed0)
    assert not np.array_equal(st.ring, ring_before)


def test_empty_batch():
    cfg = O.QsaConfig(n_heads=2)
    q_idx, packed, out = O.layer_step(
        cfg, projected_q=np.zeros((0, 2, 128)), raw_keys=np.zeros((0, 128)),
        positions=np.zeros((0, 3), int), cos_sin=np.zeros((4, 64)), q_norm_w=np.zeros(128),
        k_norm_w=np.zeros(128), ring=np.zeros((1, 4, 128)), ring_pos=None,
        ring_block_table=np.zeros((1, 1), int), token_to_req=np.zeros(0, int),
        query_start_loc=np.zeros(1, int), logical_positions=np.zeros(0, int),
        ccache=np.zeros((1, 16, 128)), compressed_slots=np.zeros(0, int),
        cblock_table=np.zeros((1, 1), int), q=np.zeros((0, 8, 128)),
        kv=np.zeros((1, 1, 16, 256)), block_table=np.zeros((1, 1), int), page=16)
    assert packed.shape == (0, cfg.packed_width) and out.shape == (0, 8, 128)


def test_within_budget_step_with_main_prepare_equals_dense_attention():
    """With the fused main-attention prepare the step's own K/V rows are
    written into the cache before stage 4, and its q and gate come from the
    projection: a within-budget step then equals dense causal attention of
    the prepared q over the cache with those rows in place."""
    spec = W.small_spec(contexts=(12, 40, 64, 3), rows_per_req=(1, 3, 2, 1), hq=8, hkv=2)
    st = OracleState(W.make_workload(spec))
    rng = np.random.default_rng(3)
    D, hq, hkv = 128, spec.hq, spec.hkv
    qkv = O.round_bf16(rng.standard_normal((spec.rows, (2 * hq + 2 * hkv) * D)))
    slots = np.array([int(st.block_table[int(st.token_to_req[r])][int(st.logical_positions[r]) // spec.page])
                      * spec.page + int(st.logical_positions[r]) % spec.page for r in range(spec.rows)])
    wq, wk = rng.standard_normal(D) * 0.1, rng.standard_normal(D) * 0.1
    main = dict(qkv=qkv, q_norm_w=wq, k_norm_w=wk, eps=1e-6, slot_mapping=slots)
    _, packed, out = st.step(main=main)
    for row in range(spec.rows):
        q, gate, k, v = O.prepare_main_row(st.cfg, qkv[row], st.positions[row], st.cos_sin, wq, wk,
                                           1e-6, hq, hkv)
        blk, off = slots[row] // spec.page, slots[row] % spec.page
        np.testing.assert_array_equal(st.kv[blk, :, off, :D], O.round_bf16(k))
        np.testing.assert_array_equal(st.kv[blk, :, off, D:], v)
        st.q[row], st.gate[row] = q, gate
        np.testing.assert_allclose(out[row], _dense_reference(st, row), atol=1e-2, rtol=1e-2)
