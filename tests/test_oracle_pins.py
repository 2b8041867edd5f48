"""Pins of the oracle to facts outside itself: library routines, closed forms,
invariants, exact arithmetic and brute force on tiny inputs.  CPU only."""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import qsa_oracle as O

RNG = np.random.default_rng(1234)


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def test_bf16_rounding_matches_torch_including_ties():
    x = RNG.standard_normal(200000).astype(np.float32) * np.float32(3.0) ** RNG.integers(-30, 30, 200000)
    x = x.astype(np.float32)
    # exact midpoints between neighbouring bf16 values (ties to even)
    b = torch.from_numpy(RNG.standard_normal(5000).astype(np.float32)).to(torch.bfloat16)
    bits = b.view(torch.int16).to(torch.int32)
    mids = ((bits << 16) | 0x8000).to(torch.int32).view(torch.float32).numpy()
    x = np.concatenate([x, mids, np.float32([0.0, -0.0, 1e-40, -3e-39, 3.3e38])])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)
    enc = O.bf16_encode(x.astype(np.float64))
    np.testing.assert_array_equal(O.bf16_decode(enc), want)


def test_e4m3_code_table_matches_torch_all_256_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode_table()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    # 254 finite codepoints (+-0 included), as the e4m3 decode patch counts them
    assert ok.sum() == 254


def test_e4m3_rounding_matches_torch_within_range():
    table = O.e4m3_decode_table()
    finite = np.unique(table[~np.isnan(table)])
    mids = (finite[1:] + finite[:-1]) / 2  # exact ties
    x = np.concatenate([finite, mids, RNG.uniform(-448, 448, 100000),
                        RNG.standard_normal(50000) * 1e-2, RNG.standard_normal(50000)])
    x = x.astype(np.float32)  # every tested value is exact in fp32
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.round_e4m3(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)
    codes = O.e4m3_encode(x.astype(np.float64))
    want_codes = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # -0 and +0 differ only in sign bit; compare values for zeros
    nz = want != 0
    np.testing.assert_array_equal(codes[nz], want_codes[nz])


def test_e4m3_saturates_instead_of_nan():
    got = O.round_e4m3(np.array([448.0, 449.0, 463.9, 464.0, 479.0, 1e6, -1e6, -470.0]))
    np.testing.assert_array_equal(got, [448, 448, 448, 448, 448, 448, -448, -448])


# --------------------------------------------------------------------------
# RMSNorm and RoPE
# --------------------------------------------------------------------------

def test_gemma_rmsnorm_matches_torch_rms_norm():
    x = RNG.standard_normal((7, 128))
    w = RNG.standard_normal(128) * 0.1
    want = F.rms_norm(torch.from_numpy(x), (128,), torch.from_numpy(1.0 + w), eps=1e-6).numpy()
    np.testing.assert_allclose(O.gemma_rmsnorm(x, w, 1e-6), want, rtol=1e-12, atol=1e-12)


def test_gemma_rmsnorm_unit_rms_and_scale_invariance():
    x = RNG.standard_normal((5, 128)) * 3.0
    y = O.gemma_rmsnorm(x, np.zeros(128), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-12)
    np.testing.assert_allclose(O.gemma_rmsnorm(17.0 * x, np.zeros(128), 0.0), y, rtol=1e-12)


def _table(max_pos=4096, rot=64):
    half = rot // 2
    inv = 10000.0 ** (-np.arange(half) * 2.0 / rot)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)


def test_rope_is_identity_at_zero_and_keeps_tail_and_norm():
    cs = _table()
    x = RNG.standard_normal(128)
    np.testing.assert_allclose(O.rope_neox(x, (0, 0, 0), cs, 64, (0, 0, 0)), x, atol=0)
    y = O.rope_neox(x, (1234, 1234, 1234), cs, 64, (0, 0, 0))
    np.testing.assert_array_equal(y[64:], x[64:])
    np.testing.assert_allclose(np.linalg.norm(y), np.linalg.norm(x), rtol=1e-12)


def test_rope_matches_complex_rotation_and_relative_position():
    cs = _table()
    x = RNG.standard_normal(128)
    k = RNG.standard_normal(128)
    m, n = 1000, 377
    # NeoX pairs (i, i + 32) as complex numbers rotated by angle pos * inv_freq_i
    z = (x[:32] + 1j * x[32:64]) * np.exp(1j * m * 10000.0 ** (-np.arange(32) / 32.0))
    y = O.rope_neox(x, (m, m, m), cs, 64, (0, 0, 0))
    np.testing.assert_allclose(y[:32], z.real, atol=1e-9)
    np.testing.assert_allclose(y[32:64], z.imag, atol=1e-9)
    d1 = O.rope_neox(x, (m,) * 3, cs, 64, (0, 0, 0)) @ O.rope_neox(k, (n,) * 3, cs, 64, (0, 0, 0))
    d2 = O.rope_neox(x, (m + 50,) * 3, cs, 64, (0, 0, 0)) @ O.rope_neox(k, (n + 50,) * 3, cs, 64, (0, 0, 0))
    assert abs(d1 - d2) < 1e-9


def test_mrope_with_equal_components_equals_1d_rope():
    cs = _table()
    x = RNG.standard_normal((3, 128))
    for p in (0, 5, 999, 4095):
        np.testing.assert_array_equal(O.rope_neox(x, (p, p, p), cs, 64, (8, 12, 12)),
                                      O.rope_neox(x, (p, p, p), cs, 64, (0, 0, 0)))


def test_mrope_section_table_golden():
    """Hand-derived component of each of the 32 frequencies for [8, 12, 12]
    (tests/golden/mrope_components_8_12_12.txt)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "mrope_components_8_12_12.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    want = {int(i): "THW".index(c) for i, c in rows}
    assert len(want) == 32
    for i in range(32):
        assert O.mrope_component(i, (8, 12, 12)) == want[i]


def test_mrope_changes_only_its_section():
    cs = _table()
    x = RNG.standard_normal(128)
    a = O.rope_neox(x, (100, 200, 300), cs, 64, (8, 12, 12))
    b = O.rope_neox(x, (100, 250, 300), cs, 64, (8, 12, 12))
    changed = {i for i in range(32) if a[i] != b[i] or a[32 + i] != b[32 + i]}
    assert changed == {i for i in range(32) if O.mrope_component(i, (8, 12, 12)) == 1}


# --------------------------------------------------------------------------
# Compress (stage 1)
# --------------------------------------------------------------------------

def _cfg(**kw):
    base = dict(n_heads=4, head_dim=128, rotary_dim=64, compress_ratio=4, token_topk=16,
                eps=1e-6, index_dtype=O.DTYPE_BF16, state_size=8, cpage=4)
    base.update(kw)
    return O.QsaConfig(**base)


def test_compress_equal_members_pool_to_the_member():
    cfg = _cfg()
    cs = _table()
    key = RNG.standard_normal(128)
    w = RNG.standard_normal(128) * 0.1
    got = O.compress_key(cfg, np.stack([key] * 4), (40, 40, 40), cs, w)
    want = O.round_bf16(O.rope_neox(O.gemma_rmsnorm(key, w, 1e-6), (40,) * 3, cs, 64, (0, 0, 0)))
    np.testing.assert_array_equal(got, want)


def _history_case(r=4, S=8, split_at=None):
    """A request with token history h[0..p]; the step holds tokens
    split_at..p, older tokens sit in the ring."""
    cfg = _cfg(compress_ratio=r, state_size=S)
    cs = _table()
    p = 4 * 10 + r - 1  # completes group 10
    hist = RNG.standard_normal((p + 1, 128))
    wq = RNG.standard_normal(128) * 0.1
    wk = RNG.standard_normal(128) * 0.1
    start = split_at
    rows = p - start + 1
    ring = np.zeros((2, S, 128))
    for t in range(max(0, start - S), start):
        ring[1, t % S] = hist[t]
    ccache = np.zeros((8, cfg.cpage, 128))
    slots = np.full(rows, -1)
    g = (p + 1) // r - 1
    slots[-1] = 3 * cfg.cpage + 1
    args = dict(projected_q=None, raw_keys=hist[start:p + 1],
                positions=np.stack([np.arange(start, p + 1)] * 3, axis=1), cos_sin=cs,
                q_norm_w=wq, k_norm_w=wk, ring=ring, ring_pos=None,
                ring_block_table=np.array([[1]]), token_to_req=np.zeros(rows, dtype=int),
                query_start_loc=np.array([0, rows]), logical_positions=np.arange(start, p + 1),
                ccache=ccache, compressed_slots=slots)
    return cfg, cs, hist, p, g, wk, args


@pytest.mark.parametrize("split_at_back", [0, 1, 2, 3, 5])
def test_compress_member_source_ring_or_step_is_transparent(split_at_back):
    """The compressed key of group g depends only on the token history, not
    on how many of its members arrived in this step (brute force)."""
    cfg, cs, hist, p, g, wk, args = _history_case(split_at=None or (43 - split_at_back))
    O.compress_stage(cfg, **args)
    want = O.round_bf16(O.rope_neox(O.gemma_rmsnorm(hist[g * 4:g * 4 + 4].mean(0), wk, 1e-6),
                                    (g * 4,) * 3, cs, 64, (0, 0, 0)))
    np.testing.assert_array_equal(args["ccache"][3, 1], want)
    # every row's raw key now sits in the ring at t mod S
    for t in range(43 - split_at_back, p + 1):
        np.testing.assert_array_equal(args["ring"][1, t % 8], hist[t])


def test_compress_ring_writes_happen_after_pooling_reads():
    """S = r and a 6-row step: later rows overwrite ring slots the first
    group still needs; pooling must see the pre-step ring (R14)."""
    cfg = _cfg(compress_ratio=4, state_size=4)
    cs = _table()
    hist = RNG.standard_normal((48, 128))
    wk = RNG.standard_normal(128) * 0.1
    start, p_last = 42, 47          # groups 10 (40..43) and 11 (44..47)
    ring = np.zeros((1, 4, 128))
    for t in range(38, 42):
        ring[0, t % 4] = hist[t]
    rows = p_last - start + 1
    slots = np.full(rows, -1)
    slots[43 - start] = 0
    slots[47 - start] = 1
    ccache = np.zeros((1, 4, 128))
    O.compress_stage(cfg, projected_q=None, raw_keys=hist[start:], positions=np.zeros((rows, 3), int),
                     cos_sin=cs, q_norm_w=np.zeros(128), k_norm_w=wk, ring=ring, ring_pos=None,
                     ring_block_table=np.array([[0]]), token_to_req=np.zeros(rows, int),
                     query_start_loc=np.array([0, rows]), logical_positions=np.arange(start, 48),
                     ccache=ccache, compressed_slots=slots)
    for slot, g in ((0, 10), (1, 11)):
        want = O.round_bf16(O.rope_neox(O.gemma_rmsnorm(hist[4 * g:4 * g + 4].mean(0), wk, 1e-6),
                                        (4 * g,) * 3, cs, 64, (0, 0, 0)))
        np.testing.assert_array_equal(ccache[0, slot], want)
    for t in range(44, 48):
        np.testing.assert_array_equal(ring[0, t % 4], hist[t])


def test_prep_query_e4m3_values_are_codes():
    cfg = _cfg(index_dtype=O.DTYPE_E4M3)
    q = O.prep_query(cfg, RNG.standard_normal((4, 128)), (9, 9, 9), _table(), np.zeros(128))
    table = O.e4m3_decode_table()
    assert np.isin(q, table[~np.isnan(table)]).all()


# --------------------------------------------------------------------------
# Index logits, selection, expand
# --------------------------------------------------------------------------

def test_index_logits_relu_identity_and_library_check():
    cfg = _cfg(n_heads=4)
    q = O.round_e4m3(RNG.standard_normal((4, 128)))
    k = O.round_e4m3(RNG.standard_normal((50, 128)))
    s_pos = O.index_logits_row(cfg, q, k)
    s_neg = O.index_logits_row(cfg, -q, k)
    scale = 1.0 / (4 * math.sqrt(128))
    # relu(x) - relu(-x) = x  and  relu(x) + relu(-x) = |x|
    np.testing.assert_allclose(s_pos - s_neg, (k @ q.sum(0)) * scale, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s_pos + s_neg, np.abs(k @ q.T).sum(1) * scale, rtol=1e-12, atol=1e-12)
    lib = torch.relu(torch.einsum("hd,cd->ch", torch.from_numpy(q), torch.from_numpy(k))).sum(1) * scale
    np.testing.assert_allclose(s_pos, lib.numpy(), rtol=1e-12)


def test_index_logits_exact_for_e4m3_inputs():
    """e4m3 x e4m3 products and their sums are exact in float64 here, so the
    oracle equals exact rational arithmetic."""
    cfg = _cfg(n_heads=2)
    q = O.round_e4m3(RNG.standard_normal((2, 128)))
    k = O.round_e4m3(RNG.standard_normal((3, 128)))
    s = O.index_logits_row(cfg, q, k)
    for c in range(3):
        tot = Fraction(0)
        for h in range(2):
            d = sum(Fraction(q[h, i]) * Fraction(k[c, i]) for i in range(128))
            tot += max(d, Fraction(0))
        assert float(tot) / (2 * math.sqrt(128)) == pytest.approx(s[c], rel=1e-15)


def test_select_matches_torch_topk_for_distinct_scores():
    for V, kb in ((100, 16), (5000, 512), (16, 16), (3, 16), (0, 4)):
        s = RNG.permutation(V).astype(np.float64) / 7.0
        got = O.select_blocks(s, V, kb)
        if V <= kb:
            np.testing.assert_array_equal(got, np.arange(V))
        else:
            want = np.sort(torch.topk(torch.from_numpy(s), kb).indices.numpy())
            np.testing.assert_array_equal(got, want)


def test_select_ties_go_to_lower_index():
    s = np.array([1.0, 5.0, 3.0, 5.0, 3.0, 3.0, 0.0])
    np.testing.assert_array_equal(O.select_blocks(s, 7, 3), [1, 2, 3])
    np.testing.assert_array_equal(O.select_blocks(s, 7, 4), [1, 2, 3, 4])


def test_expand_golden_rows():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "expand_rows.txt")
    n = 0
    for ln in open(path):
        if not ln.strip() or ln.startswith("#"):
            continue
        r, topk, p, blocks, want = ln.split("|")
        cfg = _cfg(compress_ratio=int(r), token_topk=int(topk))
        blocks = [int(b) for b in blocks.split(",") if b.strip()]
        want = [int(v) for v in want.split(",")]
        np.testing.assert_array_equal(O.expand_row(cfg, blocks, int(p)), want)
        n += 1
    assert n >= 4


@pytest.mark.parametrize("p", [0, 1, 2, 3, 4, 7, 62, 63, 64, 65, 255, 299, 1000])
def test_expand_count_closed_form_and_causality(p):
    cfg = _cfg(compress_ratio=4, token_topk=64)
    V = O.visible_blocks(p, 4)
    scores = RNG.standard_normal(V)
    blocks = O.select_blocks(scores, V, cfg.block_topk)
    row = O.expand_row(cfg, blocks, p)
    n = row[-1]
    assert n == O.expected_count(cfg, p)
    toks = row[:n]
    assert len(set(toks.tolist())) == n
    assert (toks >= 0).all() and (toks <= p).all()
    assert (row[n:-1] == -1).all()
    assert len(row) == cfg.token_topk + 4 - 1 + 1
    if V <= cfg.block_topk:  # everything within budget is selected
        np.testing.assert_array_equal(np.sort(toks), np.arange(p + 1))


# --------------------------------------------------------------------------
# Sparse GQA
# --------------------------------------------------------------------------

def _kv_case(L=200, Hq=8, Hkv=2, page=16, D=128):
    nb = -(-L // page) + 3
    kv = O.round_bf16(RNG.standard_normal((nb, Hkv, page, 2 * D)))
    bt = RNG.permutation(nb)[: -(-L // page)]
    q = O.round_bf16(RNG.standard_normal((Hq, D)))
    return kv, bt, q


def test_sparse_gqa_all_selected_equals_dense_sdpa():
    L, page, D = 200, 16, 128
    kv, bt, q = _kv_case(L=L)
    toks = np.arange(L)
    got = O.sparse_gqa_row(q, kv, bt, toks, page)
    blocks = bt[toks // page]
    k = kv[blocks, :, toks % page, :D]  # [L, Hkv, D]
    v = kv[blocks, :, toks % page, D:]
    kk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(4, 0)  # [Hq, L, D]
    vv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(4, 0)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[:, None, :], kk, vv)[:, 0]
    np.testing.assert_array_equal(got, O.round_bf16(ref.numpy()))


def test_sparse_gqa_order_invariant_and_empty():
    kv, bt, q = _kv_case()
    toks = RNG.choice(200, size=37, replace=False)
    a = O.sparse_gqa_row(q, kv, bt, toks, 16)
    b = O.sparse_gqa_row(q, kv, bt, toks[::-1], 16)
    np.testing.assert_allclose(a, b, atol=1e-2)  # equal up to bf16 tie rounding
    assert np.abs(a - b).max() <= 2.0 ** -7 * np.abs(a).max()
    np.testing.assert_array_equal(O.sparse_gqa_row(q, kv, bt, [], 16), np.zeros_like(q))


def test_sparse_gqa_gate_limits():
    kv, bt, q = _kv_case()
    toks = np.arange(50)
    plain = O.sparse_gqa_row(q, kv, bt, toks, 16)
    np.testing.assert_array_equal(O.sparse_gqa_row(q, kv, bt, toks, 16, np.full(q.shape, 60.0)), plain)
    np.testing.assert_array_equal(O.sparse_gqa_row(q, kv, bt, toks, 16, np.full(q.shape, -800.0)),
                                  np.zeros_like(plain))
    half = O.sparse_gqa_row(q, kv, bt, toks, 16, np.zeros(q.shape))
    np.testing.assert_array_equal(half, O.round_bf16(plain * 0.5))


def test_sparse_gqa_single_token_returns_its_value():
    kv, bt, q = _kv_case()
    out = O.sparse_gqa_row(q, kv, bt, [77], 16)
    v = kv[bt[77 // 16], :, 77 % 16, 128:]
    np.testing.assert_array_equal(out, np.repeat(v, 4, axis=0))


# --------------------------------------------------------------------------
# Stage-1 position sourcing, the compressed-page map and the query prep,
# each pinned against an independent restatement: RoPE as a complex
# rotation with the hand-derived [8, 12, 12] component table, the norm by
# torch's rms_norm, and values worked out by hand.
# --------------------------------------------------------------------------

def _golden_components():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "mrope_components_8_12_12.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    table = {int(i): "THW".index(c) for i, c in rows}
    return [table[i] for i in range(32)]


def _rope_complex(x, pos3, comps):
    """NeoX RoPE as a complex rotation: frequency i turns x[i] + 1j * x[i + 32]
    by pos3[comps[i]] * 10000**(-i / 32); dims 64.. pass through."""
    x = np.array(x, dtype=np.float64)
    out = x.copy()
    ang = np.array([pos3[comps[i]] for i in range(32)], dtype=np.float64) * \
        10000.0 ** (-np.arange(32) / 32.0)
    z = (x[..., :32] + 1j * x[..., 32:64]) * np.exp(1j * ang)
    out[..., :32] = z.real
    out[..., 32:64] = z.imag
    return out


def _norm(x, w, eps):
    t = torch.from_numpy(np.asarray(x, dtype=np.float64))
    return F.rms_norm(t, (t.shape[-1],), torch.from_numpy(1.0 + np.asarray(w, np.float64)),
                      eps=eps).numpy()


def _within_one_bf16_step(got, want):
    """got is a bf16 value and want an unrounded value: got must be one of
    the two bf16 neighbours of want (the rounding of an fp64 quantity that
    two evaluation orders agree on to ~1e-15)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.abs(want))[1] - 8)
    assert (np.abs(got - want) <= ulp).all(), np.abs(got - want).max()
    # and nearly always the nearest one
    assert (got == O.round_bf16(want)).mean() >= 0.99


def _image_positions(n_tokens, img_start, side):
    """3-D positions of tokens 0..n-1 with one side x side image span at
    img_start (T fixed at the span start, H and W the grid coordinates)."""
    pos = np.stack([np.arange(n_tokens)] * 3, axis=1).astype(np.int64)
    span = side * side
    for t in range(img_start, min(n_tokens, img_start + span)):
        j = t - img_start
        pos[t] = (img_start, img_start + j // side, img_start + j % side)
    return pos


@pytest.mark.parametrize("in_step", [1, 2, 3, 4, 6])
def test_compress_mrope_key_takes_first_member_position_from_step_or_ring(in_step):
    """MRoPE (reading R11): the compressed key of group g is rotated at the
    3-D position of its FIRST token g*r, read from this step's positions
    when that token is in the step, else from the ring's position cache at
    slot (g*r) mod S.  The tokens of the group sit inside an image span, so
    every member has a different (H, W): taking the last member's
    position, or reading the ring at a neighbouring slot, changes the key.
    Source: "indexer_qsa.py", apply_qsa_rope (rotation at the given
    positions); "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward,
    unfused path (RoPE of the pooled key at the group's first positions,
    qsa_store_cache_rows of the rope positions into the ring)."""
    r, S, sec = 4, 8, (8, 12, 12)
    cfg = _cfg(compress_ratio=r, state_size=S, mrope_section=sec)
    cs = _table()
    comps = _golden_components()
    p = 43                                    # completes group 10: tokens 40..43
    g = (p + 1) // r - 1
    pos3 = _image_positions(p + 1, img_start=20, side=6)
    assert len({tuple(pos3[t]) for t in range(40, 44)}) == 4
    hist = RNG.standard_normal((p + 1, 128))
    wk = RNG.standard_normal(128) * 0.1
    start = p - in_step + 1
    rows = in_step
    ring = np.zeros((2, S, 128))
    ring_pos = np.full((2, S, 3), -1, dtype=np.int64)
    for t in range(max(0, start - S), start):
        ring[1, t % S] = hist[t]
        ring_pos[1, t % S] = pos3[t]
    ccache = np.zeros((8, cfg.cpage, 128))
    slots = np.full(rows, -1)
    slots[-1] = 2 * cfg.cpage + 3
    O.compress_stage(cfg, projected_q=None, raw_keys=hist[start:], positions=pos3[start:],
                     cos_sin=cs, q_norm_w=np.zeros(128), k_norm_w=wk, ring=ring,
                     ring_pos=ring_pos, ring_block_table=np.array([[1]]),
                     token_to_req=np.zeros(rows, dtype=int), query_start_loc=np.array([0, rows]),
                     logical_positions=np.arange(start, p + 1), ccache=ccache,
                     compressed_slots=slots)
    want = _rope_complex(_norm(hist[g * r:g * r + r].mean(0), wk, cfg.eps), pos3[g * r], comps)
    _within_one_bf16_step(ccache[2, 3], want)
    # the other members' positions give a different key
    for t in range(g * r + 1, p + 1):
        other = _rope_complex(_norm(hist[g * r:g * r + r].mean(0), wk, cfg.eps), pos3[t], comps)
        assert np.abs(O.round_bf16(other) - ccache[2, 3]).max() > 1e-2
    # the ring now holds this step's raw keys and positions at t mod S
    for t in range(start, p + 1):
        np.testing.assert_array_equal(ring[1, t % S], hist[t])
        np.testing.assert_array_equal(ring_pos[1, t % S], pos3[t])


def test_gather_compressed_keys_follows_the_page_table():
    """Reading R9: compressed key c of a request is entry c mod cpage of
    physical page cblock_row[c // cpage] (the logits column count
    cdiv(max_len, block) * cdiv(block, ratio) in
    "vllm.models.qwen4_exp.nvidia.qsa", Qwen4ExpQSAAttention._run_qsa:
    one compressed page per KV block).  A cache whose key c holds the value
    c (plus d / 1000 in dim d) under a permuted page table must come back as
    0, 1, ..., V-1 in order."""
    cfg = _cfg(cpage=4)
    cblock_row = np.array([5, 2, 7, 0])
    V = 13
    ccache = np.full((8, 4, 128), -1.0)
    for c in range(16):
        ccache[cblock_row[c // 4], c % 4] = c + np.arange(128) / 1000.0
    got = O.gather_compressed_keys(cfg, ccache, cblock_row, V)
    assert got.shape == (V, 128)
    np.testing.assert_array_equal(got, np.arange(V)[:, None] + np.arange(128)[None, :] / 1000.0)


def test_prep_query_hand_worked_two_heads_mrope():
    """Query prep of one row worked out by hand: per head (reshape
    [H * D] -> [H, D]) a Gemma RMSNorm with scale 1 + w, THEN NeoX RoPE with
    MRoPE [8, 12, 12] (frequency 0 rotates at T, frequency 1 at H), then one
    bf16 rounding.  Source: "vllm.models.qwen4_exp.nvidia.qsa",
    QSAIndexer.forward, unfused path (gemma_rmsnorm(q) -> apply_qsa_rope ->
    cast); "indexer_qsa.py", apply_qsa_rope."""
    cfg = _cfg(n_heads=2, eps=0.0, mrope_section=(8, 12, 12))
    cs = _table()
    x = np.zeros(256)
    x[0], x[32] = 3.0, 4.0                        # head 0: pair of frequency 0
    x[128 + 1], x[128 + 33], x[128 + 100] = 1.0, -2.0, 2.0  # head 1: frequency 1 + a tail dim
    w = np.zeros(128)
    w[0], w[32], w[1], w[33], w[100] = 0.5, -0.25, 0.1, 0.3, -0.5
    T, H, Wd = 7, 300, 1000
    got = O.prep_query(cfg, x, (T, H, Wd), cs, w)
    want = np.zeros((2, 128))
    # head 0: mean square 25/128, so 1/rms = sqrt(128)/5; angle T * 1
    a0 = 3.0 * math.sqrt(128) / 5 * 1.5
    b0 = 4.0 * math.sqrt(128) / 5 * 0.75
    want[0, 0] = a0 * math.cos(T) - b0 * math.sin(T)
    want[0, 32] = b0 * math.cos(T) + a0 * math.sin(T)
    # head 1: mean square 9/128, so 1/rms = sqrt(128)/3; angle H * 10000^(-1/32)
    k = math.sqrt(128) / 3
    a1, b1 = 1.0 * k * 1.1, -2.0 * k * 1.3
    th = H * 10000.0 ** (-1.0 / 32.0)
    want[1, 1] = a1 * math.cos(th) - b1 * math.sin(th)
    want[1, 33] = b1 * math.cos(th) + a1 * math.sin(th)
    want[1, 100] = 2.0 * k * 0.5
    _within_one_bf16_step(got, want)
    # norm-then-rotate differs from rotate-then-norm for these weights
    swapped = O.gemma_rmsnorm(O.rope_neox(x.reshape(2, 128), (T, H, Wd), cs, 64, (8, 12, 12)),
                              w, 0.0)
    assert np.abs(O.round_bf16(swapped) - got).max() > 0.1


# --------------------------------------------------------------------------
# FP8 main KV cache (static scalar scales)
# --------------------------------------------------------------------------

def test_fp8_kv_write_matches_torch_e4m3_of_scaled_values():
    """Reading R15, the cache write: e4m3(x / scale), saturating at +-448."""
    x = RNG.standard_normal(20000).astype(np.float32).astype(np.float64)
    for scale in (1.0, 0.0625, 0.013):
        want = torch.from_numpy((x / scale).astype(np.float32)).to(torch.float8_e4m3fn)
        want = want.to(torch.float64).numpy()
        fin = np.abs(x / scale) < 440  # torch's cast is not defined to saturate
        np.testing.assert_array_equal(O.quantize_kv_e4m3(x, scale)[fin], want[fin])
    np.testing.assert_array_equal(O.quantize_kv_e4m3([1e5, -1e5], 1.0), [448.0, -448.0])


def _fp8_case(L=180, Hq=8, Hkv=2, page=16, D=128):
    nb = -(-L // page) + 2
    kv = O.round_e4m3(RNG.standard_normal((nb, Hkv, page, 2 * D)) * 20.0)  # stored values
    bt = RNG.permutation(nb)[: -(-L // page)]
    q = O.round_bf16(RNG.standard_normal((Hq, D)))
    return kv, bt, q


def test_fp8_kv_scales_fold_into_scores_and_output():
    """A k_scale applied to the scores equals the keys scaled by it, and a
    v_scale applied to the output equals the values scaled by it (the patch's
    "scaling each score is equivalent to scaling every key element" and "the
    attention output is linear in V")."""
    kv, bt, q = _fp8_case()
    toks = RNG.choice(180, size=70, replace=False)
    ks, vs = 0.0173, 0.049
    got = O.sparse_gqa_row(q, kv, bt, toks, 16, k_scale=ks, v_scale=vs)
    scaled = kv.copy()
    scaled[..., :128] *= ks
    scaled[..., 128:] *= vs
    want = O.sparse_gqa_row(q, scaled, bt, toks, 16)
    # both are bf16 roundings of the same fp64 quantity up to ~1e-15
    assert np.abs(got - want).max() <= np.abs(want).max() * 2.0 ** -7
    assert (got == want).mean() > 0.99


def test_fp8_kv_all_selected_equals_dense_sdpa_on_dequantized_cache():
    kv, bt, q = _fp8_case(L=150)
    ks, vs = 0.05, 0.031
    toks = np.arange(150)
    got = O.sparse_gqa_row(q, kv, bt, toks, 16, k_scale=ks, v_scale=vs)
    rows = kv[bt[toks // 16], :, toks % 16]  # [L, Hkv, 2D]
    k = torch.from_numpy(rows[..., :128] * ks).permute(1, 0, 2).repeat_interleave(4, 0)
    v = torch.from_numpy(rows[..., 128:] * vs).permute(1, 0, 2).repeat_interleave(4, 0)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[:, None, :], k, v)[:, 0].numpy()
    np.testing.assert_array_equal(got, O.round_bf16(ref))


# --------------------------------------------------------------------------
# Main-attention prepare (reading R16)
# --------------------------------------------------------------------------

def test_prepare_main_layout_hand_worked():
    """Each piece of the projection row lands where reading R16 puts it: per
    query head [q | gate], then the K heads, then the V heads.  Pieces hold
    distinct constants (a constant vector c has RMS |c|, so Gemma RMSNorm
    with w = 0 maps it to sign(c) everywhere, and RoPE at position 0 is the
    identity), so a swapped or shifted slice shows up directly."""
    hq, hkv, D = 3, 2, 128
    cfg = _cfg(n_heads=4, eps=0.0)
    cs = _table()
    x = np.zeros((2 * hq + 2 * hkv) * D)
    consts = {}
    for h in range(hq):
        x[(2 * h) * D:(2 * h + 1) * D] = -(h + 1.0)           # q of head h (negative)
        x[(2 * h + 1) * D:(2 * h + 2) * D] = 10.0 + h         # gate of head h
        consts[("gate", h)] = 10.0 + h
    for h in range(hkv):
        x[(2 * hq + h) * D:(2 * hq + h + 1) * D] = 5.0 + h    # k of head h
        x[(2 * hq + hkv + h) * D:(2 * hq + hkv + h + 1) * D] = 20.0 + h  # v of head h
    q, gate, k, v = O.prepare_main_row(cfg, x, (0, 0, 0), cs, np.zeros(D), np.zeros(D), 0.0,
                                       hq, hkv)
    np.testing.assert_array_equal(q, -np.ones((hq, D)))
    np.testing.assert_array_equal(gate, np.array([[10.0 + h] * D for h in range(hq)]))
    np.testing.assert_allclose(k, np.ones((hkv, D)), atol=1e-15)
    np.testing.assert_array_equal(v, np.array([[20.0 + h] * D for h in range(hkv)]))


def test_prepare_main_norm_then_rope_matches_independent_restatement():
    """q and k: Gemma RMSNorm (torch rms_norm with 1 + w) per head, then
    RoPE as a complex rotation at the row's MRoPE position; q rounded once
    to bf16."""
    hq, hkv, D = 4, 2, 128
    cfg = _cfg(n_heads=4, eps=1e-6, mrope_section=(8, 12, 12))
    cs = _table()
    comps = _golden_components()
    x = RNG.standard_normal((2 * hq + 2 * hkv) * D)
    wq, wk = RNG.standard_normal(D) * 0.1, RNG.standard_normal(D) * 0.1
    pos = (17, 900, 2100)
    q, gate, k, v = O.prepare_main_row(cfg, x, pos, cs, wq, wk, 1e-6, hq, hkv)
    qg = x[: 2 * hq * D].reshape(hq, 2, D)
    want_q = _rope_complex(_norm(qg[:, 0], wq, 1e-6), pos, comps)
    _within_one_bf16_step(q, want_q)
    kk = x[2 * hq * D: (2 * hq + hkv) * D].reshape(hkv, D)
    np.testing.assert_allclose(k, _rope_complex(_norm(kk, wk, 1e-6), pos, comps), atol=1e-12)
    np.testing.assert_array_equal(gate, qg[:, 1])


def test_write_main_kv_slot_and_dtypes():
    """The row's K/V go to block slot // page, offset slot % page, every KV
    head, K then V; bf16 rounding or e4m3(x / scale); slot < 0 writes
    nothing."""
    kv = np.zeros((5, 2, 16, 256))
    k = RNG.standard_normal((2, 128))
    v = RNG.standard_normal((2, 128))
    O.write_main_kv(kv, 3 * 16 + 9, k, v, 16)
    np.testing.assert_array_equal(kv[3, :, 9, :128], O.round_bf16(k))
    np.testing.assert_array_equal(kv[3, :, 9, 128:], O.round_bf16(v))
    assert np.count_nonzero(kv) == np.count_nonzero(kv[3, :, 9])
    kv8 = np.zeros((5, 2, 16, 256))
    O.write_main_kv(kv8, 17, k, v, 16, O.DTYPE_E4M3, 0.05, 0.02)
    want_k = torch.from_numpy((k / 0.05).astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(kv8[1, :, 1, :128], want_k)
    np.testing.assert_array_equal(kv8[1, :, 1, 128:], O.quantize_kv_e4m3(v, 0.02))
    before = kv8.copy()
    O.write_main_kv(kv8, -1, k, v, 16)
    np.testing.assert_array_equal(kv8, before)


# --------------------------------------------------------------------------
# Fused qkv + indexer projection
# --------------------------------------------------------------------------

def test_projection_exact_on_small_integers():
    """Small-integer inputs make every product and sum exact (and exactly a
    bf16 value): the oracle must equal plain integer arithmetic, done here
    with Python ints."""
    rng = np.random.default_rng(5)
    rows, hidden, qc, iq = 3, 48, 8, 6
    x = rng.integers(-3, 4, size=(rows, hidden))
    w = rng.integers(-3, 4, size=(qc + iq + 4, hidden))
    qkv, pq, rk = O.qkv_index_projection(x.astype(float), w.astype(float), qc, iq)
    full = [[sum(int(x[i, k]) * int(w[j, k]) for k in range(hidden)) for j in range(w.shape[0])]
            for i in range(rows)]
    full = np.array(full, dtype=np.float64)
    np.testing.assert_array_equal(qkv, full[:, :qc])
    np.testing.assert_array_equal(pq, full[:, qc:qc + iq])
    np.testing.assert_array_equal(rk, full[:, qc + iq:])


def test_projection_routes_columns_by_the_stacked_weights():
    """A one-hot input row k returns column k of the stacked weights; rows of
    the three weight blocks hold distinct constants, so each output lands in
    its own buffer (main qkv, then indexer q, then the indexer key)."""
    hidden, qc, iq, dk = 16, 5, 3, 2
    w = np.concatenate([np.full((qc, hidden), 1.0), np.full((iq, hidden), 2.0),
                        np.full((dk, hidden), 3.0)]) * (1 + np.arange(hidden))[None, :]
    x = np.eye(hidden)[[0, 7, 15]]
    qkv, pq, rk = O.qkv_index_projection(x, w, qc, iq)
    for i, k in enumerate([0, 7, 15]):
        np.testing.assert_array_equal(qkv[i], np.full(qc, 1.0 * (k + 1)))
        np.testing.assert_array_equal(pq[i], np.full(iq, 2.0 * (k + 1)))
        np.testing.assert_array_equal(rk[i], np.full(dk, 3.0 * (k + 1)))
