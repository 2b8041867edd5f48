"""CUDA path vs oracle on the same seeded inputs (GB300).

Stage-isolated tests feed each kernel inputs from the seeded generators or
from the oracle, never from another kernel; the full-chain tests run the
fused layer step and compare every stage's result with the oracle's own
chain under the parity rules of tests/parity.py."""

import numpy as np
import pytest
import torch

from learned_sparse_attention_gb300 import qsa as Q
from learned_sparse_attention_gb300 import workloads as W
from oracle import qsa_oracle as O
from tests.gpu_harness import (Step, cfgs, idx_dtype, max_visible, oracle_gqa_row, oracle_main,
                               random_packed)
from tests.oracle_io import OracleState, f64, i64
from tests.parity import close_bf16, close_e4m3, selection_ok

pytestmark = pytest.mark.gpu

E4, BF = W.DTYPE_E4M3, W.DTYPE_BF16

MID = {
    "tiny_bf16": W.named_spec("tiny_bf16"),
    "small_bf16_copy_path": W.small_spec("small_bf16_copy_path", seed=5),
    "small_e4m3_copy_path": W.small_spec("small_e4m3_copy_path", seed=6, index_dtype=E4),
    "mid_e4m3_r4": W.small_spec("mid_e4m3_r4", seed=11, contexts=(1999, 4096, 777, 63, 5, 2500),
                                rows_per_req=(1, 3, 2, 1, 1, 8), n_heads=32, index_dtype=E4,
                                compress_ratio=4, token_topk=256, hq=32, hkv=4, page=64),
    "mid_bf16_r8_h16": W.small_spec("mid_bf16_r8_h16", seed=12, contexts=(3001, 1024, 40, 9000),
                                    rows_per_req=(2, 1, 1, 4), n_heads=16, index_dtype=BF,
                                    compress_ratio=8, token_topk=512, hq=16, hkv=2, page=64),
    "mid_mrope_h8": W.small_spec("mid_mrope_h8", seed=13, contexts=(3000, 2048, 700),
                                 rows_per_req=(4, 4, 4), n_heads=8, index_dtype=BF,
                                 compress_ratio=4, token_topk=128, mrope_section=(8, 12, 12),
                                 image_span=64, hq=32, hkv=4, page=32),
    "mid_h64_e4m3_r2": W.small_spec("mid_h64_e4m3_r2", seed=14, contexts=(5000, 300),
                                    rows_per_req=(2, 1), n_heads=64, index_dtype=E4,
                                    compress_ratio=2, token_topk=256, hq=64, hkv=8, page=16),
    # row groups of 32 rows x 8 heads and 16 rows x 16 heads (256 MMA columns)
    "mid_h8_rows32_bf16": W.small_spec("mid_h8_rows32_bf16", seed=15, contexts=(2000, 3001),
                                       rows_per_req=(32, 21), n_heads=8, index_dtype=BF,
                                       compress_ratio=4, token_topk=256, hq=8, hkv=1, page=32),
    "mid_h16_rows16_e4m3": W.small_spec("mid_h16_rows16_e4m3", seed=16,
                                        contexts=(4000, 1501, 903), rows_per_req=(16, 9, 16),
                                        n_heads=16, index_dtype=E4, compress_ratio=4,
                                        token_topk=512, hq=16, hkv=2, page=64),
    # two row groups per logits CTA (e4m3, 256 MMA columns, >= 2 full groups
    # per request on average), with partial second groups
    "mid_e4m3_h32_two_groups": W.small_spec("mid_e4m3_h32_two_groups", seed=17,
                                            contexts=(3000, 2101), rows_per_req=(40, 23),
                                            n_heads=32, index_dtype=E4, compress_ratio=4,
                                            token_topk=512, hq=32, hkv=4, page=64),
    "mid_e4m3_h8_two_groups": W.small_spec("mid_e4m3_h8_two_groups", seed=18,
                                           contexts=(1500, 2603), rows_per_req=(70, 66),
                                           n_heads=8, index_dtype=E4, compress_ratio=4,
                                           token_topk=256, hq=8, hkv=1, page=32),
    # a decode batch (one row per request) with ragged contexts, rows that
    # see no compressed key yet among them: the logits CTAs take only the
    # (row, key chunk) items that hold keys
    "mid_decode_ragged_e4m3": W.small_spec("mid_decode_ragged_e4m3", seed=30,
                                           contexts=(3, 2000, 1, 9000, 130, 2, 4500, 700, 64,
                                                     12000),
                                           rows_per_req=(1,) * 10, n_heads=32, index_dtype=E4,
                                           compress_ratio=4, token_topk=256, hq=32, hkv=4,
                                           page=64),
    # query-head groups other than 8 (the pages only need Hq % Hkv == 0)
    "mid_group16": W.small_spec("mid_group16", seed=19, contexts=(3000, 900, 4100),
                                rows_per_req=(2, 1, 3), n_heads=16, index_dtype=E4,
                                compress_ratio=4, token_topk=512, hq=32, hkv=2, page=64),
    "mid_group4": W.small_spec("mid_group4", seed=20, contexts=(2500, 77, 3333),
                               rows_per_req=(3, 1, 2), n_heads=8, index_dtype=BF,
                               compress_ratio=4, token_topk=256, hq=16, hkv=4, page=32),
    "small_group3": W.small_spec("small_group3", seed=22, hq=6, hkv=2),
    "small_group1": W.small_spec("small_group1", seed=23, hq=4, hkv=4),
    # FP8-e4m3 main KV cache with static scales
    "mid_fp8kv_r4": W.small_spec("mid_fp8kv_r4", seed=25, contexts=(2999, 4096, 300, 1500),
                                 rows_per_req=(1, 2, 1, 4), n_heads=32, index_dtype=E4,
                                 compress_ratio=4, token_topk=512, hq=32, hkv=4, page=64,
                                 kv_dtype=E4, kv_scale=0.0625),
    "mid_fp8kv_group16": W.small_spec("mid_fp8kv_group16", seed=26, contexts=(2500, 801),
                                      rows_per_req=(3, 1), n_heads=8, index_dtype=BF,
                                      compress_ratio=8, token_topk=512, hq=32, hkv=2, page=64,
                                      kv_dtype=E4, kv_scale=0.03),
    "small_fp8kv_group4": W.small_spec("small_fp8kv_group4", seed=27, hq=8, hkv=2, kv_dtype=E4,
                                       kv_scale=0.1),
}


def _close_idx(spec, got, want):
    return close_e4m3(got, want) if spec.index_dtype == E4 else close_bf16(got, want)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    Q.load()
    Q.check_errors()
    yield
    assert Q.check_errors() == 0


# ----------------------------------------------------------------- stage 1
@pytest.mark.parametrize("name", list(MID))
def test_compress_matches_oracle(name):
    spec = MID[name]
    wl = W.make_workload(spec, device="cuda")
    st = OracleState(wl, with_kv=False)
    cc_before = st.ccache.copy()
    cfg, _ = cfgs(spec, wl)
    q_idx = torch.zeros((spec.rows, spec.n_heads, 128), dtype=idx_dtype(spec), device="cuda")
    t = wl.t
    Q.compress(cfg, t["projected_q"], q_idx, t["raw_keys"], t["positions"], t["cos_sin"],
               t["q_norm_w"], t["k_norm_w"], t["ring"], t.get("ring_pos"), t["ring_block_table"],
               t["token_to_req"], t["query_start_loc"], t["logical_positions"], t["ccache"],
               t["compressed_slots"])
    torch.cuda.synchronize()
    oq, written = st.compress()
    ok, err = _close_idx(spec, f64(q_idx), oq)
    assert ok, f"q_idx {err}"
    got_cc = f64(t["ccache"]).reshape(st.ccache.shape)
    slots = [s for _, s, _ in written]
    assert len(slots) == int((i64(t["compressed_slots"]) >= 0).sum())
    flat_got = got_cc.reshape(-1, 128)
    flat_want = st.ccache.reshape(-1, 128)
    ok, err = _close_idx(spec, flat_got[slots], flat_want[slots])
    assert ok, f"compressed keys {err}"
    untouched = np.setdiff1d(np.arange(flat_got.shape[0]), slots)
    np.testing.assert_array_equal(flat_got[untouched], cc_before.reshape(-1, 128)[untouched])
    np.testing.assert_array_equal(f64(t["ring"]).reshape(st.ring.shape), st.ring)
    if st.ring_pos is not None:
        np.testing.assert_array_equal(i64(t["ring_pos"]).reshape(st.ring_pos.shape), st.ring_pos)


# ----------------------------------------------------------------- stage 2
@pytest.mark.parametrize("name", list(MID))
def test_index_logits_matches_oracle(name):
    spec = MID[name]
    wl = W.make_workload(spec, device="cuda")
    cfg, _ = cfgs(spec, wl)
    st = OracleState(wl, with_kv=False)
    g = torch.Generator(device="cuda").manual_seed(77)
    qf = torch.randn((spec.rows, spec.n_heads, 128), generator=g, device="cuda")
    q_idx = (qf.to(torch.float8_e4m3fn).view(torch.uint8) if spec.index_dtype == E4
             else qf.to(torch.bfloat16))
    mv = max_visible(spec)
    ld = (mv + 3) // 4 * 4
    logits = torch.full((spec.rows, ld), float("nan"), device="cuda")
    ws = torch.empty(Q.workspace_bytes(cfg, cfgs(spec, wl)[1], spec.rows, spec.reqs, mv),
                     dtype=torch.uint8, device="cuda")
    t = wl.t
    Q.index_logits(cfg, q_idx, t["ccache"], t["cblock_table"], t["token_to_req"],
                   t["query_start_loc"], t["logical_positions"], logits, mv, ws)
    torch.cuda.synchronize()
    got = logits.cpu().numpy().astype(np.float64)
    qv = f64(q_idx)
    worst = 0.0
    for row in range(spec.rows):
        p = int(st.logical_positions[row])
        V = O.visible_blocks(p, spec.compress_ratio)
        if V == 0:
            continue
        req = int(st.token_to_req[row])
        keys = O.gather_compressed_keys(st.cfg, st.ccache, st.cblock_table[req], V)
        want = O.index_logits_row(st.cfg, qv[row], keys)
        # fp32 accumulation of exact products: relative error ~1e-6 of the
        # sum of |terms|; bound it by 1e-4 of the row's score scale.
        tol = 1e-4 * ((np.abs(keys) @ np.abs(qv[row]).T).sum(1) / (spec.n_heads * np.sqrt(128))
                      + 1e-3)
        e = np.abs(got[row, :V] - want)
        worst = max(worst, float((e / tol).max()))
        assert (e <= tol).all(), f"row {row}: max err {e.max():.3g}"
    print(f"{name}: worst logits error / tolerance = {worst:.3g}")


# ----------------------------------------------------------------- stage 3
@pytest.mark.parametrize("ratio,topk,positions", [
    (4, 64, [0, 2, 3, 62, 63, 64, 255, 299, 1000, 4095]),
    (4, 2048, [8191, 20000, 32767, 2046, 2047, 8000]),
    (8, 4096, [131071, 65535, 32767, 1000]),
    (2, 256, [1, 5, 511, 512, 999]),
    # enough rows for the two-CTA cluster per row (8 and 16 keys per thread)
    (4, 2048, [16384 + 207 * i for i in range(80)]),
    (8, 4096, [131071 - 997 * i for i in range(100)]),
])
@pytest.mark.parametrize("ties", [False, True, "all_equal"])
def test_topk_matches_oracle(ratio, topk, positions, ties):
    cfg_o = O.QsaConfig(n_heads=8, compress_ratio=ratio, token_topk=topk)
    cfg = Q.make_cfg(8, ratio, topk, BF, 16, 10)
    logical = np.array(positions, dtype=np.int32)
    mv = int(max((p + 1) // ratio for p in positions))
    rng = np.random.default_rng(ratio * 1000 + topk + (ties is True))
    if ties == "all_equal":  # every key ties: the lowest blocks are taken
        vals = np.full((len(positions), mv), 0.25, dtype=np.float32)
    elif ties:  # few distinct values: many exact ties at the selection boundary
        vals = rng.integers(0, 7, size=(len(positions), mv)).astype(np.float32) / 8
    else:
        vals = rng.standard_normal((len(positions), mv)).astype(np.float32)
    logits = torch.from_numpy(vals).cuda()
    packed = torch.full((len(positions), cfg_o.packed_width), -9, dtype=torch.int32, device="cuda")
    Q.topk(cfg, logits, mv, torch.from_numpy(logical).cuda(), packed)
    torch.cuda.synchronize()
    got = packed.cpu().numpy()
    for i, p in enumerate(positions):
        V = O.visible_blocks(p, ratio)
        blocks = O.select_blocks(vals[i, :V].astype(np.float64), V, cfg_o.block_topk)
        np.testing.assert_array_equal(got[i], O.expand_row(cfg_o, blocks, p))


# ----------------------------------------------------------------- stage 4
@pytest.mark.parametrize("name", ["tiny_bf16", "small_bf16_copy_path", "mid_e4m3_r4",
                                  "mid_h64_e4m3_r2", "mid_mrope_h8", "mid_group16", "mid_group4",
                                  "small_group3", "small_group1", "mid_fp8kv_r4",
                                  "mid_fp8kv_group16", "small_fp8kv_group4"])
@pytest.mark.parametrize("gate", [True, False])
def test_sparse_gqa_matches_oracle(name, gate):
    spec = MID[name]
    wl = W.make_workload(spec, device="cuda")
    st = OracleState(wl)
    _, gcfg = cfgs(spec, wl)
    rng = np.random.default_rng(5)
    packed_np = random_packed(rng, st.cfg, st.logical_positions, full_rows={0})
    packed_np[-1, :] = -1
    packed_np[-1, -1] = 0  # an empty row: output must be zero
    packed = torch.from_numpy(packed_np).cuda()
    out = torch.full_like(wl["q"], 3.0)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    Q.sparse_gqa(gcfg, wl["q"], wl["kv"], wl["block_table"], packed, wl["token_to_req"],
                 wl["gate"] if gate else None, out, ws)
    torch.cuda.synchronize()
    got = f64(out)
    for row in range(spec.rows):
        n = int(packed_np[row, -1])
        req = int(st.token_to_req[row])
        want = O.sparse_gqa_row(st.q[row], st.kv, st.block_table[req], packed_np[row, :n],
                                spec.page, st.gate[row] if gate else None, *st.kv_scales)
        ok, err = close_bf16(got[row], want)
        assert ok, f"row {row} (n={n}): max err {err:.3g}"
    assert (got[-1] == 0).all()


@pytest.mark.parametrize("hq,hkv", [(32, 4), (32, 2), (8, 4), (16, 4)])
def test_sparse_gqa_many_rows_ragged(hq, hkv):
    """Many (row, KV head) pairs (the prefill shape: several waves of CTAs,
    no split-KV), with ragged selections: counts from 0 to the full width,
    and rows whose selection is the whole prefix.  Four KV heads take one
    CTA per row (a warp per KV head), also with groups of 2 and 4 query
    heads; two KV heads (groups of 16) one CTA per (row, KV head)."""
    rows = 1400
    rng = np.random.default_rng(hq + hkv)
    contexts = [int(x) for x in rng.integers(5, 400, size=rows)]
    spec = W.small_spec("many_pairs", seed=24 + hkv, contexts=contexts, rows_per_req=[1] * rows,
                        n_heads=8, index_dtype=BF, compress_ratio=4, token_topk=64, hq=hq,
                        hkv=hkv, page=16)
    wl = W.make_workload(spec, device="cuda")
    _, gcfg = cfgs(spec, wl)
    assert Q.gqa_splits(gcfg, spec.rows, spec.packed_width) == 1
    st = OracleState(wl, with_kv=False)
    packed_np = random_packed(rng, st.cfg, st.logical_positions, full_rows=set(range(0, rows, 7)))
    packed_np[5, :] = -1
    packed_np[5, -1] = 0
    out = torch.full_like(wl["q"], 3.0)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    Q.sparse_gqa(gcfg, wl["q"], wl["kv"], wl["block_table"], torch.from_numpy(packed_np).cuda(),
                 wl["token_to_req"], wl["gate"], out, ws)
    torch.cuda.synchronize()
    got = f64(out)
    for row in list(range(0, rows, 13)) + [5, rows - 1]:
        n = int(packed_np[row, -1])
        req = int(st.token_to_req[row])
        want = oracle_gqa_row(st.q[row], wl["kv"], st.block_table[req], packed_np[row, :n],
                              spec.page, st.gate[row])
        ok, err = close_bf16(got[row], want)
        assert ok, f"row {row} (n={n}): max err {err:.3g}"
    assert (got[5] == 0).all()


def test_split_kv_invariance():
    """A row computed alone (split-KV over many CTAs + merge) equals the same
    row inside a large batch (one CTA per row and KV head)."""
    spec = W.small_spec("split", seed=21, contexts=[3000] * 80, rows_per_req=[1] * 80,
                        n_heads=8, index_dtype=BF, compress_ratio=4, token_topk=512,
                        hq=32, hkv=4, page=64)
    wl = W.make_workload(spec, device="cuda")
    _, gcfg = cfgs(spec, wl)
    st = OracleState(wl, with_kv=False)
    rng = np.random.default_rng(8)
    packed = torch.from_numpy(random_packed(rng, st.cfg, st.logical_positions,
                                            full_rows=set(range(80)))).cuda()
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    out_all = torch.empty_like(wl["q"])
    Q.sparse_gqa(gcfg, wl["q"], wl["kv"], wl["block_table"], packed, wl["token_to_req"],
                 wl["gate"], out_all, ws)
    for row in (0, 37, 79):
        one = torch.empty_like(wl["q"][row:row + 1])
        Q.sparse_gqa(gcfg, wl["q"][row:row + 1].contiguous(), wl["kv"], wl["block_table"],
                     packed[row:row + 1].contiguous(), wl["token_to_req"][row:row + 1].contiguous(),
                     wl["gate"][row:row + 1].contiguous(), one, ws)
        torch.cuda.synchronize()
        ok, err = close_bf16(f64(one[0]), f64(out_all[row]))
        assert ok, err


@pytest.mark.parametrize("hq,hkv", [(32, 4), (64, 8)])
def test_ring_plans_agree(hq, hkv):
    """Stage 4 runs a 3-stage ring at two CTAs per SM for launches of about
    one wave and a 2-stage ring at three CTAs per SM for many waves; with
    four KV heads the many-wave launch takes one CTA per row (a warp per KV
    head over all the row's tokens) instead of one per (row, KV head) (four
    warps over a quarter of the tokens each, merged).  Rows computed in a
    many-wave launch equal the same rows computed in a small launch: bit for
    bit where the arithmetic is the same (eight KV heads), within the bf16
    tolerance where the order of the sums differs (four), and every plan
    matches the oracle."""
    rows = 720
    spec = W.small_spec("plans", seed=31, contexts=[2500] * rows, rows_per_req=[1] * rows,
                        n_heads=8, index_dtype=BF, compress_ratio=4, token_topk=256,
                        hq=hq, hkv=hkv, page=64)
    wl = W.make_workload(spec, device="cuda")
    _, gcfg = cfgs(spec, wl)
    assert Q.gqa_splits(gcfg, rows, spec.packed_width) == 1
    st = OracleState(wl, with_kv=False)
    rng = np.random.default_rng(9)
    packed = torch.from_numpy(random_packed(rng, st.cfg, st.logical_positions,
                                            full_rows=set(range(0, rows, 3)))).cuda()
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    out_all = torch.empty_like(wl["q"])
    Q.sparse_gqa(gcfg, wl["q"], wl["kv"], wl["block_table"], packed, wl["token_to_req"],
                 wl["gate"], out_all, ws)
    few = 60  # at most 480 CTAs: the one-wave plan
    assert Q.gqa_splits(gcfg, few, spec.packed_width) == 1
    out_few = torch.empty_like(wl["q"][:few])
    Q.sparse_gqa(gcfg, wl["q"][:few].contiguous(), wl["kv"], wl["block_table"],
                 packed[:few].contiguous(), wl["token_to_req"][:few].contiguous(),
                 wl["gate"][:few].contiguous(), out_few, ws)
    torch.cuda.synchronize()
    if hkv == 4:
        ok, err = close_bf16(f64(out_all[:few]), f64(out_few))
        assert ok, err
    else:
        assert torch.equal(out_few, out_all[:few])
    packed_np = packed.cpu().numpy()
    for row in (0, 1, 2, few - 1, rows // 2, rows - 1):
        n = int(packed_np[row, -1])
        want = oracle_gqa_row(st.q[row], wl["kv"], st.block_table[int(st.token_to_req[row])],
                              packed_np[row, :n], spec.page, st.gate[row])
        for got in (out_all[row],) + ((out_few[row],) if row < few else ()):
            ok, err = close_bf16(f64(got), want)
            assert ok, f"row {row}: {err:.3g}"


def test_many_wave_long_selections_split_and_merged():
    """A prefill-shaped launch (many rows, four KV heads) whose selections
    are longer than one chunk of staged row ids (4099 > 2560 entries): the
    split count keeps every CTA within one chunk, so it takes two splits per
    (row, KV head), merged by the last CTA, instead of one CTA per row."""
    rows_per, reqs = 60, 12
    spec = W.small_spec("row_chunks", seed=41, contexts=[6000] * reqs, rows_per_req=[rows_per] * reqs,
                        n_heads=8, index_dtype=BF, compress_ratio=4, token_topk=4096,
                        hq=32, hkv=4, page=64)
    wl = W.make_workload(spec, device="cuda")
    _, gcfg = cfgs(spec, wl)
    assert Q.gqa_splits(gcfg, spec.rows, spec.packed_width) == 2
    st = OracleState(wl, with_kv=False)
    rng = np.random.default_rng(43)
    packed_np = random_packed(rng, st.cfg, st.logical_positions,
                              full_rows=set(range(0, spec.rows, 2)))
    assert int(packed_np[:, -1].max()) > 2560
    out = torch.full_like(wl["q"], 3.0)
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")  # split partials and tickets
    Q.sparse_gqa(gcfg, wl["q"], wl["kv"], wl["block_table"], torch.from_numpy(packed_np).cuda(),
                 wl["token_to_req"], wl["gate"], out, ws)
    torch.cuda.synchronize()
    assert Q.check_errors() == 0
    got = f64(out)
    for row in (0, 1, 2, 3, rows_per, spec.rows // 2 + 1, spec.rows - 2, spec.rows - 1):
        n = int(packed_np[row, -1])
        req = int(st.token_to_req[row])
        want = oracle_gqa_row(st.q[row], wl["kv"], st.block_table[req], packed_np[row, :n],
                              spec.page, st.gate[row])
        ok, err = close_bf16(got[row], want)
        assert ok, f"row {row} (n={n}): max err {err:.3g}"


# ----------------------------------------------------------------- full chain
def _full_chain(spec, wl, st, step, rows=None, packed_ref=None, skip=False):
    """Compare a finished GPU step with the oracle's own chain on `rows`."""
    rows = range(spec.rows) if rows is None else rows
    got_packed = step.packed.cpu().numpy()
    got_out = f64(step.out)
    tie_rows = 0
    for row in rows:
        p = int(st.logical_positions[row])
        req = int(st.token_to_req[row])
        if skip:
            opack = packed_ref[row]
            np.testing.assert_array_equal(got_packed[row], opack)
        else:
            qrow = O.prep_query(st.cfg, st.projected_q[row], st.positions[row], st.cos_sin,
                                st.q_norm_w)
            scores, _, opack = O.select_row(st.cfg, qrow, st.ccache, st.cblock_table[req], p)
            ok, ndiff = selection_ok(st.cfg, got_packed[row], opack, scores, p)
            assert ok, f"{spec.name} row {row}: selection differs beyond the tie window"
            if ndiff:
                # a block inside the tie window went the other way: stage 4 is
                # still checked, on the selection the GPU made
                tie_rows += 1
                opack = got_packed[row]
        n = int(opack[-1])
        if st.kv is not None:
            want = O.sparse_gqa_row(st.q[row], st.kv, st.block_table[req], opack[:n], spec.page,
                                    st.gate[row], *st.kv_scales)
        else:
            want = oracle_gqa_row(st.q[row], step.wl["kv"], st.block_table[req], opack[:n],
                                  spec.page, st.gate[row], st.kv_scales)
        ok, err = close_bf16(got_out[row], want)
        assert ok, f"{spec.name} row {row}: output err {err:.3g}"
    return tie_rows


@pytest.mark.parametrize("name", list(MID))
def test_layer_step_full_chain(name):
    spec = MID[name]
    wl = W.make_workload(spec, device="cuda")
    st = OracleState(wl)
    step = Step(wl).run()
    st.compress()  # the oracle's stage 1 (caches now hold this step's groups)
    ties = _full_chain(spec, wl, st, step)
    assert ties <= max(1, spec.rows // 10)
    np.testing.assert_array_equal(f64(wl["ring"]).reshape(st.ring.shape), st.ring)


def test_skip_topk_reuses_selection_and_updates_caches():
    spec = MID["mid_mrope_h8"]
    wl = W.make_workload(spec, device="cuda")
    step = Step(wl).run()
    packed0 = step.packed.cpu().numpy().copy()
    st = OracleState(wl)  # caches after step 0
    nxt = W.make_workload(spec, device="cuda", step=1, with_caches=False)
    for k in ("projected_q", "raw_keys", "q", "gate"):
        wl.t[k].copy_(nxt[k])
        setattr(st, k, f64(nxt[k]).reshape(getattr(st, k).shape))
    step.packed.copy_(torch.from_numpy(packed0))
    step.run(skip_topk=True)
    st.compress()
    _full_chain(spec, wl, st, step, packed_ref=packed0, skip=True)
    np.testing.assert_array_equal(f64(wl["ring"]).reshape(st.ring.shape), st.ring)


def test_empty_batch_is_noop():
    spec = MID["tiny_bf16"]
    wl = W.make_workload(spec, device="cuda")
    cfg, gcfg = cfgs(spec, wl)
    a = Q.QsaStepArgs()
    a.rows, a.reqs = 0, 0
    a.packed = wl["q"].data_ptr()
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    Q.layer_step(cfg, gcfg, a, ws)


def test_out_of_range_pages_are_masked_and_counted():
    spec = MID["tiny_bf16"]
    wl = W.make_workload(spec, device="cuda")
    Q.check_errors()
    wl.t["block_table"][0, 0] = 10 ** 6  # no such KV block
    Step(wl).run()
    assert Q.check_errors() > 0
    assert Q.check_errors() == 0  # the word is cleared by the read


# ----------------------------------------------------------------- full size
def _sampled(name, nsample, seed=0):
    spec = W.named_spec(name)
    wl = W.make_workload(spec, device="cuda")
    st = OracleState(wl, with_kv=False)
    step = Step(wl).run()
    assert Q.check_errors() == 0
    # oracle stage 1 keys for every row (query prep only for sampled rows)
    O.compress_stage(st.cfg, projected_q=None, raw_keys=st.raw_keys, positions=st.positions,
                     cos_sin=st.cos_sin, q_norm_w=st.q_norm_w, k_norm_w=st.k_norm_w,
                     ring=st.ring, ring_pos=st.ring_pos, ring_block_table=st.ring_block_table,
                     token_to_req=st.token_to_req, query_start_loc=st.query_start_loc,
                     logical_positions=st.logical_positions, ccache=st.ccache,
                     compressed_slots=st.compressed_slots)
    rng = np.random.default_rng(seed)
    rows = np.arange(spec.rows) if spec.rows <= nsample else np.sort(
        rng.choice(spec.rows, size=nsample, replace=False))
    ties = _full_chain(spec, wl, st, step, rows=rows)
    # compressed keys written by the step
    slots = i64(wl["compressed_slots"])
    sl = slots[slots >= 0]
    got = f64(wl["ccache"]).reshape(-1, 128)[sl]
    ok, err = _close_idx(spec, got, st.ccache.reshape(-1, 128)[sl])
    assert ok, err
    return spec, step, ties, len(rows)


@pytest.mark.parametrize("name,nsample", [("decode_batch", 64), ("long_decode", 8),
                                          ("mtp_mrope", 128), ("chunked_prefill", 192)])
def test_full_size_sampled_rows(name, nsample):
    spec, step, ties, n = _sampled(name, nsample)
    assert ties <= max(2, n // 10), f"{ties} tie rows out of {n}"
    print(f"{name}: {n} rows checked, {ties} rows differ only inside the tie window")


def test_full_size_decode_batch_fp8_kv_cache():
    """The decode batch over the FP8-e4m3 main KV cache (static scales) at
    full size, in the launch configuration the bench times."""
    spec, step, ties, n = _sampled("decode_batch_fp8kv", 64)
    assert spec.kv_dtype == W.DTYPE_E4M3
    assert ties <= max(2, n // 10), f"{ties} tie rows out of {n}"


def test_full_size_decode_batch_with_main_prepare():
    """The decode batch with the main-attention prepare fused into stage 1,
    at full size: every row's q and gate, its K/V row in the cache, and the
    whole chain's output against the oracle (stage 4 reads the cache rows
    this step wrote, which are checked first)."""
    spec = W.named_spec("decode_batch_prepare")
    assert spec.main_prep and spec.kv_dtype == W.DTYPE_BF16
    wl = W.make_workload(spec, device="cuda")
    st = OracleState(wl, with_kv=False)
    step = Step(wl, main=True).run()
    assert Q.check_errors() == 0
    O.compress_stage(st.cfg, projected_q=None, raw_keys=st.raw_keys, positions=st.positions,
                     cos_sin=st.cos_sin, q_norm_w=st.q_norm_w, k_norm_w=st.k_norm_w,
                     ring=st.ring, ring_pos=st.ring_pos, ring_block_table=st.ring_block_table,
                     token_to_req=st.token_to_req, query_start_loc=st.query_start_loc,
                     logical_positions=st.logical_positions, ccache=st.ccache,
                     compressed_slots=st.compressed_slots)
    m = oracle_main(spec, wl)
    q = np.zeros((spec.rows, spec.hq, 128))
    gate = np.zeros_like(q)
    slots = wl["slot_mapping"].cpu().numpy()
    blk = torch.as_tensor(slots // spec.page, device="cuda")
    off = torch.as_tensor(slots % spec.page, device="cuda")
    got_rows = f64(wl["kv"][blk, :, off, :])  # [rows, Hkv, 2D]
    for row in range(spec.rows):
        q[row], gate[row], k, v = O.prepare_main_row(st.cfg, m["qkv"][row], st.positions[row],
                                                     st.cos_sin, m["q_norm_w"], m["k_norm_w"],
                                                     m["eps"], spec.hq, spec.hkv)
        ok, err = close_bf16(got_rows[row, :, :128], k)
        assert ok, f"K row of row {row}: {err}"
        np.testing.assert_array_equal(got_rows[row, :, 128:], v)
    ok, err = close_bf16(f64(wl["main_q_out"]), q)
    assert ok, f"q: {err}"
    np.testing.assert_array_equal(f64(wl["main_gate_out"]), gate)
    st.q, st.gate = q, gate
    ties = _full_chain(spec, wl, st, step)
    assert ties <= max(2, spec.rows // 10), f"{ties} tie rows"


def test_full_size_invariants_decode_batch():
    """Properties that hold for every row at full size: counts, causality,
    uniqueness, -1 padding."""
    spec = W.named_spec("decode_batch")
    wl = W.make_workload(spec, device="cuda")
    step = Step(wl).run()
    pk = step.packed.cpu().numpy()
    cfg = O.QsaConfig(n_heads=32, compress_ratio=4, token_topk=2048)
    for row, p in enumerate(i64(wl["logical_positions"])):
        n = pk[row, -1]
        assert n == O.expected_count(cfg, int(p))
        toks = pk[row, :n]
        assert toks.min() >= 0 and toks.max() <= p and len(np.unique(toks)) == n
        assert (pk[row, n:-1] == -1).all()
    assert np.isfinite(f64(step.out)).all()


def test_full_size_mtp_step0_then_three_skip_topk_steps():
    """The MTP verify workload with MRoPE as the pages run it: step 0 selects,
    steps 1-3 reuse step 0's packed buffer (skip_topk) with fresh indexer
    projections, raw keys, q and gate, while stage 1 keeps writing the
    compressed cache and the ring.  Every step's caches are compared with
    the oracle's own stage 1 over the same history, and the outputs of
    sampled rows with the oracle's stage 4 on the reused selection.
    Source: "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.skip_topk (later
    steps reuse the indices while the indexer cache is still updated)."""
    spec = W.named_spec("mtp_mrope")
    wl = W.make_workload(spec, device="cuda")
    st = OracleState(wl, with_kv=False)
    step = Step(wl).run()
    assert Q.check_errors() == 0
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(spec.rows, size=32, replace=False))
    st.compress()
    _full_chain(spec, wl, st, step, rows=rows)
    packed0 = step.packed.cpu().numpy().copy()
    slots = i64(wl["compressed_slots"])
    sl = slots[slots >= 0]
    for s in (1, 2, 3):
        nxt = W.make_workload(spec, device="cuda", step=s, with_caches=False)
        for k in ("projected_q", "raw_keys", "q", "gate"):
            wl.t[k].copy_(nxt[k])
            setattr(st, k, f64(nxt[k]).reshape(getattr(st, k).shape))
        step.run(skip_topk=True)
        assert Q.check_errors() == 0
        st.compress()
        np.testing.assert_array_equal(step.packed.cpu().numpy(), packed0)
        rows = np.sort(rng.choice(spec.rows, size=32, replace=False))
        _full_chain(spec, wl, st, step, rows=rows, packed_ref=packed0, skip=True)
        ok, err = _close_idx(spec, f64(wl["ccache"]).reshape(-1, 128)[sl],
                             st.ccache.reshape(-1, 128)[sl])
        assert ok, f"step {s}: compressed keys {err}"
        np.testing.assert_array_equal(f64(wl["ring"]).reshape(st.ring.shape), st.ring)
        np.testing.assert_array_equal(i64(wl["ring_pos"]).reshape(st.ring_pos.shape), st.ring_pos)


@pytest.mark.parametrize("rows,hkv", [(3, 4), (8, 8)])
def test_split_merge_launch_matches_oracle(rows, hkv):
    """Split-KV partials merged by a separate launch (the path taken when no
    merge tickets are given, as in qsa_sparse_gqa_noalloc) against the
    oracle's stage 4, with full, partial and empty selections."""
    spec = W.small_spec("merge", seed=40 + rows, contexts=[5000 + 1000 * i for i in range(rows)],
                        rows_per_req=[1] * rows, n_heads=8, index_dtype=BF, compress_ratio=4,
                        token_topk=2048, hq=8 * hkv, hkv=hkv, page=64)
    wl = W.make_workload(spec, device="cuda")
    _, gcfg = cfgs(spec, wl)
    assert Q.gqa_splits(gcfg, spec.rows, spec.packed_width) > 1
    st = OracleState(wl, with_kv=False)
    packed_np = random_packed(np.random.default_rng(rows), st.cfg, st.logical_positions,
                              full_rows={0})
    packed_np[-1, :] = -1
    packed_np[-1, -1] = 0
    out = torch.full_like(wl["q"], 3.0)
    Q.sparse_gqa_noalloc(gcfg, wl["q"], wl["kv"], wl["block_table"],
                         torch.from_numpy(packed_np).cuda(), wl["token_to_req"], wl["gate"], out)
    torch.cuda.synchronize()
    got = f64(out)
    for row in range(spec.rows):
        n = int(packed_np[row, -1])
        req = int(st.token_to_req[row])
        want = oracle_gqa_row(st.q[row], wl["kv"], st.block_table[req], packed_np[row, :n],
                              spec.page, st.gate[row])
        ok, err = close_bf16(got[row], want)
        assert ok, f"row {row} (n={n}): max err {err:.3g}"
    assert (got[-1] == 0).all()


def test_mtp_steps_equals_step_by_step_and_oracle():
    """qsa_mtp_steps (one call for a 4-step MTP draft: step 0 selects, steps
    1-3 reuse the packed buffer) gives bit for bit what four layer_step
    calls give, and both match the oracle step by step (caches after every
    step, outputs on the reused selection)."""
    from types import SimpleNamespace

    spec = MID["mid_mrope_h8"]
    wa = W.make_workload(spec, device="cuda")
    wb = wa.clone()
    st = OracleState(wa)
    cfg, gcfg = cfgs(spec, wa)
    mv = max_visible(spec)
    k = 4
    fresh = [W.make_workload(spec, device="cuda", step=s, with_caches=False) for s in range(k)]
    names = ("projected_q", "raw_keys", "q", "gate")

    def per_step(wl):
        ts = []
        for s in range(k):
            t = dict(wl.t)
            for n in names:
                t[n] = fresh[s][n]
            ts.append(t)
        return ts

    packed_a = torch.full((spec.rows, spec.packed_width), -7, dtype=torch.int32, device="cuda")
    packed_b = packed_a.clone()
    outs_a = [torch.full_like(wa["q"], 7.0) for _ in range(k)]
    outs_b = [torch.full_like(wa["q"], 7.0) for _ in range(k)]
    nbytes = Q.workspace_bytes(cfg, gcfg, spec.rows, spec.reqs, mv)
    ws_a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ta, tb = per_step(wa), per_step(wb)
    Q.mtp_steps(cfg, gcfg, [Q.step_args(ta[s], packed_a, outs_a[s], mv) for s in range(k)], ws_a)
    for s in range(k):
        Q.layer_step(cfg, gcfg, Q.step_args(tb[s], packed_b, outs_b[s], mv), ws_b,
                     skip_topk=s > 0)
    torch.cuda.synchronize()
    assert Q.check_errors() == 0
    assert torch.equal(packed_a, packed_b)
    for s in range(k):
        assert torch.equal(outs_a[s].view(torch.int16), outs_b[s].view(torch.int16)), s
    for n in ("ring", "ring_pos", "ccache"):
        assert torch.equal(wa[n], wb[n]), n
    # the oracle, step by step, on the same inputs
    for s in range(k):
        for n in names:
            setattr(st, n, f64(fresh[s][n]).reshape(getattr(st, n).shape))
        st.compress()  # the oracle's caches now hold step s's stage 1
        view = SimpleNamespace(packed=packed_a, out=outs_a[s], wl=wa)
        if s == 0:
            _full_chain(spec, wa, st, view)  # selection from step 0's caches
            packed0 = packed_a.cpu().numpy().copy()
        else:
            _full_chain(spec, wa, st, view, packed_ref=packed0, skip=True)
    np.testing.assert_array_equal(f64(wa["ring"]).reshape(st.ring.shape), st.ring)
    np.testing.assert_array_equal(i64(wa["ring_pos"]).reshape(st.ring_pos.shape), st.ring_pos)
    sl = i64(wa["compressed_slots"])
    sl = sl[sl >= 0]
    ok, err = _close_idx(spec, f64(wa["ccache"]).reshape(-1, 128)[sl], st.ccache.reshape(-1, 128)[sl])
    assert ok, err


# ----------------------------------------------------------------- main prepare
MAIN = {
    "mid_main_bf16": W.small_spec("mid_main_bf16", seed=30, contexts=(2000, 777, 64),
                                  rows_per_req=(2, 1, 3), n_heads=16, index_dtype=E4,
                                  compress_ratio=4, token_topk=256, hq=32, hkv=4, page=64,
                                  main_prep=True),
    "mid_main_fp8_mrope_g3": W.small_spec("mid_main_fp8_mrope_g3", seed=31, contexts=(3000, 700),
                                          rows_per_req=(4, 4), n_heads=8, index_dtype=BF,
                                          compress_ratio=4, token_topk=128,
                                          mrope_section=(8, 12, 12), image_span=64, hq=24, hkv=8,
                                          page=32, kv_dtype=E4, kv_scale=0.05, main_prep=True),
    "small_main_group16": W.small_spec("small_main_group16", seed=32, hq=32, hkv=2,
                                       main_prep=True),
}


def _oracle_prepare(spec, wl, st):
    """The oracle's main-attention prepare over every row: (q, gate) per row,
    with the rows' K/V written into st.kv (the stored values)."""
    m = oracle_main(spec, wl)
    q = np.zeros((spec.rows, spec.hq, 128))
    gate = np.zeros_like(q)
    for row in range(spec.rows):
        q[row], gate[row], k, v = O.prepare_main_row(st.cfg, m["qkv"][row], st.positions[row],
                                                     st.cos_sin, m["q_norm_w"], m["k_norm_w"],
                                                     m["eps"], spec.hq, spec.hkv)
        O.write_main_kv(st.kv, int(m["slot_mapping"][row]), k, v, spec.page, spec.kv_dtype,
                        *st.kv_scales)
    return q, gate


def _kv_rows_close(spec, got_kv, want_kv, slots):
    D = 128
    for slot in slots:
        blk, off = slot // spec.page, slot % spec.page
        g, w = got_kv[blk, :, off], want_kv[blk, :, off]
        if spec.kv_dtype == E4:
            ok, err = close_e4m3(g, w)
        else:
            ok, err = close_bf16(g[:, :D], w[:, :D])
            ok = ok and np.array_equal(g[:, D:], w[:, D:])  # v is copied
        assert ok, f"KV row of slot {slot}: {err}"


@pytest.mark.parametrize("name", list(MAIN))
def test_main_prepare_matches_oracle(name):
    """qsa_main_prepare alone: q (bf16), the gate (copied) and the rows' K/V
    in the cache (bf16 or e4m3), the rest of the cache untouched."""
    spec = MAIN[name]
    wl = W.make_workload(spec, device="cuda")
    st = OracleState(wl)
    cfg, gcfg = cfgs(spec, wl)
    Q.main_prepare(cfg, gcfg, Q.main_prep(wl.t, spec.eps), wl["positions"], wl["cos_sin"])
    torch.cuda.synchronize()
    assert Q.check_errors() == 0
    q, gate = _oracle_prepare(spec, wl, st)
    ok, err = close_bf16(f64(wl["main_q_out"]), q)
    assert ok, f"q: {err}"
    np.testing.assert_array_equal(f64(wl["main_gate_out"]), gate)
    got_kv = f64(wl["kv"])
    slots = wl["slot_mapping"].cpu().numpy()
    _kv_rows_close(spec, got_kv, st.kv, slots)
    mask = np.ones(got_kv.shape[:3], dtype=bool)
    for slot in slots:
        mask[slot // spec.page, :, slot % spec.page] = False
    np.testing.assert_array_equal(got_kv[mask], st.kv[mask])


@pytest.mark.parametrize("name", list(MAIN))
def test_layer_step_with_fused_main_prepare(name):
    """The layer step with the main-attention prepare fused into stage 1:
    stage 4 attends with the prepared q and gate over the cache that holds
    this step's own K/V rows (selected as the newest tokens)."""
    spec = MAIN[name]
    wl = W.make_workload(spec, device="cuda")
    st = OracleState(wl)
    step = Step(wl, main=True).run()
    assert Q.check_errors() == 0
    st.compress()
    st.q, st.gate = _oracle_prepare(spec, wl, st)
    _full_chain(spec, wl, st, step)
    _kv_rows_close(spec, f64(wl["kv"]), st.kv, wl["slot_mapping"].cpu().numpy())
