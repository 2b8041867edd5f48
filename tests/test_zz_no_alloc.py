"""qsa_sparse_gqa_noalloc on GB300: the sparse GQA stage for callers that are
not allowed to allocate device memory where attention runs (a frozen
allocator, a pool owned by someone else, a plugin host that only hands over
the call's tensors).  Its split-KV scratch lives in a fixed array inside the
library, so the caller passes only inputs and outputs.

Checked against qsa_sparse_gqa (same kernels, caller workspace) on two calls
in a row with different inputs, so a stale scratch from the first call would
show in the second.  This file is collected last; it passes alone in a fresh
process and after the other GPU tests."""

import numpy as np
import pytest
import torch

from learned_sparse_attention_gb300 import qsa as Q
from learned_sparse_attention_gb300 import workloads as W
from tests.gpu_harness import cfgs, random_packed
from tests.oracle_io import OracleState, f64
from tests.parity import close_bf16

pytestmark = pytest.mark.gpu


def _case(rows, hkv, seed, ratio=4, topk=2048, contexts=None):
    contexts = contexts or [3000 + 997 * i for i in range(rows)]
    spec = W.small_spec("noalloc", seed=seed, contexts=contexts,
                        rows_per_req=[1] * rows, n_heads=8, index_dtype=W.DTYPE_BF16,
                        compress_ratio=ratio, token_topk=topk, hq=8 * hkv, hkv=hkv, page=64)
    wl = W.make_workload(spec, device="cuda")
    cfg, gcfg = cfgs(spec, wl)
    return spec, wl, cfg, gcfg


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    spec, wl, cfg, gcfg = _case(rows=8, hkv=4, seed=31)
    # 8 rows x 4 KV heads: few CTAs, so split-KV (and its scratch) is in use
    assert Q.gqa_splits(gcfg, spec.rows, spec.packed_width) > 1
    st = OracleState(wl, with_kv=False)
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((1, 2)):
        rng = np.random.default_rng(seed)
        packed = torch.from_numpy(random_packed(rng, st.cfg, st.logical_positions,
                                                full_rows={0, 3})).cuda()
        if call == 1:
            wl.t["q"].mul_(-1.5)  # different inputs on the second call
        ref = torch.empty_like(wl["q"])
        got = torch.full_like(wl["q"], 5.0)
        Q.sparse_gqa(gcfg, wl["q"], wl["kv"], wl["block_table"], packed, wl["token_to_req"],
                     wl["gate"], ref, ws)
        Q.sparse_gqa_noalloc(gcfg, wl["q"], wl["kv"], wl["block_table"], packed,
                             wl["token_to_req"], wl["gate"], got)
        torch.cuda.synchronize()
        ok, err = close_bf16(f64(got), f64(ref))
        assert ok, f"call {call}: max |noalloc - workspace| = {err:.3g}"
    assert Q.check_errors() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 100 rows x 8 KV heads with 4103-token selections take two splits:
    # 2 * 100 * 64 * 128 fp32 partials = 6.6 MB > 4 MiB.  Every row is empty,
    # so nothing would be read even if the call were (wrongly) launched.
    spec, wl, cfg, gcfg = _case(rows=100, hkv=8, seed=32, ratio=8, topk=4096,
                                contexts=[4200] * 100)
    assert Q.gqa_splits(gcfg, spec.rows, spec.packed_width) == 2
    packed = torch.full((spec.rows, spec.packed_width), -1, dtype=torch.int32, device="cuda")
    packed[:, -1] = 0
    out = torch.empty_like(wl["q"])
    with pytest.raises(Q.QsaError) as e:
        Q.sparse_gqa_noalloc(gcfg, wl["q"], wl["kv"], wl["block_table"], packed,
                             wl["token_to_req"], wl["gate"], out)
    assert e.value.status == 5  # QSA_ERR_WORKSPACE
