"""The fused qkv + indexer projection GEMM (tcgen05) against the oracle on
GB300, from a ragged tiny case to the decode and prefill shapes of a
32q/4kv x 128 layer with a 32-head indexer over hidden 4096 (sampled rows)."""

import numpy as np
import pytest
import torch

from learned_sparse_attention_gb300 import qsa as Q
from oracle import qsa_oracle as O
from tests.oracle_io import f64
from tests.parity import close_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,hidden,qc,iq,ik", [
    (5, 64, 100, 60, 28),          # ragged everything, one K slice
    (64, 512, 1152, 512, 128),     # decode-sized tile, 8 K slices
    (40, 960, 300, 200, 28),       # 15 K slices, ragged columns in every buffer
    (300, 1024, 640, 256, 128),    # two N tiles of 256 rows, a ragged one
    (64, 4096, 9216, 4096, 128),   # decode batch of the layer
    (2048, 4096, 9216, 4096, 128), # a prefill slice of the layer
])
def test_projection_matches_oracle(rows, hidden, qc, iq, ik):
    g = torch.Generator(device="cuda").manual_seed(rows + hidden)
    x = torch.randn((rows, hidden), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((qc + iq + ik, hidden), generator=g, device="cuda") / hidden ** 0.5).to(torch.bfloat16)
    qkv = torch.full((rows, qc), 7.0, dtype=torch.bfloat16, device="cuda")
    pq = torch.full((rows, iq), 7.0, dtype=torch.bfloat16, device="cuda")
    rk = torch.full((rows, ik), 7.0, dtype=torch.bfloat16, device="cuda")
    Q.qkv_index_proj(x, w, qkv, pq, rk)
    torch.cuda.synchronize()
    assert Q.check_errors() == 0
    rng = np.random.default_rng(rows)
    sample = np.arange(rows) if rows <= 64 else np.sort(rng.choice(rows, 24, replace=False))
    sample = np.unique(np.concatenate([sample, [0, rows - 1]]))
    want = O.qkv_index_projection(f64(x[torch.as_tensor(sample, device="cuda")]), f64(w), qc, iq)
    for got_t, want_a, name in zip((qkv, pq, rk), want, ("qkv", "projected_q", "raw_keys")):
        got = f64(got_t[torch.as_tensor(sample, device="cuda")])
        ok, err = close_bf16(got, want_a)
        assert ok, f"{name}: max err {err:.3g}"
