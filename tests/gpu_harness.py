"""Helpers for the GPU parity tests: configs from workloads, the C-ABI calls
with their buffers, and oracle evaluation of single rows (test
infrastructure)."""

from __future__ import annotations

import numpy as np
import torch

from learned_sparse_attention_gb300 import qsa as Q
from learned_sparse_attention_gb300 import workloads as W
from oracle import qsa_oracle as O
from tests.oracle_io import f64


def cfgs(spec, wl):
    cfg = Q.make_cfg(spec.n_heads, spec.compress_ratio, spec.token_topk, spec.index_dtype,
                     spec.cpage, wl["cos_sin"].shape[0], state_size=spec.S,
                     mrope_section=spec.mrope_section, eps=spec.eps)
    gcfg = Q.make_gqa_cfg(spec.hq, spec.hkv, spec.page, wl["kv"].shape[0], kv_dtype=spec.kv_dtype,
                          k_scale=kv_scales(spec)[0], v_scale=kv_scales(spec)[1])
    return cfg, gcfg


def oracle_main(spec, wl):
    """The main-attention prepare's inputs as the oracle takes them (host
    copies of the workload's generator data)."""
    return dict(qkv=f64(wl["main_qkv"]), q_norm_w=f64(wl["main_q_norm_w"]),
                k_norm_w=f64(wl["main_k_norm_w"]), eps=spec.eps,
                slot_mapping=wl["slot_mapping"].cpu().numpy(), kv_dtype=spec.kv_dtype)


def kv_scales(spec):
    """(k_scale, v_scale) of the workload's main KV cache (1, 1 for bf16)."""
    return (spec.kv_scale, spec.kv_scale) if spec.kv_dtype == W.DTYPE_E4M3 else (1.0, 1.0)


def max_visible(spec) -> int:
    return max(spec.contexts) // spec.compress_ratio


def idx_dtype(spec):
    return torch.uint8 if spec.index_dtype == W.DTYPE_E4M3 else torch.bfloat16


class Step:
    """One GPU layer step of a workload through the C ABI."""

    def __init__(self, wl, gate=True, main=False):
        self.wl = wl
        s = wl.spec
        dev = wl["q"].device
        self.cfg, self.gcfg = cfgs(s, wl)
        self.mv = max_visible(s)
        self.packed = torch.full((s.rows, s.packed_width), -7, dtype=torch.int32, device=dev)
        self.out = torch.full_like(wl["q"], 7.0)
        nbytes = Q.workspace_bytes(self.cfg, self.gcfg, s.rows, s.reqs, self.mv)
        assert nbytes > 0
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.gate = gate
        self.main = main  # fuse the main-attention prepare into stage 1

    def run(self, skip_topk=False):
        t = dict(self.wl.t)
        if not self.gate:
            t["gate"] = None
        m = Q.main_prep(t, self.wl.spec.eps) if self.main else None
        Q.layer_step(self.cfg, self.gcfg, Q.step_args(t, self.packed, self.out, self.mv, main=m),
                     self.ws, skip_topk=skip_topk)
        torch.cuda.synchronize()
        return self


def gather_token_kv(kv: torch.Tensor, block_row, tokens, page: int) -> np.ndarray:
    """K|V rows of the given request-relative tokens: [n, Hkv, 1, 2D] float64
    (input marshalling for the oracle: a device gather of generator data)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    if len(tokens) == 0:
        return np.zeros((0, kv.shape[1], 1, kv.shape[3]))
    blocks = torch.as_tensor(np.asarray(block_row)[tokens // page], device=kv.device)
    offs = torch.as_tensor(tokens % page, device=kv.device)
    rows = kv[blocks, :, offs, :]  # [n, Hkv, 2D]
    return f64(rows)[:, :, None, :]


def oracle_gqa_row(q_row, kv: torch.Tensor, block_row, tokens, page, gate_row, scales=(1.0, 1.0)):
    """Oracle stage 4 on one row, with the KV rows of its tokens gathered
    from the device cache and re-indexed as one-token pages."""
    compact = gather_token_kv(kv, block_row, tokens, page)
    n = len(tokens)
    return O.sparse_gqa_row(q_row, compact, np.arange(n), np.arange(n), 1, gate_row,
                            k_scale=scales[0], v_scale=scales[1])


def random_packed(rng, cfg: O.QsaConfig, logical, full_rows=()):
    """Seeded valid packed rows: a random subset of tokens 0..p of at most
    output_width entries in random order, -1 padded, count last."""
    Wd = cfg.output_width
    out = np.full((len(logical), Wd + 1), -1, dtype=np.int32)
    for i, p in enumerate(logical):
        p = int(p)
        if i in full_rows:
            n = min(Wd, p + 1)
        else:
            n = int(rng.integers(0, min(Wd, p + 1) + 1))
        toks = rng.choice(p + 1, size=n, replace=False) if n else np.zeros(0, dtype=np.int64)
        out[i, :n] = toks
        out[i, Wd] = n
    return out
