"""Marshalling between seeded workloads (torch tensors) and the oracle
(float64 numpy arrays).  Test infrastructure: no QSA arithmetic here."""

from __future__ import annotations

import numpy as np
import torch

from oracle import qsa_oracle as O


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 / fp32 / e4m3(uint8 storage) tensor."""
    t = t.detach().cpu()
    if t.dtype == torch.uint8:
        return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return t.to(torch.float64).numpy()


def i64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.int64).numpy()


def oracle_cfg(spec) -> O.QsaConfig:
    return O.QsaConfig(n_heads=spec.n_heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim,
                       compress_ratio=spec.compress_ratio, token_topk=spec.token_topk,
                       eps=spec.eps, index_dtype=spec.index_dtype,
                       mrope_section=spec.mrope_section, state_size=spec.S, cpage=spec.cpage)


class OracleState:
    """Host float64 copy of a workload's inputs and caches."""

    def __init__(self, wl, with_kv=True):
        s = wl.spec
        self.spec = s
        self.cfg = oracle_cfg(s)
        t = wl.t
        D = s.head_dim
        self.projected_q = f64(t["projected_q"]).reshape(s.rows, s.n_heads, D)
        self.raw_keys = f64(t["raw_keys"]).reshape(s.rows, D)
        self.positions = i64(t["positions"]).reshape(s.rows, 3)
        self.cos_sin = f64(t["cos_sin"])
        self.q_norm_w = f64(t["q_norm_w"])
        self.k_norm_w = f64(t["k_norm_w"])
        self.ring = f64(t["ring"]).reshape(t["ring"].shape[0], s.S, D)
        self.ring_pos = i64(t["ring_pos"]).reshape(-1, s.S, 3) if "ring_pos" in t else None
        self.ring_block_table = i64(t["ring_block_table"])
        self.token_to_req = i64(t["token_to_req"])
        self.query_start_loc = i64(t["query_start_loc"])
        self.logical_positions = i64(t["logical_positions"])
        self.ccache = f64(t["ccache"]).reshape(t["ccache"].shape[0], s.cpage, D)
        self.compressed_slots = i64(t["compressed_slots"])
        self.cblock_table = i64(t["cblock_table"])
        self.block_table = i64(t["block_table"])
        self.q = f64(t["q"])
        self.gate = f64(t["gate"])
        self.kv = f64(t["kv"]) if with_kv else None  # e4m3 caches: the stored values
        self.kv_scales = ((s.kv_scale, s.kv_scale) if getattr(s, "kv_dtype", 0) == 1
                          else (1.0, 1.0))

    def step(self, skip_topk=False, packed=None, rows_to_score=None, gate=True, main=None):
        return O.layer_step(
            self.cfg, projected_q=self.projected_q, raw_keys=self.raw_keys,
            positions=self.positions, cos_sin=self.cos_sin, q_norm_w=self.q_norm_w,
            k_norm_w=self.k_norm_w, ring=self.ring, ring_pos=self.ring_pos,
            ring_block_table=self.ring_block_table, token_to_req=self.token_to_req,
            query_start_loc=self.query_start_loc, logical_positions=self.logical_positions,
            ccache=self.ccache, compressed_slots=self.compressed_slots,
            cblock_table=self.cblock_table, q=self.q, kv=self.kv,
            block_table=self.block_table, page=self.spec.page,
            gate=self.gate if gate else None, packed=packed, skip_topk=skip_topk,
            rows_to_score=rows_to_score, k_scale=self.kv_scales[0], v_scale=self.kv_scales[1],
            main=main)

    def compress(self):
        return O.compress_stage(
            self.cfg, projected_q=self.projected_q, raw_keys=self.raw_keys,
            positions=self.positions, cos_sin=self.cos_sin, q_norm_w=self.q_norm_w,
            k_norm_w=self.k_norm_w, ring=self.ring, ring_pos=self.ring_pos,
            ring_block_table=self.ring_block_table, token_to_req=self.token_to_req,
            query_start_loc=self.query_start_loc, logical_positions=self.logical_positions,
            ccache=self.ccache, compressed_slots=self.compressed_slots)
