"""Seeded synthetic QSA workloads.

This module holds only input generation: shapes, request metadata (token to
request maps, logical positions, block tables as seeded page permutations,
compressed and ring slots) and random fills of activations and caches.  It
contains none of the QSA arithmetic and is shared by the tests, the bench
and the smoke check.

Workload recipe (all values seeded):
* activations (indexer projections, raw keys, main Q, gate) ~ N(0, 1), bf16;
* RMSNorm weights ~ N(0, 0.1), bf16;
* main paged K/V cache ~ N(0, 1), bf16, layout [blocks, Hkv, page, 2*D]; the
  FP8 variant stores e4m3(x / kv_scale) of the same values (kv_scale = 1/16
  for K and V: the stored values span about +-64, inside e4m3's +-448);
* compressed-key cache ~ N(0, 1) rounded to the indexer dtype (e4m3 or
  bf16), layout [cpages, cpage, 1, D] with cpage = page / compress_ratio;
* compressor-state ring ~ N(0, 1), bf16, layout [ring_blocks, S, 1, D]
  with S = 2 * compress_ratio, one ring block per request;
* block tables are seeded random permutations of the physical pages, so
  gathers are not sequential;
* RoPE cos/sin table: theta = 10000, fp32, [max_pos, rotary_dim] with cos
  in the first half and sin in the second;
* with the main-attention prepare: the qkv projection rows ~ N(0, 1) bf16
  ([rows, (2 Hq + 2 Hkv) * 128]), its q/k norm weights ~ N(0, 0.1), and the
  slot of each row's own token (its block-table page and offset);
* the "peaked" long-context workload picks a seeded 1% of each request's
  token positions and scales by 8 the raw indexer key, the main-cache K row
  and the compressed key of the group holding each of them (the prefix of
  the compressed cache is a seeded fill, not stage 1 run over the history,
  so the peak is placed there directly: the index scores of those groups
  are then about 8 times the others');
* the MTP/MRoPE workload gives each request one 1024-token image span laid
  out as a 32x32 (H, W) grid at fixed T; text tokens have T = H = W = t.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

DTYPE_BF16 = 0
DTYPE_E4M3 = 1


@dataclass
class WorkloadSpec:
    name: str
    seed: int
    contexts: list            # per request: final context length L (incl. this step's rows)
    rows_per_req: list        # per request: query rows in this step (last positions)
    n_heads: int = 32         # indexer heads H_i
    head_dim: int = 128
    rotary_dim: int = 64
    compress_ratio: int = 4
    token_topk: int = 2048
    index_dtype: int = DTYPE_E4M3
    mrope_section: tuple = (0, 0, 0)
    hq: int = 32
    hkv: int = 4
    page: int = 64
    eps: float = 1e-6
    peak_frac: float = 0.0    # fraction of positions scaled x8 (raw key and main K)
    image_span: int = 0       # MRoPE image-span length per request (0 = text only)
    mtp_steps: int = 1        # steps 1.. reuse step 0's selection (skip_topk)
    state_size: int = 0       # 0 -> 2 * compress_ratio
    main_prep: bool = False   # inputs of the fused main-attention prepare (qkv projection, slots)
    kv_dtype: int = DTYPE_BF16  # main KV cache: bf16, or e4m3 with a static scale
    kv_scale: float = 1.0 / 16  # e4m3 cache: stored value = e4m3(x / kv_scale), K and V alike

    @property
    def cpage(self) -> int:
        return self.page // self.compress_ratio

    @property
    def S(self) -> int:
        return self.state_size or 2 * self.compress_ratio

    @property
    def rows(self) -> int:
        return int(sum(self.rows_per_req))

    @property
    def reqs(self) -> int:
        return len(self.contexts)

    @property
    def block_topk(self) -> int:
        return self.token_topk // self.compress_ratio

    @property
    def packed_width(self) -> int:
        return self.token_topk + self.compress_ratio - 1 + 1


def _decode_contexts(seed: int) -> list:
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(8192, 32768, size=64, endpoint=True)]


def named_spec(name: str) -> WorkloadSpec:
    """The five named workloads (the pages' model shapes with synthetic data)."""
    if name == "tiny_bf16":
        return WorkloadSpec(name, 0, [256, 300], [1, 1], n_heads=8, index_dtype=DTYPE_BF16,
                            compress_ratio=4, token_topk=64, hq=8, hkv=1, page=16)
    if name == "decode_batch":
        return WorkloadSpec(name, 1, _decode_contexts(1), [1] * 64)
    if name == "chunked_prefill":
        return WorkloadSpec(name, 2, [32768 + 16384], [16384])
    if name == "long_decode":
        return WorkloadSpec(name, 3, [131072] * 8, [1] * 8, compress_ratio=8, token_topk=4096,
                            hq=64, hkv=8, peak_frac=0.01)
    if name == "mtp_mrope":
        return WorkloadSpec(name, 4, [65536] * 32, [4] * 32, index_dtype=DTYPE_BF16,
                            mrope_section=(8, 12, 12), image_span=1024, mtp_steps=4)
    if name == "decode_batch_fp8kv":  # the decode batch over an FP8-e4m3 main KV cache
        return WorkloadSpec(name, 1, _decode_contexts(1), [1] * 64, kv_dtype=DTYPE_E4M3)
    if name == "decode_batch_prepare":  # the decode batch with the fused main-attention prepare
        return WorkloadSpec(name, 1, _decode_contexts(1), [1] * 64, main_prep=True)
    raise KeyError(name)


NAMED = ("tiny_bf16", "decode_batch", "chunked_prefill", "long_decode", "mtp_mrope",
         "decode_batch_fp8kv", "decode_batch_prepare")


def rope_cos_sin(max_pos: int, rotary_dim: int, theta: float = 10000.0) -> torch.Tensor:
    """Caller-side RoPE table [max_pos, rotary_dim] fp32: cos | sin halves."""
    half = rotary_dim // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / rotary_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))


def _positions3(spec: WorkloadSpec, req_image_start: int, t: np.ndarray) -> np.ndarray:
    """3-D (T, H, W) positions of logical tokens t of one request."""
    t = np.asarray(t, dtype=np.int64)
    pos = np.stack([t, t, t], axis=-1)
    if spec.image_span and req_image_start >= 0:
        a = req_image_start
        inside = (t >= a) & (t < a + spec.image_span)
        j = t - a
        side = int(math.isqrt(spec.image_span))
        pos[inside, 0] = a
        pos[inside, 1] = a + j[inside] // side
        pos[inside, 2] = a + j[inside] % side
    return pos


@dataclass
class Workload:
    spec: WorkloadSpec
    t: dict = field(default_factory=dict)   # name -> torch tensor
    image_start: list = field(default_factory=list)

    def to(self, device) -> "Workload":
        return Workload(self.spec, {k: v.to(device) for k, v in self.t.items()}, list(self.image_start))

    def clone(self) -> "Workload":
        return Workload(self.spec, {k: v.clone() for k, v in self.t.items()}, list(self.image_start))

    def __getitem__(self, k):
        return self.t[k]


def _randn(gen, shape, device, dtype=torch.bfloat16, std=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def make_workload(spec: WorkloadSpec, device="cpu", step: int = 0, with_caches: bool = True,
                  with_kv: bool = True) -> Workload:
    """Build every input of one layer step.  Metadata and small tensors come
    from a CPU generator seeded by (seed, step); the large caches from a
    generator on ``device`` seeded by seed (so they do not depend on step).
    """
    rng = np.random.default_rng([spec.seed, 17])
    r = spec.compress_ratio
    reqs, rows = spec.reqs, spec.rows
    D = spec.head_dim

    token_to_req = np.repeat(np.arange(reqs), spec.rows_per_req).astype(np.int32)
    qsl = np.zeros(reqs + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(spec.rows_per_req)
    logical = np.concatenate([np.arange(L - n, L) for L, n in zip(spec.contexts, spec.rows_per_req)]
                             ).astype(np.int32)

    # Main KV blocks: ceil(L / page) per request, a seeded permutation of the pool.
    kv_need = [-(-L // spec.page) for L in spec.contexts]
    n_kv_blocks = int(sum(kv_need))
    perm = rng.permutation(n_kv_blocks).astype(np.int32)
    bt_stride = max(kv_need)
    block_table = np.zeros((reqs, bt_stride), dtype=np.int32)
    o = 0
    for i, n in enumerate(kv_need):
        block_table[i, :n] = perm[o:o + n]
        o += n

    # Compressed pages: ceil(V_final / cpage) per request (at least 1).
    c_need = [max(1, -(-(L // r) // spec.cpage)) for L in spec.contexts]
    n_cpages = int(sum(c_need))
    cperm = rng.permutation(n_cpages).astype(np.int32)
    cbt_stride = max(c_need)
    cblock_table = np.zeros((reqs, cbt_stride), dtype=np.int32)
    o = 0
    for i, n in enumerate(c_need):
        cblock_table[i, :n] = cperm[o:o + n]
        o += n

    # One ring block per request.
    ring_block_table = rng.permutation(reqs).astype(np.int32).reshape(reqs, 1)

    # Compressed slot of the group each row completes (-1 when none).
    slots = np.full(rows, -1, dtype=np.int64)
    for row in range(rows):
        p = int(logical[row])
        if (p + 1) % r == 0:
            g = (p + 1) // r - 1
            req = int(token_to_req[row])
            slots[row] = int(cblock_table[req, g // spec.cpage]) * spec.cpage + g % spec.cpage

    image_start = []
    for L in spec.contexts:
        if spec.image_span and L > 2 * spec.image_span + 16:
            image_start.append(int(rng.integers(0, L - 2 * spec.image_span)))
        else:
            image_start.append(-1)
    positions = np.zeros((rows, 1, 3), dtype=np.int64)
    for row in range(rows):
        req = int(token_to_req[row])
        positions[row, 0] = _positions3(spec, image_start[req], np.array([logical[row]]))[0]
    max_pos = int(max(spec.contexts)) + 1

    S = spec.S
    ring_pos = None
    if any(spec.mrope_section):
        ring_pos = np.zeros((reqs, S, 1, 3), dtype=np.int64)
        for req in range(reqs):
            first = int(spec.contexts[req] - spec.rows_per_req[req])
            # The ring holds tokens first-S .. first-1 at slot t mod S.
            ts = np.arange(max(0, first - S), first)
            if len(ts):
                rb = int(ring_block_table[req, 0])
                ring_pos[rb, ts % S, 0] = _positions3(spec, image_start[req], ts)

    g = torch.Generator(device="cpu").manual_seed(spec.seed * 1000 + step)
    t = {}
    t["token_to_req"] = torch.from_numpy(token_to_req)
    t["query_start_loc"] = torch.from_numpy(qsl)
    t["logical_positions"] = torch.from_numpy(logical)
    t["positions"] = torch.from_numpy(positions)
    t["compressed_slots"] = torch.from_numpy(slots)
    t["block_table"] = torch.from_numpy(block_table)
    t["cblock_table"] = torch.from_numpy(cblock_table)
    t["ring_block_table"] = torch.from_numpy(ring_block_table)
    t["projected_q"] = _randn(g, (rows, spec.n_heads * D), "cpu")
    t["raw_keys"] = _randn(g, (rows, 1, D), "cpu")
    t["q"] = _randn(g, (rows, spec.hq, D), "cpu")
    t["gate"] = _randn(g, (rows, spec.hq, D), "cpu")
    gw = torch.Generator(device="cpu").manual_seed(spec.seed * 1000 + 999)
    t["q_norm_w"] = _randn(gw, (D,), "cpu", std=0.1)
    t["k_norm_w"] = _randn(gw, (D,), "cpu", std=0.1)
    t["cos_sin"] = rope_cos_sin(max_pos, spec.rotary_dim)
    t["ring"] = _randn(gw, (reqs, S, 1, D), "cpu")
    if ring_pos is not None:
        t["ring_pos"] = torch.from_numpy(ring_pos)

    if spec.main_prep:
        gm = torch.Generator(device="cpu").manual_seed(spec.seed * 1000 + 500 + step)
        t["main_qkv"] = _randn(gm, (rows, (2 * spec.hq + 2 * spec.hkv) * D), "cpu")
        gw2 = torch.Generator(device="cpu").manual_seed(spec.seed * 1000 + 501)
        t["main_q_norm_w"] = _randn(gw2, (D,), "cpu", std=0.1)
        t["main_k_norm_w"] = _randn(gw2, (D,), "cpu", std=0.1)
        slot_map = np.array([int(block_table[int(token_to_req[r]), int(logical[r]) // spec.page])
                             * spec.page + int(logical[r]) % spec.page for r in range(rows)],
                            dtype=np.int64)
        t["slot_mapping"] = torch.from_numpy(slot_map)
        t["main_q_out"] = torch.zeros((rows, spec.hq, D), dtype=torch.bfloat16)
        t["main_gate_out"] = torch.zeros((rows, spec.hq, D), dtype=torch.bfloat16)
    dev = torch.device(device)
    if not with_caches:
        t = {k: v.to(dev) for k, v in t.items() if k != "ring"}
        return Workload(spec, t, image_start)
    gd = torch.Generator(device=dev).manual_seed(spec.seed * 1000 + 7)
    # without the main KV cache (index-only studies) a one-block stand-in keeps the keys valid
    t["kv"] = _randn(gd, (n_kv_blocks if with_kv else 1, spec.hkv, spec.page, 2 * D), dev)
    cc = torch.randn((n_cpages, spec.cpage, 1, D), generator=gd, device=dev, dtype=torch.float32)
    peaks = []  # per request: the peaked token positions
    if spec.peak_frac > 0:
        gp = np.random.default_rng([spec.seed, 99])
        for req in range(reqs):
            L = spec.contexts[req]
            npk = max(1, int(round(spec.peak_frac * L)))
            peaks.append(np.sort(gp.choice(L, size=npk, replace=False)))
        # compressed keys of the groups holding a peaked token
        for req, tok in enumerate(peaks):
            grp = np.unique(tok // r)
            flat = cblock_table[req, grp // spec.cpage].astype(np.int64) * spec.cpage + grp % spec.cpage
            idx = torch.from_numpy(flat).to(dev)
            ccf = cc.view(-1, D)
            ccf[idx] = ccf[idx] * 8
    if spec.index_dtype == DTYPE_E4M3:
        t["ccache"] = cc.to(torch.float8_e4m3fn).view(torch.uint8)
    else:
        t["ccache"] = cc.to(torch.bfloat16)

    if spec.peak_frac > 0 and with_kv:
        assert spec.kv_dtype == DTYPE_BF16, "peaked positions are placed in a bf16 cache"
        for req in range(reqs):
            tok = peaks[req]
            L = spec.contexts[req]
            blk = torch.from_numpy(block_table[req, tok // spec.page].astype(np.int64)).to(dev)
            off = torch.from_numpy((tok % spec.page).astype(np.int64)).to(dev)
            kv = t["kv"]
            kv[blk, :, off, :D] = kv[blk, :, off, :D] * 8
            peaked = set(int(x) for x in tok)
            # this step's raw keys at peaked positions
            for row in range(qsl[req], qsl[req + 1]):
                if int(logical[row]) in peaked:
                    t["raw_keys"][row] *= 8
            # ring entries holding peaked tokens
            firstpos = int(L - spec.rows_per_req[req])
            rb = int(ring_block_table[req, 0])
            for tt in range(max(0, firstpos - S), firstpos):
                if tt in peaked:
                    t["ring"][rb, tt % S] *= 8
    if spec.kv_dtype == DTYPE_E4M3:
        # the same N(0, 1) values, stored as e4m3(x / kv_scale) (all inside +-448)
        kv = t["kv"]
        q8 = torch.empty(kv.shape, dtype=torch.uint8, device=kv.device)
        for b0 in range(0, kv.shape[0], 4096):  # bounded temporaries
            x = kv[b0:b0 + 4096].float() / spec.kv_scale
            q8[b0:b0 + 4096] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        t["kv"] = q8
    t = {k: (v.to(dev) if v.device != dev else v) for k, v in t.items()}
    return Workload(spec, t, image_start)


def small_spec(name="small", seed=5, contexts=(37, 64, 301, 5), rows_per_req=(1, 3, 2, 1),
               **kw) -> WorkloadSpec:
    """A small mixed case: several requests, ragged lengths, multi-row steps."""
    base = dict(n_heads=8, index_dtype=DTYPE_BF16, compress_ratio=4, token_topk=64,
                hq=16, hkv=2, page=16)
    base.update(kw)
    return WorkloadSpec(name, seed, list(contexts), list(rows_per_req), **base)
