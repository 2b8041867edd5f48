"""QSA oracle: a plain, slow, float64 CPU restatement of the QSA layer step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library and
imports nothing from the package.

Sources (web pages, cited by page title and symbol):

* "vllm.models.qwen4_exp.nvidia.qsa" (vLLM PR docs) -- ``QSAIndexer``:
  ``output_width`` / ``packed_output_width`` properties, ``forward`` and its
  "Unfused reference path"; ``Qwen4ExpQSAImpl.forward``.
* "vllm/models/qwen4_exp/nvidia/indexer_qsa.py" (fork page) -- ``apply_qsa_rope``
  and ``_supports_fused_pre_indexer``.
* "vllm.models.qwen4_exp.nvidia.ops.qsa" (vLLM PR docs) --
  ``qsa_compress_groups_with_ratio``, ``qsa_sparse_paged_attention``,
  ``qsa_store_cache_rows``.
* "0002-qwen4_exp-FP8-E4M3-KV-reader-for-QSA..." patch page --
  ``_qsa_sparse_paged_gqa_splitk_kernel`` (score scale, masking, softmax,
  normalisation and gate epilogue).

All arithmetic is float64.  Values are rounded to bf16 / e4m3 only where the
readings below say so, each once.  Readings of points the pages leave open:

R1  pooling operator: arithmetic mean of the ``compress_ratio`` raw keys.
R2  one rounding: query prep and compressed keys stay unrounded through
    norm and RoPE and are rounded once to the indexer dtype.
R3  index score: s(row, c) = (1 / (H * sqrt(D))) * sum_h max(0, q_h . k_c).
R4  ties in the block top-k go to the lower block index.
R5  no forced blocks: the only unselected-by-score tokens kept are the
    at most ratio-1 tokens of the still-open group (the tail).
R6  packed row order: selected blocks ascending, each block's tokens
    ascending, then the tail ascending.
R7  visible blocks V(p) = floor((p + 1) / ratio); a group completed by this
    very row is visible to it.
R8  ring slot of token t: ring_block_table[req, 0] * S + (t mod S).
R9  compressed page holds ``cpage`` consecutive compressed keys; compressed
    key c of a request lives at page cblock_table[req, c // cpage],
    offset c % cpage.
R10 interleaved MRoPE: frequency i uses the H component if i % 3 == 1 and
    i < 3 * section[1], the W component if i % 3 == 2 and
    i < 3 * section[2], the T component otherwise.
R11 1-D RoPE (all sections 0): the query uses positions[row, 0, 0]; a
    compressed key uses the logical position of its group's first token.
    MRoPE: both use 3-D positions; a key takes its first token's 3-D
    position from this step's ``positions`` or, for older tokens, from the
    ring's position cache.
R12 e4m3: round to nearest even, saturate to +-448 (OCP FP8 E4M3FN), never
    NaN.  bf16: round to nearest even.
R13 gate: out = bf16(bf16(attn) * sigmoid(gate)); no gate: bf16(attn).
R16 main-attention prepare (the fused qsa_prepare of QSAIndexer.forward):
    the projection row is [Hq heads x (q | gate), Hkv heads x k, Hkv heads
    x v], each piece head_dim wide (the sigmoid gate packed next to each
    query head); q and k take Gemma RMSNorm (q_norm / k_norm) per head, then
    the indexer's rotary embedding at the row's position, and are rounded
    once (q to bf16, k to the cache dtype); the gate is passed through for
    stage 4's sigmoid; v is stored as is (bf16) or as e4m3(v / v_scale).
R15 FP8 main KV cache: stored value e4m3(x / scale) with a static scalar
    scale per tensor (k_scale for K, v_scale for V); attention reads the
    stored values unscaled, multiplies each score by k_scale (with
    head_dim^-0.5) and the normalised output by v_scale before its bf16
    rounding.
R14 the pooled group of a row is the ratio tokens ending at its logical
    position p; members at or after the first logical position of the
    request's rows in this step are read from this step's raw keys, older
    members from the ring.  All ring writes happen after all pooling reads,
    and later rows overwrite earlier rows at the same ring slot.
"""

from __future__ import annotations

import math

import numpy as np

DTYPE_BF16 = 0
DTYPE_E4M3 = 1

E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# Floating-point formats (R12)
# ---------------------------------------------------------------------------

def _round_to_format(x, sig_bits: int, min_exp: int) -> np.ndarray:
    """Round float64 values to the nearest value with ``sig_bits`` significant
    bits (ties to even) and a smallest normal exponent of ``min_exp``.

    x = m * 2**e with m in [0.5, 1): the quantum of a normal value is
    2**(e - sig_bits); below the normal range it is fixed at
    2**(min_exp + 1 - sig_bits) (gradual underflow).  Division by a power of
    two is exact, and numpy's rint rounds half to even.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, min_exp + 1)
    quantum = np.ldexp(1.0, e - sig_bits)
    return np.rint(x / quantum) * quantum


def round_bf16(x) -> np.ndarray:
    """Nearest bf16 value (8 significant bits, fp32 exponent range)."""
    return _round_to_format(x, 8, -126)


def round_e4m3(x) -> np.ndarray:
    """Nearest e4m3fn value (4 significant bits, min normal 2**-6), saturated."""
    return np.clip(_round_to_format(x, 4, -6), -E4M3_MAX, E4M3_MAX)


def round_index_dtype(x, index_dtype: int) -> np.ndarray:
    if index_dtype == DTYPE_BF16:
        return round_bf16(x)
    if index_dtype == DTYPE_E4M3:
        return round_e4m3(x)
    raise ValueError(f"unknown index dtype {index_dtype}")


def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 e4m3fn codes (sign, 4-bit exponent with bias
    7, 3-bit mantissa; exponent field 0 is subnormal; S.1111.111 is NaN)."""
    table = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        man = code & 0x7
        if exp_field == 0xF and man == 0x7:
            table[code] = np.nan
        elif exp_field == 0:
            table[code] = sign * (man / 8.0) * 2.0 ** -6
        else:
            table[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp_field - 7)
    return table


def e4m3_decode(codes) -> np.ndarray:
    return e4m3_decode_table()[np.asarray(codes, dtype=np.uint8)]


def quantize_kv_e4m3(x, scale: float) -> np.ndarray:
    """FP8 KV-cache write with a static per-tensor scale: the stored value is
    e4m3(x / scale), saturated to +-448 ("vllm.models.qwen4_exp.nvidia.qsa",
    Qwen4ExpQSABackend: e4m3 bytes written by reshape_and_cache with the
    layer's per-tensor scales; the patch notes the writer clamps to +-448).
    Returns the stored (unscaled) values."""
    return round_e4m3(np.asarray(x, dtype=np.float64) / float(scale))


def e4m3_encode(x) -> np.ndarray:
    """Codes of round_e4m3(x); +0 for zero."""
    v = round_e4m3(x)
    table = e4m3_decode_table()
    finite = np.where(np.isnan(table), np.inf, table)
    order = np.argsort(finite[:128], kind="stable")  # non-negative codes
    mags = finite[:128][order]
    idx = np.searchsorted(mags, np.abs(v))
    codes = order[idx].astype(np.uint8)
    codes = np.where((v < 0) & (np.abs(v) > 0), codes | 0x80, codes)
    return codes.astype(np.uint8)


def bf16_decode(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_encode(x) -> np.ndarray:
    """Bit patterns of round_bf16(x)."""
    v = round_bf16(x).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# Stage 1 pieces: Gemma RMSNorm and NeoX RoPE / interleaved MRoPE
# ---------------------------------------------------------------------------

def gemma_rmsnorm(x, w, eps: float) -> np.ndarray:
    """Gemma RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * (1 + w).

    Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.__init__
    (q_layernorm / k_layernorm are GemmaRMSNorm(head_dim, eps=rms_norm_eps))
    and the unfused path's gemma_rmsnorm calls.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * (1.0 + np.asarray(w, dtype=np.float64))


def mrope_component(i: int, section) -> int:
    """Position component (0 = T, 1 = H, 2 = W) used by rotary frequency i
    (reading R10).  All-zero sections mean 1-D RoPE: always component 0."""
    if not any(section):
        return 0
    if i % 3 == 1 and i < 3 * section[1]:
        return 1
    if i % 3 == 2 and i < 3 * section[2]:
        return 2
    return 0


def rope_neox(x, pos3, cos_sin, rotary_dim: int, section) -> np.ndarray:
    """NeoX-style rotary embedding on the first ``rotary_dim`` dims of the
    last axis; the remaining dims pass through unchanged.

    Follows "indexer_qsa.py", apply_qsa_rope: the caller's cos/sin cache row
    at a position is split in two halves (cos first, then sin); frequency i
    rotates the pair (x[i], x[i + rotary_dim/2]).  With MRoPE each frequency
    takes the position of its component (R10).

    x: [..., D]; pos3: 3 ints (T, H, W) for this vector; cos_sin:
    [max_pos, rotary_dim].
    """
    x = np.array(x, dtype=np.float64, copy=True)
    half = rotary_dim // 2
    out = x.copy()
    for i in range(half):
        p = int(pos3[mrope_component(i, section)])
        c = float(cos_sin[p, i])
        s = float(cos_sin[p, half + i])
        a = x[..., i]
        b = x[..., half + i]
        out[..., i] = a * c - b * s
        out[..., half + i] = b * c + a * s
    return out


# ---------------------------------------------------------------------------
# Configuration
# ---------------------------------------------------------------------------

class QsaConfig:
    """Indexer configuration (QSAIndexer.__init__ attributes plus cache
    geometry)."""

    def __init__(self, n_heads, head_dim=128, rotary_dim=64, compress_ratio=4,
                 token_topk=64, eps=1e-6, index_dtype=DTYPE_BF16,
                 mrope_section=(0, 0, 0), state_size=None, cpage=16):
        self.n_heads = int(n_heads)
        self.head_dim = int(head_dim)
        self.rotary_dim = int(rotary_dim)
        self.compress_ratio = int(compress_ratio)
        self.token_topk = int(token_topk)
        self.eps = float(eps)
        self.index_dtype = int(index_dtype)
        self.mrope_section = tuple(int(s) for s in mrope_section)
        self.state_size = int(state_size if state_size is not None else compress_ratio)
        self.cpage = int(cpage)

    @property
    def block_topk(self) -> int:
        """Selected compressed blocks per row: token_topk // compress_ratio."""
        return self.token_topk // self.compress_ratio

    @property
    def output_width(self) -> int:
        """Selection columns per row: token_topk + compress_ratio - 1
        (QSAIndexer.output_width)."""
        return self.token_topk + self.compress_ratio - 1

    @property
    def packed_width(self) -> int:
        """output_width + 1: the trailing column is the valid count
        (QSAIndexer.packed_output_width)."""
        return self.output_width + 1

    @property
    def mrope(self) -> bool:
        return any(self.mrope_section)


def visible_blocks(p: int, r: int) -> int:
    """V(p) = floor((p + 1) / r) (reading R7)."""
    return (int(p) + 1) // int(r)


# ---------------------------------------------------------------------------
# Stage 1: query prep, group compress, ring commit
# ---------------------------------------------------------------------------

def prep_query(cfg: QsaConfig, projected_q_row, pos3, cos_sin, q_norm_w) -> np.ndarray:
    """Indexer query of one row: Gemma-RMSNorm(q_layernorm) per head, RoPE at
    the row's position, one rounding to the indexer dtype.

    Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward, unfused
    reference path (gemma_rmsnorm -> apply_qsa_rope -> .to(indexer_dtype)),
    with R2, R11.  projected_q_row: [H, D] -> [H, D] float64 (rounded values).
    """
    q = np.asarray(projected_q_row, dtype=np.float64).reshape(cfg.n_heads, cfg.head_dim)
    q = gemma_rmsnorm(q, q_norm_w, cfg.eps)
    q = rope_neox(q, pos3, cos_sin, cfg.rotary_dim, cfg.mrope_section)
    return round_index_dtype(q, cfg.index_dtype)


def compress_key(cfg: QsaConfig, member_keys, first_pos3, cos_sin, k_norm_w) -> np.ndarray:
    """One compressed key: mean of the group's raw keys (R1),
    Gemma-RMSNorm(k_layernorm), RoPE at the group's first-token position,
    one rounding (R2).

    Follows "vllm.models.qwen4_exp.nvidia.ops.qsa",
    qsa_compress_groups_with_ratio (completed groups are pooled), then the
    unfused path's gemma_rmsnorm / apply_qsa_rope(first_positions) /
    qsa_store_cache_rows.  member_keys: [r, D].
    """
    pooled = np.mean(np.asarray(member_keys, dtype=np.float64), axis=0)
    k = gemma_rmsnorm(pooled, k_norm_w, cfg.eps)
    k = rope_neox(k, first_pos3, cos_sin, cfg.rotary_dim, cfg.mrope_section)
    return round_index_dtype(k, cfg.index_dtype)


def compress_stage(cfg: QsaConfig, *, projected_q, raw_keys, positions, cos_sin,
                   q_norm_w, k_norm_w, ring, ring_pos, ring_block_table,
                   token_to_req, query_start_loc, logical_positions, ccache,
                   compressed_slots):
    """Stage 1 for a batch of rows.  Mutates ``ring`` / ``ring_pos`` /
    ``ccache`` in place and returns q_idx [rows, H, D] (None when
    projected_q is None) plus the list of (row, slot, key) written.

    projected_q: [rows, H, D] or None; raw_keys: [rows, D]; positions:
    [rows, 3] ints; ring: [nb, S, D]; ring_pos: [nb, S, 3] or None;
    ccache: [cpages, cpage, D] (values).  Readings R1, R2, R8, R11, R14.
    """
    rows = len(token_to_req)
    r = cfg.compress_ratio
    S = cfg.state_size
    q_idx = None
    if projected_q is not None:
        q_idx = np.zeros((rows, cfg.n_heads, cfg.head_dim))
        for row in range(rows):
            q_idx[row] = prep_query(cfg, projected_q[row], positions[row], cos_sin, q_norm_w)

    written = []
    for row in range(rows):
        slot = int(compressed_slots[row])
        if slot < 0:
            continue
        req = int(token_to_req[row])
        p = int(logical_positions[row])
        first_row = int(query_start_loc[req])
        step_start = int(logical_positions[first_row])
        ring_block = int(ring_block_table[req][0])
        members = []
        member_pos = []
        for t in range(p - r + 1, p + 1):
            if t >= step_start:
                src = first_row + (t - step_start)
                members.append(raw_keys[src])
                member_pos.append(positions[src])
            else:
                members.append(ring[ring_block, t % S])
                if cfg.mrope:
                    member_pos.append(ring_pos[ring_block, t % S])
                else:
                    member_pos.append((t, t, t))
        first = member_pos[0] if cfg.mrope else (p - r + 1,) * 3
        key = compress_key(cfg, np.stack(members), first, cos_sin, k_norm_w)
        written.append((row, slot, key))

    for row, slot, key in written:
        ccache[slot // cfg.cpage, slot % cfg.cpage] = key
    for row in range(rows):
        req = int(token_to_req[row])
        p = int(logical_positions[row])
        ring_block = int(ring_block_table[req][0])
        ring[ring_block, p % S] = raw_keys[row]
        if ring_pos is not None:
            ring_pos[ring_block, p % S] = positions[row]
    return q_idx, written


def prepare_main_row(cfg: QsaConfig, qkv_row, pos3, cos_sin, q_norm_w, k_norm_w, eps: float,
                     hq: int, hkv: int):
    """Main-attention prepare of one row (R16): returns (q [Hq, D] bf16 values,
    gate [Hq, D], k [Hkv, D] unrounded, v [Hkv, D]).

    Follows "vllm.models.qwen4_exp.nvidia.qsa": Qwen4ExpQSAAttention.__init__
    (qkv_proj packs the output gate next to Q: total_num_heads * (1 +
    attn_output_gate) query-sized heads, then the K and V heads; q_norm and
    k_norm are GemmaRMSNorm(head_dim); the indexer shares rotary_emb) and
    QSAIndexer.forward (qsa_prepare with main_qkv, main_q_norm_weight,
    main_k_norm_weight, main_eps: the main QK-norm/RoPE/gate in the same
    launch as the indexer prepare).
    """
    D = cfg.head_dim
    x = np.asarray(qkv_row, dtype=np.float64)
    qg = x[: 2 * hq * D].reshape(hq, 2, D)
    q, gate = qg[:, 0], qg[:, 1]
    k = x[2 * hq * D: 2 * hq * D + hkv * D].reshape(hkv, D)
    v = x[2 * hq * D + hkv * D: 2 * hq * D + 2 * hkv * D].reshape(hkv, D)
    q = round_bf16(rope_neox(gemma_rmsnorm(q, q_norm_w, eps), pos3, cos_sin, cfg.rotary_dim,
                             cfg.mrope_section))
    k = rope_neox(gemma_rmsnorm(k, k_norm_w, eps), pos3, cos_sin, cfg.rotary_dim,
                  cfg.mrope_section)
    return q, gate.copy(), k, v.copy()


def write_main_kv(kv, slot: int, k, v, page: int, kv_dtype: int = DTYPE_BF16,
                  k_scale: float = 1.0, v_scale: float = 1.0) -> None:
    """The main K/V cache write of one row (R16, R15) at flat slot
    block * page + offset ("vllm.models.qwen4_exp.nvidia.qsa",
    Qwen4ExpQSAImpl.do_kv_cache_update: reshape_and_cache_flash at
    slot_mapping with the layer's scales).  kv: [blocks, Hkv, page, 2D]
    (values; mutated)."""
    if slot < 0:
        return
    D = kv.shape[-1] // 2
    blk, off = slot // page, slot % page
    if kv_dtype == DTYPE_E4M3:
        kv[blk, :, off, :D] = quantize_kv_e4m3(k, k_scale)
        kv[blk, :, off, D:] = quantize_kv_e4m3(v, v_scale)
    else:
        kv[blk, :, off, :D] = round_bf16(k)
        kv[blk, :, off, D:] = round_bf16(v)


def qkv_index_projection(x, w, qkv_cols: int, index_q_cols: int):
    """The fused projection of the main attention and the indexer: one GEMM
    y = x . w^T over the stacked weights [w_qkv; w_index_q; w_index_k], the
    output rounded once to bf16 and split into (main qkv rows, the indexer's
    projected_q, its raw keys).

    Follows "vllm.models.qwen4_exp.nvidia.qsa": Qwen4ExpQSAQKVIndexerLinear
    (sharded Q/gate, K and V and the replicated indexer Q/K computed by one
    GEMM, the indexer's weights as shard 3), Qwen4ExpQSAAttention.forward (qkv,
    projected_qk = qkv.split([2 * q_size + 2 * kv_size, index_qk_size])) and
    QSAIndexer.forward (projected_q, raw_keys = projected_qk.split(
    (index_n_heads * D, index_kv_heads * D))).  x: [rows, hidden]; w:
    [qkv_cols + index_q_cols + D_k, hidden] (values).
    """
    y = round_bf16(np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T)
    return (y[:, :qkv_cols], y[:, qkv_cols:qkv_cols + index_q_cols],
            y[:, qkv_cols + index_q_cols:])


# ---------------------------------------------------------------------------
# Stage 2: index logits; stage 3: block top-k and expand
# ---------------------------------------------------------------------------

def gather_compressed_keys(cfg: QsaConfig, ccache, cblock_row, V: int) -> np.ndarray:
    """Compressed keys 0..V-1 of one request (R9): [V, D]."""
    c = np.arange(V)
    return ccache[np.asarray(cblock_row)[c // cfg.cpage], c % cfg.cpage]


def index_logits_row(cfg: QsaConfig, q_idx_row, keys) -> np.ndarray:
    """Index scores of one row against its visible compressed keys (R3):
    s(c) = (1/(H sqrt(D))) sum_h max(0, q_h . k_c).

    Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward
    (qsa_select_paged_decode / qsa_select_paged_prefill score the indexer
    query against the paged compressed-key cache; the selection is
    "weight-free").  q_idx_row: [H, D]; keys: [V, D] -> [V].
    """
    dots = np.asarray(keys, dtype=np.float64) @ np.asarray(q_idx_row, dtype=np.float64).T
    return np.maximum(dots, 0.0).sum(axis=1) / (cfg.n_heads * math.sqrt(cfg.head_dim))


def select_blocks(scores, V: int, block_topk: int) -> np.ndarray:
    """The block_topk highest-scoring blocks among 0..V-1, ascending (R4, R6).
    All visible blocks when V <= block_topk."""
    if V <= block_topk:
        return np.arange(V, dtype=np.int64)
    s = np.asarray(scores, dtype=np.float64)[:V]
    order = np.lexsort((np.arange(V), -s))  # by score desc, then index asc
    return np.sort(order[:block_topk]).astype(np.int64)


def expand_row(cfg: QsaConfig, blocks, p: int) -> np.ndarray:
    """Packed selection row [output_width + 1] (R5, R6, R7).

    Follows "vllm.models.qwen4_exp.nvidia.qsa", QSAIndexer.forward /
    expand_qsa_block_indices and the packed_output_width docstring: leading
    columns are request-relative token indices padded with -1, the trailing
    column is the valid count.
    """
    r = cfg.compress_ratio
    V = visible_blocks(p, r)
    tokens = [int(b) * r + j for b in blocks for j in range(r)]
    tokens += list(range(V * r, p + 1))
    out = np.full(cfg.packed_width, -1, dtype=np.int64)
    out[: len(tokens)] = tokens
    out[-1] = len(tokens)
    return out


def expected_count(cfg: QsaConfig, p: int) -> int:
    """Closed form of the valid count: min(V, K_b) * r + (p + 1 - V * r)."""
    r = cfg.compress_ratio
    V = visible_blocks(p, r)
    return min(V, cfg.block_topk) * r + (p + 1 - V * r)


def select_row(cfg: QsaConfig, q_idx_row, ccache, cblock_row, p: int):
    """Stages 2-3 for one row: (scores [V], blocks, packed row)."""
    V = visible_blocks(p, cfg.compress_ratio)
    if V == 0:
        scores = np.zeros(0)
    else:
        keys = gather_compressed_keys(cfg, ccache, cblock_row, V)
        scores = index_logits_row(cfg, q_idx_row, keys)
    blocks = select_blocks(scores, V, cfg.block_topk)
    return scores, blocks, expand_row(cfg, blocks, p)


def inert_row(cfg: QsaConfig) -> np.ndarray:
    """Packed row of a row without metadata: all -1, count 0 (QSAIndexer.forward,
    profiling/dummy branch)."""
    out = np.full(cfg.packed_width, -1, dtype=np.int64)
    out[-1] = 0
    return out


# ---------------------------------------------------------------------------
# Stage 4: sparse paged GQA with the output gate
# ---------------------------------------------------------------------------

def sigmoid(x):
    """Logistic function, evaluated without overflow for large |x|."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def sparse_gqa_row(q_row, kv, block_row, tokens, page: int, gate_row=None,
                   k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """Sparse GQA for one row over its selected tokens.

    Follows "0002-qwen4_exp-FP8-E4M3-KV-reader-for-QSA..." patch,
    _qsa_sparse_paged_gqa_splitk_kernel (scores scaled by head_dim^-0.5,
    softmax over the valid entries only, output divided by the normaliser,
    zero when nothing is valid, bf16 rounding of the attention output before
    the gate) and "vllm.models.qwen4_exp.nvidia.qsa", Qwen4ExpQSAImpl.forward
    (K and V are the two halves of the last axis of the paged cache).

    FP8 cache (the same patch, KV_DTYPE branches): K and V hold the decoded
    e4m3 values as stored (unscaled); the static scalar k_scale multiplies
    every score (together with head_dim^-0.5) and v_scale the normalised
    attention output, before its bf16 rounding.  A bf16 cache uses 1 for both.

    q_row: [Hq, D]; kv: [blocks, Hkv, page, 2D] (values); tokens:
    request-relative token indices; gate_row: [Hq, D] or None.  Returns bf16
    values [Hq, D].
    """
    q_row = np.asarray(q_row, dtype=np.float64)
    Hq, D = q_row.shape
    Hkv = kv.shape[1]
    group = Hq // Hkv
    tokens = np.asarray(tokens, dtype=np.int64)
    attn = np.zeros((Hq, D))
    if len(tokens):
        blocks = np.asarray(block_row)[tokens // page]
        offs = tokens % page
        for hq in range(Hq):
            kvh = hq // group
            rows = np.asarray(kv[blocks, kvh, offs], dtype=np.float64)  # [n, 2D]
            k = rows[:, :D]
            v = rows[:, D:]
            z = (k @ q_row[hq]) * (float(k_scale) / math.sqrt(D))
            w = np.exp(z - z.max())
            attn[hq] = ((w / w.sum()) @ v) * float(v_scale)
    out = round_bf16(attn)
    if gate_row is not None:
        out = round_bf16(out * sigmoid(gate_row))
    return out


# ---------------------------------------------------------------------------
# The layer step
# ---------------------------------------------------------------------------

def layer_step(cfg: QsaConfig, *, projected_q, raw_keys, positions, cos_sin,
               q_norm_w, k_norm_w, ring, ring_pos, ring_block_table,
               token_to_req, query_start_loc, logical_positions, ccache,
               compressed_slots, cblock_table, q, kv, block_table, page,
               gate=None, packed=None, skip_topk=False, rows_to_score=None,
               k_scale=1.0, v_scale=1.0, main=None):
    """O1..O7 in order: stage 1 on every row, then (unless skip_topk) stages
    2-3, then stage 4.  With skip_topk the given ``packed`` buffer (from the
    step that selected) feeds stage 4 unchanged (QSAIndexer.skip_topk:
    "later steps reuse them while continuing to update the QSA indexer
    cache").  Mutates the caches; returns (q_idx, packed, out).
    ``rows_to_score`` restricts stages 2-4 to a subset of rows (the others
    keep packed = inert and out = 0).  ``main`` (optional) is the fused
    main-attention prepare (R16): a dict with qkv [rows, (2Hq + 2Hkv) D],
    q_norm_w, k_norm_w, eps, slot_mapping [rows], kv_dtype; its q and gate
    replace ``q`` / ``gate`` and its K/V rows are written into ``kv`` before
    stage 4.
    """
    rows = len(token_to_req)
    q_idx, _ = compress_stage(
        cfg, projected_q=projected_q, raw_keys=raw_keys, positions=positions,
        cos_sin=cos_sin, q_norm_w=q_norm_w, k_norm_w=k_norm_w, ring=ring,
        ring_pos=ring_pos, ring_block_table=ring_block_table,
        token_to_req=token_to_req, query_start_loc=query_start_loc,
        logical_positions=logical_positions, ccache=ccache,
        compressed_slots=compressed_slots)
    todo = range(rows) if rows_to_score is None else rows_to_score
    if main is not None:
        hq, hkv = q.shape[1], kv.shape[1]
        q = np.zeros((rows, hq, cfg.head_dim))
        gate = np.zeros((rows, hq, cfg.head_dim))
        for row in range(rows):
            q[row], gate[row], k, v = prepare_main_row(
                cfg, main["qkv"][row], positions[row], cos_sin, main["q_norm_w"],
                main["k_norm_w"], main["eps"], hq, hkv)
            write_main_kv(kv, int(main["slot_mapping"][row]), k, v, page,
                          main.get("kv_dtype", DTYPE_BF16), k_scale, v_scale)
    if skip_topk:
        if packed is None:
            raise ValueError("skip_topk needs the packed buffer of the selecting step")
        packed = np.asarray(packed)
    else:
        packed = np.stack([inert_row(cfg) for _ in range(rows)]) if rows else \
            np.zeros((0, cfg.packed_width), dtype=np.int64)
        for row in todo:
            req = int(token_to_req[row])
            _, _, packed[row] = select_row(cfg, q_idx[row], ccache, cblock_table[req],
                                           int(logical_positions[row]))
    Hq, D = q.shape[1], q.shape[2]
    out = np.zeros((rows, Hq, D))
    for row in todo:
        req = int(token_to_req[row])
        n = int(packed[row, -1])
        out[row] = sparse_gqa_row(q[row], kv, block_table[req], packed[row, :n], page,
                                  None if gate is None else gate[row], k_scale, v_scale)
    return q_idx, packed, out
