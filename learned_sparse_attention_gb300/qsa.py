"""Thin Python binding of the QSA C ABI (include/qsa.h).

Argument marshalling only: every step of the layer runs in the CUDA kernels
of libqsa.so.  Tensors are torch CUDA tensors (torch provides device memory
and the current stream); nothing here computes on the host.  The library is
required: if it is missing or a tensor is not on a CUDA device, the calls
raise instead of falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

QSA_OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "shape", 3: "dtype", 4: "unsupported",
          5: "workspace", 6: "cuda", 7: "device fault"}
DTYPE_BF16 = 0
DTYPE_E4M3 = 1

_c_int = ctypes.c_int32
_p = ctypes.c_void_p


class QsaError(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status


class QsaCfg(ctypes.Structure):
    _fields_ = [("n_heads", _c_int), ("head_dim", _c_int), ("rotary_dim", _c_int),
                ("compress_ratio", _c_int), ("token_topk", _c_int), ("eps", ctypes.c_float),
                ("index_dtype", _c_int), ("mrope_section", _c_int * 3), ("state_size", _c_int),
                ("cpage", _c_int), ("max_position", _c_int)]


class QsaGqaCfg(ctypes.Structure):
    _fields_ = [("num_q_heads", _c_int), ("num_kv_heads", _c_int), ("head_dim", _c_int),
                ("page_size", _c_int), ("num_blocks", _c_int), ("kv_dtype", _c_int),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class QsaMainPrep(ctypes.Structure):
    _fields_ = [("qkv", _p), ("q_norm_w", _p), ("k_norm_w", _p), ("eps", ctypes.c_float),
                ("q_out", _p), ("gate_out", _p), ("kv", _p), ("slot_mapping", _p)]


class QsaStepArgs(ctypes.Structure):
    _fields_ = [("rows", _c_int), ("reqs", _c_int), ("max_visible", _c_int),
                ("projected_q", _p), ("raw_keys", _p), ("positions", _p), ("cos_sin", _p),
                ("q_norm_w", _p), ("k_norm_w", _p), ("ring", _p), ("ring_blocks", _c_int),
                ("ring_pos", _p), ("ring_block_table", _p), ("ring_bt_stride", _c_int),
                ("ccache", _p), ("cpages", _c_int), ("cblock_table", _p), ("cbt_stride", _c_int),
                ("compressed_slots", _p), ("token_to_req", _p), ("query_start_loc", _p),
                ("logical_positions", _p), ("packed", _p), ("q", _p), ("kv", _p),
                ("block_table", _p), ("bt_stride", _c_int), ("gate", _p), ("out", _p),
                ("main", _p)]


_LIB = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libqsa.so (building it in-tree first when it is missing)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise RuntimeError(f"QSA CUDA library missing: {_build.LIB}")
        _build.build_library()
    lib = ctypes.CDLL(_build.LIB)
    P, I, Z = _p, _c_int, ctypes.c_size_t
    sig = {
        "qsa_compress": [P, P, P, P, P, P, P, P, P, I, P, P, I, P, P, P, P, I, P, I, I, P],
        "qsa_index_logits": [P, P, P, I, P, I, P, P, P, P, ctypes.c_int64, I, I, I, P, Z, P],
        "qsa_topk": [P, P, ctypes.c_int64, I, P, P, I, P],
        "qsa_sparse_gqa": [P, P, P, P, I, P, I, P, P, P, I, P, Z, P],
        "qsa_layer_step": [P, P, P, I, P, Z, P],
        "qsa_mtp_steps": [P, P, P, I, P, Z, P],
        "qsa_main_prepare": [P, P, P, P, P, I, P],
        "qsa_qkv_index_proj": [P, P, I, I, I, I, I, P, P, P, P],
        "qsa_workspace_bytes": [P, P, I, I, I],
        "qsa_status_string": [I],
        "qsa_check_errors": [ctypes.POINTER(ctypes.c_int64)],
        "qsa_version": [],
        "qsa_step_launches": [P, P, I, I, I],
        "qsa_gqa_splits": [P, I, I],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.qsa_workspace_bytes.restype = ctypes.c_size_t
    lib.qsa_status_string.restype = ctypes.c_char_p
    lib.qsa_version.restype = ctypes.c_char_p
    _LIB = lib
    return lib


def _check(fn, status):
    if status != QSA_OK:
        text = load().qsa_status_string(status).decode()
        raise QsaError(fn, status, text)


def make_cfg(n_heads, compress_ratio, token_topk, index_dtype, cpage, max_position,
             state_size=None, mrope_section=(0, 0, 0), eps=1e-6, head_dim=128,
             rotary_dim=64) -> QsaCfg:
    c = QsaCfg()
    c.n_heads, c.head_dim, c.rotary_dim = n_heads, head_dim, rotary_dim
    c.compress_ratio, c.token_topk, c.eps = compress_ratio, token_topk, eps
    c.index_dtype = index_dtype
    c.mrope_section[:] = list(mrope_section)
    c.state_size = state_size if state_size is not None else 2 * compress_ratio
    c.cpage, c.max_position = cpage, max_position
    return c


def make_gqa_cfg(num_q_heads, num_kv_heads, page_size, num_blocks, head_dim=128,
                 kv_dtype=DTYPE_BF16, k_scale=1.0, v_scale=1.0) -> QsaGqaCfg:
    g = QsaGqaCfg()
    g.num_q_heads, g.num_kv_heads, g.head_dim = num_q_heads, num_kv_heads, head_dim
    g.page_size, g.num_blocks = page_size, num_blocks
    g.kv_dtype, g.k_scale, g.v_scale = kv_dtype, k_scale, v_scale
    return g


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


_IDX = (torch.uint8, torch.bfloat16)


def compress(cfg, projected_q, q_idx, raw_keys, positions, cos_sin, q_norm_w, k_norm_w, ring,
             ring_pos, ring_block_table, token_to_req, query_start_loc, logical_positions, ccache,
             compressed_slots, stream=None):
    rows = raw_keys.shape[0]
    reqs = query_start_loc.shape[0] - 1
    st = load().qsa_compress(
        ctypes.byref(cfg), _ptr(projected_q, torch.bfloat16, "projected_q"),
        _ptr(q_idx, _IDX, "q_idx"), _ptr(raw_keys, torch.bfloat16, "raw_keys"),
        _ptr(positions, torch.int64, "positions"), _ptr(cos_sin, torch.float32, "cos_sin"),
        _ptr(q_norm_w, torch.bfloat16), _ptr(k_norm_w, torch.bfloat16),
        _ptr(ring, torch.bfloat16, "ring"), ring.shape[0], _ptr(ring_pos, torch.int64),
        _ptr(ring_block_table, torch.int32), ring_block_table.shape[1],
        _ptr(token_to_req, torch.int32), _ptr(query_start_loc, torch.int32),
        _ptr(logical_positions, torch.int32), _ptr(ccache, _IDX, "ccache"), ccache.shape[0],
        _ptr(compressed_slots, torch.int64), rows, reqs, _stream(stream))
    _check("qsa_compress", st)


def index_logits(cfg, q_idx, ccache, cblock_table, token_to_req, query_start_loc,
                 logical_positions, logits, max_visible, ws, stream=None):
    rows = token_to_req.shape[0]
    reqs = query_start_loc.shape[0] - 1
    st = load().qsa_index_logits(
        ctypes.byref(cfg), _ptr(q_idx, _IDX), _ptr(ccache, _IDX), ccache.shape[0],
        _ptr(cblock_table, torch.int32), cblock_table.shape[1], _ptr(token_to_req, torch.int32),
        _ptr(query_start_loc, torch.int32), _ptr(logical_positions, torch.int32),
        _ptr(logits, torch.float32), logits.shape[1], max_visible, rows, reqs,
        _ptr(ws, torch.uint8), ws.numel(), _stream(stream))
    _check("qsa_index_logits", st)


def topk(cfg, logits, max_visible, logical_positions, packed, stream=None):
    rows = logical_positions.shape[0]
    st = load().qsa_topk(ctypes.byref(cfg), _ptr(logits, torch.float32),
                         logits.shape[1] if logits is not None else 0, max_visible,
                         _ptr(logical_positions, torch.int32), _ptr(packed, torch.int32), rows,
                         _stream(stream))
    _check("qsa_topk", st)


def sparse_gqa(gcfg, q, kv, block_table, packed, token_to_req, gate, out, ws, stream=None):
    st = load().qsa_sparse_gqa(
        ctypes.byref(gcfg), _ptr(q, torch.bfloat16), _ptr(kv, _IDX),
        _ptr(block_table, torch.int32), block_table.shape[1], _ptr(packed, torch.int32),
        packed.shape[1], _ptr(token_to_req, torch.int32), _ptr(gate, torch.bfloat16),
        _ptr(out, torch.bfloat16), q.shape[0], _ptr(ws, torch.uint8),
        0 if ws is None else ws.numel(), _stream(stream))
    _check("qsa_sparse_gqa", st)


NOALLOC_SCRATCH_BYTES = 4 << 20


def sparse_gqa_noalloc(gcfg, q, kv, block_table, packed, token_to_req, gate, out, stream=None):
    """Stage 4 without a workspace: for callers that may not allocate device
    memory; the split-KV scratch is a fixed array inside the library (see
    qsa_sparse_gqa_noalloc in include/qsa.h for its limit and sharing rules)."""
    lib = load()
    f = lib.qsa_sparse_gqa_noalloc
    f.argtypes = [_p, _p, _p, _p, _c_int, _p, _c_int, _p, _p, _p, _c_int, _p]
    f.restype = ctypes.c_int
    st = f(ctypes.byref(gcfg), _ptr(q, torch.bfloat16), _ptr(kv, _IDX),
           _ptr(block_table, torch.int32), block_table.shape[1], _ptr(packed, torch.int32),
           packed.shape[1], _ptr(token_to_req, torch.int32), _ptr(gate, torch.bfloat16),
           _ptr(out, torch.bfloat16), q.shape[0], _stream(stream))
    _check("qsa_sparse_gqa_noalloc", st)


def workspace_bytes(cfg, gcfg, rows, reqs, max_visible) -> int:
    return int(load().qsa_workspace_bytes(ctypes.byref(cfg), ctypes.byref(gcfg), rows, reqs,
                                          max_visible))


def main_prep(t: dict, eps: float = 1e-6) -> QsaMainPrep:
    """The main-attention prepare's argument struct from named CUDA tensors
    (main_qkv, main_q_norm_w, main_k_norm_w, main_q_out, main_gate_out, kv,
    slot_mapping) and the norms' epsilon."""
    m = QsaMainPrep()
    m.qkv = _ptr(t["main_qkv"], torch.bfloat16, "main_qkv")
    m.q_norm_w = _ptr(t["main_q_norm_w"], torch.bfloat16)
    m.k_norm_w = _ptr(t["main_k_norm_w"], torch.bfloat16)
    m.eps = float(eps)
    m.q_out = _ptr(t["main_q_out"], torch.bfloat16, "main_q_out")
    m.gate_out = _ptr(t["main_gate_out"], torch.bfloat16, "main_gate_out")
    m.kv = _ptr(t["kv"], _IDX)
    m.slot_mapping = _ptr(t["slot_mapping"], torch.int64, "slot_mapping")
    m._tensors = dict(t)
    return m


def main_prepare(cfg, gcfg, m: QsaMainPrep, positions, cos_sin, stream=None):
    """The main-attention prepare alone (qsa_main_prepare)."""
    st = load().qsa_main_prepare(ctypes.byref(cfg), ctypes.byref(gcfg), ctypes.byref(m),
                                 _ptr(positions, torch.int64), _ptr(cos_sin, torch.float32),
                                 positions.shape[0], _stream(stream))
    _check("qsa_main_prepare", st)


def step_args(t: dict, packed, out, max_visible, main: QsaMainPrep | None = None) -> QsaStepArgs:
    """Fill the step argument struct from named CUDA tensors (keys as produced
    by learned_sparse_attention_gb300.workloads); `main` fuses the
    main-attention prepare into stage 1."""
    a = QsaStepArgs()
    a.rows = t["raw_keys"].shape[0]
    a.reqs = t["query_start_loc"].shape[0] - 1
    a.max_visible = max_visible
    a.projected_q = _ptr(t["projected_q"], torch.bfloat16)
    a.raw_keys = _ptr(t["raw_keys"], torch.bfloat16)
    a.positions = _ptr(t["positions"], torch.int64)
    a.cos_sin = _ptr(t["cos_sin"], torch.float32)
    a.q_norm_w = _ptr(t["q_norm_w"], torch.bfloat16)
    a.k_norm_w = _ptr(t["k_norm_w"], torch.bfloat16)
    a.ring = _ptr(t["ring"], torch.bfloat16)
    a.ring_blocks = t["ring"].shape[0]
    a.ring_pos = _ptr(t.get("ring_pos"), torch.int64)
    a.ring_block_table = _ptr(t["ring_block_table"], torch.int32)
    a.ring_bt_stride = t["ring_block_table"].shape[1]
    a.ccache = _ptr(t["ccache"], _IDX)
    a.cpages = t["ccache"].shape[0]
    a.cblock_table = _ptr(t["cblock_table"], torch.int32)
    a.cbt_stride = t["cblock_table"].shape[1]
    a.compressed_slots = _ptr(t["compressed_slots"], torch.int64)
    a.token_to_req = _ptr(t["token_to_req"], torch.int32)
    a.query_start_loc = _ptr(t["query_start_loc"], torch.int32)
    a.logical_positions = _ptr(t["logical_positions"], torch.int32)
    a.packed = _ptr(packed, torch.int32)
    a.q = _ptr(t["q"], torch.bfloat16)
    a.kv = _ptr(t["kv"], _IDX)
    a.block_table = _ptr(t["block_table"], torch.int32)
    a.bt_stride = t["block_table"].shape[1]
    a.gate = _ptr(t.get("gate"), torch.bfloat16)
    a.out = _ptr(out, torch.bfloat16)
    a.main = ctypes.addressof(main) if main is not None else None
    # the struct holds raw device addresses: keep the tensors (and the
    # prepare's struct) behind them alive for as long as the struct is
    a._tensors = (dict(t), packed, out, main)
    return a


def layer_step(cfg, gcfg, args: QsaStepArgs, ws, skip_topk=False, stream=None):
    st = load().qsa_layer_step(ctypes.byref(cfg), ctypes.byref(gcfg), ctypes.byref(args),
                               1 if skip_topk else 0, _ptr(ws, torch.uint8), ws.numel(),
                               _stream(stream))
    _check("qsa_layer_step", st)


MTP_MAX_STEPS = 16


def mtp_steps(cfg, gcfg, steps, ws, stream=None):
    """The k layer steps of one MTP draft (qsa_mtp_steps): steps[0] selects,
    the later steps reuse its packed buffer.  `steps` is a list of
    QsaStepArgs sharing rows, reqs and the packed buffer."""
    k = len(steps)
    arr = (QsaStepArgs * k)(*steps)
    st = load().qsa_mtp_steps(ctypes.byref(cfg), ctypes.byref(gcfg), arr, k, _ptr(ws, torch.uint8),
                              ws.numel(), _stream(stream))
    _check("qsa_mtp_steps", st)


def qkv_index_proj(x, w, qkv_out, index_q_out, index_k_out, stream=None):
    """The fused projection GEMM (qsa_qkv_index_proj): x [rows, hidden] .
    w^T with w = [w_qkv; w_index_q; w_index_k], into the three outputs."""
    rows, hidden = x.shape
    st = load().qsa_qkv_index_proj(
        _ptr(x, torch.bfloat16, "x"), _ptr(w, torch.bfloat16, "w"), rows, hidden,
        qkv_out.shape[-1], index_q_out.shape[-1], index_k_out.shape[-1],
        _ptr(qkv_out, torch.bfloat16), _ptr(index_q_out, torch.bfloat16),
        _ptr(index_k_out, torch.bfloat16), _stream(stream))
    _check("qsa_qkv_index_proj", st)


def step_launches(cfg, gcfg, rows, reqs, skip_topk=False) -> int:
    """Kernel launches made by one layer_step call."""
    return int(load().qsa_step_launches(ctypes.byref(cfg), ctypes.byref(gcfg), rows, reqs,
                                        1 if skip_topk else 0))


def gqa_splits(gcfg, rows, packed_width) -> int:
    """Split-KV factor of the sparse GQA stage for these sizes."""
    return int(load().qsa_gqa_splits(ctypes.byref(gcfg), rows, packed_width))


def check_errors() -> int:
    """Synchronise and return (and clear) the device error count; raises on
    a CUDA error, returns the count (non-zero means masked accesses)."""
    n = ctypes.c_int64(0)
    st = load().qsa_check_errors(ctypes.byref(n))
    if st not in (QSA_OK, 7):
        _check("qsa_check_errors", st)
    return int(n.value)


def version() -> str:
    return load().qsa_version().decode()
