"""The C-ABI library builds, loads and exports every symbol include/qsa.h
declares; host-side validation rejects bad arguments before any CUDA call.
No compute call runs here (CPU only)."""

import ctypes
import os
import re

import pytest

from learned_sparse_attention_gb300 import build as B
from learned_sparse_attention_gb300 import qsa as Q

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "qsa.h")


@pytest.fixture(scope="module")
def lib():
    B.build_library()
    return Q.load(build_if_missing=False)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"qsa_compress", "qsa_index_logits", "qsa_topk", "qsa_sparse_gqa",
            "qsa_layer_step", "qsa_workspace_bytes", "qsa_status_string",
            "qsa_check_errors"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    for s in range(8):
        assert lib.qsa_status_string(s)
    assert b"unknown" in lib.qsa_status_string(99)
    assert b"sm_103a" in lib.qsa_version()


def _cfg(**kw):
    base = dict(n_heads=32, compress_ratio=4, token_topk=2048, index_dtype=Q.DTYPE_E4M3,
                cpage=16, max_position=40000)
    base.update(kw)
    return Q.make_cfg(**base)


def test_workspace_bytes(lib):
    g = Q.make_gqa_cfg(32, 4, 64, 1000)
    n1 = Q.workspace_bytes(_cfg(), g, 64, 64, 8192)
    # q_idx (64 x 32 x 128 B) + logits (64 x 8192 x 4 B) at least
    assert n1 >= 64 * 32 * 128 + 64 * 8192 * 4
    assert n1 % 256 == 0
    assert Q.workspace_bytes(_cfg(), g, 128, 64, 8192) > n1
    assert Q.workspace_bytes(_cfg(head_dim=64), g, 64, 64, 8192) == 0
    assert Q.workspace_bytes(_cfg(), Q.make_gqa_cfg(32, 3, 64, 10), 64, 64, 8192) == 0


@pytest.mark.parametrize("bad,status", [
    (dict(head_dim=64), 4), (dict(rotary_dim=32), 4), (dict(n_heads=12), 4),
    (dict(compress_ratio=3), 4), (dict(compress_ratio=1), 4), (dict(token_topk=2050), 1),
    (dict(index_dtype=5), 3), (dict(mrope_section=(8, 12, 11)), 4), (dict(state_size=2), 2),
    (dict(cpage=12), 4),
])
def test_compress_rejects_bad_config_before_launch(lib, bad, status):
    cfg = _cfg(**bad)
    dummy = ctypes.c_void_p(256)
    st = lib.qsa_compress(ctypes.byref(cfg), None, None, dummy, dummy, dummy, dummy, dummy,
                          dummy, 1, None, dummy, 1, dummy, dummy, dummy, dummy, 1, dummy, 4, 1,
                          None)
    assert st == status


def test_null_and_shape_errors(lib):
    cfg = _cfg()
    d = ctypes.c_void_p(256)
    # raw_keys missing
    assert lib.qsa_compress(ctypes.byref(cfg), None, None, None, d, d, d, d, d, 1, None, d, 1, d,
                            d, d, d, 1, d, 4, 1, None) == 1
    # projected_q without q_idx
    assert lib.qsa_compress(ctypes.byref(cfg), d, None, d, d, d, d, d, d, 1, None, d, 1, d,
                            d, d, d, 1, d, 4, 1, None) == 1
    # MRoPE needs the ring position cache
    mcfg = _cfg(mrope_section=(8, 12, 12))
    assert lib.qsa_compress(ctypes.byref(mcfg), None, None, d, d, d, d, d, d, 1, None, d, 1, d,
                            d, d, d, 1, d, 4, 1, None) == 1
    # misaligned raw keys
    assert lib.qsa_compress(ctypes.byref(cfg), None, None, ctypes.c_void_p(258), d, d, d, d, d, 1,
                            None, d, 1, d, d, d, d, 1, d, 4, 1, None) == 1
    # rows == 0 is a no-op
    assert lib.qsa_compress(ctypes.byref(cfg), None, None, None, None, None, None, None, None, 0,
                            None, None, 0, None, None, None, None, 0, None, 0, 0, None) == 0
    g = Q.make_gqa_cfg(32, 4, 64, 10)
    # packed width must hold selections plus the count column
    assert lib.qsa_sparse_gqa(ctypes.byref(g), d, d, d, 1, d, 1, d, None, d, 4, None, 0,
                              None) == 2
    # GQA groups: 1..8 and 16 run (a few rows split the selection over CTAs and
    # need the workspace: refused without one); other groups are unsupported;
    # Hq % Hkv != 0 is a shape error
    g2 = Q.make_gqa_cfg(16, 4, 64, 10)
    assert lib.qsa_sparse_gqa(ctypes.byref(g2), d, d, d, 1, d, 68, d, None, d, 4, None, 0,
                              None) == 5
    g12 = Q.make_gqa_cfg(48, 4, 64, 10)
    assert lib.qsa_sparse_gqa(ctypes.byref(g12), d, d, d, 1, d, 68, d, None, d, 4, None, 0,
                              None) == 4
    g_odd = Q.make_gqa_cfg(30, 4, 64, 10)
    assert lib.qsa_sparse_gqa(ctypes.byref(g_odd), d, d, d, 1, d, 68, d, None, d, 4, None, 0,
                              None) == 2
    # the no-workspace entry point makes the same configuration checks
    assert lib.qsa_sparse_gqa_noalloc(ctypes.byref(g12), d, d, d, 1, d, 68, d, None, d, 4,
                                      None) == 4
    assert lib.qsa_sparse_gqa_noalloc(ctypes.byref(g_odd), d, d, d, 1, d, 68, d, None, d, 4,
                                      None) == 2
    # page size not a multiple of 16
    g3 = Q.make_gqa_cfg(32, 4, 40, 10)
    assert lib.qsa_sparse_gqa(ctypes.byref(g3), d, d, d, 1, d, 68, d, None, d, 4, None, 0,
                              None) == 2
    # logits: ld smaller than max_visible; negative rows
    assert lib.qsa_index_logits(ctypes.byref(cfg), d, d, 1, d, 1, d, d, d, d, 100, 200, 4, 1, d,
                                1 << 20, None) == 2
    assert lib.qsa_index_logits(ctypes.byref(cfg), d, d, 1, d, 1, d, d, d, d, 256, 200, -1, 1,
                                None, 0, None) == 2
    # misaligned compressed cache
    assert lib.qsa_index_logits(ctypes.byref(cfg), d, ctypes.c_void_p(264), 1, d, 1, d, d, d, d,
                                256, 200, 4, 1, None, 0, None) == 1
    # top-k beyond the shared-memory limit of this build
    assert lib.qsa_topk(ctypes.byref(cfg), d, 1 << 20, 1 << 20, d, d, 4, None) == 4


def test_layer_step_argument_checks(lib):
    cfg = _cfg()
    g = Q.make_gqa_cfg(32, 4, 64, 10)
    a = Q.QsaStepArgs()
    a.rows, a.reqs = 4, 1
    # no packed buffer (skip_topk without a buffer, or a plain step without one)
    assert lib.qsa_layer_step(ctypes.byref(cfg), ctypes.byref(g), ctypes.byref(a), 1,
                              ctypes.c_void_p(256), 1 << 30, None) == 1
    a.packed = 256
    a.max_visible = 100
    # workspace too small
    assert lib.qsa_layer_step(ctypes.byref(cfg), ctypes.byref(g), ctypes.byref(a), 0,
                              ctypes.c_void_p(256), 16, None) == 5
    a.rows = 0
    assert lib.qsa_layer_step(ctypes.byref(cfg), ctypes.byref(g), ctypes.byref(a), 0, None, 0,
                              None) == 0


def test_binding_rejects_host_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        Q._ptr(torch.zeros(4), torch.float32, "x")


def test_mtp_steps_rejects_bad_step_lists(lib):
    g = Q.make_gqa_cfg(32, 4, 64, 1000)
    a, b = Q.QsaStepArgs(), Q.QsaStepArgs()
    a.rows = b.rows = 4
    a.reqs = b.reqs = 1
    a.packed, b.packed = 4096, 8192          # different packed buffers
    arr = (Q.QsaStepArgs * 2)(a, b)
    assert lib.qsa_mtp_steps(ctypes.byref(_cfg()), ctypes.byref(g), arr, 2, None, 0, None) == 1
    b.rows = 5
    b.packed = 4096
    arr = (Q.QsaStepArgs * 2)(a, b)
    assert lib.qsa_mtp_steps(ctypes.byref(_cfg()), ctypes.byref(g), arr, 2, None, 0, None) == 1
    assert lib.qsa_mtp_steps(ctypes.byref(_cfg()), ctypes.byref(g), arr, 0, None, 0, None) == 1
    assert lib.qsa_mtp_steps(ctypes.byref(_cfg()), ctypes.byref(g), None, 1, None, 0, None) == 1
    big = (Q.QsaStepArgs * 17)(*([a] * 17))
    assert lib.qsa_mtp_steps(ctypes.byref(_cfg()), ctypes.byref(g), big, 17, None, 0, None) == 1
