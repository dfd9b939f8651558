"""te_encoder_block_fwd_static: the encoder block for callers that cannot
allocate device memory (an application whose device memory all belongs to
its own allocator, or a loop that must never allocate).  It takes no
workspace and uses the library's fixed scratch array
(TE_STATIC_SCRATCH_BYTES, 32 MiB) instead.

Both entry points run the same deterministic kernels on the same inputs, so
the static one must give the same bits as te_encoder_block_fwd with a
caller-provided workspace, on two calls in a row (the second call finds the
first call's leftovers in the shared array; a stale read there would show as
a difference).  This file is collected last so that a run stopping at the
first failure has already run every other test.
"""
import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

import transformer_encoder_forward_gb300 as te
from transformer_encoder_forward_gb300 import synth
from tests.gpu_util import rel_frob, to_dev, to_np

TOL = 5e-3   # the whole-block tolerance of the other block tests (diagnostic here)


def _stack(lens):
    from transformer_encoder_forward_gb300.model import EncoderStack
    cfg = synth.small_config("c2", layers=2, window=40, lens=tuple(lens))
    ps = [synth.draw_layer(cfg, i, 31) for i in range(cfg.layers)]
    return cfg, EncoderStack(cfg, ps, lens, synth.rope_tables(cfg, lens))


@pytest.mark.gpu
def test_static_scratch_block_matches_workspace_block_on_two_calls():
    import torch
    lens = [37, 64, 101, 300]
    cfg, st = _stack(lens)
    need = te.block_workspace(st.descs[0], st.T)
    assert 0 < need <= te.TE_STATIC_SCRATCH_BYTES
    for call, seed in enumerate((3, 4)):
        x0 = to_dev(synth.draw_x(st.T, cfg.d, seed))
        a0 = torch.empty(st.T, cfg.d, dtype=torch.bfloat16, device="cuda")
        st.input_norm(x0, a0)
        # the existing entry point, caller-provided workspace
        x_ref, a_ref = x0.clone(), a0.clone()
        te.encoder_block_fwd(st.descs[0], x_ref, a_ref, st.cu_host, st.cu_dev, st.workspace)
        # the allocation-free entry point, library scratch
        x_st, a_st = x0.clone(), a0.clone()
        te.encoder_block_fwd_static(st.descs[0], x_st, a_st, st.cu_host, st.cu_dev)
        te.check()
        assert np.all(np.isfinite(to_np(x_st)))
        # the same kernels on the same bytes: the same bits
        assert torch.equal(x_st, x_ref), (call, rel_frob(to_np(x_st), to_np(x_ref)))
        assert torch.equal(a_st, a_ref), (call, rel_frob(to_np(a_st), to_np(a_ref)))
        assert not torch.equal(x_st, x0), call   # the block did change x
        assert rel_frob(to_np(x_st) - to_np(x0), to_np(x_ref) - to_np(x0)) < TOL, call


def _shaped_desc(cfg):
    """A descriptor with valid shapes and non-NULL, aligned (never
    dereferenced) pointers: host validation passes and the size check decides."""
    d = te.te_block_desc()
    d.d, d.n_heads, d.n_kv_heads, d.head_dim, d.ffn = cfg.d, cfg.heads, cfg.kv_heads, cfg.hd, cfg.ffn
    d.gated, d.norm_kind, d.resid_form, d.act = 1, te.TE_NORM_RMS, te.TE_RESID_PLAIN, te.TE_ACT_GELU_TANH
    d.eps, d.attn_scale, d.post, d.q_mul = 1e-6, cfg.scale, 1.0, 1.0
    base = 0x100000
    qw, kw = cfg.heads * cfg.hd, cfg.kv_heads * cfg.hd
    for i, (key, n, k) in enumerate((("wq", qw, cfg.d), ("wk", kw, cfg.d), ("wv", kw, cfg.d),
                                     ("wo", cfg.d, qw), ("wg", cfg.ffn, cfg.d), ("wu", cfg.ffn, cfg.d),
                                     ("wd", cfg.d, cfg.ffn))):
        setattr(d, key, te.te_q8w(base * (i + 1), base * (i + 11), None, n, k, None, None))
    d.ffn_norm_w = base * 30
    return d


def test_static_scratch_block_rejects_rows_beyond_its_array():
    # validated on the host before anything is launched: no GPU needed
    L = te.lib()
    cfg = synth.CONFIGS["c2"]
    d = _shaped_desc(cfg)
    per_row = L.te_encoder_block_workspace(ctypes.byref(d), 1)
    assert per_row >= 3 * 512 * 2 + 512 * 2 + 512 * 4 + 2048 * 2   # qkv, o, tmp, m
    rows = te.TE_STATIC_SCRATCH_BYTES // (3 * 512 * 2 + 512 * 2 + 512 * 4 + 2048 * 2) + 64
    cu = synth.cu_seqlens([rows])
    need = L.te_encoder_block_workspace(ctypes.byref(d), rows)
    assert need > te.TE_STATIC_SCRATCH_BYTES
    st = L.te_encoder_block_fwd_static(ctypes.byref(d), 0x10000, 0x20000,
                                       cu.ctypes.data_as(ctypes.c_void_p), 0x30000, 1, None)
    assert st == te.TE_EWORKSPACE, L.te_last_error().decode()
    assert "TE_STATIC_SCRATCH_BYTES" in L.te_last_error().decode()
    # a malformed descriptor is reported as such, not as a scratch overflow
    d.head_dim = -64
    st = L.te_encoder_block_fwd_static(ctypes.byref(d), 0x10000, 0x20000,
                                       cu.ctypes.data_as(ctypes.c_void_p), 0x30000, 1, None)
    assert st == te.TE_ESHAPE, L.te_last_error().decode()


def test_static_scratch_size_constant_matches_the_header():
    hdr = (Path(__file__).resolve().parents[1] / "include" / "tefwd.h").read_text()
    m = re.search(r"#define\s+TE_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", hdr)
    assert m, "TE_STATIC_SCRATCH_BYTES not found in tefwd.h"
    assert int(m.group(1)) << int(m.group(2)) == te.TE_STATIC_SCRATCH_BYTES
