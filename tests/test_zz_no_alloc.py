"""te_encoder_block_fwd_static: the encoder block for callers that cannot
allocate device memory (an application whose device memory all belongs to
its own allocator, or a loop that must never allocate).  It takes no
workspace and uses the library's fixed 32 MiB scratch array instead.

Its results must equal those of te_encoder_block_fwd with a caller-provided
workspace, on two calls in a row (the second call finds the first call's
leftovers in the shared array).  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import transformer_encoder_forward_gb300 as te
from transformer_encoder_forward_gb300 import synth
from tests.gpu_util import rel_frob, to_dev, to_np

TOL = 5e-3   # the whole-block tolerance of the other block tests


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
    assert 0 < need <= 32 << 20
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
        assert rel_frob(to_np(x_st), to_np(x_ref)) < TOL, call
        assert rel_frob(to_np(a_st), to_np(a_ref)) < TOL, call
        assert rel_frob(to_np(x_st) - to_np(x0), to_np(x_ref) - to_np(x0)) < TOL, call


def test_static_scratch_block_rejects_rows_beyond_its_array():
    # validated on the host before anything is launched: no GPU needed
    L = te.lib()
    cfg = synth.CONFIGS["c2"]
    d = te.te_block_desc()
    d.d, d.n_heads, d.n_kv_heads, d.head_dim, d.ffn = cfg.d, cfg.heads, cfg.kv_heads, cfg.hd, cfg.ffn
    d.gated = 1
    cu = synth.cu_seqlens([4000])
    need = L.te_encoder_block_workspace(ctypes.byref(d), 4000)
    assert need > 32 << 20
    st = L.te_encoder_block_fwd_static(ctypes.byref(d), 0x10000, 0x20000,
                                       cu.ctypes.data_as(ctypes.c_void_p), 0x30000, 1, None)
    assert st == te.TE_EWORKSPACE
    assert "32" in L.te_last_error().decode() or "static" in L.te_last_error().decode()
