"""The C-ABI library builds, loads, exports what include/tefwd.h declares, and
rejects bad arguments on the host before launching anything (no GPU needed:
every call here must fail validation)."""
import ctypes
import os
import re

import numpy as np
import pytest

import transformer_encoder_forward_gb300 as te
from transformer_encoder_forward_gb300 import build as tebuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(te.LIB_PATH):
        tebuild.build()
    return te.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tefwd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(te_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(te.EXPORTS), "binding and header disagree"


def test_version_and_empty_error(L):
    assert "sm_103a" in te.version()


def test_binding_structs_match_the_compiled_abi(L):
    # the ctypes mirrors of te_q8w, te_q8_item and te_block_desc have the
    # library's own sizes (a field added on one side only shows here)
    assert te.abi_sizes() == (ctypes.sizeof(te.te_q8w), ctypes.sizeof(te.te_q8_item),
                              ctypes.sizeof(te.te_block_desc))
    assert L.te_abi_sizes(None, 0) == 3
    src = open(os.path.join(ROOT, "include", "tefwd.h")).read()
    assert int(re.search(r"#define TE_BLOCK_PROF_EVENTS (\d+)", src).group(1)) == te.TE_BLOCK_PROF_EVENTS
    assert len(te.EncoderStack.STEP_CLASSES) + 1 == te.TE_BLOCK_PROF_EVENTS


FAKE = 0x10000   # never dereferenced: every call below fails validation first


def _call(L, name, *args):
    st = getattr(L, name)(*args)
    return st, L.te_last_error().decode()


def test_q8_linear_rejects_bad_arguments(L):
    item = te.te_q8_item(te.te_q8w(FAKE, FAKE, None, 64, 128), FAKE, 64, te.TE_F32, 0, None, 0)
    arr = (te.te_q8_item * 1)(item)
    st, msg = _call(L, "te_q8_linear", FAKE, 128, 16, 128, arr, 0, None)
    assert st == te.TE_ESHAPE and "z=" in msg
    st, msg = _call(L, "te_q8_linear", FAKE, 128, 16, 100, arr, 1, None)
    assert st == te.TE_ESHAPE and "k=100" in msg
    st, msg = _call(L, "te_q8_linear", FAKE + 2, 128, 16, 128, arr, 1, None)
    assert st == te.TE_EALIGN
    bad_k = (te.te_q8_item * 1)(te.te_q8_item(te.te_q8w(FAKE, FAKE, None, 64, 64), FAKE, 64,
                                              te.TE_F32, 0, None, 0))
    st, msg = _call(L, "te_q8_linear", FAKE, 128, 16, 128, bad_k, 1, None)
    assert st == te.TE_ESHAPE and "item 0" in msg
    bad_n = (te.te_q8_item * 1)(te.te_q8_item(te.te_q8w(FAKE, FAKE, None, 40, 128), FAKE, 64,
                                              te.TE_F32, 0, None, 0))
    assert _call(L, "te_q8_linear", FAKE, 128, 16, 128, bad_n, 1, None)[0] == te.TE_ESHAPE
    inplace_bf16 = (te.te_q8_item * 1)(te.te_q8_item(te.te_q8w(FAKE, FAKE, None, 64, 128), FAKE,
                                                     64, te.TE_BF16, 0, FAKE, 64))
    assert _call(L, "te_q8_linear", FAKE, 128, 16, 128, inplace_bf16, 1, None)[0] == te.TE_EINVAL
    null_y = (te.te_q8_item * 1)(te.te_q8_item(te.te_q8w(FAKE, FAKE, None, 64, 128), None, 64,
                                               te.TE_F32, 0, None, 0))
    assert _call(L, "te_q8_linear", FAKE, 128, 16, 128, null_y, 1, None)[0] == te.TE_EINVAL


def test_gated_linear_and_epilogue_reject_bad_arguments(L):
    wg = te.te_q8w(FAKE, FAKE, None, 256, 128)
    wu = te.te_q8w(FAKE, FAKE, None, 256, 128)
    assert _call(L, "te_q8_gated_linear", FAKE, 128, 16, 128, ctypes.byref(wg), ctypes.byref(wu), 7,
                 FAKE, 256, None)[0] == te.TE_EINVAL                           # bad act
    wu_bad = te.te_q8w(FAKE, FAKE, None, 192, 128)
    st, msg = _call(L, "te_q8_gated_linear", FAKE, 128, 16, 128, ctypes.byref(wg), ctypes.byref(wu_bad),
                    te.TE_ACT_SILU, FAKE, 256, None)
    assert st == te.TE_ESHAPE and "wu" in msg
    assert _call(L, "te_q8_gated_linear", FAKE, 128, 16, 128, ctypes.byref(wg), ctypes.byref(wu),
                 te.TE_ACT_SILU, FAKE + 8, 256, None)[0] == te.TE_EALIGN
    act_res = (te.te_q8_item * 1)(te.te_q8_item(te.te_q8w(FAKE, FAKE, None, 64, 128), FAKE, 64,
                                                te.TE_BF16, te.TE_EPI_SILU, FAKE, 64))
    assert _call(L, "te_q8_linear", FAKE, 128, 16, 128, act_res, 1, None)[0] == te.TE_EINVAL
    bad_epi = (te.te_q8_item * 1)(te.te_q8_item(te.te_q8w(FAKE, FAKE, None, 64, 128), FAKE, 64,
                                                te.TE_BF16, 9, None, 0))
    assert _call(L, "te_q8_linear", FAKE, 128, 16, 128, bad_epi, 1, None)[0] == te.TE_EINVAL


def _cu(vals):
    a = np.asarray(vals, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def test_attention_rejects_bad_cu_seqlens_and_shapes(L):
    a, p = _cu([0, 5, 5, 9])            # an empty sequence
    st, msg = _call(L, "te_attn_varlen_fwd", FAKE, 192, 0, 64, 128, p, FAKE, 3, 1, 1, 64, 0,
                    1.0, FAKE * 4, 64, None)
    assert st == te.TE_EINVAL and "length 0" in msg
    a, p = _cu([1, 5])                   # does not start at 0
    assert _call(L, "te_attn_varlen_fwd", FAKE, 192, 0, 64, 128, p, FAKE, 1, 1, 1, 64, 0, 1.0,
                 FAKE * 4, 64, None)[0] == te.TE_EINVAL
    a, p = _cu([0, 9, 5])                # decreasing
    assert _call(L, "te_attn_varlen_fwd", FAKE, 192, 0, 64, 128, p, FAKE, 2, 1, 1, 64, 0, 1.0,
                 FAKE * 4, 64, None)[0] == te.TE_EINVAL
    a, p = _cu([0, 9])
    assert _call(L, "te_attn_varlen_fwd", FAKE, 288, 0, 96, 192, p, FAKE, 1, 1, 1, 96, 0, 1.0,
                 FAKE * 4, 96, None)[0] == te.TE_ESHAPE                       # hd = 96
    assert _call(L, "te_attn_varlen_fwd", FAKE, 192, 0, 64, 128, p, FAKE, 1, 3, 2, 64, 0, 1.0,
                 FAKE * 4, 192, None)[0] == te.TE_ESHAPE                      # 3 % 2 heads
    assert _call(L, "te_attn_varlen_fwd", FAKE, 192, 0, 64, 128, p, FAKE, 1, 1, 1, 64, -1, 1.0,
                 FAKE * 4, 64, None)[0] == te.TE_EINVAL                       # window < 0
    assert _call(L, "te_attn_varlen_fwd", FAKE, 192, 0, 64, 128, p, FAKE, 1, 1, 1, 64, 0, 1.0,
                 FAKE + 64, 64, None)[0] == te.TE_EINVAL                      # out overlaps qkv
    assert _call(L, "te_attn_varlen_fwd", FAKE, 100, 0, 64, 128, p, FAKE, 1, 1, 1, 64, 0, 1.0,
                 FAKE * 4, 64, None)[0] == te.TE_ESHAPE                       # ld too small


def test_row_ops_reject_bad_arguments(L):
    assert _call(L, "te_rownorm", FAKE, te.TE_F32, 100, FAKE, None, te.TE_NORM_RMS, 1e-6, 1.0,
                 FAKE, te.TE_BF16, 100, 4, 100, None)[0] == te.TE_ESHAPE      # d % 8
    assert _call(L, "te_rownorm", FAKE, te.TE_F32, 64, FAKE, None, 7, 1e-6, 1.0, FAKE, te.TE_BF16,
                 64, 4, 64, None)[0] == te.TE_EINVAL                          # bad kind
    assert _call(L, "te_rownorm", FAKE + 4, te.TE_F32, 64, FAKE, None, te.TE_NORM_RMS, 1e-6, 1.0,
                 FAKE, te.TE_BF16, 64, 4, 64, None)[0] == te.TE_EALIGN
    assert _call(L, "te_add_norm", FAKE, None, FAKE, 1.0, None, None, te.TE_NORM_RMS, 1e-6, None,
                 te.TE_BF16, 4, 64, None)[0] == te.TE_EINVAL                  # w_post without t
    assert _call(L, "te_qk_prep_rope", FAKE, 384, 0, 128, 2, 2, 64, None, None, 1e-6, FAKE, FAKE,
                 None, 4, 48, 1.0, 8, None)[0] == te.TE_ESHAPE                # sec = 48
    assert _call(L, "te_qk_prep_rope", FAKE, 384, 0, 128, 2, 2, 64, None, None, 1e-6, FAKE, FAKE,
                 None, 4, 64, 1.0, 8, None)[0] == te.TE_ESHAPE                # table too short
    assert _call(L, "te_gate_act", FAKE, 64, 60, te.TE_ACT_SILU, FAKE, 32, 4, 32, None)[0] \
        == te.TE_ESHAPE                                                      # u runs past ld
    assert _call(L, "te_gate_act", FAKE, 64, 32, 5, FAKE, 32, 4, 32, None)[0] == te.TE_EINVAL
    a, p = _cu([0, 3, 3])
    assert _call(L, "te_pool_mean", FAKE, 64, p, FAKE, 2, None, 1e-6, FAKE, None)[0] == te.TE_EINVAL


def test_block_formats_reject_bad_arguments(L):
    no_scale = (te.te_q8_item * 1)()
    no_scale[0] = te.te_q8_item(te.te_q8w(FAKE, None, None, 128, 128, None), FAKE, 128, te.TE_F32, 0, None, 0)
    assert _call(L, "te_q8_linear", FAKE, 128, 16, 128, no_scale, 1, None)[0] == te.TE_EINVAL
    bad_bs = (te.te_q8_item * 1)()
    bad_bs[0] = te.te_q8_item(te.te_q8w(FAKE, None, None, 128, 128, FAKE + 2), FAKE, 128, te.TE_F32, 0, None, 0)
    assert _call(L, "te_q8_linear", FAKE, 128, 16, 128, bad_bs, 1, None)[0] == te.TE_EALIGN
    assert _call(L, "te_q8_0_unpack", FAKE, 4, 48, FAKE, FAKE, None)[0] == te.TE_ESHAPE      # k % 32
    assert _call(L, "te_q4_0_unpack", FAKE + 1, 4, 64, FAKE, FAKE, None)[0] == te.TE_EALIGN
    assert _call(L, "te_q8_0_unpack", None, 4, 64, FAKE, FAKE, None)[0] == te.TE_EINVAL


def test_attention_items_reject_bad_arguments(L):
    import numpy as np
    def items(*rows):
        arr = np.asarray(rows, np.int32).reshape(-1, 4)
        return arr, arr.ctypes.data_as(ctypes.c_void_p)
    a, p = items([0, 33, 40, 10])                     # first range not a multiple of 32
    assert _call(L, "te_attn_items_fwd", FAKE, 384, 0, 128, 256, p, FAKE, 1, 100, 2, 2, 64, 0, 0.125,
                 FAKE * 2, 128, None)[0] == te.TE_ESHAPE
    a, p = items([0, 32, 90, 20])                     # second range past the rows
    assert _call(L, "te_attn_items_fwd", FAKE, 384, 0, 128, 256, p, FAKE, 1, 100, 2, 2, 64, 0, 0.125,
                 FAKE * 2, 128, None)[0] == te.TE_EINVAL
    a, p = items([0, 32, 40, 20])                     # items on the device must be 16-byte aligned
    assert _call(L, "te_attn_items_fwd", FAKE, 384, 0, 128, 256, p, FAKE + 4, 1, 100, 2, 2, 64, 0,
                 0.125, FAKE * 2, 128, None)[0] == te.TE_EALIGN


def test_adaln_row_ops_reject_bad_arguments(L):
    # scale without a next norm, gate without a branch, misaligned vectors
    assert _call(L, "te_add_norm_mod", FAKE, FAKE, FAKE, None, 1.0, None, None, FAKE, te.TE_NORM_RMS,
                 1e-6, None, te.TE_BF16, 4, 64, None)[0] == te.TE_EINVAL
    assert _call(L, "te_add_norm_mod", FAKE, None, None, FAKE, 1.0, None, None, None, te.TE_NORM_RMS,
                 1e-6, None, te.TE_BF16, 4, 64, None)[0] == te.TE_EINVAL
    assert _call(L, "te_add_norm_mod", FAKE, FAKE, FAKE, FAKE + 4, 1.0, FAKE, None, None,
                 te.TE_NORM_RMS, 1e-6, FAKE, te.TE_BF16, 4, 64, None)[0] == te.TE_EALIGN
    assert _call(L, "te_rownorm_mod", FAKE, te.TE_F32, 64, FAKE, None, FAKE + 8, te.TE_NORM_RMS,
                 1e-6, 1.0, FAKE, te.TE_BF16, 64, 4, 64, None)[0] == te.TE_EALIGN
    assert _call(L, "te_rownorm_mod", FAKE, te.TE_F32, 100, FAKE, None, FAKE, te.TE_NORM_RMS,
                 1e-6, 1.0, FAKE, te.TE_BF16, 100, 4, 100, None)[0] == te.TE_ESHAPE


def _desc(**over):
    d = te.te_block_desc()
    d.d, d.n_heads, d.n_kv_heads, d.head_dim, d.ffn = 256, 4, 4, 64, 1024
    d.gated, d.eps, d.attn_scale, d.post = 1, 1e-6, 0.125, 1.0
    for key, (n, k) in dict(wq=(256, 256), wk=(256, 256), wv=(256, 256), wo=(256, 256),
                            wg=(1024, 256), wu=(1024, 256), wd=(256, 1024)).items():
        setattr(d, key, te.te_q8w(FAKE, FAKE, None, n, k))
    d.ffn_norm_w = FAKE
    for k, v in over.items():
        setattr(d, k, v)
    return d


def test_block_validation_and_workspace(L):
    a, p = _cu([0, 37, 101])
    d = _desc()
    ws = L.te_encoder_block_workspace(ctypes.byref(d), 101)
    expect = sum(((101 * w + 255) // 256) * 256 for w in (768 * 2, 256 * 2, 256 * 4, 1024 * 2))
    assert ws == expect
    st, msg = _call(L, "te_encoder_block_fwd", ctypes.byref(d), FAKE, FAKE, p, FAKE, 2, FAKE * 256,
                    ws - 1, None)
    assert st == te.TE_EWORKSPACE
    bad = _desc(wo=te.te_q8w(FAKE, FAKE, None, 256, 512))
    st, msg = _call(L, "te_encoder_block_fwd", ctypes.byref(bad), FAKE, FAKE, p, FAKE, 2,
                    FAKE * 256, ws, None)
    assert st == te.TE_ESHAPE and "wo" in msg
    sand = _desc(resid_form=te.TE_RESID_SANDWICH)
    assert _call(L, "te_encoder_block_fwd", ctypes.byref(sand), FAKE, FAKE, p, FAKE, 2,
                 FAKE * 256, ws, None)[0] == te.TE_EINVAL
    qn_only = _desc(q_norm=FAKE)
    assert _call(L, "te_encoder_block_fwd", ctypes.byref(qn_only), FAKE, FAKE, p, FAKE, 2,
                 FAKE * 256, ws, None)[0] == te.TE_EINVAL
    unal = _desc()
    assert _call(L, "te_encoder_block_fwd", ctypes.byref(unal), FAKE, FAKE, p, FAKE, 2,
                 FAKE * 256 + 16, ws, None)[0] == te.TE_EALIGN
    # adaLN modulation: sandwich form only, aligned, next scale needs a next norm
    plain_mod = _desc(mod=FAKE)
    assert _call(L, "te_encoder_block_fwd", ctypes.byref(plain_mod), FAKE, FAKE, p, FAKE, 2,
                 FAKE * 256, ws, None)[0] == te.TE_EINVAL
    sand_ok = dict(resid_form=te.TE_RESID_SANDWICH, post_attn_w=FAKE, post_ffn_w=FAKE)
    mod_unal = _desc(mod=FAKE + 4, **sand_ok)
    assert _call(L, "te_encoder_block_fwd", ctypes.byref(mod_unal), FAKE, FAKE, p, FAKE, 2,
                 FAKE * 256, ws, None)[0] == te.TE_EALIGN
    plain_ple = _desc(ple_dim=64, ple_norm_w=FAKE, ple_post_w=FAKE, ple_x=FAKE)
    assert _call(L, "te_encoder_block_fwd", ctypes.byref(plain_ple), FAKE, FAKE, p, FAKE, 2,
                 FAKE * 256, ws, None)[0] == te.TE_EINVAL
    odd_ple = _desc(ple_dim=100, **sand_ok)
    assert _call(L, "te_encoder_block_fwd", ctypes.byref(odd_ple), FAKE, FAKE, p, FAKE, 2,
                 FAKE * 256, ws, None)[0] == te.TE_ESHAPE
    next_s_only = _desc(mod=FAKE, next_mod_scale=FAKE, **sand_ok)
    assert _call(L, "te_encoder_block_fwd", ctypes.byref(next_s_only), FAKE, FAKE, p, FAKE, 2,
                 FAKE * 256, ws, None)[0] == te.TE_EINVAL


def test_mma_peak_rejects_bad_arguments(L):
    ms = ctypes.c_float(0.0)
    st, msg = _call(L, "te_mma_peak", 100, 10, ctypes.byref(ms), None)
    assert st == te.TE_EINVAL and "bn=100" in msg
    st, msg = _call(L, "te_mma_peak", 192, 0, ctypes.byref(ms), None)
    assert st == te.TE_EINVAL and "stages=0" in msg
    assert _call(L, "te_mma_peak", 192, 10, None, None)[0] == te.TE_EINVAL
