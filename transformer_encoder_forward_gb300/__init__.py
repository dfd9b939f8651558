"""Python binding of libtefwd (the C-ABI in include/tefwd.h).

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of libtefwd.so.  PyTorch supplies device memory and the current CUDA
stream.  There is no CPU or library fallback: if the shared library is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtefwd.so")

TE_OK, TE_EINVAL, TE_ESHAPE, TE_EALIGN, TE_EWORKSPACE, TE_ECUDA, TE_EDEVICE = range(7)
TE_F32, TE_BF16 = 0, 1
TE_NORM_RMS, TE_NORM_LN = 0, 1
TE_ACT_GELU_TANH, TE_ACT_SILU = 0, 1
TE_RESID_PLAIN, TE_RESID_SANDWICH = 0, 1
TE_EPI_NONE, TE_EPI_GELU_TANH, TE_EPI_SILU = 0, 1, 2
# TE_STATIC_SCRATCH_BYTES of tefwd.h: the scratch array of te_encoder_block_fwd_static
TE_STATIC_SCRATCH_BYTES = 32 << 20
# TE_BLOCK_PROF_EVENTS of tefwd.h: the step-boundary events of te_block_desc.prof_events
TE_BLOCK_PROF_EVENTS = 9

_STATUS = {0: "TE_OK", 1: "TE_EINVAL", 2: "TE_ESHAPE", 3: "TE_EALIGN", 4: "TE_EWORKSPACE",
           5: "TE_ECUDA", 6: "TE_EDEVICE"}


class TEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


c_i32, c_i64, c_f32, c_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p


class te_q8w(ctypes.Structure):
    _fields_ = [("q", c_p), ("scale", c_p), ("bias", c_p), ("n", c_i32), ("k", c_i32),
                ("block_scale", c_p), ("col", c_p)]


class te_q8_item(ctypes.Structure):
    _fields_ = [("w", te_q8w), ("y", c_p), ("ldy", c_i64), ("y_dtype", c_i32),
                ("epilogue", c_i32), ("residual", c_p), ("ldr", c_i64)]


class te_block_desc(ctypes.Structure):
    _fields_ = [("d", c_i32), ("n_heads", c_i32), ("n_kv_heads", c_i32), ("head_dim", c_i32),
                ("ffn", c_i32), ("norm_kind", c_i32), ("resid_form", c_i32), ("act", c_i32),
                ("gated", c_i32), ("window", c_i32), ("eps", c_f32), ("attn_scale", c_f32),
                ("post", c_f32), ("q_mul", c_f32),
                ("wq", te_q8w), ("wk", te_q8w), ("wv", te_q8w), ("wo", te_q8w), ("wg", te_q8w),
                ("wu", te_q8w), ("wd", te_q8w),
                ("ffn_norm_w", c_p), ("ffn_norm_b", c_p), ("post_attn_w", c_p),
                ("post_ffn_w", c_p), ("next_norm_w", c_p), ("next_norm_b", c_p),
                ("q_norm", c_p), ("k_norm", c_p), ("rope_cos", c_p), ("rope_sin", c_p),
                ("rope_pos", c_p), ("rope_sec", c_i32), ("rope_rows", c_i32),
                ("mod", c_p), ("next_mod_scale", c_p), ("v_norm", c_i32),
                ("ple_dim", c_i32), ("ple_scale", c_f32), ("ple_in", te_q8w), ("ple_gate", te_q8w),
                ("ple_proj", te_q8w), ("ple_norm_w", c_p), ("ple_post_w", c_p), ("ple_x", c_p),
                ("attn_items_host", c_p), ("attn_items_dev", c_p), ("n_attn_items", c_i32),
                ("prof_events", c_p)]


_lib = None

EXPORTS = {
    "te_q8_linear": (ctypes.c_int, [c_p, c_i64, c_i32, c_i32, ctypes.POINTER(te_q8_item), c_i32, c_p]),
    "te_q8_gated_linear": (ctypes.c_int, [c_p, c_i64, c_i32, c_i32, ctypes.POINTER(te_q8w),
                                          ctypes.POINTER(te_q8w), c_i32, c_p, c_i64, c_p]),
    "te_attn_varlen_fwd": (ctypes.c_int, [c_p, c_i64, c_i32, c_i32, c_i32, c_p, c_p, c_i32, c_i32,
                                          c_i32, c_i32, c_i32, c_f32, c_p, c_i64, c_p]),
    "te_attn_items_fwd": (ctypes.c_int, [c_p, c_i64, c_i32, c_i32, c_i32, c_p, c_p, c_i32, c_i32,
                                         c_i32, c_i32, c_i32, c_i32, c_f32, c_p, c_i64, c_p]),
    "te_rownorm": (ctypes.c_int, [c_p, c_i32, c_i64, c_p, c_p, c_i32, c_f32, c_f32, c_p, c_i32,
                                  c_i64, c_i32, c_i32, c_p]),
    "te_add_norm": (ctypes.c_int, [c_p, c_p, c_p, c_f32, c_p, c_p, c_i32, c_f32, c_p, c_i32, c_i32,
                                   c_i32, c_p]),
    "te_q8_0_unpack": (ctypes.c_int, [c_p, c_i32, c_i32, c_p, c_p, c_p]),
    "te_q4_0_unpack": (ctypes.c_int, [c_p, c_i32, c_i32, c_p, c_p, c_p]),
    "te_rownorm_mod": (ctypes.c_int, [c_p, c_i32, c_i64, c_p, c_p, c_p, c_i32, c_f32, c_f32, c_p,
                                      c_i32, c_i64, c_i32, c_i32, c_p]),
    "te_add_norm_mod": (ctypes.c_int, [c_p, c_p, c_p, c_p, c_f32, c_p, c_p, c_p, c_i32, c_f32, c_p,
                                       c_i32, c_i32, c_i32, c_p]),
    "te_qk_prep_rope": (ctypes.c_int, [c_p, c_i64, c_i32, c_i32, c_i32, c_i32, c_i32, c_p, c_p,
                                       c_f32, c_p, c_p, c_p, c_i32, c_i32, c_f32, c_i32, c_p]),
    "te_qkv_prep_rope": (ctypes.c_int, [c_p, c_i64, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_p,
                                        c_p, c_i32, c_f32, c_p, c_p, c_p, c_i32, c_i32, c_f32, c_i32,
                                        c_p]),
    "te_selftest_wait_timeout": (ctypes.c_int, [c_i32, c_p]),
    "te_mma_peak": (ctypes.c_int, [c_i32, c_i32, c_p, c_p]),
    "te_cast_bf16": (ctypes.c_int, [c_p, c_i64, c_p, c_i64, c_i32, c_i32, c_p]),
    "te_gate_act": (ctypes.c_int, [c_p, c_i64, c_i32, c_i32, c_p, c_i64, c_i32, c_i32, c_p]),
    "te_pool_mean": (ctypes.c_int, [c_p, c_i32, c_p, c_p, c_i32, c_p, c_f32, c_p, c_p]),
    "te_encoder_block_workspace": (ctypes.c_size_t, [ctypes.POINTER(te_block_desc), c_i32]),
    "te_encoder_block_fwd": (ctypes.c_int, [ctypes.POINTER(te_block_desc), c_p, c_p, c_p, c_p, c_i32,
                                            c_p, ctypes.c_size_t, c_p]),
    "te_encoder_block_fwd_static": (ctypes.c_int, [ctypes.POINTER(te_block_desc), c_p, c_p, c_p,
                                                   c_p, c_i32, c_p]),
    "te_check": (ctypes.c_int, [c_p]),
    "te_last_error": (ctypes.c_char_p, []),
    "te_version": (ctypes.c_char_p, []),
    "te_abi_sizes": (c_i32, [ctypes.POINTER(ctypes.c_size_t), c_i32]),
}


def lib() -> ctypes.CDLL:
    """The loaded libtefwd.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtefwd.so is not built ({LIB_PATH}); run "
                               "python -m transformer_encoder_forward_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ok(st: int):
    if st != TE_OK:
        raise TEError(st, lib().te_last_error().decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _host_i32(a):
    """A host int32 array pointer for cu_seqlens (numpy array or CPU tensor)."""
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr, arr.ctypes.data_as(c_p)


# --------------------------------------------------------------------- ops

def q8w(q, s, b=None, block_scale=None, col=None) -> te_q8w:
    """Descriptor of one quantised weight held in device tensors (q int8
    [n, k], s f32 [n] or None, optional b f32 [n]; block_scale: f16 bits
    [n, k/32] for the 32-element block formats; col: f32 [k], the q8_2f
    column field; both None for q8_row)."""
    return te_q8w(_ptr(q), _ptr(s), _ptr(b), q.shape[0], q.shape[1], _ptr(block_scale), _ptr(col))


def q8_0_unpack(packed, n, k, q, block_scale, stream=None):
    """Packed Q8_0 bytes (uint8 device tensor) -> q int8 [n, k], block_scale [n, k/32]."""
    _ok(lib().te_q8_0_unpack(packed.data_ptr(), n, k, q.data_ptr(), block_scale.data_ptr(),
                             _stream(stream)))


def q4_0_unpack(packed, n, k, q, block_scale, stream=None):
    """Packed Q4_0 bytes (uint8 device tensor) -> q int8 [n, k], block_scale [n, k/32]."""
    _ok(lib().te_q4_0_unpack(packed.data_ptr(), n, k, q.data_ptr(), block_scale.data_ptr(),
                             _stream(stream)))


def q8_linear(x, items: Sequence[dict], stream=None):
    """Grouped q8 GEMM.  items: dicts with keys w (te_q8w), y (tensor view
    whose data_ptr is the first output element), ldy, optional residual/ldr.
    y_dtype follows the tensor's dtype."""
    import torch
    arr = (te_q8_item * len(items))()
    for i, it in enumerate(items):
        y = it["y"]
        r = it.get("residual")
        arr[i] = te_q8_item(it["w"], y.data_ptr(), it["ldy"],
                            TE_F32 if y.dtype == torch.float32 else TE_BF16,
                            it.get("epilogue", TE_EPI_NONE), _ptr(r), it.get("ldr", 0))
    _ok(lib().te_q8_linear(x.data_ptr(), it_ld(x), x.shape[0], x.shape[1], arr, len(items),
                           _stream(stream)))


def q8_gated_linear(x, wg: te_q8w, wu: te_q8w, act, out, stream=None):
    """m = act(bf16(x Wg^T)) * bf16(x Wu^T) in one GEMM (bf16 out)."""
    _ok(lib().te_q8_gated_linear(x.data_ptr(), x.stride(0), x.shape[0], x.shape[1],
                                 ctypes.byref(wg), ctypes.byref(wu), act, out.data_ptr(),
                                 out.stride(0), _stream(stream)))


def it_ld(t) -> int:
    return t.stride(0)


def attn_varlen_fwd(qkv, ld, q_off, k_off, v_off, cu_host, cu_dev, nq, nkv, hd, window, scale,
                    out, ldo, stream=None):
    arr, hp = _host_i32(cu_host)
    _ok(lib().te_attn_varlen_fwd(qkv.data_ptr(), ld, q_off, k_off, v_off, hp, cu_dev.data_ptr(),
                                 len(arr) - 1, nq, nkv, hd, window, scale, out.data_ptr(), ldo,
                                 _stream(stream)))


def attn_items_fwd(qkv, ld, q_off, k_off, v_off, items_host, items_dev, rows, nq, nkv, hd, window,
                   scale, out, ldo, stream=None):
    """Attention over two-range items: items int32 [n, 4] = off1, len1, off2, len2
    (host numpy array and the same on the device)."""
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(items_host, dtype=np.int32).reshape(-1, 4))
    _ok(lib().te_attn_items_fwd(qkv.data_ptr(), ld, q_off, k_off, v_off, arr.ctypes.data_as(c_p),
                                items_dev.data_ptr(), arr.shape[0], rows, nq, nkv, hd, window, scale,
                                out.data_ptr(), ldo, _stream(stream)))


def selftest_wait_timeout(limit_us, stream=None):
    """Launch the bounded-wait self-test (a wait that can only time out)."""
    _ok(lib().te_selftest_wait_timeout(limit_us, _stream(stream)))


def mma_peak(bn, stages, stream=None):
    """Device ms of `stages` x 8 back-to-back 2-SM MMAs (N = bn) on every SM
    pair: the q8 GEMM's tensor ceiling without loads (te_mma_peak)."""
    ms = ctypes.c_float(0.0)
    _ok(lib().te_mma_peak(bn, stages, ctypes.byref(ms), _stream(stream)))
    return float(ms.value)


def sm_count(device=0):
    import torch
    return torch.cuda.get_device_properties(device).multi_processor_count


def cast_bf16(x, y, stream=None):
    """y (bf16) = x (f32), rows of the same width."""
    _ok(lib().te_cast_bf16(x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0), x.shape[0], x.shape[1],
                           _stream(stream)))


def _dt(t) -> int:
    import torch
    return TE_F32 if t.dtype == torch.float32 else TE_BF16


def rownorm(x, w, b, kind, eps, y, pre=1.0, stream=None):
    _ok(lib().te_rownorm(x.data_ptr(), _dt(x), x.stride(0), _ptr(w), _ptr(b), kind, eps, pre,
                         y.data_ptr(), _dt(y), y.stride(0), x.shape[0], x.shape[1],
                         _stream(stream)))


def add_norm(h, t, w_post, post, w_next, b_next, kind, eps, a, stream=None):
    _ok(lib().te_add_norm(h.data_ptr(), _ptr(t), _ptr(w_post), post, _ptr(w_next), _ptr(b_next),
                          kind, eps, _ptr(a), _dt(a) if a is not None else TE_BF16, h.shape[0],
                          h.shape[1], _stream(stream)))


def rownorm_mod(x, w, b, mod_scale, kind, eps, y, pre=1.0, stream=None):
    """rownorm with the adaLN scale: y = (Norm(x) w (+b)) (1 + mod_scale)."""
    _ok(lib().te_rownorm_mod(x.data_ptr(), _dt(x), x.stride(0), _ptr(w), _ptr(b), _ptr(mod_scale),
                             kind, eps, pre, y.data_ptr(), _dt(y), y.stride(0), x.shape[0],
                             x.shape[1], _stream(stream)))


def add_norm_mod(h, t, w_post, gate, post, w_next, b_next, mod_scale, kind, eps, a, stream=None):
    """add_norm with the adaLN gate on the branch and scale on the next norm."""
    _ok(lib().te_add_norm_mod(h.data_ptr(), _ptr(t), _ptr(w_post), _ptr(gate), post, _ptr(w_next),
                              _ptr(b_next), _ptr(mod_scale), kind, eps, _ptr(a),
                              _dt(a) if a is not None else TE_BF16, h.shape[0], h.shape[1],
                              _stream(stream)))


def qkv_prep_rope(qkv, ld, q_off, k_off, v_off, nq, nkv, hd, qn, kn, v_norm, eps, cos, sin, pos,
                  sec, q_mul, rows, stream=None):
    """qk_prep_rope plus (v_norm) the unweighted RMS norm of the v heads."""
    table_rows = cos.shape[0] if cos is not None else 0
    _ok(lib().te_qkv_prep_rope(qkv.data_ptr(), ld, q_off, k_off, v_off, nq, nkv, hd, _ptr(qn),
                               _ptr(kn), 1 if v_norm else 0, eps, _ptr(cos), _ptr(sin), _ptr(pos),
                               table_rows, sec, q_mul, rows, _stream(stream)))


def qk_prep_rope(qkv, ld, q_off, k_off, nq, nkv, hd, qn, kn, eps, cos, sin, pos, sec, q_mul,
                 rows, stream=None):
    table_rows = cos.shape[0] if cos is not None else 0
    _ok(lib().te_qk_prep_rope(qkv.data_ptr(), ld, q_off, k_off, nq, nkv, hd, _ptr(qn), _ptr(kn),
                              eps, _ptr(cos), _ptr(sin), _ptr(pos), table_rows, sec, q_mul, rows,
                              _stream(stream)))


def gate_act(gu, ld, u_off, act, m, ldm, rows, f, stream=None):
    _ok(lib().te_gate_act(gu.data_ptr(), ld, u_off, act, m.data_ptr(), ldm, rows, f,
                          _stream(stream)))


def pool_mean(x, cu_host, cu_dev, w_final, eps, out, stream=None):
    arr, hp = _host_i32(cu_host)
    _ok(lib().te_pool_mean(x.data_ptr(), x.shape[1], hp, cu_dev.data_ptr(), len(arr) - 1,
                           _ptr(w_final), eps, out.data_ptr(), _stream(stream)))


def block_workspace(desc: te_block_desc, t: int) -> int:
    return int(lib().te_encoder_block_workspace(ctypes.byref(desc), t))


def encoder_block_fwd(desc: te_block_desc, x, a, cu_host, cu_dev, workspace, stream=None):
    arr, hp = _host_i32(cu_host)
    _ok(lib().te_encoder_block_fwd(ctypes.byref(desc), x.data_ptr(), a.data_ptr(), hp,
                                   cu_dev.data_ptr(), len(arr) - 1, workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))


def encoder_block_fwd_static(desc: te_block_desc, x, a, cu_host, cu_dev, stream=None):
    """The block with the library's fixed scratch array instead of a
    workspace (for callers that cannot allocate device memory)."""
    arr, hp = _host_i32(cu_host)
    _ok(lib().te_encoder_block_fwd_static(ctypes.byref(desc), x.data_ptr(), a.data_ptr(), hp,
                                          cu_dev.data_ptr(), len(arr) - 1, _stream(stream)))


def check(stream=None):
    """Synchronises the stream and raises on a pending CUDA error or a
    device-side error word (bounded wait timeout, bad RoPE index)."""
    _ok(lib().te_check(_stream(stream)))


def version() -> str:
    return lib().te_version().decode()


def abi_sizes():
    """(sizeof te_q8w, te_q8_item, te_block_desc) as the library was compiled."""
    out = (ctypes.c_size_t * 3)()
    n = lib().te_abi_sizes(out, 3)
    return tuple(int(v) for v in out[:n])


from .model import EncoderStack, LayerWeights  # noqa: E402,F401
