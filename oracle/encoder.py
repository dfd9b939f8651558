"""CPU oracle of the pre-norm transformer encoder block forward (f64).

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
baseline leg may import this module.  It shares no code with the CUDA
library and imports nothing from it: it is the plain definition of what the
library computes, written out with numpy in float64 so that a reader can check
it against the pages by eye.

Sources (the three pages the method is described on):

* "cortiq-engine 0.8.39 src/gpu_metal/egemma2.rs" - the EmbeddingGemma 2
  text and vision encoders on Metal: the program builder (``Prog::rms``,
  ``Prog::add_norm``, ``Prog::gelu``, ``Prog::qkv``, ``Prog::attention``),
  ``att_plan`` (sliding-window key span) and ``TextGpu::forward`` (the layer
  loop, final norm and mean-pool).
* "cortiq-engine 0.7.6 src/gpu_metal/zimage.rs" - the Z-Image DiT on Metal:
  the module doc (q8_row weights, "Measured"), ``Enc::block`` / ``Enc::rowop``
  (post-norm residual + next pre-norm, q/k norm + RoPE, SwiGLU) and
  ``bench_gemm`` / ``bench_flash`` (their f64 host checks).
* "cera 0.2.4 src/model/vision_encoder_gpu.rs" - the LFM2-VL ViT encoder:
  ``trait VitGpuOps`` (layernorm, gelu, attention, bias_add, add) and the block
  loop of ``encode_image_gpu``.

Storage precision (the CUDA path stores these, so the oracle rounds at the
same points): the residual stream and the outputs of the O and down
projections that feed a norm are f32; normed activations, the q|k|v panel,
the attention output, the gate|up output and the FFN hidden are bf16
(round-to-nearest-even).  Everything between two storage points is f64 here.

Readings where the pages are silent or ambiguous:
RMSNorm multiplies by the stored weight (not 1 + w) with eps inside the root;
LayerNorm uses the biased variance; a key j is visible to query i iff both
lie in the same sequence and (window == 0 or |i - j| <= window); q/k norm is
applied before RoPE; RoPE is rotate-half within sections of ``sec`` channels;
the first half of the gate|up panel is the gate; pooling divides by the
sequence length after the final norm; the DiT's adaLN scale s multiplies a
normed row by (1 + s) and its gate g multiplies the post-normed branch before
the residual add (the pages print only the vectors' layout and that the
unmodulated block is s = 0, gate = 1).

Parity pins: every function here is pinned in tests/test_oracle.py against
something other than itself (brute-force loops, closed forms, invariants or
a library routine).  The whole block has no worked example on the pages;
its parity rests on the pinned parts plus block-level invariants.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# storage rounding


def round_bf16(a):
    """Round to the nearest bfloat16 value, ties to even; returned as f64.

    bfloat16 keeps 8 significant bits and float32's exponent range, so the
    quantum of a value with binary exponent e (a = m*2^e, 0.5 <= |m| < 1) is
    2^(e-8); below the smallest normal (2^-126) the quantum stays 2^-133.
    A result that reaches 2^128 is past the largest finite value: infinity.
    """
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)
    e = np.maximum(e, -125)
    quantum = np.ldexp(1.0, e - 8)
    out = np.rint(a / quantum) * quantum
    return np.where(np.abs(out) >= 2.0 ** 128, np.copysign(np.inf, a), out)


def round_f32(a):
    """Round to the nearest float32 (ties to even); returned as f64."""
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def widen_int8(q):
    """int8 -> real value; every int8 is exact in bf16, f32 and f64
    (zimage.rs module doc: the int8 tile is staged as half "exact")."""
    return np.asarray(q, dtype=np.int8).astype(np.float64)


# ---------------------------------------------------------------------------
# q8_row linear


def q8_linear(x, q, s, b=None, residual=None):
    """y[t, o] = s[o] * sum_k x[t, k] * q[o, k]  (+ b[o])  (+ residual[t, o]).

    q8_row weights: int8 [n, k] row-major and one scale per output row,
    dequantised as W[o, k] = s[o] * q[o, k] (zimage.rs module doc; the f64
    form of ``bench_gemm``'s host check).  The bias follows the ViT's biased
    linears (``bias_add`` of ``VitGpuOps``), the residual the plain pre-norm
    block's ``x += proj`` (``encode_image_gpu``).
    """
    x = np.asarray(x, dtype=np.float64)
    y = (x @ widen_int8(q).T) * np.asarray(s, dtype=np.float64)[None, :]
    if b is not None:
        y = y + np.asarray(b, dtype=np.float64)[None, :]
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float64)
    return y


# ---------------------------------------------------------------------------
# norms


def decode_q8_0(packed, n, k):
    """Q8_0 bytes -> (q int8 [n, k], d f64 [n, k/32]) (vision_encoder_gpu.rs
    ``q8_0_weight``: 34 bytes a block, the f16 scale first, then 32 int8)."""
    raw = np.frombuffer(bytes(packed), dtype=np.uint8).reshape(n, k // 32, 34)
    d = raw[:, :, 0:2].copy().view("<f2")[:, :, 0].astype(np.float64)
    q = raw[:, :, 2:].copy().view(np.int8).reshape(n, k)
    return q, d


def decode_q4_0(packed, n, k):
    """Q4_0 bytes -> (q int8 [n, k] in [-8, 7], d f64 [n, k/32])
    (``q4_0_weight``: 18 bytes a block, the f16 scale, then 16 bytes whose
    low nibble is element i and high nibble element i + 16, stored + 8)."""
    raw = np.frombuffer(bytes(packed), dtype=np.uint8).reshape(n, k // 32, 18)
    d = raw[:, :, 0:2].copy().view("<f2")[:, :, 0].astype(np.float64)
    by = raw[:, :, 2:].astype(np.int16)
    q = np.concatenate([(by & 15) - 8, (by >> 4) - 8], axis=2).astype(np.int8).reshape(n, k)
    return q, d


def q8_block_linear(x, q, d, s=None, b=None):
    """The GEMM with 32-element block scales: y[t, o] = s[o] * sum_k x[t, k] *
    bf16(q[o, k] * d[o, k // 32]) (+ b[o]).  The library feeds the tensor
    cores bf16 operands, so the dequantised weight is rounded once to bf16
    (q * d itself is exact); s = None is 1."""
    q = widen_int8(q)
    n, k = q.shape
    wdq = round_bf16(q * np.repeat(np.asarray(d, dtype=np.float64), 32, axis=1)[:, :k])
    y = np.asarray(x, dtype=np.float64) @ wdq.T
    if s is not None:
        y = y * np.asarray(s, dtype=np.float64)[None, :]
    if b is not None:
        y = y + np.asarray(b, dtype=np.float64)[None, :]
    return y


def q8_2f_linear(x, q, col, s, b=None, residual=None):
    """The q8_2f GEMM: y[t, o] = s[o] * sum_k x[t, k] * bf16(q[o, k] * col[k])
    (+ b[o]) (+ residual).  zimage.rs ``ensure_dev`` (q8_2f = q8_row bytes +
    f16 row scales + an f16 field per column); the library folds the column
    field into the widened weight and rounds that product once to the bf16
    tensor-core operand."""
    wq = round_bf16(widen_int8(q) * np.asarray(col, dtype=np.float64)[None, :])
    y = np.asarray(x, dtype=np.float64) @ wq.T
    y = y * np.asarray(s, dtype=np.float64)[None, :]
    if b is not None:
        y = y + np.asarray(b, dtype=np.float64)[None, :]
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float64)
    return y


def linear(x, w, residual=None):
    """One projection of the block in its weight's format: q8_row
    (``q8_linear``) or the packed 32-element block formats (decoded, then
    ``q8_block_linear``)."""
    if "packed" in w:
        dec = decode_q8_0 if w["fmt"] == "q8_0" else decode_q4_0
        q, d = dec(w["packed"], w["n"], w["k"])
        y = q8_block_linear(x, q, d, w.get("s"), w.get("b"))
        return y if residual is None else y + np.asarray(residual, dtype=np.float64)
    if w.get("col") is not None:
        return q8_2f_linear(x, w["q"], w["col"], w["s"], w["b"], residual=residual)
    return q8_linear(x, w["q"], w["s"], w["b"], residual=residual)


def rms_norm(x, w, eps, pre=1.0):
    """y = rms(pre*x) * w with rms(v) = v / sqrt(mean(v^2) + eps)
    (egemma2.rs ``Prog::rms``; the weight multiplies as stored)."""
    v = pre * np.asarray(x, dtype=np.float64)
    inv = 1.0 / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)
    return v * inv * np.asarray(w, dtype=np.float64)


def layer_norm(x, w, b, eps):
    """(x - mean) * inv_std * w + b per row, biased variance
    (vision_encoder_gpu.rs ``VitGpuOps::layernorm``)."""
    x = np.asarray(x, dtype=np.float64)
    mu = np.mean(x, axis=-1, keepdims=True)
    var = np.mean((x - mu) ** 2, axis=-1, keepdims=True)
    y = (x - mu) / np.sqrt(var + eps) * np.asarray(w, dtype=np.float64)
    if b is not None:
        y = y + np.asarray(b, dtype=np.float64)
    return y


def norm(kind, x, w, b, eps, mod_scale=None):
    """The block's pre-norm; with the DiT's adaLN scale s the normed row is
    then multiplied by (1 + s) (zimage.rs ``Enc::rowop`` pre mode with
    ``has_s``; ``refine_caption``: unmodulated is s = 0)."""
    if kind == "rms":
        y = rms_norm(x, w, eps)
    elif kind == "ln":
        y = layer_norm(x, w, b, eps)
    else:
        raise ValueError(kind)
    if mod_scale is not None:
        y = y * (1.0 + np.asarray(mod_scale, dtype=np.float64))
    return y


def add_norm_sandwich(h, t, w_post, post, eps, gate=None):
    """H = (H + g * rms(T) * w_post) * post  (egemma2.rs ``Prog::add_norm``;
    zimage.rs ``Enc::rowop`` post-norm mode, the adaLN gate g with ``has_g``;
    unmodulated g = 1)."""
    branch = rms_norm(t, w_post, eps)
    if gate is not None:
        branch = branch * np.asarray(gate, dtype=np.float64)
    return (np.asarray(h, dtype=np.float64) + branch) * post


# ---------------------------------------------------------------------------
# q/k norm + RoPE


def rope(x, cos, sin, sec):
    """Rotate-half RoPE within each section of ``sec`` channels.

    x: [rows, hd]; cos/sin: [rows, hd/2] (each row's angles).  For section s
    and i < sec/2 the pair (x[s*sec+i], x[s*sec+i+sec/2]) rotates by the angle
    at table column s*sec/2 + i (egemma2.rs ``EgQkv.sec``: 1-D uses sec = hd,
    the vision tower's 2-D form sec = hd/2, "the column half, then the row
    half").
    """
    x = np.asarray(x, dtype=np.float64)
    cos = np.asarray(cos, dtype=np.float64)
    sin = np.asarray(sin, dtype=np.float64)
    hd = x.shape[-1]
    half = sec // 2
    out = np.empty_like(x)
    for sct in range(hd // sec):
        x1 = x[:, sct * sec: sct * sec + half]
        x2 = x[:, sct * sec + half: (sct + 1) * sec]
        c = cos[:, sct * half: (sct + 1) * half]
        s = sin[:, sct * half: (sct + 1) * half]
        out[:, sct * sec: sct * sec + half] = x1 * c - x2 * s
        out[:, sct * sec + half: (sct + 1) * sec] = x2 * c + x1 * s
    return out


def qk_prep(qkv, nq, nkv, hd, q_off, k_off, qn, kn, eps, cos, sin, pos, sec, q_mul,
            v_off=None):
    """q/k RMSNorm per head with [hd] weights, then RoPE, then q * q_mul;
    the panel is returned rounded to bf16 (egemma2.rs ``Prog::qkv``;
    zimage.rs ``Enc::block`` "qk-norm + RoPE in place", q pre-multiplied).
    With ``v_off`` the v heads are RMS-normalised too, without a weight and
    without RoPE (egemma2.rs ``Prog::qkv`` "v norm": the pass covers the
    nq + 2 nkv heads and takes weights for q and k only).

    ``pos`` selects each row's table row (None = the row index).
    """
    out = np.array(qkv, dtype=np.float64, copy=True)
    rows = out.shape[0]
    if sec:
        idx = np.arange(rows) if pos is None else np.asarray(pos, dtype=np.int64)
        c_rows = np.asarray(cos, dtype=np.float64)[idx]
        s_rows = np.asarray(sin, dtype=np.float64)[idx]
    for off, nh, w, mul in ((q_off, nq, qn, q_mul), (k_off, nkv, kn, 1.0)):
        for h in range(nh):
            sl = slice(off + h * hd, off + (h + 1) * hd)
            v = out[:, sl]
            if w is not None:
                v = rms_norm(v, w, eps)
            if sec:
                v = rope(v, c_rows, s_rows, sec)
            out[:, sl] = v * mul
    if v_off is not None:
        for h in range(nkv):
            sl = slice(v_off + h * hd, v_off + (h + 1) * hd)
            out[:, sl] = rms_norm(out[:, sl], np.ones(hd), eps)
    return round_bf16(out)


# ---------------------------------------------------------------------------
# attention


def visible_mask(n, window):
    """Key j visible to query i of one sequence iff window == 0 or
    |i - j| <= window (egemma2.rs ``att_plan``: keys of a query block span
    [q0 - W, q_last + W], W = 0 meaning the whole sequence)."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    if window == 0:
        return np.ones((n, n), dtype=bool)
    return np.abs(i - j) <= window


def softmax_probs(q, k, scale, visible):
    """p[i, j] = exp(scale*q_i.k_j - max_j) / sum_j, invisible keys exactly 0."""
    s = scale * (np.asarray(q, dtype=np.float64) @ np.asarray(k, dtype=np.float64).T)
    s = np.where(visible, s, -np.inf)
    s = s - np.max(s, axis=1, keepdims=True)
    p = np.where(visible, np.exp(s), 0.0)
    return p / np.sum(p, axis=1, keepdims=True)


def attention_varlen(qkv, cu, nq, nkv, hd, q_off, k_off, v_off, window, scale,
                     rows=None):
    """Bidirectional multi-head attention over a packed batch.

    o[i, h] = sum_j softmax_j(scale * q[i,h] . k[j,kvh]) v[j,kvh] over the
    visible keys j of i's own sequence, kvh = h // (nq/nkv) (egemma2.rs
    ``Prog::attention`` / ``att_plan``; vision_encoder_gpu.rs
    ``VitGpuOps::attention``).  Returns f64 [T, nq*hd]; with ``rows`` only
    those query rows are computed (the others stay NaN).
    """
    qkv = np.asarray(qkv, dtype=np.float64)
    cu = np.asarray(cu, dtype=np.int64)
    T = qkv.shape[0]
    out = np.full((T, nq * hd), np.nan)
    group = nq // nkv
    want = None if rows is None else np.zeros(T, dtype=bool)
    if want is not None:
        want[np.asarray(rows)] = True
    for sidx in range(len(cu) - 1):
        r0, r1 = int(cu[sidx]), int(cu[sidx + 1])
        n = r1 - r0
        if n == 0:
            continue
        vis = visible_mask(n, window)
        qi = np.arange(n) if want is None else np.nonzero(want[r0:r1])[0]
        if len(qi) == 0:
            continue
        for h in range(nq):
            kvh = h // group
            Q = qkv[r0 + qi, q_off + h * hd: q_off + (h + 1) * hd]
            K = qkv[r0:r1, k_off + kvh * hd: k_off + (kvh + 1) * hd]
            V = qkv[r0:r1, v_off + kvh * hd: v_off + (kvh + 1) * hd]
            P = softmax_probs(Q, K, scale, vis[qi])
            out[r0 + qi, h * hd:(h + 1) * hd] = P @ V
    return out


def attention_items(qkv, items, nq, nkv, hd, q_off, k_off, v_off, window, scale):
    """Attention over two-range items (zimage.rs ``PFa``: an item's image rows
    [off1, off1+len1) and caption rows [off2, off2+len2) attend as one
    sequence in that joint order; the window counts joint positions).  Each
    item's rows are gathered into one sequence, attended as such, and the
    outputs scattered back to their own rows; rows in no item stay NaN."""
    qkv = np.asarray(qkv, dtype=np.float64)
    out = np.full((qkv.shape[0], nq * hd), np.nan)
    for off1, len1, off2, len2 in np.asarray(items, dtype=np.int64).reshape(-1, 4):
        rows = np.r_[np.arange(off1, off1 + len1), np.arange(off2, off2 + len2)].astype(np.int64)
        o = attention_varlen(qkv[rows], [0, len(rows)], nq, nkv, hd, q_off, k_off, v_off, window, scale)
        out[rows] = o
    return out


# ---------------------------------------------------------------------------
# gating


def gelu_tanh(g):
    """0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) (egemma2.rs
    ``Prog::gelu``; vision_encoder_gpu.rs ``VitGpuOps::gelu``)."""
    g = np.asarray(g, dtype=np.float64)
    return 0.5 * g * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)))


def silu(g):
    """g / (1 + e^-g) (zimage.rs SwiGLU: h = silu(w1 x) * (w3 x))."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def gate_act(gu, f, gated, act):
    """m = act(g) * u with g = gu[:, :f], u = gu[:, f:2f]; ungated m = act(gu)."""
    gu = np.asarray(gu, dtype=np.float64)
    fn = gelu_tanh if act == "gelu_tanh" else silu
    if gated:
        return fn(gu[:, :f]) * gu[:, f:2 * f]
    return fn(gu[:, :f])


# ---------------------------------------------------------------------------
# pooling


def pool_mean(x, cu, w, eps):
    """out[s] = (1/len_s) sum_{r in s} rms(x_r) * w  (egemma2.rs
    ``TextGpu::forward``: ``row_inv`` then ``pool``; None = no final norm)."""
    x = np.asarray(x, dtype=np.float64)
    cu = np.asarray(cu, dtype=np.int64)
    out = np.zeros((len(cu) - 1, x.shape[1]))
    for sidx in range(len(cu) - 1):
        seg = x[cu[sidx]:cu[sidx + 1]]
        if w is not None:
            seg = rms_norm(seg, w, eps)
        out[sidx] = seg.mean(axis=0)
    return out


# ---------------------------------------------------------------------------
# the block


def block_forward(cfg, p, x, a, cu, layer, tables, next_norm=None, rows=None, mod=None,
                  next_mod_scale=None, ple=None, items=None):
    """One encoder block, step by step; returns every stored intermediate.

    cfg: a BlockConfig-like object (d, heads, kv_heads, hd, ffn, gated, act,
    norm, form, qk_norm, eps, post, scale, window_of(layer)); p: the layer's
    weights; x: f32 residual stream [T, d]; a: this block's normed input
    (bf16 values); tables: RoPE inputs; next_norm: (w, b) of the next block's
    pre-norm or None.

    Plain form (vision_encoder_gpu.rs ``encode_image_gpu``):
        x += o Wo^T (+b);  a = Norm2(x);  x += act-FFN(a);  a = Norm1'(x)
    Sandwich form (egemma2.rs ``TextGpu::forward``; zimage.rs ``Enc::block``):
        x = (x + rms(o Wo^T) w_pa) post;  a = rms(x) w_2;
        x = (x + rms(FFN(a)) w_pf) post;  a = rms(x) w_next
    adaLN-modulated DiT block (zimage.rs ``Enc::block``: ``mods`` =
    [s_msa | g_msa | s_mlp | g_mlp], sandwich form only): ``mod`` [4, d] gates
    the two residual branches with g_msa, g_mlp and scales the FFN input by
    (1 + s_mlp); s_msa scales this block's input ``a`` (made by the caller)
    and ``next_mod_scale`` (the next block's s_msa) the returned ``a_out``.
    Per-layer input path (egemma2.rs ``TextGpu::forward`` "per-layer input";
    ``ple`` = {x_in: the stack's input as bf16, norm_w, scale}, sandwich form):
    after the FFN residual (taken with post 1) pin = rms(scale * x_in W_in^T)
    ple_norm, z = gelu_tanh(bf16(x) W_gate^T) * pin, and
    x = (x + rms(z W_proj^T) w_ple) * post.
    Two-range attention items (zimage.rs module doc "The chain": the CFG pair
    is one batch-2 program over rows [img0 | img1 | cap0 | cap1], every
    row-local step runs once over all rows and attention runs per item over
    its two row ranges; ``PFa``): with ``items`` ([n, 4] = off1, len1, off2,
    len2) the attention step is ``attention_items`` instead of the
    per-sequence attention; ``cu`` then only gives the row count.
    ``rows`` restricts the block to sampled query rows: q|k|v is computed for
    every row (all keys are needed), everything after attention only for the
    sampled rows (it is row-local), and the returned post-attention
    intermediates hold those rows only, in the order given.
    """
    hd, H, KV, d, F = cfg.hd, cfg.heads, cfg.kv_heads, cfg.d, cfg.ffn
    eps = cfg.eps
    if (mod is not None or next_mod_scale is not None) and cfg.form != "sandwich":
        raise ValueError("adaLN modulation applies to the sandwich (post-norm) form")
    g_msa = s_mlp = g_mlp = None
    if mod is not None:
        mod = np.asarray(mod, dtype=np.float64).reshape(4, d)
        g_msa, s_mlp, g_mlp = mod[1], mod[2], mod[3]
    r = {}
    x = round_f32(x)
    a = round_bf16(a)
    qw, kw = H * hd, KV * hd
    qkv = np.concatenate([
        linear(a, p["wq"]),
        linear(a, p["wk"]),
        linear(a, p["wv"]),
    ], axis=1)
    r["qkv_raw"] = qkv = round_bf16(qkv)
    v_norm = getattr(cfg, "v_norm", False)
    if cfg.qk_norm or tables["sec"] or v_norm:
        qkv = qk_prep(qkv, H, KV, hd, 0, qw,
                      p["q_norm"] if cfg.qk_norm else None,
                      p["k_norm"] if cfg.qk_norm else None,
                      eps, tables["cos"], tables["sin"], tables["pos"], tables["sec"], 1.0,
                      v_off=qw + kw if v_norm else None)
    r["qkv"] = qkv
    if items is not None:
        o = attention_items(qkv, items, H, KV, hd, 0, qw, qw + kw, cfg.window_of(layer), cfg.scale)
    else:
        o = attention_varlen(qkv, cu, H, KV, hd, 0, qw, qw + kw, cfg.window_of(layer),
                             cfg.scale, rows=rows)
    if rows is not None:
        rows = np.asarray(rows)
        o, x = o[rows], x[rows]
    r["o"] = o = round_bf16(o)
    if cfg.form == "plain":
        x = round_f32(linear(o, p["wo"], residual=x))
    else:
        t = round_f32(linear(o, p["wo"]))
        r["t"] = t
        x = round_f32(add_norm_sandwich(x, t, p["post_attn_w"], cfg.post, eps, gate=g_msa))
    r["x_mid"] = x
    r["a_mid"] = a2 = round_bf16(norm(cfg.norm, x, p["norm2_w"], p["norm2_b"], eps, mod_scale=s_mlp))
    parts = [linear(a2, p["wg"])]
    if cfg.gated:
        parts.append(linear(a2, p["wu"]))
    r["gu"] = gu = round_bf16(np.concatenate(parts, axis=1))
    r["m"] = m = round_bf16(gate_act(gu, F, cfg.gated, cfg.act))
    if cfg.form == "plain":
        x = round_f32(linear(m, p["wd"], residual=x))
    else:
        f = round_f32(linear(m, p["wd"]))
        r["f"] = f
        if ple is None:
            x = round_f32(add_norm_sandwich(x, f, p["post_ffn_w"], cfg.post, eps, gate=g_mlp))
        else:
            x = round_f32(add_norm_sandwich(x, f, p["post_ffn_w"], 1.0, eps, gate=g_mlp))
            x_in = ple["x_in"] if rows is None else np.asarray(ple["x_in"])[rows]
            t1 = round_f32(linear(round_bf16(x_in), p["ple_in"]))
            pin = round_bf16(rms_norm(t1, ple["norm_w"], eps, pre=ple["scale"]))
            g = round_bf16(linear(round_bf16(x), p["ple_gate"]))
            r["ple_z"] = z = round_bf16(gelu_tanh(g) * pin)
            tp = round_f32(linear(z, p["ple_proj"]))
            x = round_f32(add_norm_sandwich(x, tp, p["ple_post_w"], cfg.post, eps))
    r["x_out"] = x
    if next_norm is not None:
        r["a_out"] = round_bf16(norm(cfg.norm, x, next_norm[0], next_norm[1], eps,
                                     mod_scale=next_mod_scale))
    else:
        r["a_out"] = None
    return r
