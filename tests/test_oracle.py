"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against brute force on tiny inputs, a
closed form, an invariant the pages' definitions imply, or a library routine
that computes the same textbook quantity, chosen so that a plausible slip in
the oracle (a dropped term, a wrong sign or index, a transposed operand)
fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from oracle import encoder as O
from transformer_encoder_forward_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- rounding

def test_round_bf16_matches_torch_rne_on_f32_inputs():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),       # subnormal range
        np.array([0.0, -0.0, 1.0, -1.0, 1.00390625, 1.01171875, 3.4e38, 1e-45],
                 dtype=np.float32),
    ])
    # exact ties: f32 values halfway between two bf16 values
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32) \
        .astype(np.float32)
    ties = np.concatenate([ties, (np.arange(0x3F80, 0x3FA0, dtype=np.uint32) << 16 | 0x8000)
                           .view(np.float32)])
    vals = np.concatenate([vals, ties])
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(vals.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_round_f32_is_float32_cast():
    v = np.array([1.0 + 2.0 ** -30, math.pi, -1e-40])
    np.testing.assert_array_equal(O.round_f32(v), v.astype(np.float32).astype(np.float64))


def test_int8_widening_is_exact_for_all_values():
    q = np.arange(-128, 128, dtype=np.int8)
    w = O.widen_int8(q)
    np.testing.assert_array_equal(w, np.arange(-128, 128, dtype=np.float64))
    # every int8 is a bf16 value: rounding changes nothing
    np.testing.assert_array_equal(O.round_bf16(w), w)
    ref = torch.from_numpy(q).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(w, ref)


# ---------------------------------------------------------------- q8 linear

def _q8_brute(x, q, s, b, r):
    t, k = x.shape
    n = q.shape[0]
    y = [[0.0] * n for _ in range(t)]
    for i in range(t):
        for o in range(n):
            acc = 0.0
            for kk in range(k):
                acc += float(x[i, kk]) * int(q[o, kk])
            v = float(s[o]) * acc
            if b is not None:
                v += float(b[o])
            if r is not None:
                v += float(r[i, o])
            y[i][o] = v
    return np.array(y)


def test_q8_linear_brute_force_tiny():
    rng = np.random.default_rng(2)
    x = O.round_bf16(rng.standard_normal((5, 24)))
    q = rng.integers(-127, 128, (7, 24), dtype=np.int8)
    s = rng.uniform(0.01, 0.02, 7).astype(np.float32)
    b = rng.standard_normal(7).astype(np.float32)
    r = rng.standard_normal((5, 7)).astype(np.float32)
    for bb, rr in ((None, None), (b, None), (b, r), (None, r)):
        np.testing.assert_allclose(O.q8_linear(x, q, s, bb, rr), _q8_brute(x, q, s, bb, rr),
                                   rtol=1e-13, atol=1e-13)


def test_q8_linear_exact_integer_case():
    # integer activations |x| <= 16, unit scale, K <= 1024: every partial sum
    # is an integer below 2^24, so the result is exact in f32 as well.
    rng = np.random.default_rng(3)
    k = 1024
    x = rng.integers(-16, 17, (9, k)).astype(np.float64)
    q = rng.integers(-127, 128, (11, k), dtype=np.int8)
    y = O.q8_linear(x, q, np.ones(11, np.float32))
    exact = x.astype(np.int64) @ q.astype(np.int64).T
    np.testing.assert_array_equal(y, exact.astype(np.float64))
    assert np.all(np.abs(exact) < 2 ** 24)


def test_q8_linear_row_scale_is_per_output_row():
    # a transposed scale (per input column) would break this
    q = np.eye(4, dtype=np.int8)
    s = np.array([1.0, 2.0, 3.0, 4.0], dtype=np.float32)
    x = np.array([[1.0, 1.0, 1.0, 1.0]])
    np.testing.assert_array_equal(O.q8_linear(x, q, s), [[1.0, 2.0, 3.0, 4.0]])
    x = np.array([[1.0, 0.0, 0.0, 0.0]])
    q2 = np.array([[0, 0, 0, 0], [5, 0, 0, 0], [0, 0, 0, 0], [0, 0, 0, 0]], dtype=np.int8)
    np.testing.assert_array_equal(O.q8_linear(x, q2, s), [[0.0, 10.0, 0.0, 0.0]])


# ---------------------------------------------------------------- norms

def test_rms_norm_constant_row_closed_form():
    for c in (0.5, -3.0, 1e-4):
        w = np.linspace(0.5, 1.5, 16)
        y = O.rms_norm(np.full((1, 16), c), w, 1e-6)
        np.testing.assert_allclose(y[0], c / math.sqrt(c * c + 1e-6) * w, rtol=1e-14)


def test_rms_norm_unit_rms_without_eps_and_pre_scale():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 40)) * 5
    y = O.rms_norm(x, np.ones(40), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-13)
    # scale invariance: rms(c x) = rms(x) when eps = 0, and pre multiplies before
    np.testing.assert_allclose(O.rms_norm(3 * x, np.ones(40), 0.0), y, rtol=1e-13)
    np.testing.assert_allclose(O.rms_norm(x, np.ones(40), 1e-3, pre=2.0),
                               O.rms_norm(2 * x, np.ones(40), 1e-3), rtol=1e-14)
    # eps enters under the root: rms of a zero row is zero, not NaN
    assert np.all(O.rms_norm(np.zeros((1, 8)), np.ones(8), 1e-6) == 0)


def test_layer_norm_against_torch_and_constant_row():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 48)) * 2 + 1
    w = rng.standard_normal(48)
    b = rng.standard_normal(48)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (48,), torch.from_numpy(w),
                                         torch.from_numpy(b), 1e-5).numpy()
    np.testing.assert_allclose(O.layer_norm(x, w, b, 1e-5), ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.layer_norm(np.full((1, 48), 7.0), w, b, 1e-5)[0], b,
                               atol=1e-12)
    y = O.layer_norm(x, np.ones(48), None, 0.0)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-13)
    np.testing.assert_allclose(y.var(axis=1), 1, rtol=1e-12)


def test_add_norm_sandwich_closed_form():
    h = np.array([[1.0, 2.0, 3.0, 4.0]])
    t = np.full((1, 4), 2.0)
    w = np.array([1.0, 0.5, 2.0, 1.0])
    out = O.add_norm_sandwich(h, t, w, 0.5, 0.0)
    np.testing.assert_allclose(out, (h + w) * 0.5, rtol=1e-15)


# ---------------------------------------------------------------- RoPE / qk prep

def _rope_complex(x, ang, sec):
    # independent formulation: pair (x1, x2) as x1 + i x2 times e^{i angle}
    hd = x.shape[1]
    half = sec // 2
    out = np.empty_like(x)
    for s in range(hd // sec):
        z = x[:, s * sec: s * sec + half] + 1j * x[:, s * sec + half:(s + 1) * sec]
        z = z * np.exp(1j * ang[:, s * half:(s + 1) * half])
        out[:, s * sec: s * sec + half] = z.real
        out[:, s * sec + half:(s + 1) * sec] = z.imag
    return out


@pytest.mark.parametrize("sec", [16, 8])
def test_rope_matches_complex_rotation_and_preserves_pair_norms(sec):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((9, 16))
    ang = rng.uniform(-4, 4, (9, 8))
    y = O.rope(x, np.cos(ang), np.sin(ang), sec)
    np.testing.assert_allclose(y, _rope_complex(x, ang, sec), rtol=1e-13, atol=1e-13)
    half = sec // 2
    for s in range(16 // sec):
        a, b = slice(s * sec, s * sec + half), slice(s * sec + half, (s + 1) * sec)
        np.testing.assert_allclose(x[:, a] ** 2 + x[:, b] ** 2, y[:, a] ** 2 + y[:, b] ** 2,
                                   rtol=1e-12)
    # angle 0 is the identity
    np.testing.assert_allclose(O.rope(x, np.ones((9, 8)), np.zeros((9, 8)), sec), x)


def test_rope_1d_tables_give_relative_positions():
    cfg = synth.small_config("c2", hd=16)
    lens = [40]
    tb = synth.rope_tables(cfg, lens)
    rng = np.random.default_rng(7)
    q = rng.standard_normal(16)
    k = rng.standard_normal(16)
    def at(v, p):
        return O.rope(v[None, :], tb["cos"][p:p + 1], tb["sin"][p:p + 1], 16)[0]
    d1 = at(q, 10) @ at(k, 3)
    d2 = at(q, 27) @ at(k, 20)
    assert abs(d1 - d2) < 1e-5 * (abs(d1) + 1)


def test_qk_prep_heads_and_q_mul():
    rng = np.random.default_rng(8)
    hd, nq, nkv = 8, 2, 1
    qkv = O.round_bf16(rng.standard_normal((3, (nq + 2 * nkv) * hd)))
    # no norm, no RoPE, q_mul = 1: the identity on bf16 values
    same = O.qk_prep(qkv, nq, nkv, hd, 0, nq * hd, None, None, 1e-6, None, None, None, 0, 1.0)
    np.testing.assert_array_equal(same, qkv)
    # q_mul touches q only (v, at the tail, never changes)
    two = O.qk_prep(qkv, nq, nkv, hd, 0, nq * hd, None, None, 1e-6, None, None, None, 0, 2.0)
    np.testing.assert_array_equal(two[:, :nq * hd], 2 * qkv[:, :nq * hd])
    np.testing.assert_array_equal(two[:, nq * hd:], qkv[:, nq * hd:])
    # norm acts per head: each q head, rescaled alone, has unit RMS
    qn = np.ones(hd)
    nrm = O.qk_prep(qkv, nq, nkv, hd, 0, nq * hd, qn, qn, 0.0, None, None, None, 0, 1.0)
    for h in range(nq + nkv):
        blk = nrm[:, h * hd:(h + 1) * hd]
        np.testing.assert_allclose(np.sqrt(np.mean(blk ** 2, axis=1)), 1.0, rtol=1e-2)


# ---------------------------------------------------------------- attention

def _attn_brute(q, k, v, scale, vis):
    n, hd = q.shape
    out = np.zeros_like(q)
    for i in range(n):
        sc = [scale * sum(q[i, c] * k[j, c] for c in range(hd)) if vis[i, j] else None
              for j in range(k.shape[0])]
        mx = max(s for s in sc if s is not None)
        w = [math.exp(s - mx) if s is not None else 0.0 for s in sc]
        tot = sum(w)
        for c in range(hd):
            out[i, c] = sum(w[j] * v[j, c] for j in range(k.shape[0])) / tot
    return out


def _panel(rng, T, nq, nkv, hd):
    return O.round_bf16(rng.standard_normal((T, (nq + 2 * nkv) * hd)))


def test_attention_brute_force_with_window_and_two_sequences():
    rng = np.random.default_rng(9)
    hd, nq = 4, 2
    cu = np.array([0, 7, 12])
    qkv = _panel(rng, 12, nq, nq, hd)
    for window in (0, 2):
        o = O.attention_varlen(qkv, cu, nq, nq, hd, 0, nq * hd, 2 * nq * hd, window, 0.7)
        for s in range(2):
            r0, r1 = cu[s], cu[s + 1]
            n = r1 - r0
            vis = np.array([[window == 0 or abs(i - j) <= window for j in range(n)]
                            for i in range(n)])
            for h in range(nq):
                ref = _attn_brute(qkv[r0:r1, h * hd:(h + 1) * hd],
                                  qkv[r0:r1, nq * hd + h * hd: nq * hd + (h + 1) * hd],
                                  qkv[r0:r1, 2 * nq * hd + h * hd: 2 * nq * hd + (h + 1) * hd],
                                  0.7, vis)
                np.testing.assert_allclose(o[r0:r1, h * hd:(h + 1) * hd], ref, rtol=1e-12,
                                           atol=1e-12)


def test_attention_matches_torch_sdpa_with_mask():
    rng = np.random.default_rng(10)
    n, hd = 33, 16
    q, k, v = (rng.standard_normal((n, hd)) for _ in range(3))
    vis = O.visible_mask(n, 5)
    p = O.softmax_probs(q, k, 0.25, vis)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=torch.from_numpy(vis)[None], scale=0.25)[0].numpy()
    np.testing.assert_allclose(p @ v, ref, rtol=1e-12, atol=1e-12)


def test_softmax_rows_sum_to_one_and_masked_weights_are_zero():
    rng = np.random.default_rng(11)
    q, k = rng.standard_normal((20, 8)) * 4, rng.standard_normal((20, 8)) * 4
    vis = O.visible_mask(20, 3)
    p = O.softmax_probs(q, k, 1.0, vis)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-14)
    assert np.all(p[~vis] == 0.0)
    assert np.all(p[vis] > 0.0)


def test_identical_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(12)
    hd, n, W = 8, 17, 4
    qkv = np.zeros((n, 3 * hd))
    qkv[:, :hd] = rng.standard_normal((n, hd))
    qkv[:, hd:2 * hd] = rng.standard_normal(hd)          # every key identical
    qkv[:, 2 * hd:] = rng.standard_normal((n, hd))
    o = O.attention_varlen(qkv, [0, n], 1, 1, hd, 0, hd, 2 * hd, W, 1.0)
    for i in range(n):
        lo, hi = max(0, i - W), min(n, i + W + 1)
        np.testing.assert_allclose(o[i], qkv[lo:hi, 2 * hd:].mean(axis=0), rtol=1e-12)


def test_length_one_sequence_returns_v_and_sequences_are_independent():
    rng = np.random.default_rng(13)
    hd = 8
    qkv = rng.standard_normal((10, 3 * hd))
    cu = [0, 1, 6, 10]
    o = O.attention_varlen(qkv, cu, 1, 1, hd, 0, hd, 2 * hd, 0, 1.0)
    np.testing.assert_allclose(o[0], qkv[0, 2 * hd:])
    qkv2 = qkv.copy()
    qkv2[6:] = rng.standard_normal((4, 3 * hd))          # change the last sequence
    o2 = O.attention_varlen(qkv2, cu, 1, 1, hd, 0, hd, 2 * hd, 0, 1.0)
    np.testing.assert_array_equal(o[:6], o2[:6])


def test_out_of_window_keys_have_no_effect_and_wide_window_is_full():
    rng = np.random.default_rng(14)
    hd, n, W = 8, 30, 5
    qkv = rng.standard_normal((n, 3 * hd))
    o = O.attention_varlen(qkv, [0, n], 1, 1, hd, 0, hd, 2 * hd, W, 0.5)
    # perturb every key/value farther than W from row 0: row 0 is unchanged
    qkv2 = qkv.copy()
    qkv2[W + 1:, hd:] = rng.standard_normal((n - W - 1, 2 * hd)) * 100
    o2 = O.attention_varlen(qkv2, [0, n], 1, 1, hd, 0, hd, 2 * hd, W, 0.5)
    np.testing.assert_array_equal(o[0], o2[0])
    full = O.attention_varlen(qkv, [0, n], 1, 1, hd, 0, hd, 2 * hd, 0, 0.5)
    wide = O.attention_varlen(qkv, [0, n], 1, 1, hd, 0, hd, 2 * hd, n - 1, 0.5)
    np.testing.assert_array_equal(full, wide)


def test_gqa_head_grouping():
    rng = np.random.default_rng(15)
    hd, nq, nkv, n = 4, 4, 2, 6
    qkv = rng.standard_normal((n, (nq + 2 * nkv) * hd))
    o = O.attention_varlen(qkv, [0, n], nq, nkv, hd, 0, nq * hd, (nq + nkv) * hd, 0, 1.0)
    # q head 3 uses kv head 1
    q = qkv[:, 3 * hd:4 * hd]
    k = qkv[:, nq * hd + hd: nq * hd + 2 * hd]
    v = qkv[:, (nq + nkv) * hd + hd:(nq + nkv) * hd + 2 * hd]
    ref = _attn_brute(q, k, v, 1.0, np.ones((n, n), bool))
    np.testing.assert_allclose(o[:, 3 * hd:], ref, rtol=1e-12)


# ---------------------------------------------------------------- gating

def test_gelu_tanh_and_silu_against_torch_and_symmetries():
    x = np.linspace(-8, 8, 1001)
    tx = torch.from_numpy(x)
    np.testing.assert_allclose(O.gelu_tanh(x),
                               torch.nn.functional.gelu(tx, approximate="tanh").numpy(),
                               rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(O.silu(x), torch.nn.functional.silu(tx).numpy(),
                               rtol=1e-14, atol=1e-15)
    assert O.gelu_tanh(0.0) == 0.0 and O.silu(0.0) == 0.0
    np.testing.assert_allclose(O.gelu_tanh(x) - O.gelu_tanh(-x), x, atol=1e-14)
    np.testing.assert_allclose(O.silu(x) - O.silu(-x), x, atol=1e-14)
    # closed form at 1: 0.5 (1 + tanh(sqrt(2/pi) * 1.044715))
    assert abs(O.gelu_tanh(1.0) - 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * 1.044715))) < 1e-16


def test_gate_act_takes_gate_first():
    gu = np.array([[1.0, -2.0, 3.0, 4.0]])      # f = 2: g = [1, -2], u = [3, 4]
    m = O.gate_act(gu, 2, True, "silu")
    np.testing.assert_allclose(m, [[O.silu(1.0) * 3.0, O.silu(-2.0) * 4.0]])
    np.testing.assert_allclose(O.gate_act(gu, 2, False, "gelu_tanh"),
                               [[O.gelu_tanh(1.0), O.gelu_tanh(-2.0)]])


# ---------------------------------------------------------------- pooling

def test_pool_mean_identical_rows_and_plain_mean():
    rng = np.random.default_rng(16)
    row = rng.standard_normal(12)
    x = np.vstack([np.tile(row, (5, 1)), rng.standard_normal((3, 12))])
    w = rng.uniform(0.5, 1.5, 12)
    out = O.pool_mean(x, [0, 5, 8], w, 1e-6)
    np.testing.assert_allclose(out[0], O.rms_norm(row[None], w, 1e-6)[0], rtol=1e-13)
    plain = O.pool_mean(x, [0, 5, 8], None, 1e-6)
    np.testing.assert_allclose(plain[1], x[5:8].sum(axis=0) / 3, rtol=1e-13)


# ---------------------------------------------------------------- the block

def _tiny(form, norm, gated, act, rope, qk_norm, window=0, bias=False):
    return synth.BlockConfig("tiny", 1, 32, 2, 2, 16, 48, gated, act, norm, form, qk_norm,
                             rope, window, "all", bias, False, (9, 14))


def _torch_block(cfg, p, x, cu, tables, next_norm, ple=None):
    """The same block written with torch's own library ops (linear, layer_norm,
    scaled_dot_product_attention, gelu/silu, complex rotation for RoPE).

    With ``ple`` ({x_in, norm_w, scale}) the per-layer input path follows the
    FFN residual as egemma2.rs ``TextGpu::forward`` "per-layer input" chains
    it: mm(x_in, W_in) -> rms with pre-scale and the stack's norm weight ->
    mm(h, W_gate) -> gelu of that gate times pin -> mm(z, W_proj) -> add_norm
    with the layer's own post-norm weight and the layer scalar (the FFN's
    add_norm before it takes scalar 1)."""
    t = lambda a: torch.as_tensor(np.asarray(a, np.float64))
    bf = lambda v: v.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    f32 = lambda v: v.to(torch.float32).to(torch.float64)
    F = torch.nn.functional

    def lin(v, w):
        out = F.linear(v, t(w["q"].astype(np.float64)) * t(w["s"])[:, None])
        return out + t(w["b"]) if w["b"] is not None else out

    def nrm(v, w, b):
        if cfg.norm == "ln":
            return F.layer_norm(v, (v.shape[-1],), t(w), None if b is None else t(b), cfg.eps)
        return F.rms_norm(v, (v.shape[-1],), t(w), cfg.eps)

    x = f32(t(x))
    a = bf(nrm(x, p["norm1_w"], p["norm1_b"]))
    H, hd = cfg.heads, cfg.hd
    qkv = bf(torch.cat([lin(a, p["wq"]), lin(a, p["wk"]), lin(a, p["wv"])], 1))
    q, k, v = qkv[:, :H * hd], qkv[:, H * hd:2 * H * hd], qkv[:, 2 * H * hd:]
    def prep(u, w):
        u = u.reshape(-1, H, hd)
        if cfg.qk_norm:
            u = F.rms_norm(u, (hd,), t(w), cfg.eps)
        if tables["sec"]:
            ang = torch.atan2(t(tables["sin"]), t(tables["cos"]))[t(tables["pos"]).long()]
            sec = tables["sec"]
            half = sec // 2
            parts = []
            for s in range(hd // sec):
                z = torch.complex(u[..., s * sec:s * sec + half], u[..., s * sec + half:(s + 1) * sec])
                z = z * torch.polar(torch.ones_like(ang[:, None, s * half:(s + 1) * half]),
                                    ang[:, None, s * half:(s + 1) * half])
                parts.append((z.real, z.imag))
            u = torch.cat([c for pr in parts for c in pr], -1)
        return u.reshape(-1, H * hd)
    if cfg.qk_norm or tables["sec"]:
        q, k = bf(prep(q, p.get("q_norm"))), bf(prep(k, p.get("k_norm")))
    o = torch.zeros_like(q)
    for s in range(len(cu) - 1):
        r0, r1 = int(cu[s]), int(cu[s + 1])
        n = r1 - r0
        ii = torch.arange(n)
        mask = torch.ones(n, n, dtype=torch.bool) if cfg.window == 0 else \
            (ii[:, None] - ii[None, :]).abs() <= cfg.window
        qs = q[r0:r1].reshape(n, H, hd).transpose(0, 1)
        ks = k[r0:r1].reshape(n, H, hd).transpose(0, 1)
        vs = v[r0:r1].reshape(n, H, hd).transpose(0, 1)
        os_ = F.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=cfg.scale)
        o[r0:r1] = os_.transpose(0, 1).reshape(n, H * hd)
    o = bf(o)
    if cfg.form == "plain":
        x = f32(x + lin(o, p["wo"]))
    else:
        x = f32((x + F.rms_norm(f32(lin(o, p["wo"])), (cfg.d,), t(p["post_attn_w"]), cfg.eps)) * cfg.post)
    a2 = bf(nrm(x, p["norm2_w"], p["norm2_b"]))
    g = lin(a2, p["wg"])
    actf = (lambda u: F.gelu(u, approximate="tanh")) if cfg.act == "gelu_tanh" else F.silu
    m = bf(actf(bf(g)) * bf(lin(a2, p["wu"]))) if cfg.gated else bf(actf(bf(g)))
    if cfg.form == "plain":
        x = f32(x + lin(m, p["wd"]))
    elif ple is None:
        x = f32((x + F.rms_norm(f32(lin(m, p["wd"])), (cfg.d,), t(p["post_ffn_w"]), cfg.eps)) * cfg.post)
    else:
        x = f32(x + F.rms_norm(f32(lin(m, p["wd"])), (cfg.d,), t(p["post_ffn_w"]), cfg.eps))
        P = p["ple_in"]["q"].shape[0]
        src = f32(lin(bf(t(ple["x_in"])), p["ple_in"]))
        pin = bf(F.rms_norm(ple["scale"] * src, (P,), t(ple["norm_w"]), cfg.eps))
        gate = bf(lin(bf(x), p["ple_gate"]))
        z = bf(F.gelu(gate, approximate="tanh") * pin)
        proj = f32(lin(z, p["ple_proj"]))
        x = f32((x + F.rms_norm(proj, (cfg.d,), t(p["ple_post_w"]), cfg.eps)) * cfg.post)
    a_out = bf(nrm(x, *next_norm)) if next_norm is not None else None
    return x.numpy(), (a_out.numpy() if a_out is not None else None), a.numpy()


@pytest.mark.parametrize("form,norm,gated,act,rope,qk,window,bias", [
    ("plain", "rms", True, "gelu_tanh", None, False, 0, False),     # c1 form
    ("plain", "ln", False, "gelu_tanh", None, False, 0, True),      # c3 form
    ("sandwich", "rms", True, "gelu_tanh", "1d", True, 4, False),   # c2 form
    ("sandwich", "rms", True, "silu", "2d", True, 0, False),        # c4/c5 form
])
def test_block_matches_torch_library_composition(form, norm, gated, act, rope, qk, window, bias):
    cfg = _tiny(form, norm, gated, act, rope, qk, window, bias)
    lens = cfg.lens
    cu = synth.cu_seqlens(lens)
    T = int(cu[-1])
    p = synth.draw_layer(cfg, 0, 99)
    x = synth.draw_x(T, cfg.d, 5)
    tables = synth.rope_tables(cfg, lens)
    nxt = synth.draw_norm(np.random.default_rng(3), cfg.d, cfg.norm == "ln")
    x_ref, a_ref, a_in = _torch_block(cfg, p, x, cu, tables, nxt)
    r = O.block_forward(cfg, p, x, a_in, cu, 0, tables, next_norm=nxt)
    np.testing.assert_allclose(r["x_out"], x_ref, rtol=2e-5, atol=2e-5)
    np.testing.assert_allclose(r["a_out"], a_ref, rtol=2e-2, atol=2e-2)
    rel = np.linalg.norm(r["a_out"] - a_ref) / np.linalg.norm(a_ref)
    assert rel < 1e-4


def test_block_with_zero_weights_is_identity_on_residual():
    for form in ("plain", "sandwich"):
        cfg = _tiny(form, "rms", True, "silu", None, False)
        p = synth.draw_layer(cfg, 0, 1)
        for key in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
            p[key]["s"] = np.zeros_like(p[key]["s"])
        cu = synth.cu_seqlens(cfg.lens)
        x = synth.draw_x(int(cu[-1]), cfg.d, 2)
        a = O.round_bf16(O.rms_norm(x, p["norm1_w"], cfg.eps))
        r = O.block_forward(cfg, p, x, a, cu, 0, synth.rope_tables(cfg, cfg.lens))
        np.testing.assert_array_equal(r["x_out"], x.astype(np.float64))


def test_block_is_equivariant_to_sequence_order():
    cfg = _tiny("sandwich", "rms", True, "gelu_tanh", "1d", True, 3)
    p = synth.draw_layer(cfg, 0, 4)
    lens = (9, 14)
    cu = synth.cu_seqlens(lens)
    x = synth.draw_x(23, cfg.d, 6)
    a = O.round_bf16(O.rms_norm(x, p["norm1_w"], cfg.eps))
    r = O.block_forward(cfg, p, x, a, cu, 0, synth.rope_tables(cfg, lens))
    perm = np.r_[9:23, 0:9]
    lens2 = (14, 9)
    r2 = O.block_forward(cfg, p, x[perm], a[perm], synth.cu_seqlens(lens2), 0,
                         synth.rope_tables(cfg, lens2))
    np.testing.assert_allclose(r2["x_out"], r["x_out"][perm], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- adaLN (DiT)
# The pages fix two things about the modulation (zimage.rs Enc::block /
# refine_caption): the per-block layout [s_msa | g_msa | s_mlp | g_mlp] and that
# the unmodulated block is s = 0, gate = 1.  The pins below check the oracle's
# modulated block against those facts and against the block's structure: which
# vector acts on which branch, that s scales through (1 + s), that g multiplies
# the whole post-normed branch.

def _dit_case(seed=7):
    cfg = _tiny("sandwich", "rms", True, "silu", "2d", True, 0)
    p = synth.draw_layer(cfg, 0, seed)
    cu = synth.cu_seqlens(cfg.lens)
    x = synth.draw_x(int(cu[-1]), cfg.d, seed + 1)
    tables = synth.rope_tables(cfg, cfg.lens)
    return cfg, p, cu, x, tables


def test_adaln_identity_modulation_is_the_unmodulated_block():
    cfg, p, cu, x, tables = _dit_case()
    d = cfg.d
    nxt = synth.draw_norm(np.random.default_rng(3), d, False)
    a = O.round_bf16(O.norm("rms", x, p["norm1_w"], None, cfg.eps, mod_scale=np.zeros(d)))
    ident = np.stack([np.zeros(d), np.ones(d), np.zeros(d), np.ones(d)])
    r0 = O.block_forward(cfg, p, x, a, cu, 0, tables, next_norm=nxt)
    r1 = O.block_forward(cfg, p, x, a, cu, 0, tables, next_norm=nxt, mod=ident,
                         next_mod_scale=np.zeros(d))
    for key in ("x_mid", "a_mid", "x_out", "a_out"):
        np.testing.assert_array_equal(r1[key], r0[key])


def test_adaln_zero_gates_leave_the_residual_stream_unchanged():
    cfg, p, cu, x, tables = _dit_case(11)
    d = cfg.d
    rng = np.random.default_rng(2)
    mod = np.stack([rng.normal(0, .3, d), np.zeros(d), rng.normal(0, .3, d), np.zeros(d)])
    a = O.round_bf16(O.norm("rms", x, p["norm1_w"], None, cfg.eps, mod_scale=mod[0]))
    r = O.block_forward(cfg, p, x, a, cu, 0, tables, mod=mod)
    np.testing.assert_array_equal(r["x_mid"], x.astype(np.float64))
    np.testing.assert_array_equal(r["x_out"], x.astype(np.float64))


def test_adaln_gate_scales_only_its_own_branch():
    # g_msa acts on the attention branch: x_mid - x = g_msa * rms(t) w_pa,
    # so dividing the delta by g_msa gives the unmodulated delta; g_mlp does
    # not touch x_mid
    cfg, p, cu, x, tables = _dit_case(13)
    d = cfg.d
    rng = np.random.default_rng(4)
    a = O.round_bf16(O.norm("rms", x, p["norm1_w"], None, cfg.eps))
    base = O.block_forward(cfg, p, x, a, cu, 0, tables)
    g = rng.uniform(0.5, 1.5, d) * rng.choice([-1, 1], d)
    mod = np.stack([np.zeros(d), g, np.zeros(d), rng.uniform(0.5, 1.5, d)])
    r = O.block_forward(cfg, p, x, a, cu, 0, tables, mod=mod)
    x64 = x.astype(np.float64)
    delta_mod = (r["x_mid"] - x64) / g
    delta_ref = base["x_mid"] - x64
    np.testing.assert_allclose(delta_mod, delta_ref, rtol=1e-5, atol=1e-6)
    np.testing.assert_array_equal(r["t"], base["t"])      # same attention branch input


def test_adaln_scale_multiplies_the_normed_ffn_input_by_one_plus_s():
    cfg, p, cu, x, tables = _dit_case(17)
    d = cfg.d
    rng = np.random.default_rng(5)
    a = O.round_bf16(O.norm("rms", x, p["norm1_w"], None, cfg.eps))
    s = rng.normal(0, .5, d)
    mod = np.stack([np.zeros(d), np.ones(d), s, np.ones(d)])
    r = O.block_forward(cfg, p, x, a, cu, 0, tables, mod=mod)
    # a_mid is stored bf16: compare with the unrounded reference within bf16
    ref = O.rms_norm(r["x_mid"], p["norm2_w"], cfg.eps) * (1.0 + s)
    np.testing.assert_allclose(r["a_mid"], ref, rtol=2 ** -8, atol=1e-30)
    # s = -1 on every channel zeroes the FFN input, hence the FFN branch
    mod2 = np.stack([np.zeros(d), np.ones(d), -np.ones(d), np.ones(d)])
    r2 = O.block_forward(cfg, p, x, a, cu, 0, tables, mod=mod2)
    assert not np.any(r2["a_mid"])
    np.testing.assert_array_equal(r2["f"], np.zeros_like(r2["f"]))


def test_adaln_rejects_the_plain_form():
    cfg = _tiny("plain", "rms", True, "silu", None, False)
    p = synth.draw_layer(cfg, 0, 1)
    cu = synth.cu_seqlens(cfg.lens)
    x = synth.draw_x(int(cu[-1]), cfg.d, 2)
    with pytest.raises(ValueError):
        O.block_forward(cfg, p, x, x, cu, 0, synth.rope_tables(cfg, cfg.lens),
                        mod=np.zeros((4, cfg.d)))


# ------------------------------------------------- 32-element block formats
# vision_encoder_gpu.rs' test quantisers fix the byte layouts: Q8_0 = f16 scale
# + 32 int8; Q4_0 = f16 scale + 16 bytes (low nibble element i, high nibble
# element i + 16, each + 8).  The pins build blocks by hand, round-trip the
# pages' quantiser rule, and check the block GEMM by brute force.

def test_decode_q8_0_hand_built_block():
    payload = np.arange(-16, 16, dtype=np.int8)
    blk = np.concatenate([np.array([0x00, 0x38], np.uint8), payload.view(np.uint8)])   # f16 0.5
    q, d = O.decode_q8_0(blk.tobytes(), 1, 32)
    np.testing.assert_array_equal(q[0], payload)
    assert d.shape == (1, 1) and d[0, 0] == 0.5


def test_decode_q4_0_nibble_layout():
    lo = np.arange(16, dtype=np.uint8)             # element i   -> i - 8
    hi = (15 - np.arange(16)).astype(np.uint8)     # element 16+i -> 7 - i
    blk = np.concatenate([np.array([0x00, 0x3C], np.uint8), lo | (hi << 4)])           # f16 1.0
    q, d = O.decode_q4_0(blk.tobytes(), 1, 32)
    np.testing.assert_array_equal(q[0, :16], np.arange(16) - 8)
    np.testing.assert_array_equal(q[0, 16:], 7 - np.arange(16))
    assert d[0, 0] == 1.0


def _quantize_like_the_pages(w, fmt):
    """Per 32-element block: d = amax / qmax, q = round(w / d) clamped
    (Q8_0: +-127; Q4_0: stored q + 8 in [0, 15]), d stored as f16."""
    n, k = w.shape
    out = bytearray()
    for row in w:
        for blk in row.reshape(-1, 32):
            amax = np.abs(blk).max()
            d = amax / (127.0 if fmt == "q8_0" else 7.0)
            inv = 1.0 / d if d else 0.0
            out += np.float16(d).tobytes()
            if fmt == "q8_0":
                out += np.clip(np.round(blk * inv), -127, 127).astype(np.int8).tobytes()
            else:
                u = np.clip(np.round(blk * inv) + 8, 0, 15).astype(np.uint8)
                out += (u[:16] | (u[16:] << 4)).astype(np.uint8).tobytes()
    return bytes(out)


@pytest.mark.parametrize("fmt,qmax", [("q8_0", 127), ("q4_0", 7)])
def test_block_decode_round_trips_the_quantiser_within_half_a_step(fmt, qmax):
    rng = np.random.default_rng(12)
    w = rng.standard_normal((6, 128))
    dec = O.decode_q8_0 if fmt == "q8_0" else O.decode_q4_0
    q, d = dec(_quantize_like_the_pages(w, fmt), 6, 128)
    wd = q.astype(np.float64) * np.repeat(d, 32, axis=1)
    step = np.repeat(np.abs(w).reshape(6, 4, 32).max(axis=2) / qmax, 32, axis=1)
    # half a quantisation step, plus the f16 rounding of the scale
    assert np.all(np.abs(w - wd) <= 0.5 * step + qmax * step * 2.0 ** -11 + 1e-12)


def test_block_linear_matches_brute_force_with_bf16_weights():
    rng = np.random.default_rng(13)
    m, n, k = 3, 5, 64
    x = rng.standard_normal((m, k))
    q = rng.integers(-127, 128, (n, k)).astype(np.int8)
    d = rng.uniform(0.001, 0.01, (n, k // 32)).astype(np.float16).astype(np.float64)
    s = rng.uniform(0.5, 2.0, n)
    b = rng.standard_normal(n)
    y = O.q8_block_linear(x, q, d, s, b)
    for t in range(m):
        for o in range(n):
            acc = 0.0
            for j in range(k):
                acc += x[t, j] * float(O.round_bf16(np.float64(q[o, j]) * d[o, j // 32]))
            assert abs(y[t, o] - (s[o] * acc + b[o])) <= 1e-12 * (1 + abs(y[t, o]))


def test_block_linear_exact_cases():
    rng = np.random.default_rng(14)
    x = rng.integers(-16, 17, (7, 96)).astype(np.float64)
    q = rng.integers(-127, 128, (8, 96)).astype(np.int8)
    exact = x @ q.astype(np.float64).T
    # unit scales: the integer product; a power-of-two scale: the same, scaled
    np.testing.assert_array_equal(O.q8_block_linear(x, q, np.ones((8, 3))), exact)
    np.testing.assert_array_equal(O.q8_block_linear(x, q, np.full((8, 3), 2.0 ** -7)), exact * 2.0 ** -7)


# ---------------------------------------------------------------- q8_2f
# zimage.rs ensure_dev: q8_2f = the q8_row bytes + a per-column f16 field;
# W[o, k] = s[o] q[o, k] col[k].

def test_q8_2f_unit_field_is_q8_row():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((4, 64))
    q = rng.integers(-127, 128, (6, 64)).astype(np.int8)
    s = rng.uniform(0.5, 2, 6)
    np.testing.assert_array_equal(O.q8_2f_linear(x, q, np.ones(64), s), O.q8_linear(x, q, s))


def test_q8_2f_power_of_two_field_scales_columns_exactly():
    # col[k] = 2^e_k: bf16(q col) = q col exactly, so y = (x * col) q^T s
    rng = np.random.default_rng(22)
    x = rng.integers(-16, 17, (5, 64)).astype(np.float64)
    q = rng.integers(-127, 128, (7, 64)).astype(np.int8)
    col = 2.0 ** rng.integers(-3, 4, 64)
    y = O.q8_2f_linear(x, q, col, np.ones(7))
    np.testing.assert_array_equal(y, (x * col[None, :]) @ q.astype(np.float64).T)


def test_q8_2f_matches_brute_force():
    rng = np.random.default_rng(23)
    x = rng.standard_normal((3, 64))
    q = rng.integers(-127, 128, (4, 64)).astype(np.int8)
    col = rng.uniform(0.5, 1.5, 64).astype(np.float16).astype(np.float64)
    s = rng.uniform(0.5, 2, 4)
    b = rng.standard_normal(4)
    y = O.q8_2f_linear(x, q, col, s, b)
    for t in range(3):
        for o in range(4):
            acc = sum(x[t, j] * float(O.round_bf16(float(q[o, j]) * col[j])) for j in range(64))
            assert abs(y[t, o] - (s[o] * acc + b[o])) <= 1e-12 * (1 + abs(y[t, o]))


# ------------------------------------------------------------------ v norm
# egemma2.rs Prog::qkv normalises q, k and v heads in one pass with weights
# for q and k only: v is RMS-normalised without a weight, without RoPE.

def test_v_norm_gives_unit_rms_v_heads_and_leaves_q_k_alone():
    rng = np.random.default_rng(31)
    nq, nkv, hd = 4, 2, 64
    qkv = O.round_bf16(rng.standard_normal((9, (nq + 2 * nkv) * hd)) * 3)
    qn, kn = 1 + 0.1 * rng.standard_normal(hd), 1 + 0.1 * rng.standard_normal(hd)
    base = O.qk_prep(qkv, nq, nkv, hd, 0, nq * hd, qn, kn, 1e-6, None, None, None, 0, 1.0)
    vn = O.qk_prep(qkv, nq, nkv, hd, 0, nq * hd, qn, kn, 1e-6, None, None, None, 0, 1.0,
                   v_off=(nq + nkv) * hd)
    qk = slice(0, (nq + nkv) * hd)
    np.testing.assert_array_equal(vn[:, qk], base[:, qk])
    v = vn[:, (nq + nkv) * hd:].reshape(9, nkv, hd)
    rms = np.sqrt(np.mean(v ** 2, axis=2))
    np.testing.assert_allclose(rms, 1.0, atol=4e-3)           # bf16-rounded unit rows
    # a constant head c maps to c / sqrt(c^2 + eps) (times the unit weight)
    const = np.zeros((1, (nq + 2 * nkv) * hd))
    const[0, (nq + nkv) * hd:] = 0.25
    out = O.qk_prep(const, nq, nkv, hd, 0, nq * hd, None, None, 1e-6, None, None, None, 0, 1.0,
                    v_off=(nq + nkv) * hd)
    np.testing.assert_allclose(out[0, (nq + nkv) * hd:], O.round_bf16(0.25 / np.sqrt(0.0625 + 1e-6)))


# -------------------------------------------------------- two-range items
# zimage.rs PFa {img_off, n_img, cap_off, n_cap}: image and caption rows of
# one item attend as one sequence.

def test_two_range_items_reduce_to_varlen_and_ignore_range_order_without_window():
    rng = np.random.default_rng(41)
    nq, nkv, hd = 2, 1, 64
    qkv = rng.standard_normal((70, (nq + 2 * nkv) * hd))
    scale = hd ** -0.5
    args = (nq, nkv, hd, 0, nq * hd, (nq + nkv) * hd)
    # len2 = 0: exactly the packed-sequence attention
    one = O.attention_items(qkv, [[0, 30, 0, 0], [30, 40, 0, 0]], *args, 0, scale)
    np.testing.assert_array_equal(one, O.attention_varlen(qkv, [0, 30, 70], *args, 0, scale))
    # an item = its rows attended as one sequence, wherever they lie
    it = O.attention_items(qkv, [[40, 30, 0, 12]], *args, 0, scale)
    rows = np.r_[40:70, 0:12]
    ref = O.attention_varlen(qkv[rows], [0, 42], *args, 0, scale)
    np.testing.assert_allclose(it[rows], ref, rtol=0, atol=0)
    assert np.all(np.isnan(it[12:40]))
    # full attention: swapping the two ranges changes nothing per row
    sw = O.attention_items(qkv, [[0, 12, 40, 30]], *args, 0, scale)
    np.testing.assert_allclose(sw[rows], it[rows], rtol=1e-12, atol=1e-12)


# ------------------------------------------- two-range items inside the block
# zimage.rs module doc "The chain": the CFG pair is one batch-2 program over
# rows [img0 | img1 | cap0 | cap1]; row-local steps run once over all rows and
# attention runs per item over its two row ranges.

def _cfg_pair_case(window=0):
    import dataclasses
    cfg = dataclasses.replace(_tiny("sandwich", "rms", True, "silu", "2d", True, window),
                              lens=(12, 12, 5, 3), cfg_pair=True)
    p = synth.draw_layer(cfg, 0, 71)
    lens = cfg.lens
    cu = synth.cu_seqlens(lens)
    x = synth.draw_x(int(cu[-1]), cfg.d, 72)
    a = O.round_bf16(O.rms_norm(x, p["norm1_w"], cfg.eps))
    return cfg, p, lens, cu, x, a


@pytest.mark.parametrize("window", [0, 4])
def test_cfg_pair_block_equals_the_gathered_items_as_sequences(window):
    # the block over [img0 | img1 | cap0 | cap1] with items equals, row for
    # row, the plain block over the rows gathered as [img0 | cap0 | img1 |
    # cap1] with one sequence per item and each row keeping its RoPE angles
    import dataclasses
    cfg, p, lens, cu, x, a = _cfg_pair_case(window)
    items = synth.attn_items(cfg, lens)
    assert items.tolist() == [[0, 12, 24, 5], [12, 12, 29, 3]]
    tables = synth.rope_tables(cfg, lens)
    r = O.block_forward(cfg, p, x, a, cu, 0, tables, next_norm=(p["norm1_w"], None), items=items)
    perm = np.r_[0:12, 24:29, 12:24, 29:32]
    plain = dataclasses.replace(cfg, cfg_pair=False, lens=(17, 15))
    tab_g = dict(tables, cos=tables["cos"][perm], sin=tables["sin"][perm])
    g = O.block_forward(plain, p, x[perm], a[perm], synth.cu_seqlens([17, 15]), 0, tab_g,
                        next_norm=(p["norm1_w"], None))
    np.testing.assert_array_equal(r["x_out"][perm], g["x_out"])
    np.testing.assert_array_equal(r["a_out"][perm], g["a_out"])
    # and it is not the per-range attention: the caption rows see the image
    sep = O.block_forward(cfg, p, x, a, cu, 0, tables, next_norm=(p["norm1_w"], None))
    assert not np.allclose(sep["x_out"][24:], r["x_out"][24:])


def test_block_with_single_range_items_equals_the_sequence_block():
    cfg, p, lens, cu, x, a = _cfg_pair_case()
    tables = synth.rope_tables(cfg, lens)
    items = np.asarray([[int(cu[i]), int(lens[i]), 0, 0] for i in range(len(lens))], dtype=np.int32)
    r = O.block_forward(cfg, p, x, a, cu, 0, tables, items=items)
    q = O.block_forward(cfg, p, x, a, cu, 0, tables)
    np.testing.assert_array_equal(r["x_out"], q["x_out"])


# ------------------------------------------------------ per-layer input (PLE)
# egemma2.rs TextGpu::forward "per-layer input": pin = rms(ple_scale * x W_in^T)
# ple_norm; z = gelu(h W_gate^T) * pin; H = (H + rms(z W_proj^T) w) * scalar.

def _ple_case(seed=51):
    cfg = _tiny("sandwich", "rms", True, "gelu_tanh", "1d", True, 0)
    import dataclasses
    cfg = dataclasses.replace(cfg, ple_dim=64)
    p = synth.draw_layer(cfg, 0, seed)
    cu = synth.cu_seqlens(cfg.lens)
    x = synth.draw_x(int(cu[-1]), cfg.d, seed + 1)
    a = O.round_bf16(O.rms_norm(x, p["norm1_w"], cfg.eps))
    ple = dict(synth.draw_ple(cfg, seed), x_in=O.round_bf16(x))
    return cfg, p, cu, x, a, ple, synth.rope_tables(cfg, cfg.lens)


def test_ple_block_matches_torch_library_composition():
    # the per-layer input chain against torch's own ops, with a layer scalar
    # other than 1 (it must follow the PLE residual, not the FFN's), pin as
    # wide as d so that swapping the two norm weights would still run, and
    # distinct, non-unit norm weights; a gelu on pin instead of the gate, the
    # norm weights swapped or the scalar on the FFN residual all fail here
    import dataclasses
    cfg = dataclasses.replace(_tiny("sandwich", "rms", True, "gelu_tanh", "1d", True, 0),
                              ple_dim=32, post=1.5)
    p = synth.draw_layer(cfg, 0, 61)
    lens = cfg.lens
    cu = synth.cu_seqlens(lens)
    x = synth.draw_x(int(cu[-1]), cfg.d, 62)
    tables = synth.rope_tables(cfg, lens)
    ple = dict(synth.draw_ple(cfg, 61), x_in=O.round_bf16(x))
    ple["norm_w"] = ple["norm_w"] * 2.0 - 0.5            # far from ple_post_w
    assert np.max(np.abs(ple["norm_w"] - p["ple_post_w"])) > 0.5
    nxt = synth.draw_norm(np.random.default_rng(3), cfg.d, False)
    x_ref, a_ref, a_in = _torch_block(cfg, p, x, cu, tables, nxt, ple=ple)
    r = O.block_forward(cfg, p, x, a_in, cu, 0, tables, next_norm=nxt, ple=ple)
    np.testing.assert_allclose(r["x_out"], x_ref, rtol=2e-5, atol=2e-5)
    # a_out is bf16: the two sides may round a value on either side of a tie
    # (one bf16 step, 2^-7 relative at most), and only rarely
    diff = np.abs(r["a_out"] - a_ref)
    assert np.all(diff <= 2.0 ** -7 * np.abs(a_ref) + 1e-30)
    assert np.mean(diff > 0) < 0.05
    # the branch is far from negligible, so the comparison sees it
    base = O.block_forward(dataclasses.replace(cfg, ple_dim=0), p, x, a_in, cu, 0, tables)
    assert np.linalg.norm(r["x_out"] - base["x_out"]) > 0.1 * np.linalg.norm(r["x_out"])


@pytest.mark.parametrize("zeroed", ["ple_in", "ple_gate", "ple_proj"])
def test_ple_path_with_a_zero_weight_adds_nothing(zeroed):
    # any of the three projections at zero makes the branch exactly 0
    # (pin = 0, or gelu(0) = 0, or rms(0) = 0): the block without the path
    cfg, p, cu, x, a, ple, tables = _ple_case()
    p[zeroed] = dict(p[zeroed], s=np.zeros_like(p[zeroed]["s"]))
    r = O.block_forward(cfg, p, x, a, cu, 0, tables, ple=ple)
    import dataclasses
    base = O.block_forward(dataclasses.replace(cfg, ple_dim=0), p, x, a, cu, 0, tables)
    np.testing.assert_array_equal(r["x_out"], base["x_out"])


def test_ple_pin_ignores_the_scale_of_its_source():
    # rms(c v) = rms(v) up to eps: scaling the per-layer source by a power of
    # two (exact in bf16) barely moves the result, while the branch itself is
    # far from zero
    cfg, p, cu, x, a, ple, tables = _ple_case(53)
    r1 = O.block_forward(cfg, p, x, a, cu, 0, tables, ple=ple)
    r2 = O.block_forward(cfg, p, x, a, cu, 0, tables, ple=dict(ple, x_in=ple["x_in"] * 4.0))
    import dataclasses
    base = O.block_forward(dataclasses.replace(cfg, ple_dim=0), p, x, a, cu, 0, tables)
    assert np.max(np.abs(r1["x_out"] - base["x_out"])) > 0.05
    # equal up to bf16 rounding flips of pin (eps moves it by ~1e-4 relative)
    d_scaled, d_branch = r2["x_out"] - r1["x_out"], r1["x_out"] - base["x_out"]
    assert np.linalg.norm(d_scaled) < 0.02 * np.linalg.norm(d_branch)
    assert np.any(r1["ple_z"])
