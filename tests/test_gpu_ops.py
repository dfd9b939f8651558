"""Per-op parity of the CUDA kernels (called through the C-ABI) against the
CPU oracle on the same seeded inputs.

Tolerances (relative Frobenius): 1e-3 per GEMM with a bf16 output, 3e-3 for
attention (bf16 P), 2e-3 for row ops with bf16 outputs (the oracle rounds at
the same storage points, so only rare rounding flips differ).  A GEMM with an
f32 output reads the same bf16 x and exact int8 weights as the oracle, so only
the f32 accumulation order differs: its gate is 20x the pages' own error level
for that comparison (zimage.rs module doc, Measured: zi_q8mm against f64,
5e-7).  Integer work (int8 widening, index/mask computation) is compared bit
for bit.
"""
import numpy as np
import pytest

import transformer_encoder_forward_gb300 as te
from oracle import encoder as O
from transformer_encoder_forward_gb300 import synth
from tests.gpu_util import bf16_input, page_constant, q8_dev, record_margin, rel_frob, to_dev, to_np

pytestmark = pytest.mark.gpu

# f32-output GEMM gate: 20x the pages' rel. error of the q8 GEMM against f64
GEMM_F32_TOL = 20 * page_constant("q8_gemm_rel_error_vs_f64")["value"]


def _gemm_gate(ydt):
    return GEMM_F32_TOL if ydt == "f32" else 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    torch.cuda.init()
    te.lib()
    yield
    te.check()


def _torch():
    import torch
    return torch


# ------------------------------------------------------------------ q8 GEMM

GEMM_CASES = [
    # m, k, item widths, bias, residual, out dtype
    (1, 64, [32], False, False, "f32"),
    (37, 256, [256, 256, 256], False, False, "bf16"),
    (101, 256, [1024, 1024], False, False, "bf16"),
    (101, 1024, [256], False, True, "f32"),
    (300, 512, [96, 160], True, False, "f32"),
    (777, 768, [768, 768, 768], True, False, "bf16"),
    (1000, 192, [64, 128, 192, 288], True, True, "f32"),
    (2112, 3840, [384], False, False, "f32"),
    (4100, 320, [640], False, False, "bf16"),
    # two 192-token tiles per weight stage (many feature tiles, ragged last pair)
    (3000, 256, [3840, 3840], True, False, "bf16"),
    (3000, 256, [3840, 3840], False, True, "f32"),
    # a residual other than y (f32 and bf16 y), rows wider than n
    (300, 512, [96, 160], True, "sep", "f32"),
    (777, 256, [256, 512], False, "sep", "bf16"),
    # long K, 128-token tiles two a unit (the choice that saves a wave here)
    (2111, 2048, [3840], False, True, "f32"),
    # the DiT out projection at 8448 tokens: whole waves of two-tile units,
    # then the rows left in a second launch (in-place residual)
    (8448, 3840, [3840], False, True, "f32"),
    # a split with a separate residual and a bf16 output
    (2111, 2048, [3840], True, "sep", "bf16"),
    # two 192-token tiles a unit at long K, bf16 out: the second tile partly
    # drained by converter warps (whole waves, then a second launch)
    (6000, 3072, [768, 768, 768], True, False, "bf16"),
    # resident weights over long runs of token tiles that cross feature pairs
    (5000, 512, [512, 512, 512], False, False, "bf16"),
    (5000, 512, [512], True, True, "f32"),
    (6001, 448, [1536], False, False, "bf16"),
]


@pytest.mark.parametrize("m,k,ns,bias,resid,ydt", GEMM_CASES)
def test_q8_linear_matches_oracle(m, k, ns, bias, resid, ydt):
    torch = _torch()
    rng = np.random.default_rng([m, k, len(ns)])
    x, x64 = bf16_input(rng, (m, k))
    ws = [synth.draw_q8(rng, n, k, True, bias) for n in ns]
    dt = torch.float32 if ydt == "f32" else torch.bfloat16
    items, outs, refs = [], [], []
    for w in ws:
        q, s, b = q8_dev(w)
        n = w["q"].shape[0]
        r_np = rng.standard_normal((m, n)).astype(np.float32) if resid else None
        if resid == "sep":
            # separate residual and output, both with padded rows
            r_dev = torch.zeros(m, n + 8, dtype=torch.float32, device="cuda")
            r_dev[:, :n] = to_dev(r_np)
            y_full = torch.full((m, n + 16), float("nan"), dtype=dt, device="cuda")
            y = y_full[:, :n]
            it = {"w": te.q8w(q, s, b), "y": y, "ldy": n + 16, "residual": r_dev, "ldr": n + 8}
            outs_keep = (r_dev, y_full)
        else:
            y = to_dev(r_np) if resid else torch.full((m, n), float("nan"), dtype=dt, device="cuda")
            it = {"w": te.q8w(q, s, b), "y": y, "ldy": n}
            outs_keep = None
            if resid:
                it.update(residual=y, ldr=n)       # in place: y = y + s*acc + b
        items.append(it)
        outs.append((y, (q, s, b, outs_keep)))
        ref = O.q8_linear(x64, w["q"], w["s"], w["b"], r_np)
        refs.append(O.round_bf16(ref) if ydt == "bf16" else ref)
    te.q8_linear(x, items)
    te.check()
    gate = _gemm_gate(ydt)
    for i, ((y, (_, _, _, keep)), ref) in enumerate(zip(outs, refs)):
        got = to_np(y)
        assert np.all(np.isfinite(got))
        e = record_margin("q8_linear", f"m={m} k={k} item {i} {ydt}", rel_frob(got, ref), gate)
        assert e < gate, e
        if keep is not None:                   # the row padding of y is untouched
            assert bool(torch.isnan(keep[1][:, y.shape[1]:]).all())


def test_q8_linear_exact_integer_case_is_bit_exact():
    # integer x with |x| <= 16, unit scale, K = 1024: every partial sum is an
    # integer below 2^24, so f32 accumulation is exact and so is the result
    torch = _torch()
    rng = np.random.default_rng(5)
    m, k = 333, 1024
    xi = rng.integers(-16, 17, (m, k)).astype(np.float32)
    x = torch.from_numpy(xi).to(torch.bfloat16).cuda()
    q_np = rng.integers(-127, 128, (256, k), dtype=np.int8)
    q = to_dev(q_np)
    s = torch.ones(256, dtype=torch.float32, device="cuda")
    y = torch.empty(m, 256, dtype=torch.float32, device="cuda")
    te.q8_linear(x, [{"w": te.q8w(q, s), "y": y, "ldy": 256}])
    exact = xi.astype(np.int64) @ q_np.astype(np.int64).T
    np.testing.assert_array_equal(to_np(y), exact.astype(np.float64))


def test_q8_linear_split_launch_is_bit_exact_on_integers():
    # 2111 rows at K = 2048, N = 3840 run as whole waves of two-tile units
    # and a second launch for the rest: integer x with |x| <= 4 keeps every
    # partial sum an integer below 2^24, so each row must be exact in both
    torch = _torch()
    rng = np.random.default_rng(6)
    m, k, n = 2111, 2048, 3840
    xi = rng.integers(-4, 5, (m, k)).astype(np.float32)
    x = torch.from_numpy(xi).to(torch.bfloat16).cuda()
    q_np = rng.integers(-127, 128, (n, k), dtype=np.int8)
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    te.q8_linear(x, [{"w": te.q8w(to_dev(q_np), torch.ones(n, device="cuda")), "y": y, "ldy": n}])
    te.check()
    exact = xi.astype(np.int64) @ q_np.astype(np.int64).T
    np.testing.assert_array_equal(to_np(y), exact.astype(np.float64))


@pytest.mark.parametrize("reps", [2, 4])
def test_int8_widening_and_indexing_are_bit_exact(reps):
    # one-hot activation rows pick single weight columns: y[t, o] = q[o, j_t]
    # exactly, for every int8 value (including -128) and every row/column;
    # with 4 repetitions (1027 tokens) the weights are widened into the
    # shared-memory-resident tile
    torch = _torch()
    k, n = 256, 256
    q_np = (np.arange(n * k, dtype=np.int64).reshape(n, k) * 37 % 256 - 128).astype(np.int8)
    m = reps * k + 3
    cols = np.r_[np.tile(np.r_[np.arange(k), np.arange(k)[::-1]], reps // 2), [0, 17, 255]]
    xi = np.zeros((m, k), np.float32)
    xi[np.arange(m), cols] = 1.0
    x = torch.from_numpy(xi).to(torch.bfloat16).cuda()
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    te.q8_linear(x, [{"w": te.q8w(to_dev(q_np), torch.ones(n, device="cuda")), "y": y, "ldy": n}])
    np.testing.assert_array_equal(to_np(y), q_np[:, cols].T.astype(np.float64))
    assert set(np.unique(q_np)) == set(range(-128, 128))


@pytest.mark.parametrize("m,k,f,act,bias", [(37, 256, 1024, "gelu_tanh", False),
                                            (1000, 512, 2048, "gelu_tanh", True),
                                            (2112, 3840, 10240, "silu", False),
                                            (101, 256, 96, "silu", True),
                                            (300, 192, 32, "gelu_tanh", False),
                                            (5000, 512, 2048, "gelu_tanh", False),
                                            # resident weights with 192-token tiles
                                            (1500, 256, 768, "silu", True),
                                            (2100, 192, 512, "gelu_tanh", False),
                                            # long K, 128-token tiles two a unit
                                            (2300, 2048, 1024, "silu", True),
                                            # whole waves of two-tile units, then a second launch
                                            (2400, 3072, 3840, "silu", False)])
def test_gated_linear_matches_oracle(m, k, f, act, bias):
    # m = act(bf16(g)) * bf16(u): the same storage points as the g|u panel
    # followed by the gate, without the panel
    torch = _torch()
    rng = np.random.default_rng([m, k, f])
    x, x64 = bf16_input(rng, (m, k))
    wg = synth.draw_q8(rng, f, k, True, bias)
    wu = synth.draw_q8(rng, f, k, True, bias)
    dg, du = q8_dev(wg), q8_dev(wu)
    out = torch.full((m, f), float("nan"), dtype=torch.bfloat16, device="cuda")
    te.q8_gated_linear(x, te.q8w(*dg), te.q8w(*du),
                       te.TE_ACT_SILU if act == "silu" else te.TE_ACT_GELU_TANH, out)
    te.check()
    g = O.round_bf16(O.q8_linear(x64, wg["q"], wg["s"], wg["b"]))
    u = O.round_bf16(O.q8_linear(x64, wu["q"], wu["s"], wu["b"]))
    ref = O.round_bf16(O.gate_act(np.concatenate([g, u], axis=1), f, True, act))
    got = to_np(out)
    assert np.all(np.isfinite(got))
    assert rel_frob(got, ref) < 2e-3, rel_frob(got, ref)


@pytest.mark.parametrize("m,k,n,act,ydt", [(4096, 768, 3072, "gelu_tanh", "bf16"), (77, 256, 96, "silu", "bf16"),
                                            # f32 out: 16-token halves (192-token tiles), and
                                            # two tiles a unit at long K
                                            (4096, 768, 512, "gelu_tanh", "f32"),
                                            (6000, 3072, 768, "silu", "f32"),
                                            (6000, 3072, 768, "gelu_tanh", "bf16")])
def test_q8_linear_epilogue_activation_matches_oracle(m, k, n, act, ydt):
    # y = act(bf16(s * acc + b)), stored as y's type
    torch = _torch()
    rng = np.random.default_rng([m, n])
    x, x64 = bf16_input(rng, (m, k))
    w = synth.draw_q8(rng, n, k, True, True)
    dw = q8_dev(w)
    dt = torch.float32 if ydt == "f32" else torch.bfloat16
    y = torch.full((m, n), float("nan"), dtype=dt, device="cuda")
    te.q8_linear(x, [{"w": te.q8w(*dw), "y": y, "ldy": n,
                      "epilogue": te.TE_EPI_SILU if act == "silu" else te.TE_EPI_GELU_TANH}])
    te.check()
    pre = O.round_bf16(O.q8_linear(x64, w["q"], w["s"], w["b"]))
    ref = O.gate_act(pre, n, False, act)
    if ydt == "bf16":
        ref = O.round_bf16(ref)
    assert rel_frob(to_np(y), ref) < 2e-3


# ---------------------------------------------------------------- attention

ATTN_CASES = [
    # lens, nq, nkv, hd, window
    ([1], 2, 2, 64, 0),
    ([37, 64], 4, 4, 64, 0),
    ([5, 130, 64, 1, 200], 3, 3, 64, 0),
    ([5, 130, 64, 1, 200], 2, 2, 128, 17),
    ([300, 77], 4, 2, 64, 64),
    ([700, 129], 2, 1, 128, 512),
    ([1056, 1056], 2, 2, 128, 0),
    ([955, 16, 400], 2, 2, 64, 512),
    # many heads with grouped K/V: more work items (480) than CTAs resident
    # at once (two an SM), in several waves
    ([955, 16, 400, 130, 64, 1, 200, 37], 24, 8, 64, 0),
    ([955, 16, 400, 130, 64, 1, 200, 37], 24, 24, 64, 100),
]


def _attn_run(qkv_t, cu, nq, nkv, hd, window, scale):
    torch = _torch()
    T = qkv_t.shape[0]
    out = torch.full((T, nq * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    te.attn_varlen_fwd(qkv_t, qkv_t.shape[1], 0, nq * hd, (nq + nkv) * hd, cu, to_dev(cu), nq,
                       nkv, hd, window, scale, out, nq * hd)
    return out


@pytest.mark.parametrize("lens,nq,nkv,hd,window", ATTN_CASES)
def test_attention_matches_oracle(lens, nq, nkv, hd, window):
    rng = np.random.default_rng([len(lens), nq, hd, window])
    cu = synth.cu_seqlens(lens)
    T = int(cu[-1])
    W = (nq + 2 * nkv) * hd
    qkv_t, qkv = bf16_input(rng, (T, W), 1.5)
    scale = 1.0 / np.sqrt(hd)
    out = _attn_run(qkv_t, cu, nq, nkv, hd, window, scale)
    te.check()
    ref = O.attention_varlen(qkv, cu, nq, nkv, hd, 0, nq * hd, (nq + nkv) * hd, window, scale)
    got = to_np(out)
    assert np.all(np.isfinite(got))
    e = record_margin("attention", f"lens={lens[:4]} hd={hd} W={window}", rel_frob(got, O.round_bf16(ref)), 3e-3)
    assert e < 3e-3, e


# More (sequence, query block) pairs than the launch parameters carry as a
# longest-first work list: the launcher falls back to the plain grid
# (query block, head, sequence).  A text batch of many short sequences.
MANY_SEQ_CASES = [(700, 64, 1, 1, 0), (700, 64, 2, 2, 37), (660, 128, 2, 1, 0), (660, 128, 2, 2, 21)]


@pytest.mark.parametrize("nseq,hd,nq,nkv,window", MANY_SEQ_CASES)
def test_attention_many_short_sequences_plain_grid(nseq, hd, nq, nkv, window):
    torch = _torch()
    rng = np.random.default_rng([nseq, hd, nq, window])
    lens = rng.integers(1, 201, nseq)
    lens[:3] = [1, 200, 129]
    qb = 128 if hd == 64 else 256                     # queries per CTA
    assert int(np.sum((lens + qb - 1) // qb)) > 640   # beyond the work list
    cu = synth.cu_seqlens(lens)
    T = int(cu[-1])
    W = (nq + 2 * nkv) * hd
    qkv_t, qkv = bf16_input(rng, (T, W), 1.5)
    scale = 1.0 / np.sqrt(hd)
    out = _attn_run(qkv_t, cu, nq, nkv, hd, window, scale).clone()
    te.check()
    ref = O.attention_varlen(qkv, cu, nq, nkv, hd, 0, nq * hd, (nq + nkv) * hd, window, scale)
    got = to_np(out)
    assert np.all(np.isfinite(got))
    e = record_margin("attention plain grid", f"{nseq} seqs hd={hd} W={window}",
                      rel_frob(got, O.round_bf16(ref)), 3e-3)
    assert e < 3e-3, e
    # other sequences and out-of-window keys have no effect, bit for bit:
    # change every key/value row of the odd sequences and, with a window, the
    # keys/values past each even sequence's first window + 1 rows
    pert = qkv_t.clone()
    keep = np.zeros(T, dtype=bool)       # query rows whose visible keys are unchanged
    for s in range(nseq):
        r0, r1 = int(cu[s]), int(cu[s + 1])
        if s % 2:
            pert[r0:r1, nq * hd:] = (torch.randn(r1 - r0, 2 * nkv * hd, device="cuda") * 40).to(torch.bfloat16)
        elif window and r1 - r0 > 2 * window + 2:
            cut = r0 + window + 1                      # rows from cut on change
            pert[cut:r1, nq * hd:] = (torch.randn(r1 - cut, 2 * nkv * hd, device="cuda") * 40).to(torch.bfloat16)
            keep[r0] = True                            # row r0 sees keys r0 .. r0 + window only
        else:
            keep[r0:r1] = True
    out2 = _attn_run(pert, cu, nq, nkv, hd, window, scale)
    te.check()
    idx = torch.from_numpy(np.nonzero(keep)[0]).cuda()
    assert idx.numel() > 0
    assert torch.equal(out2[idx], out[idx])


def test_attention_scale_one_and_length_one_sequences():
    rng = np.random.default_rng(21)
    lens = [1, 1, 3, 1]
    cu = synth.cu_seqlens(lens)
    qkv_t, qkv = bf16_input(rng, (6, 3 * 64))
    out = to_np(_attn_run(qkv_t, cu, 1, 1, 64, 0, 1.0))
    for r in (0, 1, 5):                      # a length-1 sequence returns its own v exactly
        np.testing.assert_array_equal(out[r], qkv[r, 128:])
    ref = O.attention_varlen(qkv, cu, 1, 1, 64, 0, 64, 128, 0, 1.0)
    assert rel_frob(out, O.round_bf16(ref)) < 3e-3


def test_attention_masked_keys_and_other_sequences_have_no_effect():
    torch = _torch()
    rng = np.random.default_rng(22)
    lens = [200, 150]
    cu = synth.cu_seqlens(lens)
    nq, hd, W = 2, 64, 20
    qkv_t, _ = bf16_input(rng, (350, 3 * nq * hd))
    base = _attn_run(qkv_t, cu, nq, nq, hd, W, 0.125).clone()
    pert = qkv_t.clone()
    # keys/values of rows 100.. of sequence 0 and all of sequence 1 change
    pert[100:200, nq * hd:] = torch.randn(100, 2 * nq * hd, device="cuda").to(torch.bfloat16) * 50
    pert[200:, :] = torch.randn(150, 3 * nq * hd, device="cuda").to(torch.bfloat16)
    out = _attn_run(pert, cu, nq, nq, hd, W, 0.125)
    # rows 0 .. 100-W-1 of sequence 0 see none of the changed keys: bit-identical
    assert torch.equal(out[:100 - W], base[:100 - W])
    assert not torch.equal(out[100 - W:200], base[100 - W:200])


def test_attention_wide_window_equals_full():
    torch = _torch()
    rng = np.random.default_rng(23)
    lens = [130, 61]
    cu = synth.cu_seqlens(lens)
    qkv_t, _ = bf16_input(rng, (191, 3 * 128))
    full = _attn_run(qkv_t, cu, 1, 1, 128, 0, 0.1)
    wide = _attn_run(qkv_t, cu, 1, 1, 128, 129, 0.1)
    assert torch.equal(full, wide)


# ----------------------------------------------------------------- row ops

@pytest.mark.parametrize("d,kind,xdt", [(256, "rms", "f32"), (768, "ln", "f32"),
                                        (3840, "rms", "f32"), (512, "ln", "bf16"),
                                        (4096, "rms", "bf16")])
def test_rownorm_matches_oracle(d, kind, xdt):
    torch = _torch()
    rng = np.random.default_rng([d, len(kind)])
    t = 203
    if xdt == "f32":
        x64 = rng.standard_normal((t, d)).astype(np.float32) * 2 + 0.3
        x = to_dev(x64)
    else:
        x, x64 = bf16_input(rng, (t, d), 2.0)
    w, b = synth.draw_norm(rng, d, kind == "ln")
    y = torch.empty(t, d, dtype=torch.bfloat16, device="cuda")
    te.rownorm(x, to_dev(w), to_dev(b) if b is not None else None,
               te.TE_NORM_LN if kind == "ln" else te.TE_NORM_RMS, 1e-5, y, pre=0.5)
    ref = O.round_bf16(O.norm(kind, 0.5 * np.asarray(x64, np.float64), w, b, 1e-5))
    assert rel_frob(to_np(y), ref) < 2e-3


@pytest.mark.parametrize("d,sandwich,nxt,kind", [(512, True, True, "rms"), (3840, True, False, "rms"),
                                                 (768, False, True, "ln"), (256, False, False, "rms"),
                                                 (3840, True, True, "rms"), (2048, False, True, "ln"),
                                                 (4096, True, True, "ln"), (1032, True, True, "rms"),
                                                 (1024, True, True, "rms"), (520, False, True, "ln"),
                                                 (1024, False, False, "ln")])
def test_add_norm_matches_oracle(d, sandwich, nxt, kind):
    torch = _torch()
    rng = np.random.default_rng([d, int(sandwich), int(nxt)])
    rows = 157
    h = rng.standard_normal((rows, d)).astype(np.float32)
    t = rng.standard_normal((rows, d)).astype(np.float32) * 3
    wp, _ = synth.draw_norm(rng, d, False)
    wn, bn = synth.draw_norm(rng, d, kind == "ln")
    h_t, t_t = to_dev(h), to_dev(t)
    a = torch.zeros(rows, d, dtype=torch.bfloat16, device="cuda")
    te.add_norm(h_t, t_t, to_dev(wp) if sandwich else None, 0.75,
                to_dev(wn) if nxt else None, to_dev(bn) if (nxt and bn is not None) else None,
                te.TE_NORM_LN if kind == "ln" else te.TE_NORM_RMS, 1e-6, a)
    h_ref = O.add_norm_sandwich(h, t, wp, 0.75, 1e-6) if sandwich else h.astype(np.float64) + t
    assert rel_frob(to_np(h_t), h_ref) < 1e-6
    if nxt:
        a_ref = O.round_bf16(O.norm(kind, O.round_f32(h_ref), wn, bn, 1e-6))
        assert rel_frob(to_np(a), a_ref) < 2e-3
    else:
        assert torch.count_nonzero(a) == 0


@pytest.mark.parametrize("d,sandwich,kind", [(512, True, "rms"), (3840, True, "rms"),
                                            (768, False, "ln"), (2048, False, "rms"),
                                            (1024, True, "rms")])
def test_add_norm_with_adaln_gate_and_scale_matches_oracle(d, sandwich, kind):
    torch = _torch()
    rng = np.random.default_rng([d, 77, int(sandwich)])
    rows = 141
    h = rng.standard_normal((rows, d)).astype(np.float32)
    t = rng.standard_normal((rows, d)).astype(np.float32) * 3
    wp, _ = synth.draw_norm(rng, d, False)
    wn, bn = synth.draw_norm(rng, d, kind == "ln")
    mod = synth.draw_mods(rng, d)
    g, s = mod[1], mod[2]
    h_t, t_t = to_dev(h), to_dev(t)
    a = torch.zeros(rows, d, dtype=torch.bfloat16, device="cuda")
    te.add_norm_mod(h_t, t_t, to_dev(wp) if sandwich else None, to_dev(g), 0.75, to_dev(wn),
                    to_dev(bn) if bn is not None else None, to_dev(s),
                    te.TE_NORM_LN if kind == "ln" else te.TE_NORM_RMS, 1e-6, a)
    if sandwich:
        h_ref = O.add_norm_sandwich(h, t, wp, 0.75, 1e-6, gate=g)
    else:
        h_ref = h.astype(np.float64) + g.astype(np.float64) * t
    assert rel_frob(to_np(h_t), h_ref) < 1e-6
    a_ref = O.round_bf16(O.norm(kind, O.round_f32(h_ref), wn, bn, 1e-6, mod_scale=s))
    assert rel_frob(to_np(a), a_ref) < 2e-3
    # rownorm with the scale alone
    y = torch.empty(rows, d, dtype=torch.bfloat16, device="cuda")
    te.rownorm_mod(h_t, to_dev(wn), to_dev(bn) if bn is not None else None, to_dev(s),
                   te.TE_NORM_LN if kind == "ln" else te.TE_NORM_RMS, 1e-6, y)
    y_ref = O.round_bf16(O.norm(kind, to_np(h_t), wn, bn, 1e-6, mod_scale=s))
    assert rel_frob(to_np(y), y_ref) < 2e-3


@pytest.mark.parametrize("d", [256, 768, 3840])
def test_adaln_identity_vectors_are_bit_exact_no_ops(d):
    # s = 0 and g = 1 must give exactly the unmodulated row ops (one width of
    # each add_norm layout: a warp, four warps and eight warps a row)
    torch = _torch()
    rng = np.random.default_rng([91, d])
    rows = 99
    h = to_dev(rng.standard_normal((rows, d)).astype(np.float32))
    t = to_dev(rng.standard_normal((rows, d)).astype(np.float32))
    wp, _ = synth.draw_norm(rng, d, False)
    wn, _ = synth.draw_norm(rng, d, False)
    zeros, ones = torch.zeros(d, device="cuda"), torch.ones(d, device="cuda")
    h1, h2 = h.clone(), h.clone()
    a1 = torch.empty(rows, d, dtype=torch.bfloat16, device="cuda")
    a2 = torch.empty_like(a1)
    te.add_norm(h1, t, to_dev(wp), 1.0, to_dev(wn), None, te.TE_NORM_RMS, 1e-6, a1)
    te.add_norm_mod(h2, t, to_dev(wp), ones, 1.0, to_dev(wn), None, zeros, te.TE_NORM_RMS, 1e-6, a2)
    te.check()
    assert torch.equal(h1, h2) and torch.equal(a1, a2)


@pytest.mark.parametrize("hd,nq,nkv,rope,qk", [(64, 8, 8, "1d", True), (128, 4, 4, "2d", True),
                                               (64, 4, 2, None, False), (128, 30, 30, "2d", True)])
def test_qkv_prep_with_v_norm_matches_oracle(hd, nq, nkv, rope, qk):
    torch = _torch()
    rng = np.random.default_rng([hd, nq, nkv, 5])
    lens = [37, 64, 100]
    cfg = synth.small_config("c2", hd=hd, rope=rope)
    tb = synth.rope_tables(cfg, lens)
    T = sum(lens)
    W = (nq + 2 * nkv) * hd
    x, x64 = bf16_input(rng, (T, W), 2.0)
    qn = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32) if qk else None
    kn = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32) if qk else None
    dv = lambda a, dt=None: to_dev(a, dt) if a is not None else None
    te.qkv_prep_rope(x, W, 0, nq * hd, (nq + nkv) * hd, nq, nkv, hd, dv(qn), dv(kn), True, 1e-6,
                     dv(tb["cos"]), dv(tb["sin"]), dv(tb["pos"], torch.int32), tb["sec"], 0.5, T)
    te.check()
    ref = O.qk_prep(x64, nq, nkv, hd, 0, nq * hd, qn, kn, 1e-6, tb["cos"], tb["sin"], tb["pos"],
                    tb["sec"], 0.5, v_off=(nq + nkv) * hd)
    assert rel_frob(to_np(x), ref) < 2e-3


@pytest.mark.parametrize("hd,nq,nkv,rope,qk", [(64, 8, 8, "1d", True), (128, 4, 4, "2d", True),
                                               (64, 4, 2, "2d", False), (128, 2, 1, None, True)])
def test_qk_prep_rope_matches_oracle(hd, nq, nkv, rope, qk):
    torch = _torch()
    rng = np.random.default_rng([hd, nq, nkv])
    lens = [37, 64, 100]
    cfg = synth.small_config("c2", hd=hd, rope=rope)
    tb = synth.rope_tables(cfg, lens)
    T = sum(lens)
    W = (nq + 2 * nkv) * hd
    qkv_t, qkv = bf16_input(rng, (T, W), 2.0)
    qn, _ = synth.draw_norm(rng, hd, False)
    kn, _ = synth.draw_norm(rng, hd, False)
    cos = to_dev(tb["cos"]) if rope else None
    sin = to_dev(tb["sin"]) if rope else None
    pos = to_dev(tb["pos"]) if rope else None
    te.qk_prep_rope(qkv_t, W, 0, nq * hd, nq, nkv, hd, to_dev(qn) if qk else None,
                    to_dev(kn) if qk else None, 1e-6, cos, sin, pos, tb["sec"], 1.25, T)
    ref = O.qk_prep(qkv, nq, nkv, hd, 0, nq * hd, qn if qk else None, kn if qk else None, 1e-6,
                    tb["cos"], tb["sin"], tb["pos"], tb["sec"], 1.25)
    got = to_np(qkv_t)
    assert rel_frob(got, ref) < 2e-3
    np.testing.assert_array_equal(got[:, (nq + nkv) * hd:], qkv[:, (nq + nkv) * hd:])  # v untouched


@pytest.mark.parametrize("act,gated,f", [("gelu_tanh", True, 1024), ("silu", True, 10240),
                                         ("gelu_tanh", False, 3072), ("silu", False, 64)])
def test_gate_act_matches_oracle(act, gated, f):
    torch = _torch()
    rng = np.random.default_rng([f, int(gated)])
    rows = 211
    ld = 2 * f if gated else f
    gu_t, gu = bf16_input(rng, (rows, ld), 2.0)
    m = torch.empty(rows, f, dtype=torch.bfloat16, device="cuda")
    te.gate_act(gu_t, ld, f if gated else -1, te.TE_ACT_SILU if act == "silu" else te.TE_ACT_GELU_TANH,
                m, f, rows, f)
    ref = O.round_bf16(O.gate_act(gu, f, gated, act))
    assert rel_frob(to_np(m), ref) < 2e-3


@pytest.mark.parametrize("d,norm", [(512, True), (256, False), (3840, True)])
def test_pool_mean_matches_oracle(d, norm):
    torch = _torch()
    rng = np.random.default_rng([d, int(norm)])
    lens = synth.draw_lens(synth.CONFIGS["c2"])[:7]
    cu = synth.cu_seqlens(lens)
    x = rng.standard_normal((int(cu[-1]), d)).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    out = torch.empty(len(lens), d, dtype=torch.float32, device="cuda")
    te.pool_mean(to_dev(x), cu, to_dev(cu), to_dev(w) if norm else None, 1e-6, out)
    ref = O.pool_mean(x, cu, w if norm else None, 1e-6)
    assert rel_frob(to_np(out), ref) < 1e-5


# ------------------------------------------------- 32-element block formats

@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_block_unpack_is_bit_exact(fmt):
    torch = _torch()
    rng = np.random.default_rng([len(fmt), 3])
    n, k = 77, 640
    w = synth.draw_block_packed(rng, n, k, fmt)
    packed = torch.from_numpy(w["packed"]).cuda()
    q = torch.empty(n, k, dtype=torch.int8, device="cuda")
    bs = torch.empty(n, k // 32, dtype=torch.int16, device="cuda")
    (te.q8_0_unpack if fmt == "q8_0" else te.q4_0_unpack)(packed, n, k, q, bs)
    te.check()
    q_ref, d_ref = (O.decode_q8_0 if fmt == "q8_0" else O.decode_q4_0)(w["packed"], n, k)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    d_got = bs.cpu().numpy().view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(d_got, d_ref)


def _block_weight(rng, n, k, fmt, with_scale, bias):
    """Device operands of one block-format weight (unpacked on the GPU) and
    the oracle's decode of the same bytes."""
    torch = _torch()
    w = synth.draw_block_packed(rng, n, k, fmt)
    q = torch.empty(n, k, dtype=torch.int8, device="cuda")
    bs = torch.empty(n, k // 32, dtype=torch.int16, device="cuda")
    (te.q8_0_unpack if fmt == "q8_0" else te.q4_0_unpack)(torch.from_numpy(w["packed"]).cuda(), n, k, q, bs)
    q_np, d_np = (O.decode_q8_0 if fmt == "q8_0" else O.decode_q4_0)(w["packed"], n, k)
    s = rng.uniform(0.5, 2.0, n).astype(np.float32) if with_scale else None
    b = (rng.standard_normal(n) * 0.02).astype(np.float32) if bias else None
    dev = (q, to_dev(s) if s is not None else None, to_dev(b) if b is not None else None, bs)
    return dev, (q_np, d_np, s, b)


@pytest.mark.parametrize("m,k,specs,ydt", [
    (37, 256, [("q8_0", True, False, 384)], "f32"),
    (300, 512, [("q4_0", False, True, 384), ("q8_0", True, False, 256)], "bf16"),
    (1000, 3840, [("q8_0", False, False, 384)], "bf16"),
    # enough feature tiles for two 192-token tiles per weight stage, ragged tail
    (2200, 3840, [("q4_0", True, False, 3840), ("q8_0", False, False, 3840)], "bf16"),
    # K <= 512 with enough tokens: resident weights (128- and 192-token tiles)
    (2000, 512, [("q4_0", True, True, 512), ("q8_0", False, False, 256)], "bf16"),
    (1500, 256, [("q8_0", True, False, 384), ("q4_0", False, True, 256)], "f32"),
])
def test_block_format_gemm_matches_oracle(m, k, specs, ydt):
    torch = _torch()
    rng = np.random.default_rng([m, k, len(specs)])
    x, x64 = bf16_input(rng, (m, k))
    dt = torch.float32 if ydt == "f32" else torch.bfloat16
    items, checks = [], []
    for fmt, with_scale, bias, n in specs:
        dev, ref = _block_weight(rng, n, k, fmt, with_scale, bias)
        y = torch.full((m, n), float("nan"), dtype=dt, device="cuda")
        items.append({"w": te.q8w(dev[0], dev[1], dev[2], dev[3]), "y": y, "ldy": n})
        r = O.q8_block_linear(x64, ref[0], ref[1], ref[2], ref[3])
        checks.append((y, O.round_bf16(r) if ydt == "bf16" else r, dev))
    te.q8_linear(x, items)
    te.check()
    gate = _gemm_gate(ydt)
    for i, (y, ref, _) in enumerate(checks):
        got = to_np(y)
        assert np.all(np.isfinite(got))
        e = record_margin("block-format GEMM", f"m={m} k={k} item {i} {ydt}", rel_frob(got, ref), gate)
        assert e < gate, e


@pytest.mark.parametrize("m,k,f", [(777, 768, 512), (1500, 384, 512), (1800, 256, 256)])
def test_block_format_gated_linear_matches_oracle(m, k, f):
    torch = _torch()
    rng = np.random.default_rng(71)
    x, x64 = bf16_input(rng, (m, k))
    dg, rg = _block_weight(rng, f, k, "q8_0", False, False)
    du, ru = _block_weight(rng, f, k, "q4_0", True, False)
    out = torch.empty(m, f, dtype=torch.bfloat16, device="cuda")
    te.q8_gated_linear(x, te.q8w(*dg), te.q8w(*du), te.TE_ACT_SILU, out)
    te.check()
    g = O.round_bf16(O.q8_block_linear(x64, *rg))
    u = O.round_bf16(O.q8_block_linear(x64, *ru))
    ref = O.round_bf16(O.gate_act(np.concatenate([g, u], axis=1), f, True, "silu"))
    assert rel_frob(to_np(out), ref) < 1e-3


def test_block_format_gemm_unit_scales_is_bit_exact():
    # d = 1 (f16 0x3C00) and integer x: every product and partial sum is an
    # integer below 2^24, so the result is exact
    torch = _torch()
    rng = np.random.default_rng(72)
    m, k, n = 129, 512, 256
    xi = rng.integers(-16, 17, (m, k)).astype(np.float32)
    x = torch.from_numpy(xi).to(torch.bfloat16).cuda()
    q_np = rng.integers(-127, 128, (n, k), dtype=np.int8)
    bs = torch.full((n, k // 32), 0x3C00, dtype=torch.int16, device="cuda")
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    te.q8_linear(x, [{"w": te.q8w(to_dev(q_np), None, None, bs), "y": y, "ldy": n}])
    np.testing.assert_array_equal(to_np(y), (xi.astype(np.int64) @ q_np.astype(np.int64).T).astype(np.float64))


# ------------------------------------------------------------------- q8_2f

@pytest.mark.parametrize("m,k,ns,ydt", [(101, 256, [256], "f32"), (777, 768, [768, 512], "bf16"),
                                        (2200, 3840, [3840, 3840], "bf16"), (300, 320, [96], "f32"),
                                        (2000, 448, [384, 256], "f32"), (1500, 192, [256, 512], "bf16")])
def test_q8_2f_gemm_matches_oracle(m, k, ns, ydt):
    torch = _torch()
    rng = np.random.default_rng([m, k, 2])
    x, x64 = bf16_input(rng, (m, k))
    dt = torch.float32 if ydt == "f32" else torch.bfloat16
    items, checks, keep = [], [], []
    for n in ns:
        w = synth.draw_q8(rng, n, k, True, True)
        col = rng.uniform(0.5, 1.5, k).astype(np.float16).astype(np.float32)
        dev = (to_dev(w["q"]), to_dev(w["s"]), to_dev(w["b"]), None, to_dev(col))
        keep.append(dev)
        y = torch.full((m, n), float("nan"), dtype=dt, device="cuda")
        items.append({"w": te.q8w(*dev), "y": y, "ldy": n})
        r = O.q8_2f_linear(x64, w["q"], col, w["s"], w["b"])
        checks.append((y, O.round_bf16(r) if ydt == "bf16" else r))
    te.q8_linear(x, items)
    te.check()
    gate = _gemm_gate(ydt)
    for i, (y, ref) in enumerate(checks):
        got = to_np(y)
        assert np.all(np.isfinite(got))
        e = record_margin("q8_2f GEMM", f"m={m} k={k} item {i} {ydt}", rel_frob(got, ref), gate)
        assert e < gate, e


# ------------------------------------------------------- two-range items

def _items_case(rng, hd, nq, nkv, n_img, n_cap, nitems=2):
    """A CFG-like packing [img0 | img1 | cap0 | cap1]: item i = (img_i, cap_i)."""
    W = (nq + 2 * nkv) * hd
    T = nitems * (n_img + n_cap)
    items = [[i * n_img, n_img, nitems * n_img + i * n_cap, n_cap] for i in range(nitems)]
    x, x64 = bf16_input(rng, (T, W))
    return np.asarray(items, np.int32), x, x64, T, W


@pytest.mark.parametrize("hd,nq,nkv,n_img,n_cap,window", [
    (128, 4, 4, 96, 70, 0),      # query / key tiles spanning the two ranges
    (128, 2, 1, 256, 33, 0),
    (64, 4, 2, 160, 200, 0),
    (64, 2, 2, 224, 61, 50),     # windowed over joint positions
])
def test_attention_two_range_items_match_oracle(hd, nq, nkv, n_img, n_cap, window):
    torch = _torch()
    rng = np.random.default_rng([hd, n_img, n_cap])
    items, x, x64, T, W = _items_case(rng, hd, nq, nkv, n_img, n_cap)
    out = torch.full((T, nq * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    scale = hd ** -0.5
    te.attn_items_fwd(x, W, 0, nq * hd, (nq + nkv) * hd, items, to_dev(items), T, nq, nkv, hd, window,
                      scale, out, nq * hd)
    te.check()
    ref = O.attention_items(x64, items, nq, nkv, hd, 0, nq * hd, (nq + nkv) * hd, window, scale)
    got = to_np(out)
    assert np.all(np.isfinite(got))
    assert rel_frob(got, ref) < 3e-3, rel_frob(got, ref)


def test_attention_two_range_items_many_heads():
    """More work items (8 query blocks x 48 heads = 384) than hd-64 CTAs
    resident at once, over four two-range items."""
    torch = _torch()
    rng = np.random.default_rng(47)
    hd, nq, nkv = 64, 48, 16
    items, x, x64, T, W = _items_case(rng, hd, nq, nkv, 160, 96, nitems=4)
    out = torch.full((T, nq * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    scale = hd ** -0.5
    te.attn_items_fwd(x, W, 0, nq * hd, (nq + nkv) * hd, items, to_dev(items), T, nq, nkv, hd, 0, scale, out,
                      nq * hd)
    te.check()
    ref = O.attention_items(x64, items, nq, nkv, hd, 0, nq * hd, (nq + nkv) * hd, 0, scale)
    got = to_np(out)
    assert np.all(np.isfinite(got))
    e = record_margin("attention", "two-range items, 48 heads", rel_frob(got, ref), 3e-3)
    assert e < 3e-3, e


def test_attention_items_equal_varlen_on_gathered_rows_bit_exactly():
    torch = _torch()
    rng = np.random.default_rng(43)
    hd, nq, nkv = 128, 2, 2
    items, x, x64, T, W = _items_case(rng, hd, nq, nkv, 128 + 32, 77, nitems=2)
    out = torch.empty(T, nq * hd, dtype=torch.bfloat16, device="cuda")
    te.attn_items_fwd(x, W, 0, nq * hd, (nq + nkv) * hd, items, to_dev(items), T, nq, nkv, hd, 0,
                      hd ** -0.5, out, nq * hd)
    # the same rows gathered in joint order, as two packed sequences
    rows = np.concatenate([np.r_[o1:o1 + l1, o2:o2 + l2] for o1, l1, o2, l2 in items])
    xg = x[torch.from_numpy(rows).cuda()].contiguous()
    lens = [int(l1 + l2) for _, l1, _, l2 in items]
    cu = synth.cu_seqlens(lens)
    og = torch.empty_like(out)
    te.attn_varlen_fwd(xg, W, 0, nq * hd, (nq + nkv) * hd, cu, torch.from_numpy(cu).cuda(), nq, nkv,
                       hd, 0, hd ** -0.5, og, nq * hd)
    te.check()
    assert torch.equal(out[torch.from_numpy(rows).cuda()], og)
    # single-range items are the packed sequences themselves
    it1 = np.asarray([[0, 100, 0, 0], [100, 37, 0, 0]], np.int32)
    o1 = torch.empty(137, nq * hd, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    te.attn_items_fwd(x, W, 0, nq * hd, (nq + nkv) * hd, it1, to_dev(it1), T, nq, nkv, hd, 0,
                      hd ** -0.5, o1, nq * hd)
    cu2 = synth.cu_seqlens([100, 37])
    te.attn_varlen_fwd(x[:137], W, 0, nq * hd, (nq + nkv) * hd, cu2, torch.from_numpy(cu2).cuda(), nq,
                       nkv, hd, 0, hd ** -0.5, o2, nq * hd)
    te.check()
    assert torch.equal(o1, o2)


def test_mma_peak_runs_at_every_width():
    """The MMA-form ceiling runs on every SM pair and reports a rate within
    what the tensor cores can do: 8192 dense bf16 flops a cycle an SM, at
    most 2.6 PFLOP/s at the 2070 MHz top clock of 152 SMs."""
    pairs = te.sm_count() // 2
    for bn in (64, 128, 192, 256):
        ms = te.mma_peak(bn, 200)
        te.check()
        tf = pairs * 200 * 8 * 2 * 256 * bn * 16 / (ms * 1e-3) / 1e12
        assert 50.0 < tf < 2700.0, (bn, ms, tf)

