"""Whole-block and stack parity of the CUDA path (te_encoder_block_fwd through
the C-ABI) against the CPU oracle.

Gate: relative Frobenius error <= 5e-3 on the block output x (also checked on
the residual-free delta x_out - x_in, the stricter diagnostic) and on the next
block's normed input a.  Stacks are compared teacher-forced: the oracle takes
the GPU's input to each checked layer.  At the largest workload the oracle
runs on sampled query rows (all keys).
"""
import numpy as np
import pytest

import transformer_encoder_forward_gb300 as te
from oracle import encoder as O
from transformer_encoder_forward_gb300 import synth
from transformer_encoder_forward_gb300.model import EncoderStack
from tests.gpu_util import record_margin, rel_frob, to_dev, to_np

pytestmark = pytest.mark.gpu

TOL = 5e-3


def _stack(cfg, lens, layers, seed=11, jitter=True):
    ps = [synth.draw_layer(cfg, i, seed, jitter) for i in range(layers)]
    tables = synth.rope_tables(cfg, lens)
    fin = synth.draw_final_norm(cfg, seed) if cfg.pool else None
    ple = synth.draw_ple(cfg, seed) if cfg.ple_dim else None
    st = EncoderStack(cfg, ps, lens, tables, fin, ple=ple, items=synth.attn_items(cfg, lens))
    st.ple_host = ple
    return st, ps, tables


def _next_norm(ps, i):
    return (ps[i + 1]["norm1_w"], ps[i + 1]["norm1_b"]) if i + 1 < len(ps) else None


def _mods(ps, i):
    """(this block's adaLN vectors, the next block's s_msa), or Nones."""
    mod = ps[i].get("mod")
    nxt = ps[i + 1]["mod"][0] if mod is not None and i + 1 < len(ps) else None
    return mod, nxt


def _check_layer(cfg, st, ps, tables, i, x, a, rows=None, tag=None):
    """Runs GPU layer i in place on (x, a) and compares against the oracle on
    the same inputs."""
    import torch
    x_in, a_in = to_np(x), to_np(a)
    te.encoder_block_fwd(st.descs[i], x, a, st.cu_host, st.cu_dev, st.workspace)
    te.check()
    mod, next_s = _mods(ps, i)
    ple = None
    if st.ple_x is not None:
        ple = dict(st.ple_host, x_in=to_np(st.ple_x))
    r = O.block_forward(cfg, ps[i], x_in, a_in, st.cu_host, i, tables, _next_norm(ps, i),
                        rows=rows, mod=mod, next_mod_scale=next_s, ple=ple, items=st.items_host)
    sel = slice(None) if rows is None else np.asarray(rows)
    got_x = to_np(x)[sel]
    xin = x_in[sel]
    assert np.all(np.isfinite(got_x))
    tag = f"{tag or cfg.name} layer {i}"
    e_x = record_margin("block", f"{tag} x_out", rel_frob(got_x, r["x_out"]), TOL)
    e_d = record_margin("block", f"{tag} x_out - x_in", rel_frob(got_x - xin, r["x_out"] - xin), 2 * TOL)
    assert e_x < TOL, (i, e_x)
    assert e_d < 2 * TOL, (i, e_d)
    if r["a_out"] is not None:
        e_a = record_margin("block", f"{tag} a_out", rel_frob(to_np(a)[sel], r["a_out"]), TOL)
        assert e_a < TOL, (i, e_a)
    return e_x, e_d


FORMS = {
    "c1_full": ("c1", {}, (37, 64)),
    "c2_small": ("c2", dict(layers=2, window=40), (100, 1, 300, 37)),
    "c3_small": ("c3", dict(layers=2), (200, 129)),
    "c4_small": ("c4", dict(d=512, heads=4, kv_heads=4, ffn=1024), (150, 133)),
    "gqa_small": ("c2", dict(layers=2, kv_heads=2, window=0), (64, 65)),
    # the DiT block with adaLN modulation (gates on both branches, scales on
    # every pre-norm including the next block's input)
    "c4m_small": ("c4m", dict(layers=3, d=512, heads=4, kv_heads=4, ffn=1024), (150, 133)),
    # the ViT block with the 32-element block weight formats
    "c3q8_small": ("c3q8", dict(layers=2), (200, 129)),
    "c3q4_small": ("c3q4", dict(layers=2), (200, 129)),
    # the text block with the v heads normalised too
    "c2v_small": ("c2v", dict(layers=2, window=40), (100, 1, 300, 37)),
    # the text block with the per-layer input path
    "c2p_small": ("c2p", dict(layers=2, window=40), (100, 1, 300, 37)),
    # the DiT block with q8_2f weights (column field)
    "c4f_small": ("c4f", dict(layers=2, d=512, heads=4, kv_heads=4, ffn=1024), (150, 133)),
    # the DiT block as the CFG pair's batch-2 program: rows [img0 | img1 |
    # cap0 | cap1], attention per two-range item
    "c4c_small": ("c4c", dict(layers=2, d=512, heads=4, kv_heads=4, ffn=1024), (256, 256, 64, 32)),
}


@pytest.mark.parametrize("name", list(FORMS))
def test_block_forms_match_oracle(name):
    key, over, lens = FORMS[name]
    cfg = synth.small_config(key, lens=lens, **over)
    st, ps, tables = _stack(cfg, lens, cfg.layers)
    x = to_dev(synth.draw_x(st.T, cfg.d, 3))
    import torch
    a = torch.empty(st.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    if st.ple_x is not None:
        te.cast_bf16(x, st.ple_x)        # the per-layer inputs' source, as a forward makes it
    st.input_norm(x, a)
    s0 = ps[0]["mod"][0] if cfg.adaln else None
    a0 = O.round_bf16(O.norm(cfg.norm, to_np(x), ps[0]["norm1_w"], ps[0]["norm1_b"], cfg.eps,
                             mod_scale=s0))
    assert rel_frob(to_np(a), a0) < 2e-3
    for i in range(cfg.layers):
        _check_layer(cfg, st, ps, tables, i, x, a, tag=name)


def test_text_stack_24_layers_teacher_forced_and_pooled():
    import torch
    cfg = synth.CONFIGS["c2"]
    lens = synth.draw_lens(cfg)
    st, ps, tables = _stack(cfg, lens, cfg.layers)
    x = to_dev(synth.draw_x(st.T, cfg.d, 4))
    a = torch.empty(st.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    st.input_norm(x, a)
    check = {0, 1, 12, 23}
    for i in range(cfg.layers):
        if i in check:
            _check_layer(cfg, st, ps, tables, i, x, a)
        else:
            te.encoder_block_fwd(st.descs[i], x, a, st.cu_host, st.cu_dev, st.workspace)
    out = torch.empty(len(lens), cfg.d, dtype=torch.float32, device="cuda")
    te.pool_mean(x, st.cu_host, st.cu_dev, st.final_norm, cfg.eps, out)
    te.check()
    ref = O.pool_mean(to_np(x), st.cu_host, synth.draw_final_norm(cfg, 11), cfg.eps)
    assert rel_frob(to_np(out), ref) < 1e-5


def test_vit_stack_16_layers_teacher_forced():
    import torch
    cfg = synth.CONFIGS["c3"]
    lens = synth.draw_lens(cfg)
    st, ps, tables = _stack(cfg, lens, cfg.layers)
    x = to_dev(synth.draw_x(st.T, cfg.d, 5))
    a = torch.empty(st.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    st.input_norm(x, a)
    for i in range(cfg.layers):
        if i in (0, 8, 15):
            _check_layer(cfg, st, ps, tables, i, x, a)
        else:
            te.encoder_block_fwd(st.descs[i], x, a, st.cu_host, st.cu_dev, st.workspace)


def test_dit_block_full_size():
    import torch
    cfg = synth.CONFIGS["c4"]
    lens = synth.draw_lens(cfg)
    st, ps, tables = _stack(cfg, lens, 1, jitter=False)
    x = to_dev(synth.draw_x(st.T, cfg.d, 6))
    a = torch.empty(st.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    st.input_norm(x, a)
    _check_layer(cfg, st, ps, tables, 0, x, a)


def test_dit_block_with_adaln_full_size():
    import torch
    cfg = synth.small_config("c4m", layers=2)
    lens = synth.draw_lens(cfg)
    st, ps, tables = _stack(cfg, lens, 2, jitter=False)
    x = to_dev(synth.draw_x(st.T, cfg.d, 6))
    a = torch.empty(st.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    st.input_norm(x, a)
    _check_layer(cfg, st, ps, tables, 0, x, a)


def test_dit_cfg_pair_block_full_size():
    import torch
    cfg = synth.CONFIGS["c4c"]
    lens = synth.draw_lens(cfg)
    st, ps, tables = _stack(cfg, lens, 1, jitter=False)
    assert st.items_host is not None and st.T == 2240
    x = to_dev(synth.draw_x(st.T, cfg.d, 6))
    a = torch.empty(st.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    st.input_norm(x, a)
    _check_layer(cfg, st, ps, tables, 0, x, a)


def test_cfg_pair_block_equals_the_block_over_gathered_items_bit_exactly():
    # every step but attention works per row, and an item's attention equals
    # the attention of its rows gathered into one sequence: the block over
    # [img0 | img1 | cap0 | cap1] with items must give, row for row, the same
    # bits as the block over [img0 | cap0 | img1 | cap1] with one sequence per
    # item (each row keeping its RoPE angles)
    import dataclasses
    import torch
    cfg = synth.small_config("c4c", layers=2, d=512, heads=4, kv_heads=4, ffn=1024,
                             lens=(256, 256, 96, 32))
    lens = cfg.lens
    st, ps, tables = _stack(cfg, lens, 2)
    perm = np.r_[0:256, 512:608, 256:512, 608:640]
    plain = dataclasses.replace(cfg, cfg_pair=False, lens=(352, 288))
    tab_g = dict(tables, cos=tables["cos"][perm], sin=tables["sin"][perm])
    st_g = EncoderStack(plain, ps, plain.lens, tab_g)
    assert st_g.items_host is None
    x0 = synth.draw_x(st.T, cfg.d, 13)
    x, a, _ = st.buffers()
    x.copy_(to_dev(x0))
    st.forward_device(x, a)
    xg, ag, _ = st_g.buffers()
    xg.copy_(to_dev(x0[perm]))
    st_g.forward_device(xg, ag)
    te.check()
    idx = torch.from_numpy(perm).cuda()
    assert torch.equal(x[idx], xg)
    assert torch.equal(a[idx], ag)


def test_dit_stack_layer_at_4224_tokens_sampled_rows():
    import torch
    cfg = synth.small_config("c5", layers=2)
    lens = synth.draw_lens(cfg)
    st, ps, tables = _stack(cfg, lens, 2, jitter=False)
    x = to_dev(synth.draw_x(st.T, cfg.d, 7))
    a = torch.empty(st.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    st.input_norm(x, a)
    rng = np.random.default_rng(8)
    rows = np.sort(np.r_[rng.choice(st.T, 60, replace=False), [0, 4223, 4224, 8447]])
    _check_layer(cfg, st, ps, tables, 0, x, a, rows=rows)


def test_stack_forward_is_deterministic():
    import torch
    cfg = synth.small_config("c2", layers=2, window=40, lens=(100, 300, 37))
    st, _, _ = _stack(cfg, cfg.lens, 2)
    x0 = to_dev(synth.draw_x(st.T, cfg.d, 9))
    outs = []
    for _ in range(2):
        x, a, out = st.buffers()
        x.copy_(x0)
        st.forward_device(x, a, out)
        outs.append((x.clone(), out.clone()))
    te.check()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_forward_host_graph_replay_equals_the_device_forward():
    # the public host-to-host call runs eagerly once, then replays a captured
    # graph: every call returns the device forward's result bit for bit
    import torch
    cfg = synth.small_config("c2", layers=2, window=40, lens=(100, 300, 37))
    st, _, _ = _stack(cfg, cfg.lens, 2)
    x0 = synth.draw_x(st.T, cfg.d, 9)
    x, a, out = st.buffers()
    x.copy_(to_dev(x0))
    st.forward_device(x, a, out)
    torch.cuda.synchronize()
    ref = out.cpu()
    x_host = torch.from_numpy(np.ascontiguousarray(x0)).pin_memory()
    res = torch.empty(len(cfg.lens), cfg.d, dtype=torch.float32).pin_memory()
    s = torch.cuda.Stream()
    for _ in range(3):
        res.zero_()
        st.forward_host(x_host, res, stream=s)
        s.synchronize()
        te.check()
        assert torch.equal(res, ref)
    assert len(st._graphs) == 1


def test_forward_host_stream_overlapped_copies_give_each_input_its_own_result():
    # five inputs in sequence through the overlapped path (two buffer sets,
    # copies on their own streams): each result equals the device forward of
    # that input bit for bit, for a pooled and an unpooled stack
    import torch
    for key, lens in (("c2", (100, 300, 37)), ("c3", (64, 130))):
        cfg = synth.small_config(key, layers=2, lens=lens)
        st, _, _ = _stack(cfg, cfg.lens, 2)
        xs = [synth.draw_x(st.T, cfg.d, 20 + i) for i in range(5)]
        refs = []
        for x0 in xs:
            x, a, out = st.buffers()
            x.copy_(to_dev(x0))
            st.forward_device(x, a, out)
            torch.cuda.synchronize()
            refs.append((out if cfg.pool else x).cpu())
        hosts = [torch.from_numpy(np.ascontiguousarray(x0)).pin_memory() for x0 in xs]
        shape = (len(cfg.lens), cfg.d) if cfg.pool else (st.T, cfg.d)
        res = [torch.full(shape, float("nan"), dtype=torch.float32).pin_memory() for _ in xs]
        s = torch.cuda.Stream()
        start, end = st.forward_host_stream(hosts, res, stream=s)
        end.synchronize()
        te.check()
        for i in range(len(xs)):
            assert torch.equal(res[i], refs[i]), (key, i)
        assert start.elapsed_time(end) > 0


def test_profiled_forward_times_every_step_class_and_changes_nothing():
    # the block's step-boundary events (te_block_desc.prof_events) give each
    # step class's GPU time; recording them leaves every output bit-identical
    import torch
    cfg = synth.small_config("c2", layers=2, window=40, lens=(100, 300, 37))
    st, _, _ = _stack(cfg, cfg.lens, 2)
    x0 = to_dev(synth.draw_x(st.T, cfg.d, 9))
    x, a, out = st.buffers()
    x.copy_(x0)
    st.forward_device(x, a)
    te.check()
    ref_x, ref_a = x.clone(), a.clone()
    x.copy_(x0)
    s = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s)
    ms = st.profile_forward(x, a, stream=s)
    t1.record(s)
    te.check()
    assert torch.equal(x, ref_x) and torch.equal(a, ref_a)
    assert set(ms) == set(st.STEP_CLASSES)
    for name in ("gemm_qkv", "qk_prep", "attention", "gemm_o", "norm_ffn", "gemm_gu", "gemm_down"):
        assert ms[name] > 0, (name, ms)
    assert all(v >= 0 for v in ms.values())
    assert sum(ms.values()) <= t0.elapsed_time(t1) * 1.01 + 0.01
    assert all(d.prof_events is None for d in st.descs)


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty:UserWarning")   # the refused call enqueues nothing
def test_prof_events_are_refused_during_graph_capture():
    import ctypes
    import torch
    cfg = synth.small_config("c2", layers=1, window=0, lens=(64,))
    st, _, _ = _stack(cfg, cfg.lens, 1)
    x, a, _ = st.buffers()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(te.TE_BLOCK_PROF_EVENTS)]
    s = torch.cuda.Stream()
    for e in evs:
        e.record(s)
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * te.TE_BLOCK_PROF_EVENTS)(*[e.cuda_event for e in evs])
    d = st.descs[0]
    d.prof_events = ctypes.cast(arr, ctypes.c_void_p).value
    g = torch.cuda.CUDAGraph()
    err = None
    try:
        # the call is refused before it enqueues anything: the capture ends empty
        with torch.cuda.graph(g, stream=s):
            try:
                te.encoder_block_fwd(d, x, a, st.cu_host, st.cu_dev, st.workspace, stream=s)
            except te.TEError as e:
                err = e
    finally:
        d.prof_events = None
    assert err is not None and err.status == te.TE_EINVAL and "captured" in str(err)
    torch.cuda.synchronize()
    te.check()
