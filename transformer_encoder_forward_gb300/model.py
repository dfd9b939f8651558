"""An encoder stack driven through the C-ABI: device copies of the weights,
one te_block_desc per layer, and the forward loop.

Marshalling only: the initial pre-norm, every block and the final pool are
calls into libtefwd.  The stack follows "cortiq-engine 0.8.39
src/gpu_metal/egemma2.rs" TextGpu::forward (an input norm, then the layers,
each ending with the next layer's input norm, then the final norm and
mean-pool) and "cera 0.2.4 src/model/vision_encoder_gpu.rs"
encode_image_gpu (plain pre-norm blocks).
"""
from __future__ import annotations

from typing import List, Optional

import numpy as np

from . import (TE_ACT_GELU_TANH, TE_ACT_SILU, TE_NORM_LN, TE_NORM_RMS, TE_RESID_PLAIN,
               TE_RESID_SANDWICH, block_workspace, cast_bf16, encoder_block_fwd, pool_mean,
               q4_0_unpack, q8_0_unpack, q8w, rownorm, rownorm_mod, te_block_desc)


def _dev(a, device, dtype=None):
    import torch
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


class LayerWeights:
    """Device tensors of one layer (q8 weights, scales, biases, norm vectors)."""

    def __init__(self, cfg, p: dict, device):
        import torch
        self.t = {}
        for key in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "ple_in", "ple_gate", "ple_proj"):
            w = p.get(key)
            if w is None:
                self.t[key] = None
                continue
            if "packed" in w:
                # a 32-element block format: upload the packed bytes and
                # unpack them on the device once (int8 q + f16 block scales)
                n, k = w["n"], w["k"]
                q = torch.empty(n, k, dtype=torch.int8, device=device)
                bs = torch.empty(n, k // 32, dtype=torch.int16, device=device)
                unpack = q8_0_unpack if w["fmt"] == "q8_0" else q4_0_unpack
                unpack(_dev(w["packed"], device), n, k, q, bs)
                self.t[key] = (q, _dev(w.get("s"), device), _dev(w["b"], device), bs, None)
            else:
                self.t[key] = (_dev(w["q"], device), _dev(w["s"], device), _dev(w["b"], device), None,
                               _dev(w.get("col"), device))
        for key in ("norm1_w", "norm1_b", "norm2_w", "norm2_b", "post_attn_w", "post_ffn_w",
                    "q_norm", "k_norm", "mod", "ple_post_w"):
            self.t[key] = _dev(p.get(key), device, torch.float32)
        # adaLN: s_msa (row 0 of mod) scales this layer's input norm
        self.s_msa = self.t["mod"][0] if self.t["mod"] is not None else None


class EncoderStack:
    """A stack of encoder blocks over a packed batch with fixed lengths."""

    def __init__(self, cfg, layers: List[dict], lens, tables: dict,
                 final_norm: Optional[np.ndarray] = None, device="cuda", ple: Optional[dict] = None,
                 items: Optional[np.ndarray] = None):
        """items: two-range attention items, int32 [n, 4] = (off1, len1,
        off2, len2) covering every row once (the CFG pair's batch-2 program,
        zimage.rs); None: attention per sequence of ``lens``."""
        import torch
        self.cfg = cfg
        self.device = torch.device(device)
        self.lens = np.asarray(lens, dtype=np.int32)
        cu = np.zeros(len(lens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(self.lens)
        self.cu_host = cu
        self.cu_dev = torch.from_numpy(cu).to(self.device)
        self.T = int(cu[-1])
        self.layers = [LayerWeights(cfg, p, self.device) for p in layers]
        self.final_norm = _dev(final_norm, self.device, torch.float32)
        self.rope_cos = _dev(tables.get("cos"), self.device, torch.float32)
        self.rope_sin = _dev(tables.get("sin"), self.device, torch.float32)
        self.rope_pos = _dev(tables.get("pos"), self.device, torch.int32)
        self.rope_sec = int(tables.get("sec") or 0)
        # per-layer input path: the stack's input as bf16 (filled by each
        # forward) and the stack-level norm of pin
        self.ple_x = self.ple_norm = None
        self.ple_scale = 0.0
        if getattr(cfg, "ple_dim", 0):
            if ple is None:
                raise ValueError("the per-layer input path needs the stack-level ple weights")
            self.ple_x = torch.empty(self.T, cfg.d, dtype=torch.bfloat16, device=self.device)
            self.ple_norm = _dev(ple["norm_w"], self.device, torch.float32)
            self.ple_scale = float(ple["scale"])
        self.items_host = self.items_dev = None
        if items is not None:
            self.items_host = np.ascontiguousarray(np.asarray(items, dtype=np.int32).reshape(-1, 4))
            self.items_dev = torch.from_numpy(self.items_host).to(self.device)
        self.descs = [self._desc(i) for i in range(len(self.layers))]
        ws = max(block_workspace(d, self.T) for d in self.descs)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)

    def _desc(self, i: int) -> te_block_desc:
        cfg, L = self.cfg, self.layers[i]
        nxt = self.layers[i + 1] if i + 1 < len(self.layers) else None
        ptr = lambda t: t.data_ptr() if t is not None else None
        d = te_block_desc()
        d.d, d.n_heads, d.n_kv_heads, d.head_dim, d.ffn = cfg.d, cfg.heads, cfg.kv_heads, cfg.hd, cfg.ffn
        d.norm_kind = TE_NORM_LN if cfg.norm == "ln" else TE_NORM_RMS
        d.resid_form = TE_RESID_SANDWICH if cfg.form == "sandwich" else TE_RESID_PLAIN
        d.act = TE_ACT_SILU if cfg.act == "silu" else TE_ACT_GELU_TANH
        d.gated = 1 if cfg.gated else 0
        d.window = cfg.window_of(i)
        d.eps, d.attn_scale, d.post, d.q_mul = cfg.eps, cfg.scale, cfg.post, 1.0
        for key in ("wq", "wk", "wv", "wo", "wg", "wd"):
            setattr(d, key, q8w(*L.t[key]))
        if L.t["wu"] is not None:
            d.wu = q8w(*L.t["wu"])
        d.ffn_norm_w, d.ffn_norm_b = ptr(L.t["norm2_w"]), ptr(L.t["norm2_b"])
        d.post_attn_w, d.post_ffn_w = ptr(L.t["post_attn_w"]), ptr(L.t["post_ffn_w"])
        if nxt is not None:
            d.next_norm_w, d.next_norm_b = ptr(nxt.t["norm1_w"]), ptr(nxt.t["norm1_b"])
            d.next_mod_scale = ptr(nxt.s_msa)
        d.mod = ptr(L.t["mod"])
        d.v_norm = 1 if getattr(cfg, "v_norm", False) else 0
        if self.ple_x is not None:
            d.ple_dim, d.ple_scale = cfg.ple_dim, self.ple_scale
            d.ple_in, d.ple_gate, d.ple_proj = (q8w(*L.t[k]) for k in ("ple_in", "ple_gate", "ple_proj"))
            d.ple_norm_w, d.ple_post_w = ptr(self.ple_norm), ptr(L.t["ple_post_w"])
            d.ple_x = ptr(self.ple_x)
        if self.items_host is not None:
            d.attn_items_host = self.items_host.ctypes.data
            d.attn_items_dev = ptr(self.items_dev)
            d.n_attn_items = self.items_host.shape[0]
        if cfg.qk_norm:
            d.q_norm, d.k_norm = ptr(L.t["q_norm"]), ptr(L.t["k_norm"])
        if self.rope_sec:
            d.rope_cos, d.rope_sin = ptr(self.rope_cos), ptr(self.rope_sin)
            d.rope_pos, d.rope_sec = ptr(self.rope_pos), self.rope_sec
            d.rope_rows = self.rope_cos.shape[0]
        return d

    # ------------------------------------------------------------ forward

    def buffers(self):
        import torch
        x = torch.empty(self.T, self.cfg.d, dtype=torch.float32, device=self.device)
        a = torch.empty(self.T, self.cfg.d, dtype=torch.bfloat16, device=self.device)
        out = torch.empty(len(self.lens), self.cfg.d, dtype=torch.float32, device=self.device)
        return x, a, out

    def input_norm(self, x, a, stream=None):
        L0 = self.layers[0]
        kind = TE_NORM_LN if self.cfg.norm == "ln" else TE_NORM_RMS
        if L0.s_msa is not None:
            rownorm_mod(x, L0.t["norm1_w"], L0.t["norm1_b"], L0.s_msa, kind, self.cfg.eps, a,
                        stream=stream)
        else:
            rownorm(x, L0.t["norm1_w"], L0.t["norm1_b"], kind, self.cfg.eps, a, stream=stream)

    def forward_device(self, x, a, out=None, layers=None, stream=None):
        """In place on the device: x (f32 [T, d]) goes through every layer;
        a ends as the last block's FFN input; out (f32 [nseq, d]) receives
        the final-normed mean-pool when the stack pools."""
        if self.ple_x is not None:
            cast_bf16(x, self.ple_x, stream=stream)      # the per-layer inputs' source
        self.input_norm(x, a, stream)
        n = len(self.layers) if layers is None else layers
        for i in range(n):
            encoder_block_fwd(self.descs[i], x, a, self.cu_host, self.cu_dev, self.workspace,
                              stream=stream)
        if out is not None and self.cfg.pool:
            pool_mean(x, self.cu_host, self.cu_dev, self.final_norm, self.cfg.eps, out,
                      stream=stream)

    # the block's step classes, between its TE_BLOCK_PROF_EVENTS boundaries
    STEP_CLASSES = ("gemm_qkv", "qk_prep", "attention", "gemm_o", "norm_ffn", "gemm_gu", "gemm_down",
                    "norm_next")

    def profile_forward(self, x, a, stream=None):
        """One eager forward_device with the blocks' step-boundary events
        (te_block_desc.prof_events; the pages' per-op-class GPU timing):
        GPU ms of each step class, summed over the layers (the input norm and
        the pool fall outside the classes).  Synchronises the stream."""
        import ctypes
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        n_ev = len(self.STEP_CLASSES) + 1
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in self.descs]
        for row in evs:
            for e in row:
                e.record(s)          # creates the event
        keep = []
        try:
            for d, row in zip(self.descs, evs):
                arr = (ctypes.c_void_p * n_ev)(*[e.cuda_event for e in row])
                keep.append(arr)
                d.prof_events = ctypes.cast(arr, ctypes.c_void_p).value
            self.forward_device(x, a, stream=s)
            s.synchronize()
        finally:
            for d in self.descs:
                d.prof_events = None
        ms = dict.fromkeys(self.STEP_CLASSES, 0.0)
        for row in evs:
            for k, name in enumerate(self.STEP_CLASSES):
                ms[name] += row[k].elapsed_time(row[k + 1])
        return ms

    def forward_host_stream(self, x_hosts, result_hosts, stream=None, before=None):
        """End to end for a sequence of inputs, the copies overlapped with the
        neighbouring forwards: forward i copies x_hosts[i] (pinned) in on a
        copy stream while forward i-1 computes, and its result (the pooled
        rows, else x) out to result_hosts[i] (pinned) on another while forward
        i+1 computes.  Two device buffer sets alternate; the forwards run in
        order on `stream` (the current stream when None) and share the
        workspace.  Each set's forward is replayed from a CUDA graph captured
        by forward_host on its first use (that call runs eagerly).  `before`,
        if given, is called on the compute stream ahead of each forward (the
        bench flushes L2 there).  Returns the events (start, end) that
        bracket the whole sequence; wait on `end` before reading results."""
        import torch
        n = len(x_hosts)
        if n != len(result_hosts):
            raise ValueError("forward_host_stream: as many result buffers as inputs")
        comp = stream if stream is not None else torch.cuda.current_stream(self.device)
        if getattr(self, "_pipe", None) is None:
            # two buffer sets, two copy streams and their graphs (captured
            # through forward_host on the compute stream)
            sets = [self.buffers() for _ in range(2)]
            cin = torch.cuda.Stream(device=self.device)
            cout = torch.cuda.Stream(device=self.device)
            self._pipe = (sets, cin, cout)
        sets, cin, cout = self._pipe
        for b in range(2):
            x, a, out = sets[b]
            if (x.data_ptr(), a.data_ptr(), out.data_ptr(), comp.cuda_stream) not in self.__dict__.get("_graphs", {}):
                tmp = torch.empty_like(result_hosts[0], device="cpu").pin_memory()
                self.forward_host(x_hosts[0], tmp, x, a, out, stream=comp)
                comp.synchronize()
        graphs = self._graphs
        ev = lambda: torch.cuda.Event(enable_timing=False)
        in_done = [ev(), ev()]
        comp_done = [ev(), ev()]
        out_done = [None, None]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(comp)
        cin.wait_stream(comp)
        for i in range(n):
            b = i & 1
            x, a, out = sets[b]
            src = out if self.cfg.pool else x
            # copy in once the result of the forward two back has left x
            if out_done[b] is not None:
                cin.wait_event(out_done[b])
            with torch.cuda.stream(cin):
                x.copy_(x_hosts[i], non_blocking=True)
            in_done[b].record(cin)
            comp.wait_event(in_done[b])
            with torch.cuda.stream(comp):
                if before is not None:
                    before()
                graphs[(x.data_ptr(), a.data_ptr(), out.data_ptr(), comp.cuda_stream)].replay()
            comp_done[b].record(comp)
            cout.wait_event(comp_done[b])
            with torch.cuda.stream(cout):
                result_hosts[i].copy_(src, non_blocking=True)
            out_done[b] = ev()
            out_done[b].record(cout)
        comp.wait_stream(cout)
        end.record(comp)
        return start, end

    def forward_host(self, x_host, result_host, x=None, a=None, out=None, stream=None, graph=True):
        """End to end from pinned host memory: copies the input rows in, runs
        the stack and copies the result (the pooled rows, else x) back, all on
        `stream` (a torch.cuda.Stream; the current stream when None).

        With graph=True the device part is replayed from a CUDA graph: the
        first call with a given set of device buffers runs it eagerly (that
        call's result is a normal forward) and then captures it; later calls
        replay the capture, which removes the per-layer host work of the C-ABI
        calls (validation, tensor maps, work lists) from the critical path."""
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        if x is None:
            if getattr(self, "_bufs", None) is None:
                self._bufs = self.buffers()
            x, a, out = self._bufs
        src = out if self.cfg.pool else x
        key = (x.data_ptr(), a.data_ptr(), out.data_ptr() if out is not None else 0, s.cuda_stream)
        graphs = self.__dict__.setdefault("_graphs", {})
        with torch.cuda.stream(s):
            x.copy_(x_host, non_blocking=True)
            g = graphs.get(key) if graph else None
            if g is not None:
                g.replay()
            else:
                self.forward_device(x, a, out, stream=s)
            result_host.copy_(src, non_blocking=True)
        if graph and g is None:
            # capture after the eager forward has run (capturing does not execute)
            cap = torch.cuda.Stream(device=self.device)
            cap.wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                self.forward_device(x, a, out, stream=cap)
            s.wait_stream(cap)
            graphs[key] = g
        return result_host
