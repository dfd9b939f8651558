"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module draws random numbers and lays out buffers; it holds none of the
encoder's arithmetic.  Both the CUDA path and the CPU oracle receive the
arrays it returns, so they see identical bytes.

Workloads (sizes and value recipes follow the pages' own workloads; the pages
name no public dataset, so these seeded arrays stand in for real inputs):

* ``c1`` - one pre-norm block, d=256, 4 heads x 64, gated GELU-tanh FFN 1024,
  RMSNorm, packed lengths 37+64.
* ``c2`` - text encoder stack: 24 sandwich-norm blocks, d=512, 8 heads x 64,
  gated GELU-tanh FFN 2048, q/k RMSNorm + 1-D RoPE, a 512-token sliding
  window on odd layers, 32 sequences with lengths uniform in [16, 1024],
  final norm + mean-pool (EmbeddingGemma 2 text tower, cortiq-engine
  ``egemma2.rs``, ``TextGpu::forward``).
* ``c3`` - ViT stack: 16 plain pre-norm blocks, d=768, 12 heads x 64,
  LayerNorm with bias, biased linears, GELU-tanh MLP 3072, 4 x 1024 tokens
  (cera ``vision_encoder_gpu.rs``, ``encode_image_gpu``).
* ``c4`` - one DiT block, d=3840, 30 heads x 128, q/k RMSNorm + 2-D RoPE,
  SwiGLU FFN 10240, sandwich ("post-norm") residual, 2 x 1056 tokens
  (cortiq-engine ``zimage.rs``, ``Enc::block``).
* ``c5`` - the same block shape stacked 30 deep at 2 x 4224 tokens.

Random recipe: ``x ~ N(0,1)`` f32; int8 weights uniform on [-127, 127]; row
scale ``1/(127*sqrt(K))`` (optionally jittered by a factor in [0.75, 1.25] so
that a wrong row index is visible); RMS/LN weights ``1 + N(0, 0.1)``, LN
biases ``N(0, 0.1)``, linear biases ``N(0, 0.02)``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class BlockConfig:
    """Shape and form of one encoder stack."""

    name: str
    layers: int
    d: int
    heads: int
    kv_heads: int
    hd: int
    ffn: int
    gated: bool          # gate|up pair (z=2) vs a single up projection
    act: str             # "gelu_tanh" | "silu"
    norm: str            # "rms" | "ln"
    form: str            # "plain" (x += proj) | "sandwich" (x = x + RMS(proj)*w)
    qk_norm: bool
    rope: Optional[str]  # None | "1d" | "2d"
    window: int          # sliding window on the layers it applies to (0 = full)
    window_layers: str   # "all" | "odd"
    bias: bool
    pool: bool
    lens: tuple          # fixed lengths, or () when drawn
    n_seqs: int = 0      # number of drawn lengths when ``lens`` is empty
    len_lo: int = 0
    len_hi: int = 0
    eps: float = 1e-6
    post: float = 1.0
    adaln: bool = False  # DiT adaLN modulation: per block [s_msa | g_msa | s_mlp | g_mlp]
    codec: str = "q8_row"  # weight format: "q8_row" | "q8_2f" | "q8_0" | "q4_0"
    v_norm: bool = False   # RMS-normalise the v heads too (egemma2.rs Prog::qkv "v norm")
    ple_dim: int = 0       # per-layer input width (egemma2.rs "per-layer input"), 0 = none
    # CFG pair (zimage.rs, module doc "The chain": the CFG pair is one batch-2
    # program with rows [img0 | img1 | cap0 | cap1]; attention runs per item
    # over its two row ranges): ``lens`` lists the ranges in row order, the
    # first half image ranges, the second half the matching caption ranges
    cfg_pair: bool = False

    def window_of(self, layer: int) -> int:
        if self.window == 0:
            return 0
        if self.window_layers == "all" or layer % 2 == 1:
            return self.window
        return 0

    @property
    def qkv_width(self) -> int:
        return (self.heads + 2 * self.kv_heads) * self.hd

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.hd)


CONFIGS = {
    "c1": BlockConfig("c1_block_d256", 1, 256, 4, 4, 64, 1024, True, "gelu_tanh",
                      "rms", "plain", False, None, 0, "all", False, False, (37, 64)),
    "c2": BlockConfig("c2_text_stack24_d512", 24, 512, 8, 8, 64, 2048, True, "gelu_tanh",
                      "rms", "sandwich", True, "1d", 512, "odd", False, True, (),
                      n_seqs=32, len_lo=16, len_hi=1024),
    "c3": BlockConfig("c3_vit_stack16_d768", 16, 768, 12, 12, 64, 3072, False, "gelu_tanh",
                      "ln", "plain", False, None, 0, "all", True, False, (1024,) * 4,
                      eps=1e-5),
    "c4": BlockConfig("c4_dit_block_d3840", 1, 3840, 30, 30, 128, 10240, True, "silu",
                      "rms", "sandwich", True, "2d", 0, "all", False, False, (1056, 1056)),
    "c5": BlockConfig("c5_dit_stack30_d3840", 30, 3840, 30, 30, 128, 10240, True, "silu",
                      "rms", "sandwich", True, "2d", 0, "all", False, False, (4224, 4224)),
}
# The DiT shapes with adaLN modulation (zimage.rs Enc::block ``mods``): the
# per-block vectors are synthetic (the timestep MLP that makes them lies
# outside the block).
CONFIGS["c4m"] = dataclasses.replace(CONFIGS["c4"], name="c4m_dit_block_adaln_d3840", adaln=True)
CONFIGS["c5m"] = dataclasses.replace(CONFIGS["c5"], name="c5m_dit_stack30_adaln_d3840", adaln=True)
# The text stack with the per-layer input path (256 wide).
CONFIGS["c2p"] = dataclasses.replace(CONFIGS["c2"], name="c2p_text_stack24_ple256_d512", ple_dim=256)
# The text stack with the v heads normalised as well.
CONFIGS["c2v"] = dataclasses.replace(CONFIGS["c2"], name="c2v_text_stack24_vnorm_d512", v_norm=True)
# The DiT block with q8_2f weights (zimage.rs: q8_row + a per-column field).
CONFIGS["c4f"] = dataclasses.replace(CONFIGS["c4"], name="c4f_dit_block_q8_2f_d3840", codec="q8_2f")
# The ViT stack with the 32-element block weight formats of
# vision_encoder_gpu.rs (Q8_0, Q4_0) in place of q8_row.
CONFIGS["c3q8"] = dataclasses.replace(CONFIGS["c3"], name="c3q8_vit_stack16_q8_0_d768", codec="q8_0")
CONFIGS["c3q4"] = dataclasses.replace(CONFIGS["c3"], name="c3q4_vit_stack16_q4_0_d768", codec="q4_0")
# The DiT block as the CFG batch-2 program: two items, each a 32 x 32 patch
# image (1024 rows) with its caption (160 rows for the prompt, 32 for the
# empty prompt; caption lengths padded to multiples of 32 as zimage.rs pads
# them), rows [img0 | img1 | cap0 | cap1], joint 2-D RoPE positions.
CONFIGS["c4c"] = dataclasses.replace(CONFIGS["c4"], name="c4c_dit_block_cfg_pair_d3840",
                                     lens=(1024, 1024, 160, 32), cfg_pair=True)


def config_seed(key: str) -> int:
    return BASE_SEED + int(key[1:]) if key[:1] == "c" and key[1:].isdigit() else BASE_SEED


def draw_lens(cfg: BlockConfig, seed: int = BASE_SEED) -> np.ndarray:
    """Sequence lengths of the packed batch (int32).  The text workload's 32
    lengths drawn with the base seed sum to 16238 rows (longest 955)."""
    if cfg.lens:
        return np.asarray(cfg.lens, dtype=np.int32)
    rng = np.random.default_rng(seed)
    return rng.integers(cfg.len_lo, cfg.len_hi + 1, cfg.n_seqs).astype(np.int32)


def attn_items(cfg: BlockConfig, lens) -> Optional[np.ndarray]:
    """The two-range attention items of a CFG-pair packing, int32 [n, 4] =
    (image offset, image rows, caption offset, caption rows) per item, or
    None when every range of ``lens`` is its own sequence."""
    if not cfg.cfg_pair:
        return None
    lens = np.asarray(lens, dtype=np.int64)
    n = len(lens) // 2
    cu = cu_seqlens(lens).astype(np.int64)
    return np.asarray([[cu[i], lens[i], cu[n + i], lens[n + i]] for i in range(n)], dtype=np.int32)


def unit_lens(cfg: BlockConfig, lens) -> np.ndarray:
    """Lengths of the attention units: the items' joint lengths for a
    CFG pair, else the sequences themselves."""
    it = attn_items(cfg, lens)
    if it is None:
        return np.asarray(lens, dtype=np.int64)
    return (it[:, 1].astype(np.int64) + it[:, 3])


def joint_positions(cfg: BlockConfig, lens) -> np.ndarray:
    """Each packed row's position within its attention unit (a CFG item's
    caption rows follow its image rows)."""
    it = attn_items(cfg, lens)
    lens = np.asarray(lens, dtype=np.int64)
    if it is None:
        return np.concatenate([np.arange(n) for n in lens]).astype(np.int64)
    pos = np.empty(int(lens.sum()), dtype=np.int64)
    for off1, len1, off2, len2 in it.astype(np.int64):
        pos[off1:off1 + len1] = np.arange(len1)
        pos[off2:off2 + len2] = len1 + np.arange(len2)
    return pos


def cu_seqlens(lens) -> np.ndarray:
    """Prefix offsets [0, l0, l0+l1, ...] (int32, length nseq+1)."""
    lens = np.asarray(lens, dtype=np.int64)
    cu = np.zeros(len(lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    return cu.astype(np.int32)


def draw_x(t: int, d: int, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).standard_normal((t, d)).astype(np.float32)


def draw_q8(rng: np.random.Generator, n: int, k: int, jitter: bool, bias: bool):
    """One q8_row weight: int8 [n, k] row-major, f32 scale [n], optional f32 bias [n]."""
    q = rng.integers(-127, 128, size=(n, k), dtype=np.int8)
    s = np.full(n, 1.0 / (127.0 * math.sqrt(k)), dtype=np.float64)
    if jitter:
        s = s * rng.uniform(0.75, 1.25, n)
    b = (rng.standard_normal(n) * 0.02).astype(np.float32) if bias else None
    return {"q": q, "s": s.astype(np.float32), "b": b}


def draw_block_packed(rng: np.random.Generator, n: int, k: int, fmt: str) -> dict:
    """Packed bytes of a [n, k] weight in a 32-element block format (the
    layout of vision_encoder_gpu.rs' test quantisers): per block an f16 scale
    then the payload.  q uniform on the format's range; scales U[0.5, 1.5]
    times the value that gives the weights the spread of the q8_row draws
    (standard deviation about 0.58 / sqrt(k))."""
    nb = k // 32
    if fmt == "q8_0":
        q = rng.integers(-127, 128, (n, nb, 32)).astype(np.int8)
        d = (rng.uniform(0.5, 1.5, (n, nb)) / (127 * np.sqrt(k))).astype(np.float16)
        payload = q.view(np.uint8)
    elif fmt == "q4_0":
        q = rng.integers(-8, 8, (n, nb, 32)).astype(np.int8)
        d = (rng.uniform(0.5, 1.5, (n, nb)) / (8 * np.sqrt(k))).astype(np.float16)
        u = (q.astype(np.int16) + 8).astype(np.uint8)
        payload = (u[:, :, :16] | (u[:, :, 16:] << 4)).astype(np.uint8)
    else:
        raise ValueError(fmt)
    blocks = np.concatenate([d.view(np.uint8).reshape(n, nb, 2), payload], axis=2)
    return {"packed": blocks.reshape(-1).copy(), "n": n, "k": k, "fmt": fmt}


def draw_norm(rng: np.random.Generator, d: int, with_bias: bool):
    w = (1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    b = (0.1 * rng.standard_normal(d)).astype(np.float32) if with_bias else None
    return w, b


def draw_layer(cfg: BlockConfig, layer: int, seed: int, jitter: bool = True) -> dict:
    """All weights of one layer (host numpy arrays)."""
    rng = np.random.default_rng([seed, 7919, layer])
    d, hd, F = cfg.d, cfg.hd, cfg.ffn

    def w(n, k):
        if cfg.codec == "q8_row":
            return draw_q8(rng, n, k, jitter, cfg.bias)
        if cfg.codec == "q8_2f":
            out = draw_q8(rng, n, k, jitter, cfg.bias)
            # the column field: f16 values (as the file stores them), around 1
            out["col"] = rng.uniform(0.5, 1.5, k).astype(np.float16).astype(np.float32)
            return out
        out = draw_block_packed(rng, n, k, cfg.codec)
        out["s"] = None
        out["b"] = (rng.standard_normal(n) * 0.02).astype(np.float32) if cfg.bias else None
        return out

    p = {}
    p["wq"] = w(cfg.heads * hd, d)
    p["wk"] = w(cfg.kv_heads * hd, d)
    p["wv"] = w(cfg.kv_heads * hd, d)
    p["wo"] = w(d, cfg.heads * hd)
    p["wg"] = w(F, d)
    p["wu"] = w(F, d) if cfg.gated else None
    p["wd"] = w(d, F)
    ln = cfg.norm == "ln"
    p["norm1_w"], p["norm1_b"] = draw_norm(rng, d, ln)          # attention pre-norm
    p["norm2_w"], p["norm2_b"] = draw_norm(rng, d, ln)          # FFN pre-norm
    if cfg.form == "sandwich":
        p["post_attn_w"], _ = draw_norm(rng, d, False)
        p["post_ffn_w"], _ = draw_norm(rng, d, False)
    if cfg.qk_norm:
        p["q_norm"], _ = draw_norm(rng, hd, False)
        p["k_norm"], _ = draw_norm(rng, hd, False)
    if cfg.adaln:
        p["mod"] = draw_mods(rng, d)
    if cfg.ple_dim:
        P = cfg.ple_dim
        p["ple_in"] = draw_q8(rng, P, d, jitter, False)
        p["ple_gate"] = draw_q8(rng, P, d, jitter, False)
        p["ple_proj"] = draw_q8(rng, d, P, jitter, False)
        p["ple_post_w"], _ = draw_norm(rng, d, False)
    return p


def draw_ple(cfg: BlockConfig, seed: int) -> dict:
    """The stack-level part of the per-layer input path: the norm weight of
    pin ([P]) and its pre-scale."""
    rng = np.random.default_rng([seed, 15485863])
    return {"norm_w": (1.0 + 0.1 * rng.standard_normal(cfg.ple_dim)).astype(np.float32),
            "scale": 0.0625}


def draw_mods(rng: np.random.Generator, d: int) -> np.ndarray:
    """adaLN vectors of one block, f32 [4, d] = s_msa | g_msa | s_mlp | g_mlp:
    scales s ~ 0.1 N(0, 1), gates g = tanh(N(0, 1))."""
    s = 0.1 * rng.standard_normal((2, d))
    g = np.tanh(rng.standard_normal((2, d)))
    return np.stack([s[0], g[0], s[1], g[1]]).astype(np.float32)


def draw_final_norm(cfg: BlockConfig, seed: int) -> np.ndarray:
    rng = np.random.default_rng([seed, 104729])
    return (1.0 + 0.1 * rng.standard_normal(cfg.d)).astype(np.float32)


def rope_tables(cfg: BlockConfig, lens) -> dict:
    """RoPE inputs for the boundary: cos/sin tables [P, hd/2] (f32), a per-row
    table index ``pos`` (int32 [T]) and the section width ``sec``.

    1-D (text): angle(p, i) = p * 10000^(-2i/hd); positions restart at 0 in
    every sequence, table rows indexed by position.  2-D (DiT/vision): one
    table row per packed row; (r, c) = divmod(index in sequence, 32) (for a
    CFG item, the joint index: its caption rows follow its image rows); the
    first hd/4 entries rotate by the column c, the next hd/4 by the row r,
    each with 10000^(-2i/(hd/2)); ``sec = hd/2``.
    """
    if cfg.rope is None:
        return {"cos": None, "sin": None, "pos": None, "sec": 0}
    hd = cfg.hd
    local = joint_positions(cfg, lens)
    if cfg.rope == "1d":
        P = int(local.max()) + 1
        i = np.arange(hd // 2, dtype=np.float64)
        inv = 10000.0 ** (-2.0 * i / hd)
        ang = np.arange(P, dtype=np.float64)[:, None] * inv[None, :]
        return {"cos": np.cos(ang).astype(np.float32), "sin": np.sin(ang).astype(np.float32),
                "pos": local.astype(np.int32), "sec": hd}
    quarter = hd // 4
    i = np.arange(quarter, dtype=np.float64)
    inv = 10000.0 ** (-2.0 * i / (hd // 2))
    r, c = np.divmod(local, 32)
    ang = np.concatenate([c[:, None] * inv[None, :], r[:, None] * inv[None, :]], axis=1)
    return {"cos": np.cos(ang).astype(np.float32), "sin": np.sin(ang).astype(np.float32),
            "pos": np.arange(len(local), dtype=np.int32), "sec": hd // 2}


def small_config(key: str, **over) -> BlockConfig:
    """A shrunken copy of a workload for the oracle-sized parity tests."""
    return dataclasses.replace(CONFIGS[key], **over)
