// One pre-norm transformer encoder block as a fixed sequence of launches on
// one stream (no host synchronisation, no allocation).
//
// Sources: "cortiq-engine 0.8.39 src/gpu_metal/egemma2.rs" TextGpu::forward
// (per layer: q|k|v GEMM z=3 -> q/k norm + RoPE -> attention -> O GEMM ->
// add_norm -> gate|up GEMM z=2 -> GELU-tanh gate -> down GEMM -> add_norm with
// the next layer's input norm); "cortiq-engine 0.7.6 src/gpu_metal/zimage.rs"
// Enc::block (the same chain with SwiGLU and the post-norm residual row op);
// "cera 0.2.4 src/model/vision_encoder_gpu.rs" encode_image_gpu (plain
// pre-norm block: LayerNorm, biased linears, x += proj, GELU MLP).
//
// The FFN gate runs in the gate|up GEMM's epilogue (te_q8_gated_linear; the
// ungated MLP's activation in its up projection's epilogue), so the g|u
// panel is never stored.
//
// Workspace layout (each region 256-byte aligned):
//   qkv bf16 [t, (nq + 2 nkv) hd] | o bf16 [t, nq hd] | tmp f32 [t, d] | m bf16 [t, F]
//   and with the per-layer input path: pin f32 [t, P] | panel bf16 [t, 2P] |
//   z bf16 [t, P] | bf16 copy of x [t, d]
#include <vector>

#include "common.cuh"

namespace tefwd {
namespace {

inline size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

struct WsLayout {
    size_t qkv, o, tmp, m;
    size_t pin, panel, z, hb;   // per-layer input path only
    size_t total;
};

WsLayout ws_layout(const te_block_desc &d, int32_t t) {
    WsLayout L;
    const size_t T = (size_t)t;
    const size_t qkvw = (size_t)(d.n_heads + 2 * d.n_kv_heads) * d.head_dim;
    const size_t ow = (size_t)d.n_heads * d.head_dim;
    size_t off = 0;
    L.qkv = off; off = up256(off + T * qkvw * 2);
    L.o = off;   off = up256(off + T * ow * 2);
    L.tmp = off; off = up256(off + T * d.d * 4);
    L.m = off;   off = up256(off + T * (size_t)d.ffn * 2);
    L.pin = L.panel = L.z = L.hb = 0;
    if (d.ple_dim > 0) {
        const size_t np = (size_t)d.ple_dim;
        L.pin = off;   off = up256(off + T * np * 4);        // f32 x_in . W_in^T
        L.panel = off; off = up256(off + T * 2 * np * 2);    // bf16 [gate | pin]
        L.z = off;     off = up256(off + T * np * 2);        // bf16 gelu(gate) * pin
        L.hb = off;    off = up256(off + T * (size_t)d.d * 2);   // bf16 copy of x
    }
    L.total = off;
    return L;
}

te_status check_w(const te_q8w &w, int n, int k, const char *name) {
    if (!w.q || (!w.scale && !w.block_scale))
        return fail(TE_EINVAL, "block: weight %s has a NULL q or scale (NULL scale needs block scales)", name);
    if (reinterpret_cast<uintptr_t>(w.block_scale) & 3)
        return fail(TE_EALIGN, "block: weight %s: block scales must be 4-byte aligned", name);
    if (w.col && (w.block_scale || !aligned16(w.col)))
        return fail(TE_EINVAL, "block: weight %s: the column field must be 16-byte aligned, without block scales", name);
    if (w.n != n || w.k != k)
        return fail(TE_ESHAPE, "block: weight %s is [%d, %d], need [%d, %d]", name, w.n, w.k, n, k);
    if (!aligned16(w.q) || (reinterpret_cast<uintptr_t>(w.scale) & 3) ||
        (w.bias && (reinterpret_cast<uintptr_t>(w.bias) & 3)))
        return fail(TE_EALIGN, "block: weight %s: q must be 16-byte, scale/bias 4-byte aligned", name);
    return TE_OK;
}

}  // namespace

// Host validation of a block descriptor (shapes, pointers, alignment); also
// used by te_encoder_block_fwd_static before it sizes its scratch.
te_status check_block_desc(const te_block_desc *d) {
    if (!d) return fail(TE_EINVAL, "block: NULL descriptor");
    if (d->head_dim != 64 && d->head_dim != 128) return fail(TE_ESHAPE, "block: head_dim=%d", d->head_dim);
    if (d->n_heads < 1 || d->n_kv_heads < 1 || d->n_heads % d->n_kv_heads)
        return fail(TE_ESHAPE, "block: heads %d / kv heads %d", d->n_heads, d->n_kv_heads);
    if (d->d < 64 || d->d % 64 || d->d > 4096) return fail(TE_ESHAPE, "block: d=%d (multiple of 64, <= 4096)", d->d);
    if (d->ffn < 64 || d->ffn % 64) return fail(TE_ESHAPE, "block: ffn=%d (multiple of 64)", d->ffn);
    if (d->norm_kind != TE_NORM_RMS && d->norm_kind != TE_NORM_LN) return fail(TE_EINVAL, "block: norm_kind");
    if (d->resid_form != TE_RESID_PLAIN && d->resid_form != TE_RESID_SANDWICH)
        return fail(TE_EINVAL, "block: resid_form");
    if (d->act != TE_ACT_GELU_TANH && d->act != TE_ACT_SILU) return fail(TE_EINVAL, "block: act");
    if (d->window < 0) return fail(TE_EINVAL, "block: window < 0");
    if (!d->ffn_norm_w) return fail(TE_EINVAL, "block: NULL ffn_norm_w");
    if (d->resid_form == TE_RESID_SANDWICH && (!d->post_attn_w || !d->post_ffn_w))
        return fail(TE_EINVAL, "block: sandwich form needs post_attn_w and post_ffn_w");
    if ((d->q_norm == nullptr) != (d->k_norm == nullptr))
        return fail(TE_EINVAL, "block: give both q_norm and k_norm or neither");
    if (d->rope_sec && (!d->rope_cos || !d->rope_sin))
        return fail(TE_EINVAL, "block: rope_sec set without tables");
    if ((d->mod || d->next_mod_scale) && d->resid_form != TE_RESID_SANDWICH)
        return fail(TE_EINVAL, "block: adaLN modulation needs the sandwich form");
    if (d->next_mod_scale && !d->next_norm_w)
        return fail(TE_EINVAL, "block: next_mod_scale given without next_norm_w");
    if (d->ple_dim < 0 || (d->ple_dim > 0 && (d->ple_dim % 64 || d->ple_dim > 4096)))
        return fail(TE_ESHAPE, "block: ple_dim=%d (0, or a multiple of 64 up to 4096)", d->ple_dim);
    if (d->ple_dim > 0) {
        if (d->resid_form != TE_RESID_SANDWICH) return fail(TE_EINVAL, "block: the per-layer input path needs the sandwich form");
        if (!d->ple_norm_w || !d->ple_post_w || !d->ple_x)
            return fail(TE_EINVAL, "block: the per-layer input path needs ple_norm_w, ple_post_w and ple_x");
        if (!aligned16(d->ple_norm_w) || !aligned16(d->ple_post_w) || !aligned16(d->ple_x))
            return fail(TE_EALIGN, "block: per-layer input vectors must be 16-byte aligned");
    }
    const float *vecs[] = {d->ffn_norm_w, d->ffn_norm_b, d->post_attn_w, d->post_ffn_w,
                           d->next_norm_w, d->next_norm_b, d->q_norm, d->k_norm,
                           d->mod, d->next_mod_scale};
    for (const float *v : vecs)
        if (v && !aligned16(v)) return fail(TE_EALIGN, "block: norm weights must be 16-byte aligned");
    const int hd = d->head_dim, qw = d->n_heads * hd, kw = d->n_kv_heads * hd;
    te_status st;
    if ((st = check_w(d->wq, qw, d->d, "wq")) || (st = check_w(d->wk, kw, d->d, "wk")) ||
        (st = check_w(d->wv, kw, d->d, "wv")) || (st = check_w(d->wo, d->d, qw, "wo")) ||
        (st = check_w(d->wg, d->ffn, d->d, "wg")) || (st = check_w(d->wd, d->d, d->ffn, "wd")))
        return st;
    if (d->gated && (st = check_w(d->wu, d->ffn, d->d, "wu"))) return st;
    if (d->ple_dim > 0 && ((st = check_w(d->ple_in, d->ple_dim, d->d, "ple_in")) ||
                           (st = check_w(d->ple_gate, d->ple_dim, d->d, "ple_gate")) ||
                           (st = check_w(d->ple_proj, d->d, d->ple_dim, "ple_proj"))))
        return st;
    return TE_OK;
}

// With two-range attention items every row's attention output comes from
// exactly one item: the items' ranges must tile [0, t) (the rest of each
// item's checks is te_attn_items_fwd's).
te_status check_items_cover(const te_block_desc &d, int32_t t) {
    if (!d.attn_items_host || !d.attn_items_dev) return fail(TE_EINVAL, "block: NULL attention items");
    std::vector<uint8_t> seen((size_t)t, 0);
    for (int32_t i = 0; i < d.n_attn_items; ++i) {
        const int32_t *it = d.attn_items_host + 4 * i;
        for (int r = 0; r < 2; ++r) {
            const int32_t off = it[2 * r], len = it[2 * r + 1];
            if (off < 0 || len < 0 || (int64_t)off + len > t)
                return fail(TE_EINVAL, "block: attention item %d range %d (%d, %d) outside the %d rows", i, r,
                            off, len, t);
            for (int32_t j = off; j < off + len; ++j) {
                if (seen[j]) return fail(TE_EINVAL, "block: row %d is in two attention items", j);
                seen[j] = 1;
            }
        }
    }
    for (int32_t j = 0; j < t; ++j)
        if (!seen[j]) return fail(TE_EINVAL, "block: row %d is in no attention item", j);
    return TE_OK;
}

}  // namespace tefwd

using namespace tefwd;

extern "C" int32_t te_abi_sizes(size_t *sizes, int32_t n) {
    const size_t v[3] = {sizeof(te_q8w), sizeof(te_q8_item), sizeof(te_block_desc)};
    for (int32_t i = 0; i < n && i < 3 && sizes; ++i) sizes[i] = v[i];
    return 3;
}

extern "C" size_t te_encoder_block_workspace(const te_block_desc *desc, int32_t t) {
    if (!desc || t < 0) return 0;
    return ws_layout(*desc, t).total;
}

extern "C" te_status te_encoder_block_fwd(const te_block_desc *desc, float *x, void *a,
                                          const int32_t *cu_host, const int32_t *cu_dev,
                                          int32_t nseq, void *workspace, size_t ws_bytes,
                                          te_stream stream) {
    te_status st = check_block_desc(desc);
    if (st != TE_OK) return st;
    const te_block_desc &d = *desc;
    if (!x || !a || !workspace) return fail(TE_EINVAL, "block: NULL x, a or workspace");
    int32_t t = 0, max_len = 0;
    if ((st = check_cu(cu_host, cu_dev, nseq, &t, &max_len)) != TE_OK) return st;
    if (d.rope_sec && !d.rope_pos && d.rope_rows < t)
        return fail(TE_ESHAPE, "block: RoPE table has %d rows for %d packed rows", d.rope_rows, t);
    if (d.n_attn_items < 0) return fail(TE_EINVAL, "block: n_attn_items=%d", d.n_attn_items);
    if (d.n_attn_items > 0 && (st = check_items_cover(d, t)) != TE_OK) return st;
    const WsLayout L = ws_layout(d, t);
    if (ws_bytes < L.total)
        return fail(TE_EWORKSPACE, "block: workspace %zu bytes, need %zu", ws_bytes, L.total);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(TE_EALIGN, "block: workspace must be 256-byte aligned");
    if (!aligned16(x) || !aligned16(a)) return fail(TE_EALIGN, "block: x and a must be 16-byte aligned");

    // per-step timing: every event given, and the stream not being captured
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (d.prof_events) {
        for (int k = 0; k < TE_BLOCK_PROF_EVENTS; ++k)
            if (!d.prof_events[k]) return fail(TE_EINVAL, "block: prof_events[%d] is NULL", k);
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        const cudaError_t ce = cudaStreamIsCapturing(cs, &cap);
        if (ce != cudaSuccess) return cuda_fail(ce, "block: cudaStreamIsCapturing");
        if (cap != cudaStreamCaptureStatusNone)
            return fail(TE_EINVAL, "block: prof_events while the stream is being captured");
    }
    // records step boundary k when timing is on
    auto mark = [&](int k) -> te_status {
        if (!d.prof_events) return TE_OK;
        const cudaError_t e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(d.prof_events[k]), cs);
        return e == cudaSuccess ? TE_OK : cuda_fail(e, "block: cudaEventRecord");
    };

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int hd = d.head_dim, H = d.n_heads, KV = d.n_kv_heads, D = d.d, F = d.ffn;
    const int qw = H * hd, kw = KV * hd, ldqkv = qw + 2 * kw;
    __nv_bfloat16 *qkv = reinterpret_cast<__nv_bfloat16 *>(ws + L.qkv);
    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(ws + L.o);
    float *tmp = reinterpret_cast<float *>(ws + L.tmp);
    __nv_bfloat16 *m = reinterpret_cast<__nv_bfloat16 *>(ws + L.m);
    const bool plain = d.resid_form == TE_RESID_PLAIN;

    // 1. q|k|v projections, one grouped launch (z = 3)
    te_q8_item it[3] = {};
    it[0] = {d.wq, qkv, ldqkv, TE_BF16, TE_EPI_NONE, nullptr, 0};
    it[1] = {d.wk, qkv + qw, ldqkv, TE_BF16, 0, nullptr, 0};
    it[2] = {d.wv, qkv + qw + kw, ldqkv, TE_BF16, 0, nullptr, 0};
    if ((st = mark(0)) != TE_OK || (st = te_q8_linear(a, D, t, D, it, 3, stream)) != TE_OK ||
        (st = mark(1)) != TE_OK)
        return st;
    // 2. q/k norm + RoPE (and v norm) in place
    if (d.q_norm || d.rope_sec || d.q_mul != 1.f || d.v_norm) {
        if ((st = te_qkv_prep_rope(qkv, ldqkv, 0, qw, qw + kw, H, KV, hd, d.q_norm, d.k_norm,
                                   d.v_norm ? 1 : 0, d.eps, d.rope_cos, d.rope_sin, d.rope_pos,
                                   d.rope_rows, d.rope_sec, d.q_mul, t, stream)) != TE_OK)
            return st;
    }
    if ((st = mark(2)) != TE_OK) return st;
    // 3. attention: per sequence, or per two-range item
    if (d.n_attn_items > 0)
        st = te_attn_items_fwd(qkv, ldqkv, 0, qw, qw + kw, d.attn_items_host, d.attn_items_dev,
                               d.n_attn_items, t, H, KV, hd, d.window, d.attn_scale, o, qw, stream);
    else
        st = te_attn_varlen_fwd(qkv, ldqkv, 0, qw, qw + kw, cu_host, cu_dev, nseq, H, KV, hd,
                                d.window, d.attn_scale, o, qw, stream);
    if (st != TE_OK || (st = mark(3)) != TE_OK) return st;
    // 4. O projection: plain form adds into x in the epilogue
    te_q8_item io = plain ? te_q8_item{d.wo, x, D, TE_F32, 0, x, D}
                          : te_q8_item{d.wo, tmp, D, TE_F32, 0, nullptr, 0};
    if ((st = te_q8_linear(o, qw, t, qw, &io, 1, stream)) != TE_OK || (st = mark(4)) != TE_OK) return st;
    // 5. residual + FFN pre-norm
    if (plain)
        st = te_rownorm(x, TE_F32, D, d.ffn_norm_w, d.ffn_norm_b, d.norm_kind, d.eps, 1.f, a, TE_BF16,
                        D, t, D, stream);
    else   // adaLN: gate g_msa on the attention branch, scale s_mlp on the FFN input
        st = te_add_norm_mod(x, tmp, d.post_attn_w, d.mod ? d.mod + D : nullptr, d.post, d.ffn_norm_w,
                             d.ffn_norm_b, d.mod ? d.mod + 2 * D : nullptr, d.norm_kind, d.eps, a,
                             TE_BF16, t, D, stream);
    if (st != TE_OK || (st = mark(5)) != TE_OK) return st;
    // 6-7. gate|up with the gate in the epilogue, or up with the activation
    if (d.gated) {
        st = te_q8_gated_linear(a, D, t, D, &d.wg, &d.wu, d.act, m, F, stream);
    } else {
        te_q8_item iu = {d.wg, m, F, TE_BF16, d.act == TE_ACT_SILU ? TE_EPI_SILU : TE_EPI_GELU_TANH,
                         nullptr, 0};
        st = te_q8_linear(a, D, t, D, &iu, 1, stream);
    }
    if (st != TE_OK || (st = mark(6)) != TE_OK) return st;
    // 8. down projection
    te_q8_item id = plain ? te_q8_item{d.wd, x, D, TE_F32, 0, x, D}
                          : te_q8_item{d.wd, tmp, D, TE_F32, 0, nullptr, 0};
    if ((st = te_q8_linear(m, F, t, F, &id, 1, stream)) != TE_OK || (st = mark(7)) != TE_OK) return st;
    // 9. residual + the next block's pre-norm
    if (plain) {
        if (d.next_norm_w)
            st = te_rownorm(x, TE_F32, D, d.next_norm_w, d.next_norm_b, d.norm_kind, d.eps, 1.f, a,
                            TE_BF16, D, t, D, stream);
    } else if (d.ple_dim > 0) {
        // the FFN residual (post 1, no next norm), then the per-layer input path
        if ((st = te_add_norm_mod(x, tmp, d.post_ffn_w, d.mod ? d.mod + 3 * D : nullptr, 1.f, nullptr,
                                  nullptr, nullptr, d.norm_kind, d.eps, nullptr, TE_BF16, t, D, stream)) != TE_OK)
            return st;
        const int NP = d.ple_dim;
        float *pin = reinterpret_cast<float *>(ws + L.pin);
        __nv_bfloat16 *panel = reinterpret_cast<__nv_bfloat16 *>(ws + L.panel);
        __nv_bfloat16 *z = reinterpret_cast<__nv_bfloat16 *>(ws + L.z);
        __nv_bfloat16 *hb = reinterpret_cast<__nv_bfloat16 *>(ws + L.hb);
        // pin = RMS(ple_scale * x_in W_in^T) * ple_norm, into the panel's second half
        te_q8_item ip = {d.ple_in, pin, NP, TE_F32, 0, nullptr, 0};
        if ((st = te_q8_linear(d.ple_x, D, t, D, &ip, 1, stream)) != TE_OK) return st;
        if ((st = te_rownorm(pin, TE_F32, NP, d.ple_norm_w, nullptr, TE_NORM_RMS, d.eps, d.ple_scale,
                             panel + NP, TE_BF16, 2 * NP, t, NP, stream)) != TE_OK)
            return st;
        // gate = bf16(x) W_gate^T into the first half; z = gelu_tanh(gate) * pin
        if ((st = te_cast_bf16(x, D, hb, D, t, D, stream)) != TE_OK) return st;
        te_q8_item ig = {d.ple_gate, panel, 2 * NP, TE_BF16, 0, nullptr, 0};
        if ((st = te_q8_linear(hb, D, t, D, &ig, 1, stream)) != TE_OK) return st;
        if ((st = te_gate_act(panel, 2 * NP, NP, TE_ACT_GELU_TANH, z, NP, t, NP, stream)) != TE_OK) return st;
        // x = (x + RMS(z W_proj^T) w_post) * post; a = Norm_next(x)
        te_q8_item iq = {d.ple_proj, tmp, D, TE_F32, 0, nullptr, 0};
        if ((st = te_q8_linear(z, NP, t, NP, &iq, 1, stream)) != TE_OK) return st;
        st = te_add_norm_mod(x, tmp, d.ple_post_w, nullptr, d.post, d.next_norm_w, d.next_norm_b,
                             d.next_mod_scale, d.norm_kind, d.eps, d.next_norm_w ? a : nullptr, TE_BF16, t,
                             D, stream);
    } else {
        // adaLN: gate g_mlp on the FFN branch, the next block's s_msa on its input
        st = te_add_norm_mod(x, tmp, d.post_ffn_w, d.mod ? d.mod + 3 * D : nullptr, d.post, d.next_norm_w,
                             d.next_norm_b, d.next_mod_scale, d.norm_kind, d.eps,
                             d.next_norm_w ? a : nullptr, TE_BF16, t, D, stream);
    }
    return st != TE_OK ? st : mark(8);
}
