// Varlen bidirectional multi-head attention over packed rows (flash form).
//
//     o[i, h] = sum_j softmax_j(scale * q[i, h] . k[j, g]) v[j, g],  g = h / (nq / nkv)
//
// over the keys j of i's own sequence with window == 0 or |i - j| <= window.
//
// Sources: "cortiq-engine 0.8.39 src/gpu_metal/egemma2.rs" (module doc
// "Attention", Prog::attention, att_plan: the key span of a query block is
// [q0 - W, q_last + W] clipped to the sequence, zeros outside the window and
// the padding); "cortiq-engine 0.7.6 src/gpu_metal/zimage.rs" (module doc,
// flash zi_flash_q64pf: 64 queries a group, 32-key blocks staged, running
// max and sum); "cera 0.2.4 src/model/vision_encoder_gpu.rs"
// (VitGpuOps::attention).
//
// This kernel: one CTA per (64-query tile, head, sequence); 4 warps x 16
// query rows; 64-key K/V tiles double-buffered in swizzled shared memory by
// cp.async; S = Q K^T and O += P V on mma.sync m16n8k16 (bf16 in, f32
// accumulate); online softmax in registers with exp2 and the scale folded
// with log2(e); P rounded to bf16 for the P V product and the row sum taken
// over the same rounded values.  Key tiles wholly outside the window or the
// sequence are never visited; boundary tiles are masked per element, and a
// masked key contributes exactly 0.
#include "common.cuh"

namespace tefwd {
namespace {

constexpr int BQ = 64;
constexpr int BKV = 64;

__device__ int g_attn_err;

struct AttnParams {
    const __nv_bfloat16 *qkv;
    __nv_bfloat16 *out;
    const int *cu;
    long long ld, ldo;
    int q_off, k_off, v_off, group, window;
    float scale_log2;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of (row, 16-byte chunk) in a [rows x HD] bf16 tile whose
// chunks are XOR-swizzled by the row (conflict-free ldmatrix).
template <int HD>
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
    return (uint32_t)(row * HD * 2 + ((chunk ^ (row & 7)) << 4));
}

// Loads rows [r0, r0 + 64) x columns [col, col + HD) of the panel; rows at or
// past `rend` are zero-filled.
template <int HD>
__device__ __forceinline__ void load_tile(uint32_t dst, const __nv_bfloat16 *base, long long ld,
                                          int r0, int rend, int col) {
    constexpr int CPR = HD / 8;   // 16-byte chunks per row
#pragma unroll
    for (int i = threadIdx.x; i < 64 * CPR; i += 128) {
        const int r = i / CPR, c = i % CPR;
        const bool valid = r0 + r < rend;
        const __nv_bfloat16 *src = valid ? base + (long long)(r0 + r) * ld + col + c * 8 : base;
        cp_async16(dst + tile_off<HD>(r, c), src, valid);
    }
}

template <int HD>
__global__ void __launch_bounds__(128) attn_fwd_kernel(const AttnParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int seq = blockIdx.z;
    const int r0 = p.cu[seq];
    const int len = p.cu[seq + 1] - r0;
    const int q0 = blockIdx.x * BQ;
    if (q0 >= len) return;
    const int h = blockIdx.y;
    const int g = h / p.group;
    const int W = p.window;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    constexpr int TILE = 64 * HD * 2;
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + TILE;            // 2 buffers
    const uint32_t sV = sK + 2 * TILE;        // 2 buffers

    const __nv_bfloat16 *seqbase = p.qkv + (long long)r0 * p.ld;
    int klo = 0, khi = len;
    if (W > 0) {
        klo = q0 - W > 0 ? q0 - W : 0;
        const int qlast = (q0 + BQ < len ? q0 + BQ : len) - 1;
        khi = qlast + W + 1 < len ? qlast + W + 1 : len;
    }
    const int kt0 = klo / BKV;
    const int kt1 = (khi + BKV - 1) / BKV;

    load_tile<HD>(sQ, seqbase, p.ld, q0, len, p.q_off + h * HD);
    load_tile<HD>(sK, seqbase, p.ld, kt0 * BKV, len, p.k_off + g * HD);
    load_tile<HD>(sV, seqbase, p.ld, kt0 * BKV, len, p.v_off + g * HD);
    cp_async_commit();

    float o[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    const int qa = q0 + warp * 16 + (lane >> 2);   // this thread's two query rows
    const int qb = qa + 8;
    const int qhi = (q0 + BQ < len ? q0 + BQ : len) - 1;

    for (int kt = kt0; kt < kt1; ++kt) {
        const int buf = (kt - kt0) & 1;
        if (kt + 1 < kt1) {
            load_tile<HD>(sK + (buf ^ 1) * TILE, seqbase, p.ld, (kt + 1) * BKV, len, p.k_off + g * HD);
            load_tile<HD>(sV + (buf ^ 1) * TILE, seqbase, p.ld, (kt + 1) * BKV, len, p.v_off + g * HD);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const uint32_t kbuf = sK + buf * TILE, vbuf = sV + buf * TILE;
        // ---- S = Q K^T  (16 x 64 per warp)
        float s[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
            uint32_t a0, a1, a2, a3;
            {
                const int r = warp * 16 + (lane & 15);
                ldsm_x4(sQ + tile_off<HD>(r, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
            }
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                uint32_t b0, b1, b2, b3;
                const int key = nb * 16 + (lane & 7) + ((lane >> 4) << 3);
                ldsm_x4(kbuf + tile_off<HD>(key, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
                mma16816(s[2 * nb], a0, a1, a2, a3, b0, b1);
                mma16816(s[2 * nb + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        // ---- mask, scale, online softmax
        const int kv0 = kt * BKV;
        const bool full = kv0 + BKV <= len &&
                          (W == 0 || (qhi - kv0 <= W && kv0 + BKV - 1 - q0 <= W));
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v = s[j][e] * p.scale_log2;
                if (!full) {
                    const int kj = kv0 + j * 8 + 2 * (lane & 3) + (e & 1);
                    const int qi = e < 2 ? qa : qb;
                    const int dq = qi - kj;
                    const bool vis = kj < len && (W == 0 || (dq <= W && -dq <= W));
                    if (!vis) v = -INFINITY;
                }
                s[j][e] = v;
            }
            mx_a = fmaxf(mx_a, fmaxf(s[j][0], s[j][1]));
            mx_b = fmaxf(mx_b, fmaxf(s[j][2], s[j][3]));
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xFFFFFFFFu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xFFFFFFFFu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xFFFFFFFFu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xFFFFFFFFu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float mu_a = mn_a == -INFINITY ? 0.f : mn_a;
        const float mu_b = mn_b == -INFINITY ? 0.f : mn_b;
        const float al_a = exp2f(m_a - mu_a), al_b = exp2f(m_b - mu_b);
        m_a = mn_a;
        m_b = mn_b;
        uint32_t pa[8][2];
        float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            pa[j][0] = pack_bf16x2(exp2f(s[j][0] - mu_a), exp2f(s[j][1] - mu_a));
            pa[j][1] = pack_bf16x2(exp2f(s[j][2] - mu_b), exp2f(s[j][3] - mu_b));
            rs_a += bf16_lo(pa[j][0]) + bf16_hi(pa[j][0]);
            rs_b += bf16_lo(pa[j][1]) + bf16_hi(pa[j][1]);
        }
        l_a = l_a * al_a + rs_a;
        l_b = l_b * al_b + rs_b;
#pragma unroll
        for (int i = 0; i < HD / 8; ++i) {
            o[i][0] *= al_a; o[i][1] *= al_a;
            o[i][2] *= al_b; o[i][3] *= al_b;
        }
        // ---- O += P V
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // 16 keys per step
            const uint32_t a0 = pa[2 * kk][0], a1 = pa[2 * kk][1];
            const uint32_t a2 = pa[2 * kk + 1][0], a3 = pa[2 * kk + 1][1];
#pragma unroll
            for (int nb = 0; nb < HD / 16; ++nb) {
                uint32_t b0, b1, b2, b3;
                const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                ldsm_x4_t(vbuf + tile_off<HD>(key, nb * 2 + (lane >> 4)), b0, b1, b2, b3);
                mma16816(o[2 * nb], a0, a1, a2, a3, b0, b1);
                mma16816(o[2 * nb + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    l_a += __shfl_xor_sync(0xFFFFFFFFu, l_a, 1);
    l_a += __shfl_xor_sync(0xFFFFFFFFu, l_a, 2);
    l_b += __shfl_xor_sync(0xFFFFFFFFu, l_b, 1);
    l_b += __shfl_xor_sync(0xFFFFFFFFu, l_b, 2);
    const float ia = l_a > 0.f ? 1.f / l_a : 0.f;
    const float ib = l_b > 0.f ? 1.f / l_b : 0.f;
    __nv_bfloat16 *obase = p.out + (long long)r0 * p.ldo + h * HD + 2 * (lane & 3);
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
        if (qa < len)
            *reinterpret_cast<uint32_t *>(obase + (long long)qa * p.ldo + i * 8) =
                pack_bf16x2(o[i][0] * ia, o[i][1] * ia);
        if (qb < len)
            *reinterpret_cast<uint32_t *>(obase + (long long)qb * p.ldo + i * 8) =
                pack_bf16x2(o[i][2] * ib, o[i][3] * ib);
    }
}

template <int HD>
te_status launch(const AttnParams &p, int max_len, int nq, int nseq, cudaStream_t stream) {
    const int smem = 5 * 64 * HD * 2;
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<HD>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, "attn: set shared memory size");
        attr_done = true;
    }
    const dim3 grid((max_len + BQ - 1) / BQ, nq, nseq);
    attn_fwd_kernel<HD><<<grid, 128, smem, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TE_OK : cuda_fail(e, "attn launch");
}

}  // namespace

int read_clear_attn_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_attn_err, sizeof(int)) != cudaSuccess) return -1;
    if (v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_attn_err, &zero, sizeof(int));
    }
    return v;
}

}  // namespace tefwd

using namespace tefwd;

extern "C" te_status te_attn_varlen_fwd(const void *qkv, int64_t ld, int32_t q_off, int32_t k_off,
                                        int32_t v_off, const int32_t *cu_host,
                                        const int32_t *cu_dev, int32_t nseq, int32_t nq_heads,
                                        int32_t nkv_heads, int32_t hd, int32_t window, float scale,
                                        void *out, int64_t ldo, te_stream stream) {
    if (!qkv || !out) return fail(TE_EINVAL, "attn: NULL qkv or out");
    if (hd != 64 && hd != 128) return fail(TE_ESHAPE, "attn: hd=%d (64 or 128)", hd);
    if (nq_heads < 1 || nkv_heads < 1 || nq_heads % nkv_heads)
        return fail(TE_ESHAPE, "attn: nq_heads=%d nkv_heads=%d (nq %% nkv == 0)", nq_heads, nkv_heads);
    if (nq_heads > 65535 || nseq > 65535) return fail(TE_ESHAPE, "attn: too many heads or sequences");
    if (window < 0) return fail(TE_EINVAL, "attn: window=%d (>= 0)", window);
    if (q_off < 0 || k_off < 0 || v_off < 0 || (int64_t)q_off + (int64_t)nq_heads * hd > ld ||
        (int64_t)k_off + (int64_t)nkv_heads * hd > ld || (int64_t)v_off + (int64_t)nkv_heads * hd > ld)
        return fail(TE_ESHAPE, "attn: head columns run past ld=%lld", (long long)ld);
    if (ldo < (int64_t)nq_heads * hd) return fail(TE_ESHAPE, "attn: ldo < nq_heads*hd");
    if (!aligned16(qkv) || !aligned16(out) || (ld * 2) % 16 || (ldo * 2) % 16 || q_off % 8 ||
        k_off % 8 || v_off % 8)
        return fail(TE_EALIGN, "attn: rows and head offsets must be 16-byte aligned");
    int32_t total = 0, max_len = 0;
    te_status st = check_cu(cu_host, cu_dev, nseq, &total, &max_len);
    if (st != TE_OK) return st;
    {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(qkv);
        const uintptr_t a1 = a0 + (uintptr_t)total * ld * 2;
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(out);
        const uintptr_t b1 = b0 + (uintptr_t)total * ldo * 2;
        if (a0 < b1 && b0 < a1) return fail(TE_EINVAL, "attn: out overlaps qkv");
    }
    AttnParams p;
    p.qkv = reinterpret_cast<const __nv_bfloat16 *>(qkv);
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.cu = cu_dev;
    p.ld = ld;
    p.ldo = ldo;
    p.q_off = q_off;
    p.k_off = k_off;
    p.v_off = v_off;
    p.group = nq_heads / nkv_heads;
    p.window = window;
    p.scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return hd == 64 ? launch<64>(p, max_len, nq_heads, nseq, s)
                    : launch<128>(p, max_len, nq_heads, nseq, s);
}
