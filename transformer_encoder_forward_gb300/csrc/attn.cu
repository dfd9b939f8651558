// Varlen bidirectional multi-head attention over packed rows (flash form) on
// the 5th-generation tensor cores (sm_103a).
//
//     o[i, h] = sum_j softmax_j(scale * q[i, h] . k[j, g]) v[j, g],  g = h / (nq / nkv)
//
// over the keys j of i's own sequence with window == 0 or |i - j| <= window.
//
// Sources: "cortiq-engine 0.8.39 src/gpu_metal/egemma2.rs" (module doc
// "Attention", Prog::attention, att_plan: the key span of a query block is
// [q0 - W, q_last + W] clipped to the sequence, zeros outside the window and
// the padding); "cortiq-engine 0.7.6 src/gpu_metal/zimage.rs" (module doc,
// flash zi_flash_q64pf: a query tile resident, key blocks staged, running
// max and sum, q pre-scaled so that the softmax is 2^(s - max)); "cera 0.2.4
// src/model/vision_encoder_gpu.rs" (VitGpuOps::attention).
//
// GB300 design.  One CTA per (128-query tile, head, sequence):
//   * warp 4 (one lane) loads the Q tile once and streams 128-key K and V
//     tiles with TMA (128-byte swizzle, double-buffered);
//   * warp 5 (one lane) issues S = Q K^T (tcgen05.mma kind::f16, M=128 N=128,
//     both operands K-major in shared memory) into a TMEM S buffer, and
//     O += P V (A = P from TMEM, B = V as an MN-major shared-memory operand)
//     into the TMEM O accumulator; for hd = 128, S is double-buffered so the
//     tensor core computes S(j+1) while the softmax works on S(j);
//   * warps 0-3 own one query row per thread (TMEM lane = query): they read
//     the S row with tcgen05.ld, mask it (sequence end, window), take the row
//     max, write P = 2^(s*scale*log2e - m) as bf16 back into TMEM and sum the
//     same rounded values.  The running max is only moved (and O rescaled
//     through TMEM) when it grows by more than 2^8, which keeps P in range and
//     leaves the result unchanged: O and the row sum always share one max.
//   * at the end the same threads divide O by the sum and store their row.
// Key tiles wholly outside the window or the sequence are never loaded; a
// masked key contributes exactly 0.  Every mbarrier wait is bounded (about
// 200 ms): a timeout sets an error word that te_check() reports.
#include <cuda.h>

#include "common.cuh"

namespace tefwd {
namespace {

constexpr int BQ = 128;     // queries per CTA (= TMEM lanes)
constexpr int BKV = 128;    // keys per tile
constexpr int NTHREADS = 192;

__device__ int g_attn_err;

struct AttnParams {
    CUtensorMap map;           // the bf16 q|k|v panel [T, ld], box 64 x 128
    __nv_bfloat16 *out;
    const int *cu;
    long long ldo;
    int q_off, k_off, v_off, group, window;
    float scale_log2;
};

template <int HD, int NS>
struct ALayout {
    static constexpr int NB = HD / 64;              // 64-column boxes per tile row
    static constexpr int TILE = 128 * HD * 2;       // one 128-row tile
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = TILE;              // K[2]
    static constexpr int V_OFF = 3 * TILE;          // V[2]
    static constexpr int BAR_OFF = 5 * TILE;
    // q_full, k_full[2], v_full[2], kv_empty[2], s_full[NS], s_empty[NS], p_full, pv_done, fin
    static constexpr int NBAR = 1 + 2 + 2 + 2 + 2 * NS + 3;
    static constexpr int BYTES = BAR_OFF + 8 * NBAR + 16;
    static constexpr int S_COL = 0;                 // NS x 128 f32 columns
    static constexpr int O_COL = NS * 128;          // HD f32 columns
    static constexpr int P_COL = O_COL + HD;        // 64 columns of bf16 pairs
    static constexpr int COLS = P_COL + 64 <= 256 ? 256 : 512;
    static_assert(P_COL + 64 <= COLS, "TMEM budget");
};

// Shared-memory descriptor of an MN-major operand stored as 64-element-wide
// boxes with the 128-byte swizzle: rows (along K) 128 bytes apart, 8-row
// groups 1024 bytes apart (stride byte offset), 64-element groups along MN
// `lbo` bytes apart (leading byte offset).
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int HD, int NS>
__global__ void __launch_bounds__(NTHREADS, 1) attn_tc_kernel(const __grid_constant__ AttnParams p) {
    using L = ALayout<HD, NS>;
    extern __shared__ uint8_t smem_raw[];
    const int seq = blockIdx.z;
    const int r0 = p.cu[seq];
    const int len = p.cu[seq + 1] - r0;
    const int q0 = blockIdx.x * BQ;
    if (q0 >= len) return;
    if (*reinterpret_cast<volatile int *>(&g_attn_err) != 0) return;
    const int h = blockIdx.y;
    const int g = h / p.group;
    const int W = p.window;

    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar_q = sb + L::BAR_OFF;
    const uint32_t bar_kf = bar_q + 8;             // [2]
    const uint32_t bar_vf = bar_kf + 16;           // [2]
    const uint32_t bar_kve = bar_vf + 16;          // [2]
    const uint32_t bar_sf = bar_kve + 16;          // [NS]
    const uint32_t bar_se = bar_sf + 8 * NS;       // [NS]
    const uint32_t bar_pf = bar_se + 8 * NS;
    const uint32_t bar_pv = bar_pf + 8;
    const uint32_t bar_fin = bar_pv + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * L::NBAR);

    // key tiles this query tile needs: the window's span, clipped
    int klo = 0, khi = len;
    const int qhi = (q0 + BQ < len ? q0 + BQ : len) - 1;
    if (W > 0) {
        klo = q0 - W > 0 ? q0 - W : 0;
        khi = qhi + W + 1 < len ? qhi + W + 1 : len;
    }
    const int kt0 = klo / BKV;
    const int n = (khi + BKV - 1) / BKV - kt0;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_kf + 8 * i, 1);
            mbar_init(bar_vf + 8 * i, 1);
            mbar_init(bar_kve + 8 * i, 1);
        }
        for (int i = 0; i < NS; ++i) {
            mbar_init(bar_sf + 8 * i, 1);
            mbar_init(bar_se + 8 * i, 4);
        }
        mbar_init(bar_pf, 4);
        mbar_init(bar_pv, 1);
        mbar_init(bar_fin, 1);
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(smem_u32(tmem_slot), L::COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    bool ok = true;

    if (warp == 4) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.map);
            mbar_arrive_expect_tx(bar_q, L::TILE);
            for (int c = 0; c < L::NB; ++c)
                tma_load_2d(sb + L::Q_OFF + c * 16384, &p.map, bar_q, p.q_off + h * HD + 64 * c, r0 + q0);
            int j = 0;
            for (; j < n; ++j) {
                const int st = j & 1;
                if (!mbar_wait(bar_kve + 8 * st, ((j >> 1) & 1) ^ 1)) { ok = false; break; }
                const int row = r0 + (kt0 + j) * BKV;
                mbar_arrive_expect_tx(bar_kf + 8 * st, L::TILE);
                for (int c = 0; c < L::NB; ++c)
                    tma_load_2d(sb + L::K_OFF + st * L::TILE + c * 16384, &p.map, bar_kf + 8 * st,
                                p.k_off + g * HD + 64 * c, row);
                mbar_arrive_expect_tx(bar_vf + 8 * st, L::TILE);
                for (int c = 0; c < L::NB; ++c)
                    tma_load_2d(sb + L::V_OFF + st * L::TILE + c * 16384, &p.map, bar_vf + 8 * st,
                                p.v_off + g * HD + 64 * c, row);
            }
            // no copy of ours may still be landing when the CTA exits
            mbar_wait(bar_q, 0, 20000000ull);
            for (int i = j - 2 < 0 ? 0 : j - 2; i < j; ++i) {
                mbar_wait(bar_kf + 8 * (i & 1), (i >> 1) & 1, 20000000ull);
                mbar_wait(bar_vf + 8 * (i & 1), (i >> 1) & 1, 20000000ull);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, BKV);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, HD) | (1u << 16);   // B MN-major
            auto issue_s = [&](int j) -> bool {
                const int st = j & 1, sbuf = j % NS;
                if (!mbar_wait(bar_kf + 8 * st, (j >> 1) & 1)) return false;
                if (!mbar_wait(bar_se + 8 * sbuf, ((j / NS) & 1) ^ 1)) return false;
                tc_fence_after();
                const uint32_t kb = sb + L::K_OFF + st * L::TILE;
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_ss_bf16(tbase + L::S_COL + sbuf * 128, smem_desc_sw128(sb + L::Q_OFF + off),
                                smem_desc_sw128(kb + off), idesc_s, k > 0);
                }
                mma_commit(bar_sf + 8 * sbuf);
                return true;
            };
            ok = mbar_wait(bar_q, 0) && issue_s(0);
            for (int j = 0; j < n && ok; ++j) {
                if (j + 1 < n && !issue_s(j + 1)) { ok = false; break; }
                // O += P(j) V(j)
                if (!mbar_wait(bar_pf, j & 1) || !mbar_wait(bar_vf + 8 * (j & 1), (j >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t vb = sb + L::V_OFF + (j & 1) * L::TILE;
#pragma unroll
                for (int s = 0; s < BKV / 16; ++s)
                    mma_ts_bf16(tbase + L::O_COL, tbase + L::P_COL + 8 * s,
                                smem_desc_mn_sw128(vb + s * 2048, 16384), idesc_pv, (j | s) != 0);
                mma_commit(bar_kve + 8 * (j & 1));
                mma_commit(bar_pv);
            }
            mma_commit(bar_fin);
            mbar_wait(bar_fin, 0, 20000000ull);
        }
    } else {
        // ---------------------------------------- softmax, one query per thread
        const int row = 32 * warp + lane;
        const int qi = q0 + row;
        const uint32_t tl = (uint32_t)(32 * warp) << 16;
        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; j < n; ++j) {
            const int sbuf = j % NS;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_sf + 8 * sbuf, (j / NS) & 1));
            if (!ok) break;
            tc_fence_after();
            float x[BKV];
#pragma unroll
            for (int c = 0; c < BKV / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tbase + tl + L::S_COL + sbuf * 128 + 32 * c, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) x[32 * c + e] = __uint_as_float(v[e]) * p.scale_log2;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_se + 8 * sbuf);
            // mask: keys past the sequence end or outside the window
            const int kv0 = (kt0 + j) * BKV;
            const bool full = kv0 + BKV <= len &&
                              (W == 0 || (qhi - kv0 <= W && kv0 + BKV - 1 - q0 <= W));
            if (!full) {
#pragma unroll
                for (int e = 0; e < BKV; ++e) {
                    const int dq = qi - (kv0 + e);
                    if (kv0 + e >= len || (W > 0 && (dq > W || -dq > W))) x[e] = -INFINITY;
                }
            }
            float mx = x[0];
#pragma unroll
            for (int e = 1; e < BKV; ++e) mx = fmaxf(mx, x[e]);
            const bool resc = mx > m_used + 8.f;
            bool pv_waited = false;
            if (__any_sync(0xFFFFFFFFu, resc)) {
                const float alpha = resc ? fast_exp2(m_used - mx) : 1.f;
                if (resc) m_used = mx;
                l *= alpha;
                if (j > 0) {
                    // O holds the products of the earlier tiles: wait for the
                    // last one, then rescale it in place
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_pv, (j - 1) & 1));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tbase + tl + L::O_COL + 32 * c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(tbase + tl + L::O_COL + 32 * c, v);
                    }
                    tmem_wait_st();
                    pv_waited = true;
                }
            }
            const float mu = m_used == -INFINITY ? 0.f : m_used;
            uint32_t pk[BKV / 2];
            float rs = 0.f;
#pragma unroll
            for (int e = 0; e < BKV / 2; ++e) {
                pk[e] = pack_bf16x2(fast_exp2(x[2 * e] - mu), fast_exp2(x[2 * e + 1] - mu));
                rs += bf16_lo(pk[e]) + bf16_hi(pk[e]);
            }
            l += rs;
            if (j > 0 && !pv_waited) {
                // the P buffer is free once the previous P V product is done
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_pv, (j - 1) & 1));
                if (!ok) break;
                tc_fence_after();
            }
            tmem_st32(tbase + tl + L::P_COL, *reinterpret_cast<const uint32_t(*)[32]>(pk));
            tmem_st32(tbase + tl + L::P_COL + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pf);
        }
        // ---- epilogue: O / l, one row per thread
        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_pv, (n - 1) & 1));
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *orow = p.out + (long long)(r0 + qi) * p.ldo + h * HD;
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tbase + tl + L::O_COL + 32 * c, v);
                tmem_wait_ld();
                if (qi < len) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 u;
                        u.x = pack_bf16x2(__uint_as_float(v[8 * e + 0]) * inv, __uint_as_float(v[8 * e + 1]) * inv);
                        u.y = pack_bf16x2(__uint_as_float(v[8 * e + 2]) * inv, __uint_as_float(v[8 * e + 3]) * inv);
                        u.z = pack_bf16x2(__uint_as_float(v[8 * e + 4]) * inv, __uint_as_float(v[8 * e + 5]) * inv);
                        u.w = pack_bf16x2(__uint_as_float(v[8 * e + 6]) * inv, __uint_as_float(v[8 * e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + 32 * c + 8 * e) = u;
                    }
                }
            }
        }
    }
    if (!ok) atomicExch(&g_attn_err, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tbase, L::COLS);
    }
}

template <int HD, int NS>
te_status launch(const AttnParams &p, int max_len, int nq, int nseq, cudaStream_t stream) {
    using L = ALayout<HD, NS>;
    const int smem = L::BYTES + 1024;
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, NS>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, "attn: set shared memory size");
        attr_done = true;
    }
    const dim3 grid((max_len + BQ - 1) / BQ, nq, nseq);
    attn_tc_kernel<HD, NS><<<grid, NTHREADS, smem, stream>>>(p);
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
    memset(&p, 0, sizeof(p));
    st = make_map_2d(&p.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qkv, (uint64_t)ld, (uint64_t)total,
                     (uint64_t)ld * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != TE_OK) return st;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.cu = cu_dev;
    p.ldo = ldo;
    p.q_off = q_off;
    p.k_off = k_off;
    p.v_off = v_off;
    p.group = nq_heads / nkv_heads;
    p.window = window;
    p.scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return hd == 64 ? launch<64, 1>(p, max_len, nq_heads, nseq, s)
                    : launch<128, 2>(p, max_len, nq_heads, nseq, s);
}
