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
// GB300 design.  At hd = 128 one CTA per (256 queries, head, sequence), as
// two 128-query tiles A and B that share one stream of 128-key K/V tiles; at
// hd = 64 one 128-query tile a CTA and two CTAs an SM (TL below):
//   * the last warp (one lane) loads the Q tiles once and streams K and V
//     tiles with TMA (128-byte swizzle, double-buffered);
//   * the warp before it (one lane) issues the MMAs: S_w = Q_w K^T (tcgen05.mma kind::f16,
//     M=128 N=128, both operands K-major in shared memory) into tile w's TMEM
//     S buffer, and O_w += P_w V (A = P_w from TMEM, B = V as an MN-major
//     shared-memory operand) into its TMEM O accumulator, in the order
//     PV_A(j), S_A(j+1), PV_B(j), S_B(j+1);
//   * warps 0-3 (tile A) and 4-7 (tile B) own one query row per thread (TMEM
//     lane = query): they read the S row with tcgen05.ld, mask it (sequence
//     end, window), take the row max, and write P = 2^(s*scale*log2e - m) as
//     bf16 into the first half of their own S buffer (S_w(j+1) is only issued
//     once PV_w(j) has consumed it).  The running max is only moved (and O
//     rescaled through TMEM) when it grows by more than 2^8, which keeps P in
//     range and leaves the result unchanged: O and the row sum always share
//     one max.  The two tiles' softmax passes run concurrently, each
//     overlapping the other tile's MMAs (taking turns at the exp pass paid
//     while the pass issued more instructions; with paired arithmetic it
//     costs more than it gives);
//   * at the end the same threads divide O by the sum and store their row.
// Key tiles wholly outside both tiles' windows or the sequence are never
// loaded; a masked key contributes exactly 0.  Every mbarrier wait is bounded
// (about 200 ms): a timeout sets an error word that te_check() reports.
#include <cuda.h>

#include <algorithm>
#include <vector>

#include "common.cuh"

namespace tefwd {
namespace {

constexpr int BQ = 128;     // queries per tile (= TMEM lanes); TL tiles per CTA
constexpr int BKV = 128;    // keys per tile
constexpr int MAX_WORK = 640;   // work list entries carried in the launch parameters
// the K and V bytes of all heads that the CTA order treats as one group, and
// the bytes of one group when they do not fit (see the kernel's CTA order)
constexpr long long KV_ALL_BYTES = 48ll << 20;
constexpr long long KV_GROUP_BYTES = 24ll << 20;

__device__ int g_attn_err;

struct AttnParams {
    CUtensorMap map;           // the bf16 q|k|v panel [T, ld], box 64 x 128
    CUtensorMap map32;         // the same panel, box 64 x 32 (tiles across two row ranges)
    __nv_bfloat16 *out;
    const int *cu;
    const int *items;          // two-range items [n][off1, len1, off2, len2], or NULL (cu)
    int nwork;                 // > 0: work[i] = (unit << 16) | query block, longest first
    int nq, hgroup;            // with a work list: heads, and heads per group of the CTA order
    uint32_t work[MAX_WORK];
    long long ldo;
    int q_off, k_off, v_off, group, window;
    float scale_log2;
};

// TL = query tiles per CTA: 2 (tiles A and B, one CTA per SM), or 1 (hd = 64: half the TMEM and 80 KB of shared memory,
// so that two CTAs share an SM and one's loads and latencies overlap the
// other's work - the short sequences of a text batch).  With one tile, P has
// TMEM columns of its own (S 128 | P 64 | O 64 = 256), so S(j+1) is issued as
// soon as the softmax has read S(j) into registers and runs on the tensor
// core during the softmax of block j.
template <int HD, int TL>
struct ALayout {
    static constexpr int NB = HD / 64;              // 64-column boxes per tile row
    static constexpr int TILE = 128 * HD * 2;       // one 128-row tile
    static constexpr int Q_OFF = 0;                 // Q[TL] (tiles A, B)
    static constexpr int K_OFF = TL * TILE;         // K[2]
    static constexpr int V_OFF = K_OFF + 2 * TILE;  // V[2]
    static constexpr int BAR_OFF = V_OFF + 2 * TILE;
    static constexpr int NTHREADS = 32 * (4 * TL + 2);   // softmax warps, MMA warp, TMA warp
    static constexpr int MMA_WARP = 4 * TL, TMA_WARP = 4 * TL + 1;
    // q_full, k_full[2], v_full[2], kv_empty[2] (TL = 1: V only), s_full[2], p_full[2],
    // pv_done[2], fin, k_empty[2] (TL = 1), s_free (TL = 1)
    static constexpr int NBAR = 1 + 2 + 2 + 2 + 2 + 2 + 2 + 1 + 2 + 1;
    static constexpr int BYTES = BAR_OFF + 8 * NBAR + 16;
    static constexpr int S_COL = 0;                 // S_A, S_B: TL x 128 f32 columns
    static constexpr int P_COL = TL == 1 ? 128 : 0; // TL = 1: 64 columns of its own; TL = 2: over S
    static constexpr int O_COL = TL == 1 ? 192 : TL * 128;   // O_A, O_B: TL x HD f32 columns
    static constexpr int COLS = TL == 1 ? 256 : 512;
    static_assert(TL == 2 || HD == 64, "one tile a CTA is the hd = 64 form");
    static_assert(O_COL + TL * HD <= COLS, "TMEM budget");
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

// The keys row qi sees in the block that starts at key kv0, as offsets
// [lo, hi] from kv0: key k is visible iff k < len and (W == 0 or |qi - k| <=
// W); empty when hi < lo.  Two compares per key in the masked passes.
struct KeySpan {
    int lo, hi;
    __device__ __forceinline__ bool has(int e) const { return e >= lo && e <= hi; }
};
__device__ __forceinline__ KeySpan key_span(int qi, int kv0, int len, int W) {
    // clamped before any sum, so that no window size overflows
    const int first = W > 0 && qi > W ? qi - W : 0;
    const int last = W > 0 && W < len && qi < len - 1 - W ? qi + W : len - 1;
    return {first - kv0, last - kv0};
}

// The two passes over one 128-key S row, loaded from TMEM once into registers
// (v0 = keys 0-63, v1 = keys 64-127).  Row max: keys outside the sequence or
// the window ignored when MASK, eight independent partial maxima.
template <bool MASK>
__device__ __forceinline__ float row_max_regs(const uint32_t (&v0)[64], const uint32_t (&v1)[64], int qi,
                                              int kv0, int len, int W) {
    const KeySpan sp = key_span(qi, kv0, len, W);
    float m8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
#pragma unroll
    for (int e = 0; e < 64; ++e) {
        const float x0 = __uint_as_float(v0[e]), x1 = __uint_as_float(v1[e]);
        if (!MASK) {
            m8[e & 7] = fmax3(m8[e & 7], x0, x1);
        } else {
            if (sp.has(e)) m8[e & 7] = fmaxf(m8[e & 7], x0);
            if (sp.has(64 + e)) m8[e & 7] = fmaxf(m8[e & 7], x1);
        }
    }
    return fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
}

// Exp pass: P = 2^(s*c + nm) as bf16 pairs, written over S columns the row
// has already consumed (half h of P lands in columns [32h, 32h+32)); returns
// the row sum of P over the f32 values.
template <bool MASK>
__device__ __forceinline__ float row_exp_regs(uint32_t scol, const uint32_t (&v0)[64], const uint32_t (&v1)[64],
                                              float c, float nm, int qi, int kv0, int len, int W) {
    const KeySpan sp = key_span(qi, kv0, len, W);
    // the scale, offset and the eight partial sums as f32 pairs: one paired
    // FMA and one paired add for two keys (partial sum i keeps the keys
    // with index = i mod 8, as pairs (2i', 2i' + 1))
    const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(nm, nm);
    uint64_t r4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) r4[i] = f2_pack(0.f, 0.f);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const uint32_t (&v)[64] = hh ? v1 : v0;
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), c2, nm2), a0, a1);
            float p0 = fast_exp2(a0);
            float p1 = fast_exp2(a1);
            if (MASK) {
                const int k = 64 * hh + 2 * e;
                if (!sp.has(k)) p0 = 0.f;
                if (!sp.has(k + 1)) p1 = 0.f;
            }
            r4[e & 3] = f2_add(r4[e & 3], f2_pack(p0, p1));
            pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st32(scol + 32 * hh, pk);
    }
    float r8[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) f2_unpack(r4[i], r8[2 * i], r8[2 * i + 1]);
    return ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
}

template <int HD, int TL>
__global__ void __launch_bounds__(ALayout<HD, TL>::NTHREADS, TL == 1 ? 2 : 1)
    attn_tc_kernel(const __grid_constant__ AttnParams p) {
    using L = ALayout<HD, TL>;
    extern __shared__ uint8_t smem_raw[];
    // CTA (head, work): the work list orders (unit, 256-query block) by cost,
    // longest first, so that the long blocks start early and the launch ends
    // without a tail of one long block.  The 1-D grid takes the heads in
    // groups of hgroup: within a group, work items in list order, the group's
    // heads fastest, so that the CTAs running together read the K and V of a
    // few heads (in L2) rather than of all.  Without a work list, (query
    // block, head, unit) is the grid.
    int seq, qblk, h;
    if (p.nwork) {
        const int b = blockIdx.x;
        const int per = p.hgroup * p.nwork;
        const int g = b / per;
        const int r = b - g * per;
        const int h0 = g * p.hgroup;
        const int gn = p.nq - h0 < p.hgroup ? p.nq - h0 : p.hgroup;
        const int wi = r / gn;
        const uint32_t wv = p.work[wi];
        seq = (int)(wv >> 16);
        qblk = (int)(wv & 0xFFFFu);
        h = h0 + (r - wi * gn);
    } else {
        seq = blockIdx.z;
        qblk = blockIdx.x;
        h = blockIdx.y;
    }
    // the attention unit: one packed sequence (cu), or a two-range item whose
    // joint positions 0..len1-1 are rows off1.. and len1.. are rows off2..
    int off1, len1, off2 = 0, len2 = 0;
    if (p.items) {
        const int4 it = reinterpret_cast<const int4 *>(p.items)[seq];
        off1 = it.x; len1 = it.y; off2 = it.z; len2 = it.w;
    } else {
        off1 = p.cu[seq];
        len1 = p.cu[seq + 1] - off1;
    }
    const int len = len1 + len2;
    auto row_of = [&](int j) { return j < len1 ? off1 + j : off2 + (j - len1); };
    const int q0 = qblk * TL * BQ;
    if (q0 >= len) return;
    if (*reinterpret_cast<volatile int *>(&g_attn_err) != 0) return;
    const int g = h / p.group;
    const int W = p.window;
    const int ntile = TL == 2 && q0 + BQ < len ? 2 : 1;   // tile B exists

    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar_q = sb + L::BAR_OFF;
    const uint32_t bar_kf = bar_q + 8;             // [2]
    const uint32_t bar_vf = bar_kf + 16;           // [2]
    const uint32_t bar_kve = bar_vf + 16;          // [2]
    const uint32_t bar_sf = bar_kve + 16;          // [2] per query tile
    const uint32_t bar_pf = bar_sf + 16;           // [2] per query tile
    const uint32_t bar_pv = bar_pf + 16;           // [2] per query tile
    const uint32_t bar_fin = bar_pv + 16;
    const uint32_t bar_ke = bar_fin + 8;           // [2] TL = 1: K(j) read by S(j)
    const uint32_t bar_sfree = bar_ke + 16;        // TL = 1: the softmax has read S(j)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * L::NBAR);

    // key tiles the two query tiles need: the union of their windows, clipped
    int klo = 0, khi = len;
    const int qhi = (q0 + TL * BQ < len ? q0 + TL * BQ : len) - 1;
    if (W > 0) {
        klo = q0 - W > 0 ? q0 - W : 0;
        khi = qhi + W + 1 < len ? qhi + W + 1 : len;
    }
    const int kt0 = klo / BKV;
    const int n = (khi + BKV - 1) / BKV - kt0;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 128 joint positions from j0 at column col: one box, or four 32-row
    // boxes when the tile spans the two ranges (len1 % 32 == 0); issued by
    // the lane whose e is set
    auto load_tile = [&](uint32_t dst, int col, int j0, uint32_t bar, uint32_t e) {
        if (len2 == 0 || j0 + BQ <= len1 || j0 >= len1) {
            tma_load_2d_e(dst, &p.map, bar, col, row_of(j0), e);
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r)
                tma_load_2d_e(dst + r * 32 * 128, &p.map32, bar, col, row_of(j0 + 32 * r), e);
        }
    };
    // The TMA warp initialises the barriers and starts the Q load at once:
    // its latency then overlaps the TMEM allocation and the block's sync.
    if (warp == L::TMA_WARP && lane == 0) {
        mbar_init(bar_q, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_kf + 8 * i, 1);
            mbar_init(bar_vf + 8 * i, 1);
            mbar_init(bar_kve + 8 * i, 1);
            mbar_init(bar_sf + 8 * i, 1);
            mbar_init(bar_pf + 8 * i, 4);
            mbar_init(bar_pv + 8 * i, 1);
            mbar_init(bar_ke + 8 * i, 1);
        }
        mbar_init(bar_sfree, 4);
        mbar_init(bar_fin, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_q, ntile * L::TILE);
        for (int w = 0; w < ntile; ++w)
            for (int c = 0; c < L::NB; ++c)
                load_tile(sb + L::Q_OFF + w * L::TILE + c * 16384, p.q_off + h * HD + 64 * c, q0 + w * BQ, bar_q, 1u);
    }
    if (warp == L::MMA_WARP) tmem_alloc(smem_u32(tmem_slot), L::COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    bool ok = true;

    if (warp == L::TMA_WARP) {
        // ------------------------------------------------------ TMA producer
        // (the whole warp in step, one elected lane issues)
        const uint32_t e = elect_one();
        if (e) tma_prefetch_desc(&p.map);
        // K(i) into ring slot i & 1 once its previous occupant K(i - 2) is
        // free (TL = 1: read by S(i - 2); TL = 2: K and V free together after
        // PV(i - 2)); V(i) once PV(i - 2) is done
        auto load_k = [&](int i) -> bool {
            const int st = i & 1;
            const uint32_t fb = TL == 1 ? bar_ke : bar_kve;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(fb + 8 * st, ((i >> 1) & 1) ^ 1))) return false;
            mbar_arrive_expect_tx_e(bar_kf + 8 * st, L::TILE, e);
            for (int c = 0; c < L::NB; ++c)
                load_tile(sb + L::K_OFF + st * L::TILE + c * 16384, p.k_off + g * HD + 64 * c, (kt0 + i) * BKV,
                          bar_kf + 8 * st, e);
            return true;
        };
        auto load_v = [&](int i) -> bool {
            const int st = i & 1;
            if (TL == 1 && !__all_sync(0xFFFFFFFFu, mbar_wait(bar_kve + 8 * st, ((i >> 1) & 1) ^ 1))) return false;
            mbar_arrive_expect_tx_e(bar_vf + 8 * st, L::TILE, e);
            for (int c = 0; c < L::NB; ++c)
                load_tile(sb + L::V_OFF + st * L::TILE + c * 16384, p.v_off + g * HD + 64 * c, (kt0 + i) * BKV,
                          bar_vf + 8 * st, e);
            return true;
        };
        int nk = 0, nv = 0;   // K and V tiles issued
        if (TL == 1) {
            // K runs one tile ahead of V: S(j + 1) needs it while PV(j) waits for P(j)
            if (n > 0 && (ok = load_k(0))) nk = 1;
            for (; nv < n && ok; ++nv) {
                if (nk < n) {
                    if (!(ok = load_k(nk))) break;
                    ++nk;
                }
                if (!(ok = load_v(nv))) break;
            }
        } else {
            for (; nv < n && ok; ++nv) {
                if (!(ok = load_k(nv))) break;
                ++nk;
                ok = load_v(nv);
            }
        }
        // no copy of ours may still be landing when the CTA exits
        mbar_wait(bar_q, 0, 20000000ull);
        for (int i = nk - 2 < 0 ? 0 : nk - 2; i < nk; ++i) mbar_wait(bar_kf + 8 * (i & 1), (i >> 1) & 1, 20000000ull);
        for (int i = nv - 2 < 0 ? 0 : nv - 2; i < nv; ++i) mbar_wait(bar_vf + 8 * (i & 1), (i >> 1) & 1, 20000000ull);
    } else if (warp == L::MMA_WARP) {
        // ------------------------------------------------------- MMA issuer
        // The whole warp runs the issue loop in step (waits, descriptors) and
        // one elected lane issues: the loop's values stay warp-uniform.
        const uint32_t e = elect_one();
        constexpr uint32_t idesc_s = idesc_bf16_f32(128, BKV);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, HD) | (1u << 16);   // B MN-major
        // descriptors computed once; an operand is its base plus a constant
        // (the start-address field cannot carry: shared memory < 256 KB)
        const uint64_t kd0 = smem_desc_sw128(sb + L::K_OFF), kd1 = smem_desc_sw128(sb + L::K_OFF + L::TILE);
        const uint64_t vd0 = smem_desc_mn_sw128(sb + L::V_OFF, 16384);
        const uint64_t vd1 = smem_desc_mn_sw128(sb + L::V_OFF + L::TILE, 16384);
        auto issue_s = [&](int w, int j) -> bool {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_kf + 8 * (j & 1), (j >> 1) & 1))) return false;
            tc_fence_after();
            const uint64_t k0 = (j & 1) ? kd1 : kd0;
            const uint64_t q0d = smem_desc_sw128(sb + L::Q_OFF + w * L::TILE);
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                mma_ss_bf16_e(tbase + L::S_COL + w * 128, q0d + off, k0 + off, idesc_s, k > 0, e);
            }
            mma_commit_e(bar_sf + 8 * w, e);
            if (TL == 1) mma_commit_e(bar_ke + 8 * (j & 1), e);   // K(j) read
            return true;
        };
        auto issue_pv = [&](int w, int j) {
            const uint64_t v0 = (j & 1) ? vd1 : vd0;
#pragma unroll
            for (int s2 = 0; s2 < BKV / 16; ++s2)
                mma_ts_bf16_e(tbase + L::O_COL + w * HD, tbase + L::P_COL + w * 128 + 8 * s2,
                              v0 + (uint64_t)(128 * s2), idesc_pv, (j | s2) != 0, e);
            mma_commit_e(bar_pv + 8 * w, e);
        };
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_q, 0));
        for (int w = 0; w < ntile && ok; ++w) ok = issue_s(w, 0);
        if (TL == 1) {
            // S(j+1) as soon as the softmax has read S(j) (P has columns of
            // its own), then PV(j) once P(j) is written
            for (int j = 0; j < n && ok; ++j) {
                if (j + 1 < n) {
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_sfree, j & 1))) { ok = false; break; }
                    tc_fence_after();
                    if (!(ok = issue_s(0, j + 1))) break;
                }
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_vf + 8 * (j & 1), (j >> 1) & 1)) ||
                    !__all_sync(0xFFFFFFFFu, mbar_wait(bar_pf, j & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_pv(0, j);
                mma_commit_e(bar_kve + 8 * (j & 1), e);   // V(j) read
            }
        }
        // TL = 2: issue order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): S_A(j) lands
        // first, so tile A's pass usually releases P first.  S_w(j+1)
        // overwrites the P_w(j) that PV_w(j) reads (a different
        // accumulator, so not ordered by the tensor pipe): it waits for
        // PV_w(j) to complete.
        for (int j = 0; j < n && ok && TL == 2; ++j) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_vf + 8 * (j & 1), (j >> 1) & 1))) { ok = false; break; }
            for (int w = 0; w < ntile && ok; ++w) {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_pf + 8 * w, j & 1))) { ok = false; break; }
                tc_fence_after();
                issue_pv(w, j);
                // K(j), V(j) are free once both tiles' PV(j) are done
                if (w == ntile - 1) mma_commit_e(bar_kve + 8 * (j & 1), e);
                if (j + 1 < n) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_pv + 8 * w, j & 1)) && issue_s(w, j + 1);
            }
        }
        mma_commit_e(bar_fin, e);
        __all_sync(0xFFFFFFFFu, mbar_wait(bar_fin, 0, 20000000ull));
    } else if (warp < 4 * ntile) {
        // ---------------------------------------- softmax, one query per thread
        const int w = warp >> 2;                         // query tile of this warpgroup
        const int wq = warp & 3;                         // TMEM lane quadrant
        const int row = 32 * wq + lane;
        const int tq0 = q0 + w * BQ;                     // first query of the tile
        const int qi = tq0 + row;
        const int tqhi = (tq0 + BQ < len ? tq0 + BQ : len) - 1;
        const uint32_t tl = (uint32_t)(32 * wq) << 16;
        const uint32_t scol = tbase + tl + L::S_COL + w * 128;
        const uint32_t pcol = tbase + tl + L::P_COL + w * 128;
        const uint32_t ocol = tbase + tl + L::O_COL + w * HD;
        const float c = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; j < n; ++j) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_sf + 8 * w, j & 1));
            if (!ok) break;
            // TL = 2: S_w(j) landed, so PV_w(j-1) is done: P_w and O_w may be
            // touched.  TL = 1: see below.
            tc_fence_after();
            // mask: keys past the sequence end or outside the window
            const int kv0 = (kt0 + j) * BKV;
            const bool full = kv0 + BKV <= len &&
                              (W == 0 || (tqhi - kv0 <= W && kv0 + BKV - 1 - tq0 <= W));
            // pass 1: the row max of the raw scores
            // the S row once into registers for both passes
            uint32_t v0[64], v1[64];
            tmem_ld64(scol, v0);
            tmem_ld64(scol + 64, v1);
            tmem_wait_ld();
            if (TL == 1) {
                // S(j) is in registers: the tensor core may compute S(j+1)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sfree);
            }
            float mx = full ? row_max_regs<false>(v0, v1, qi, kv0, len, W)
                            : row_max_regs<true>(v0, v1, qi, kv0, len, W);
            mx *= c;                                     // c > 0: the max of the scaled row
            if (TL == 1 && j > 0) {
                // P and O are free once PV(j-1) is done
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_pv, (j - 1) & 1));
                if (!ok) break;
                tc_fence_after();
            }
            const bool resc = mx > m_used + 8.f;
            if (__any_sync(0xFFFFFFFFu, resc)) {
                const float alpha = resc ? fast_exp2(m_used - mx) : 1.f;
                if (resc) m_used = mx;
                l *= alpha;
                if (j > 0) {
#pragma unroll
                    for (int cc = 0; cc < HD / 32; ++cc) {
                        uint32_t v[32];
                        tmem_ld32(ocol + 32 * cc, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(ocol + 32 * cc, v);
                    }
                    tmem_wait_st();
                }
            }
            // pass 2: P as bf16 (TL = 2: into the consumed S columns), and its row sum
            const float nm = m_used == -INFINITY ? 0.f : -m_used;
            const float rs = full ? row_exp_regs<false>(pcol, v0, v1, c, nm, qi, kv0, len, W)
                                  : row_exp_regs<true>(pcol, v0, v1, c, nm, qi, kv0, len, W);
            l += rs;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pf + 8 * w);
        }
        // ---- epilogue: O / l, one row per thread
        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_pv + 8 * w, (n - 1) & 1));
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *orow = p.out + (long long)(qi < len ? row_of(qi) : 0) * p.ldo + h * HD;
#pragma unroll
            for (int cc = 0; cc < HD / 32; ++cc) {
                uint32_t v[32];
                tmem_ld32(ocol + 32 * cc, v);
                tmem_wait_ld();
                if (qi < len) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 u;
                        u.x = pack_bf16x2(__uint_as_float(v[8 * e + 0]) * inv, __uint_as_float(v[8 * e + 1]) * inv);
                        u.y = pack_bf16x2(__uint_as_float(v[8 * e + 2]) * inv, __uint_as_float(v[8 * e + 3]) * inv);
                        u.z = pack_bf16x2(__uint_as_float(v[8 * e + 4]) * inv, __uint_as_float(v[8 * e + 5]) * inv);
                        u.w = pack_bf16x2(__uint_as_float(v[8 * e + 6]) * inv, __uint_as_float(v[8 * e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + 32 * cc + 8 * e) = u;
                    }
                }
            }
        }
    }
    if (!ok) atomicExch(&g_attn_err, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == L::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tbase, L::COLS);
    }
}

template <int HD, int TL>
te_status launch(const AttnParams &p, int max_len, int nq, int nseq, cudaStream_t stream) {
    using L = ALayout<HD, TL>;
    const int smem = L::BYTES + 1024;
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, TL>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, "attn: set shared memory size");
        attr_done = true;
    }
    const dim3 grid = p.nwork ? dim3(nq * p.nwork, 1, 1) : dim3((max_len + TL * BQ - 1) / (TL * BQ), nq, nseq);
    attn_tc_kernel<HD, TL><<<grid, L::NTHREADS, smem, stream>>>(p);
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

static te_status attn_common_checks(const void *qkv, int64_t ld, int32_t q_off, int32_t k_off, int32_t v_off,
                                    int32_t nq_heads, int32_t nkv_heads, int32_t hd, int32_t window,
                                    const void *out, int64_t ldo) {
    if (!qkv || !out) return fail(TE_EINVAL, "attn: NULL qkv or out");
    if (hd != 64 && hd != 128) return fail(TE_ESHAPE, "attn: hd=%d (64 or 128)", hd);
    if (nq_heads < 1 || nkv_heads < 1 || nq_heads % nkv_heads)
        return fail(TE_ESHAPE, "attn: nq_heads=%d nkv_heads=%d (nq %% nkv == 0)", nq_heads, nkv_heads);
    if (nq_heads > 65535) return fail(TE_ESHAPE, "attn: too many heads");
    if (window < 0) return fail(TE_EINVAL, "attn: window=%d (>= 0)", window);
    if (q_off < 0 || k_off < 0 || v_off < 0 || (int64_t)q_off + (int64_t)nq_heads * hd > ld ||
        (int64_t)k_off + (int64_t)nkv_heads * hd > ld || (int64_t)v_off + (int64_t)nkv_heads * hd > ld)
        return fail(TE_ESHAPE, "attn: head columns run past ld=%lld", (long long)ld);
    if (ldo < (int64_t)nq_heads * hd) return fail(TE_ESHAPE, "attn: ldo < nq_heads*hd");
    if (!aligned16(qkv) || !aligned16(out) || (ld * 2) % 16 || (ldo * 2) % 16 || q_off % 8 ||
        k_off % 8 || v_off % 8)
        return fail(TE_EALIGN, "attn: rows and head offsets must be 16-byte aligned");
    return TE_OK;
}

// The (unit, qb-query block) pairs with queries, longest first: cost =
// queries of the block x keys it can see.  Empty when there are more than
// MAX_WORK pairs (the plain grid is used then).
static int build_work(const int32_t *lens, int32_t units, int32_t window, int qb, uint32_t *work) {
    int n = 0;
    for (int32_t u = 0; u < units; ++u) n += (lens[u] + qb - 1) / qb;
    if (n > MAX_WORK || units > 65535) return 0;
    struct W { long long cost; uint32_t v; };
    W tmp[MAX_WORK];
    n = 0;
    for (int32_t u = 0; u < units; ++u) {
        for (int b = 0; b * qb < lens[u]; ++b) {
            const long long q = lens[u] - b * qb < qb ? lens[u] - b * qb : qb;
            long long keys = lens[u];
            if (window > 0 && 2LL * window + qb < keys) keys = 2LL * window + qb;
            tmp[n++] = {q * keys, ((uint32_t)u << 16) | (uint32_t)b};
        }
    }
    std::stable_sort(tmp, tmp + n, [](const W &a, const W &b) { return a.cost > b.cost; });
    for (int i = 0; i < n; ++i) work[i] = tmp[i].v;
    return n;
}

static te_status attn_launch(const void *qkv, int64_t ld, int32_t q_off, int32_t k_off, int32_t v_off,
                             const int32_t *cu_dev, const int32_t *items_dev, int32_t units, int32_t total,
                             int32_t max_len, const int32_t *unit_lens, int32_t nq_heads, int32_t nkv_heads,
                             int32_t hd, int32_t window, float scale, void *out, int64_t ldo, te_stream stream) {
    {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(qkv);
        const uintptr_t a1 = a0 + (uintptr_t)total * ld * 2;
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(out);
        const uintptr_t b1 = b0 + (uintptr_t)total * ldo * 2;
        if (a0 < b1 && b0 < a1) return fail(TE_EINVAL, "attn: out overlaps qkv");
    }
    AttnParams p;
    memset(&p, 0, sizeof(p));
    te_status st = make_map_2d(&p.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qkv, (uint64_t)ld, (uint64_t)total,
                               (uint64_t)ld * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != TE_OK) return st;
    st = make_map_2d(&p.map32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qkv, (uint64_t)ld, (uint64_t)total,
                     (uint64_t)ld * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != TE_OK) return st;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.cu = cu_dev;
    p.items = items_dev;
    p.ldo = ldo;
    p.q_off = q_off;
    p.k_off = k_off;
    p.v_off = v_off;
    p.group = nq_heads / nkv_heads;
    p.window = window;
    p.scale_log2 = scale * 1.4426950408889634f;
    // hd = 64: one 128-query tile a CTA, two CTAs an SM; hd = 128: two tiles
    // a CTA (two CTAs would not fit an SM's shared memory)
    const int tl = hd == 64 ? 1 : 2;
    p.nwork = build_work(unit_lens, units, window, tl * BQ, p.work);
    // heads per group: all when every head's K and V fit in KV_ALL_BYTES
    // together, else the kv heads whose K and V make about KV_GROUP_BYTES
    p.nq = nq_heads;
    const long long kv_head = (long long)total * hd * 4;
    long long hg = nq_heads;
    if (kv_head * nkv_heads > KV_ALL_BYTES) {
        hg = KV_GROUP_BYTES / kv_head * p.group;
        if (hg < p.group) hg = p.group;
        if (hg > nq_heads) hg = nq_heads;
    }
    p.hgroup = (int)hg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return hd == 64 ? launch<64, 1>(p, max_len, nq_heads, units, s)
                    : launch<128, 2>(p, max_len, nq_heads, units, s);
}

extern "C" te_status te_attn_varlen_fwd(const void *qkv, int64_t ld, int32_t q_off, int32_t k_off,
                                        int32_t v_off, const int32_t *cu_host,
                                        const int32_t *cu_dev, int32_t nseq, int32_t nq_heads,
                                        int32_t nkv_heads, int32_t hd, int32_t window, float scale,
                                        void *out, int64_t ldo, te_stream stream) {
    te_status st = attn_common_checks(qkv, ld, q_off, k_off, v_off, nq_heads, nkv_heads, hd, window, out, ldo);
    if (st != TE_OK) return st;
    if (nseq > 65535) return fail(TE_ESHAPE, "attn: too many sequences");
    int32_t total = 0, max_len = 0;
    if ((st = check_cu(cu_host, cu_dev, nseq, &total, &max_len)) != TE_OK) return st;
    std::vector<int32_t> lens(nseq);
    for (int32_t i = 0; i < nseq; ++i) lens[i] = cu_host[i + 1] - cu_host[i];
    return attn_launch(qkv, ld, q_off, k_off, v_off, cu_dev, nullptr, nseq, total, max_len, lens.data(),
                       nq_heads, nkv_heads, hd, window, scale, out, ldo, stream);
}

extern "C" te_status te_attn_items_fwd(const void *qkv, int64_t ld, int32_t q_off, int32_t k_off,
                                       int32_t v_off, const int32_t *items_host, const int32_t *items_dev,
                                       int32_t nitems, int32_t rows, int32_t nq_heads, int32_t nkv_heads,
                                       int32_t hd, int32_t window, float scale, void *out, int64_t ldo,
                                       te_stream stream) {
    te_status st = attn_common_checks(qkv, ld, q_off, k_off, v_off, nq_heads, nkv_heads, hd, window, out, ldo);
    if (st != TE_OK) return st;
    if (!items_host || !items_dev) return fail(TE_EINVAL, "attn_items: NULL items");
    if (nitems < 1 || nitems > 65535) return fail(TE_ESHAPE, "attn_items: nitems=%d (1..65535)", nitems);
    if (rows < 1) return fail(TE_ESHAPE, "attn_items: rows=%d", rows);
    if (reinterpret_cast<uintptr_t>(items_dev) & 15) return fail(TE_EALIGN, "attn_items: items must be 16-byte aligned");
    int32_t max_len = 0;
    std::vector<int32_t> lens(nitems);
    for (int32_t i = 0; i < nitems; ++i) {
        const int32_t o1 = items_host[4 * i], l1 = items_host[4 * i + 1];
        const int32_t o2 = items_host[4 * i + 2], l2 = items_host[4 * i + 3];
        if (o1 < 0 || l1 < 1 || o2 < 0 || l2 < 0 || (int64_t)o1 + l1 > rows || (int64_t)o2 + l2 > rows)
            return fail(TE_EINVAL, "attn_items: item %d (%d, %d, %d, %d) runs outside the %d rows", i, o1, l1,
                        o2, l2, rows);
        if (l2 > 0 && l1 % 32)
            return fail(TE_ESHAPE, "attn_items: item %d: the first range's length %d is not a multiple of 32", i, l1);
        if ((int64_t)l1 + l2 > (1 << 30)) return fail(TE_ESHAPE, "attn_items: item %d too long", i);
        if (l1 + l2 > max_len) max_len = l1 + l2;
        lens[i] = l1 + l2;
    }
    return attn_launch(qkv, ld, q_off, k_off, v_off, nullptr, items_dev, nitems, rows, max_len, lens.data(),
                       nq_heads, nkv_heads, hd, window, scale, out, ldo, stream);
}
