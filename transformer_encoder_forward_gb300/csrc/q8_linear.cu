// Grouped q8_row linear on the 5th-generation tensor cores (sm_103a).
//
//     y_i[t, o] = scale_i[o] * sum_k x[t, k] * q_i[o, k]  (+ bias_i[o]) (+ residual_i[t, o])
//
// Sources: "cortiq-engine 0.7.6 src/gpu_metal/zimage.rs", module doc ("The
// chain": each GEMM stages the int8 tile as half, exact, and applies the row
// scale in its f32 epilogue; Enc::gemm takes z <= 3 items sharing the input)
// and "cortiq-engine 0.8.39 src/gpu_metal/egemma2.rs" (Prog::mm: one dispatch
// over an item table, one item per grid z).
//
// GB300 design (not the pages' 64x64x32 simdgroup tiling).  A tile computes
// the TRANSPOSED product Y^T[o, t] = W[o, :] . X[t, :] so that its weight
// rows sit on the TMEM lanes.  Persistent 2-CTA clusters (one CTA per SM)
// walk a static list of (256 features x BN tokens) tiles: each CTA owns 128
// feature rows and half of the BN tokens, and the leader CTA issues 2-SM
// MMAs (cta_group::2, M=256) that read both CTAs' operands, so each SM only
// ingests its own weight rows and half of the activation tile.  Roles:
//   * warp 0 (one lane) streams K-slices of 128 with TMA, each as two
//     64-wide boxes: this CTA's half of the bf16 activation tile [BN/2 tokens
//     x 128] into 128-byte-swizzled shared memory (its part of the MMA's B
//     operand) and its int8 weight tile [128 x 128] (64-byte swizzle);
//   * warps 2-9 widen the int8 tile to bf16 in registers - exact, |q| <= 127
//     fits bf16's 8-bit significand - with a byte-permute / f32-add magic
//     number sequence that stays off the slow conversion pipe, and write it
//     straight into TMEM with tcgen05.st, where it is the MMA's A operand
//     (two warps per TMEM lane quadrant, each one 64-column box); the
//     widened tile never touches shared memory, which keeps shared-memory
//     bandwidth for the B reads;
//   * warp 1 (one lane of the leader) issues tcgen05.mma.cta_group::2
//     kind::f16 M=256 N=BN K=16 into one of two f32 TMEM accumulators (each
//     CTA holds its 128 rows) and releases both CTAs' stages with multicast
//     tcgen05.commit; the converters and epilogue warps of both CTAs report to
//     the leader's barriers through their cluster addresses;
//   * warps 10-13 drain the other accumulator meanwhile (tcgen05.ld): lane =
//     output feature, so the row scale and bias are per-thread constants;
//     each 32 x 32 block is written into a staging tile in the output's own
//     layout and leaves with one TMA tensor store (a TMA reduce-add when the
//     residual is y itself, the in-place x += proj of the plain block); the
//     blocks go out in chunks, one shared-memory fence a chunk.  In
//     the gated form each lane quadrant holds 16 gate rows and the same
//     features' up rows, paired by register shuffles.
// The issuing thread's instruction rate bounds the MMA rate at N <= 192 (one
// thread issues a 2-SM MMA every ~45 cycles at best), so its loop is kept
// lean.  With long K a unit can hold two token tiles: each widened weight
// stage then feeds both tiles' MMAs, each tile's accumulator is released on
// its own barrier, and the tile width follows the wave count (long_k_tile).
// With short K (every K stage fits the TMEM A stages at once) the weights stay
// resident: each cluster takes a contiguous run of units, which share their
// feature tiles except where the run crosses into the next feature pair; the
// converters widen a feature tile once, and later units of the run only
// stream activations.  The peer's warp 1 relays each of its landed stages to
// the leader's full barrier (which then counts two arrivals), so the MMA
// issuer waits on one barrier per stage.
// TMEM: 2 accumulators of BN columns + as many A stages of 64 columns as fit
// in the 512, fewer than the load stages (2 for BN = 192, 3 for 160 and for
// 128 with two token tiles a unit, 4 for 128 and 64).  A stage is 8 MMAs
// deep per token tile.  Every mbarrier wait is bounded (about 200 ms); a
// timeout sets an error word that te_check() reports, the role stops, and the
// kernel still waits for its own copies and MMAs and frees its TMEM.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"

namespace tefwd {
namespace {

constexpr int BM = 128;       // weight rows (output features) per tile = TMEM lanes
constexpr int BK = 128;       // K per pipeline stage (two 64-wide TMA boxes)
constexpr int BOX = 64;       // K width of one TMA box
constexpr int MAXZ = 4;
// activation bytes of one group of token tiles in the unit order: small
// enough that the group stays in L2 while outputs and weights stream through
constexpr long long XGROUP_BYTES = 24ll << 20;
constexpr int NWARPS = 14;    // producer, MMA, 8 converters, 4 epilogue
constexpr int NTHREADS = NWARPS * 32;

struct Item {
    const float *scale;       // NULL: 1 (block-scaled weights)
    const float *bias;
    const float *scale2;      // gated mode: the up projection's scale and bias
    const float *bias2;
    const uint16_t *bsc;      // f16 block scales [n, k/32] of the 32-element formats, or NULL
    const uint16_t *bsc2;     // gated mode: the up projection's
    const float *col;         // q8_2f column field [k], or NULL
    const float *col2;        // gated mode: the up projection's
    void *y;
    const float *resid;
    long long ldy, ldr;
    int n, ydt, tile0, ntiles, act;
};

struct Params {
    CUtensorMap tx;           // x: bf16 [m, k]
    CUtensorMap tw[MAXZ];     // q_i: int8 [n_i, k]
    CUtensorMap ty[MAXZ];     // y_i: [m, n_i] (f32 or bf16), 32-feature boxes
    Item it[MAXZ];
    int z, m, k, ttiles, nunits;
    int fpairs;               // pairs of 128-row feature tiles
    int tgroup;               // token tiles per group of the unit order
    int kb32;                 // k / 32: the row stride of the block scales
    int res;                  // resident weights (see q8_gemm_kernel)
};

__device__ int g_gemm_err;

template <int BN, int TPA>
struct Layout {
    static constexpr int HALF = BN / 2;                 // token rows each CTA of the pair holds
    // shared-memory load stages (a stage holds TPA token tiles)
    static constexpr int NST = TPA == 2 ? (BN == 128 ? 4 : 3) : (BN >= 128 ? 5 : 6);
    // TMEM stages of the widened A operand (64 columns each): what the two
    // BN-column accumulators leave of the 512 columns, at most 4 and fewer
    // than the load stages
    static constexpr int NA0 = (512 - 2 * BN) / 64 < 4 ? (512 - 2 * BN) / 64 : 4;
    static constexpr int NA = NA0 < NST - 1 ? NA0 : NST - 1;
    static constexpr int XBOX = HALF * BOX * 2;         // one 64-wide box of this CTA's activation half
    static constexpr int XTILE = 2 * XBOX;              // this CTA's half of one token tile's stage
    static constexpr int XBYTES = TPA * XTILE;          // ... of all TPA token tiles
    static constexpr int WBOX = BM * BOX;               // one 64-wide box of the int8 weight tile
    static constexpr int WBYTES = 2 * WBOX;             // int8 weight stage (own 128 rows)
    static constexpr int X_OFF = 0;
    static constexpr int W_OFF = NST * XBYTES;
    // epilogue staging, per epilogue warp: a ring of 32-token output blocks
    // (f32 32 x 32: 4 KB; bf16 32 x 32: 2 KB; gated bf16 32 x 16: 1 KB) in two
    // halves, so that one chunk's TMA stores can still be reading while the
    // next chunk is written; 8 KB a warp where shared memory allows (the
    // one-tile units of the short-K GEMMs, whose epilogue sets their pace),
    // else 4 KB; 128-byte aligned (TMA sources).  q8_2f: each stage's 128 column-field values
    // (f32), for the gate and the up weight in the gated form
    static constexpr int COL_OFF = W_OFF + NST * WBYTES;
    static constexpr int COL_BYTES = 2 * BK * 4;
    static constexpr int STG_OFF = COL_OFF + NST * COL_BYTES;
    static constexpr int STG_WARP = TPA == 1 && BN <= 128 ? 8192 : 4096;
    static constexpr int STG_BYTES = 4 * STG_WARP;
    // one-tile units at N = 128: 4 KB a warp for four converter warps that
    // help drain the gated form while the weights are resident
    static constexpr bool HELP = TPA == 1 && BN == 128;
    // two-tile units: converter warps 2-5 drain the second token tile while
    // the epilogue warps drain the first (one 2 KB
    // slot a warp: a bf16 block, two gated blocks, or an f32 16-token half)
    static constexpr bool HELP2 = TPA == 2;
    static constexpr int HSTG_OFF = STG_OFF + STG_BYTES;
    static constexpr int HSTG_BYTES = HELP ? 4 * 4096 : (HELP2 ? 4 * 2048 : 0);
    static constexpr int BAR_OFF = HSTG_OFF + HSTG_BYTES;
    // barriers: full, empty [NST]; afull, aempty [NA]; accfull, accempty [2]; done
    static constexpr int NBAR = 2 * NST + 2 * NA + 4 + 1;
    static constexpr int BYTES = BAR_OFF + 8 * NBAR + 16;
    static constexpr int A_COL = 2 * BN;                // first TMEM column of the A stages
    static constexpr int TMEM_COLS = 512;
    static_assert(NA >= 2 && 2 * BN + NA * 64 <= TMEM_COLS, "TMEM budget");
    static_assert(NA < NST, "a free A stage proves the ring passed the slot's previous use");
    static_assert(XBOX % 1024 == 0, "swizzled boxes stay 1024-byte aligned");
    static_assert(BYTES + 1024 <= 227 * 1024, "shared memory per CTA");
};

// int8 x4 -> two bf16x2 words, exactly.  (b ^ 0x80) is q + 128; placed as the
// low byte of the f32 pattern 0x4B0000xx it reads 2^23 + q + 128, and one f32
// subtraction leaves q.  |q| <= 128 needs at most 8 significant bits, so the
// upper 16 bits of that f32 are its exact bf16.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const float magic = 8388736.0f;   // 2^23 + 128
    const float f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - magic;
    const float f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - magic;
    const float f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - magic;
    const float f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - magic;
    lo = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
    hi = __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
}

// As widen4, value e multiplied by its own factor c[e] (the q8_2f column
// field) and rounded once to bf16.
__device__ __forceinline__ void widen4_col(uint32_t w, float4 c, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const float magic = 8388736.0f;   // 2^23 + 128
    const float f0 = (__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - magic) * c.x;
    const float f1 = (__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - magic) * c.y;
    const float f2 = (__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - magic) * c.z;
    const float f3 = (__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - magic) * c.w;
    lo = pack_bf16x2(f0, f1);
    hi = pack_bf16x2(f2, f3);
}

// As widen4, each value then multiplied by the block scale d (exact in f32:
// 8 x 11 significant bits) and rounded once to bf16.
__device__ __forceinline__ void widen4_scaled(uint32_t w, float d, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const float magic = 8388736.0f;   // 2^23 + 128
    const float f0 = (__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - magic) * d;
    const float f1 = (__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - magic) * d;
    const float f2 = (__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - magic) * d;
    const float f3 = (__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - magic) * d;
    lo = pack_bf16x2(f0, f1);
    hi = pack_bf16x2(f2, f3);
}

struct TileCoord {
    int zi, o0, t0;
};

// Work units are (pair of 128-row feature tiles, BN-token tile).  The two CTAs
// of a cluster take the two feature tiles of one unit: they share the token
// tile, and each CTA TMA-loads its own half of it into its own shared memory
// (no load is multicast); the 2-SM MMA reads both halves.  Units come in
// groups of tgroup token tiles; within a group, feature pair major and the
// group's token tiles fastest: clusters running together share weight tiles,
// and the group's activation rows (re-read once per feature pair) stay in L2
// while the weights stream past them once per group.  A feature tile past the
// last one (odd count) is a phantom: its weights read as zeros and its
// epilogue stores nothing.
template <bool GATED>
__device__ __forceinline__ TileCoord tile_coord(const Params &p, int unit, int rank) {
    int fp, tt;
    if (p.tgroup >= p.ttiles) {
        fp = unit / p.ttiles;
        tt = unit - fp * p.ttiles;
    } else {
        const int per = p.tgroup * p.fpairs;
        const int g = unit / per;
        const int r = unit - g * per;
        const int t0 = g * p.tgroup;
        const int gn = p.ttiles - t0 < p.tgroup ? p.ttiles - t0 : p.tgroup;
        fp = r / gn;
        tt = t0 + (r - fp * gn);
    }
    const int ft = 2 * fp + rank;
    int zi = 0;
    while (zi + 1 < p.z && ft >= p.it[zi + 1].tile0) ++zi;
    // gated: a tile holds 64 gate rows and the 64 matching up rows
    return {zi, (ft - p.it[zi].tile0) * (GATED ? BM / 2 : BM), tt};
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// tcgen05.commit (cta_group::2, multicast) and the 2-SM MMA, each issued by
// the lane whose `e` is set (the warp runs in step): the commit arrives on
// the mbarrier at `bar`'s offset in every CTA of `mask` once the 2-SM MMAs
// issued so far are done; the MMA computes D(tmem, both CTAs) (+)= A(tmem,
// both CTAs) * B(smem desc, N split across the pair).
__device__ __forceinline__ void mma_commit_pair_e(uint32_t bar, uint16_t mask, uint32_t e) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %2, 0;\n\t"
        "@q tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;\n\t}" ::"r"(bar), "h"(mask), "r"(e)
        : "memory");
}
__device__ __forceinline__ void mma_ts_pair_e(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate, uint32_t e) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(e)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

template <int BN, bool GATED, int TPA>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    q8_gemm_kernel(const __grid_constant__ Params p) {
    using L = Layout<BN, TPA>;
    constexpr int NST = L::NST;
    constexpr int NA = L::NA;
    constexpr int HALF = L::HALF;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar_full = sb + L::BAR_OFF;
    const uint32_t bar_empty = bar_full + 8 * NST;
    const uint32_t bar_afull = bar_empty + 8 * NST;
    const uint32_t bar_aempty = bar_afull + 8 * NA;
    const uint32_t bar_accfull = bar_aempty + 8 * NA;
    const uint32_t bar_accempty = bar_accfull + 16;
    const uint32_t bar_done = bar_accempty + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * L::NBAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = (p.k + BK - 1) / BK;   // a trailing half stage reads zeros past k
    const int rank = (int)cluster_rank();
    const bool leader = rank == 0;
    const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    const bool res = p.res != 0;
    // The gated form with resident weights at N = 128 is drained by the four
    // epilogue warps (blocks 0-1 of each token tile) and by converter warps
    // 2-5 (blocks 2-3), idle otherwise once the run's weights are widened:
    // one warp's drain of a unit outlasts the unit's MMAs, and each warp's
    // drain is bound by its own instruction latencies, so two warps a lane
    // quadrant halve it.
    const bool helpers = GATED && L::HELP && res;
    // once any CTA has given up a wait, the rest skip their work (the call
    // has failed; te_check reports it) instead of timing out one by one
    __shared__ int s_skip;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            // resident weights: the leader's full barriers also take the peer's relay
            mbar_init(bar_full + 8 * s, res && leader ? 2 : 1);
            mbar_init(bar_empty + 8 * s, 1);      // the leader's MMA commit, multicast
        }
        for (int a = 0; a < NA; ++a) {
            mbar_init(bar_afull + 8 * a, 16);     // every converter warp of both CTAs (leader's copy)
            mbar_init(bar_aempty + 8 * a, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_accfull + 8 * b, 1);
            // every draining warp of both CTAs (leader's copy): the epilogue
            // warps, and four converter warps too with helpers (for a
            // two-tile unit's second tile, converter warps 2-5)
            mbar_init(bar_accempty + 8 * b, helpers || (L::HELP2 && b == 1) ? 16 : 8);
        }
        mbar_init(bar_done, 1);
        fence_mbar_init();
        s_skip = *reinterpret_cast<volatile int *>(&g_gemm_err) != 0;
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), L::TMEM_COLS);
    tc_fence_before();
    cluster_sync();            // both CTAs' barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    bool ok = s_skip == 0;
    const int nunits = ok ? p.nunits : 0;
    // the leader's copies of the pair-wide barriers, as cluster addresses
    const uint32_t afull_ldr = mapa_shared(bar_afull, 0);
    const uint32_t accempty_ldr = mapa_shared(bar_accempty, 0);
    const uint32_t full_ldr = mapa_shared(bar_full, 0);
    // this cluster's units: a contiguous run with resident weights, else
    // every ncl-th unit from cid
    const int ubeg = res ? (int)((long long)cid * nunits / ncl) : cid;
    const int ucnt = res ? (int)((long long)(cid + 1) * nunits / ncl) - ubeg
                         : (cid < nunits ? (nunits - 1 - cid) / ncl + 1 : 0);
    auto unit_at = [&](int i) { return res ? ubeg + i : cid + i * ncl; };
    // whether unit i of the run widens its weights: always without resident
    // weights, else at the run's start and where the feature pair changes
    auto fills = [&](int i) {
        return !res || i == 0 || unit_at(i) / p.ttiles != unit_at(i - 1) / p.ttiles;
    };
    // With helpers: the drain of unit lt's accumulator (one token tile), blocks
    // [cb, ce), by the calling warp (lane quadrant warp & 3), in chunks of two
    // blocks through its own 4-block ring at shared address hstg (gslot: the
    // ring position); lane i stores block i of a chunk and commits its own
    // bulk group.  The arithmetic is the epilogue's gated form (see there).
    auto gated_drain = [&](int lt, int cb, int ce, uint32_t hstg, int &gslot) -> bool {
        const int q = warp & 3;
        const bool upper = lane & 16;
        const int frow = 16 * q + (lane & 15);
        const uint32_t tl = (uint32_t)(32 * q) << 16;
        const int u = unit_at(lt);
        const int b = lt & 1;
        const uint32_t ph = (lt >> 1) & 1;
        const TileCoord tc = tile_coord<GATED>(p, u, rank);
        const int o = tc.o0 + frow;
        const bool ov = o < p.it[tc.zi].n;
        const float *scale = upper ? p.it[tc.zi].scale2 : p.it[tc.zi].scale;
        const float *bias = upper ? p.it[tc.zi].bias2 : p.it[tc.zi].bias;
        const float sc = ov ? (scale ? scale[o] : 1.f) : 0.f;
        const float bi = (ov && bias) ? bias[o] : 0.f;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_accfull + 8 * b, ph))) return false;
        tc_fence_after();
        const int act = p.it[tc.zi].act;
        const int n = p.it[tc.zi].n;
        const void *ymap = &p.ty[tc.zi];
        const int acol = b * BN;
        const int t0 = tc.t0 * BN;
        const int cn = t0 >= p.m ? 0 : ((p.m - t0 + 31) / 32 < BN / 32 ? (p.m - t0 + 31) / 32 : BN / 32);
        const int cend = ce < cn ? ce : cn;
        const int fo = tc.o0 + 16 * q;
        const int jb = upper ? 16 : 0;
        const uint64_t sc2 = f2_pack(sc, sc), bi2 = f2_pack(bi, bi), half2 = f2_pack(0.5f, 0.5f);
        for (int c0 = cb; c0 < cend && fo < n; c0 += 2) {
            const int ceb = c0 + 2 < cend ? c0 + 2 : cend;
            if (lane < 2) bulk_wait_read_n<1>();
            __syncwarp();
            for (int c = c0; c < ceb; ++c) {
                uint32_t v[32];
                tmem_ld32(tbase + tl + acol + 32 * c, v);
                tmem_wait_ld();
                float gv[16], uv[16], yv[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float lo, hi;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[16 + j])), sc2, bi2), lo, hi);
                    const uint32_t b2 = pack_bf16x2(lo, hi);
                    lo = bf16_lo(b2);
                    hi = bf16_hi(b2);
                    const float got = __shfl_xor_sync(0xFFFFFFFFu, upper ? lo : hi, 16);
                    gv[j] = upper ? got : lo;
                    uv[j] = upper ? hi : got;
                }
                const bool gelu = act == TE_ACT_GELU_TANH;
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const uint64_t g2 = f2_pack(gv[j], gv[j + 1]);
                    const uint64_t z2 = gelu ? f2_mul(g2, f2_fma(f2_pack(0.035677408f, 0.035677408f), f2_mul(g2, g2),
                                                                 f2_pack(0.79788456f, 0.79788456f)))
                                             : f2_mul(half2, g2);
                    float z0, z1;
                    f2_unpack(z2, z0, z1);
                    const uint64_t h2 = f2_mul(half2, g2);
                    const uint64_t a2 = f2_fma(h2, f2_pack(hw_tanh(z0), hw_tanh(z1)), h2);
                    f2_unpack(f2_mul(a2, f2_pack(uv[j], uv[j + 1])), yv[j], yv[j + 1]);
                }
                const uint32_t so = hstg + (uint32_t)(((gslot + c - c0) & 3) * 1024);
                uint16_t *ostg_h = reinterpret_cast<uint16_t *>(smem + (so - sb));
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    ostg_h[(jb + j) * 16 + (lane & 15)] = __bfloat16_as_ushort(__float2bfloat16_rn(yv[j]));
            }
            fence_async_smem();
            __syncwarp();
            if (lane < 2) {
                const int c = c0 + lane;
                if (c < ceb) tma_store_2d(ymap, hstg + (uint32_t)(((gslot + lane) & 3) * 1024), fo, t0 + 32 * c);
                bulk_commit();
            }
            gslot += 2;
        }
        // this accumulator may take the next tile's MMAs
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(accempty_ldr + 8 * b);
        return true;
    };

    // Two-tile units: the blocks of the second token tile that the epilogue
    // warps drain themselves: none (converter warps 2-5 drain that tile while
    // the epilogue warps drain the first, which the next unit's first MMAs
    // need), or all where a residual other than y is added from global
    // memory.  Keeping its first block with the epilogue warps measured the
    // same.
    auto e_blocks2 = [&](int zi, int cn) -> int {
        const bool other_resid = p.it[zi].resid != nullptr && p.it[zi].resid != p.it[zi].y;
        return other_resid ? cn : 0;
    };
    // Two-tile units: the calling converter warp (lane quadrant warp & 3)
    // drains blocks [e_blocks2, cn) of unit lt's second token tile through
    // its own 2 KB slot at shared address hstg, with the epilogue's
    // arithmetic for the item's output form, then releases that accumulator
    // together with the epilogue warps.  Lane 0 issues the stores, one bulk
    // group each; hslot counts the gated blocks (two 1 KB slots).
    auto help2_drain = [&](int lt, uint32_t hstg, int &hslot) -> bool {
        const int q = warp & 3;
        const bool upper = GATED && (lane & 16);
        const int frow = GATED ? 16 * q + (lane & 15) : 32 * q + lane;
        const uint32_t tl = (uint32_t)(32 * q) << 16;
        const TileCoord tc = tile_coord<GATED>(p, unit_at(lt), rank);
        const Item &it = p.it[tc.zi];
        const int o = tc.o0 + frow;
        const bool ov = o < it.n;
        const float *scale = upper ? it.scale2 : it.scale;
        const float *bias = upper ? it.bias2 : it.bias;
        const float sc = ov ? (scale ? scale[o] : 1.f) : 0.f;
        const float bi = (ov && bias) ? bias[o] : 0.f;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_accfull, lt & 1))) return false;
        tc_fence_after();
        const int t0 = (tc.t0 * 2 + 1) * BN;
        const int cn = t0 >= p.m ? 0 : ((p.m - t0 + 31) / 32 < BN / 32 ? (p.m - t0 + 31) / 32 : BN / 32);
        const int fo = tc.o0 + (GATED ? 16 : 32) * q;
        const void *ymap = &p.ty[tc.zi];
        const bool f32out = it.ydt == TE_F32;
        const bool inplace = it.resid != nullptr && it.resid == it.y;
        const uint64_t sc2 = f2_pack(sc, sc), bi2 = f2_pack(bi, bi);
        for (int c = e_blocks2(tc.zi, cn); c < cn && fo < it.n; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + tl + BN + 32 * c, v);
            tmem_wait_ld();
            const int tb = t0 + 32 * c;
            if constexpr (GATED) {
                // the epilogue's gated form: scale and bias, both halves
                // rounded to bf16, gate and up lanes swap half their tokens,
                // m = act(g) * u in f32 pairs
                const uint64_t half2 = f2_pack(0.5f, 0.5f);
                float gv[16], uv[16], yv[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float lo, hi;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[16 + j])), sc2, bi2), lo, hi);
                    const uint32_t b2 = pack_bf16x2(lo, hi);
                    lo = bf16_lo(b2);
                    hi = bf16_hi(b2);
                    const float got = __shfl_xor_sync(0xFFFFFFFFu, upper ? lo : hi, 16);
                    gv[j] = upper ? got : lo;
                    uv[j] = upper ? hi : got;
                }
                const bool gelu = it.act == TE_ACT_GELU_TANH;
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const uint64_t g2 = f2_pack(gv[j], gv[j + 1]);
                    const uint64_t z2 = gelu ? f2_mul(g2, f2_fma(f2_pack(0.035677408f, 0.035677408f), f2_mul(g2, g2),
                                                                 f2_pack(0.79788456f, 0.79788456f)))
                                             : f2_mul(half2, g2);
                    float z0, z1;
                    f2_unpack(z2, z0, z1);
                    const uint64_t h2 = f2_mul(half2, g2);
                    const uint64_t a2 = f2_fma(h2, f2_pack(hw_tanh(z0), hw_tanh(z1)), h2);
                    f2_unpack(f2_mul(a2, f2_pack(uv[j], uv[j + 1])), yv[j], yv[j + 1]);
                }
                // the store two blocks back, which used this slot, has read it
                if (lane == 0) bulk_wait_read_n<1>();
                __syncwarp();
                const uint32_t so = hstg + (uint32_t)((hslot & 1) * 1024);
                uint16_t *ostg_h = reinterpret_cast<uint16_t *>(smem + (so - sb));
                const int jb = upper ? 16 : 0;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    ostg_h[(jb + j) * 16 + (lane & 15)] = __bfloat16_as_ushort(__float2bfloat16_rn(yv[j]));
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(ymap, so, fo, tb);
                    bulk_commit();
                }
                ++hslot;
            } else {
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    float a, b2;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), sc2, bi2), a, b2);
                    v[j] = __float_as_uint(a);
                    v[j + 1] = __float_as_uint(b2);
                }
                if (it.act) {   // the ungated MLP: act(bf16(s*acc + b))
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = __float_as_uint(apply_act_tanh(round_bf16(__uint_as_float(v[j])), it.act - 1));
                }
                if (f32out) {
                    // 16-token halves (the two-tile units' f32 maps have
                    // 16-row boxes), each after the previous has been read
                    float *ostg = reinterpret_cast<float *>(smem + (hstg - sb));
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if (hh == 1 && tb + 16 >= p.m) break;       // warp-uniform
                        if (lane == 0) bulk_wait_read_n<0>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 16; ++j) ostg[j * 32 + lane] = __uint_as_float(v[16 * hh + j]);
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (inplace)
                                tma_reduce_add_2d(ymap, hstg, fo, tb + 16 * hh);
                            else
                                tma_store_2d(ymap, hstg, fo, tb + 16 * hh);
                            bulk_commit();
                        }
                    }
                } else {
                    if (lane == 0) bulk_wait_read_n<0>();
                    __syncwarp();
                    uint16_t *ostg_h = reinterpret_cast<uint16_t *>(smem + (hstg - sb));
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        ostg_h[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(ymap, hstg, fo, tb);
                        bulk_commit();
                    }
                }
            }
        }
        // the second tile's accumulator may take the next unit's MMAs
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(accempty_ldr + 8);
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // (the whole warp in step, one elected lane issues: warp-uniform values)
        const uint32_t e = elect_one();
        if (e) tma_prefetch_desc(&p.tx);
        int kbg = 0;
        for (int i = 0; i < ucnt && ok; ++i) {
            const int u = unit_at(i);
            const bool fl = fills(i);   // weights (and column field) only when widened
            const TileCoord tc = tile_coord<GATED>(p, u, rank);
            const void *wmap = &p.tw[tc.zi];
            const float *cg = fl ? p.it[tc.zi].col : nullptr;
            const float *cu2 = GATED && fl ? p.it[tc.zi].col2 : nullptr;
            for (int kb = 0; kb < nkb; ++kb, ++kbg) {
                const int s = kbg % NST;
                const uint32_t fb = bar_full + 8 * s;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_empty + 8 * s, ((kbg / NST) & 1) ^ 1))) {
                    ok = false;
                    break;
                }
                // the column field slice of this stage (the last stage may hold 64)
                const uint32_t cbytes = (uint32_t)((p.k - kb * BK < BK ? p.k - kb * BK : BK) * 4);
                mbar_arrive_expect_tx_e(fb, L::XBYTES + (fl ? L::WBYTES : 0) + (cg ? cbytes : 0) + (cu2 ? cbytes : 0),
                                        e);
                if (cg) bulk_load_e(sb + L::COL_OFF + s * L::COL_BYTES, cg + kb * BK, cbytes, fb, e);
                if (cu2) bulk_load_e(sb + L::COL_OFF + s * L::COL_BYTES + BK * 4, cu2 + kb * BK, cbytes, fb, e);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint32_t wdst = sb + L::W_OFF + s * L::WBYTES + c * L::WBOX;
#pragma unroll
                    for (int tt = 0; tt < TPA; ++tt)
                        tma_load_2d_e(sb + L::X_OFF + s * L::XBYTES + tt * L::XTILE + c * L::XBOX, &p.tx, fb,
                                      kb * BK + c * BOX, (tc.t0 * TPA + tt) * BN + rank * HALF, e);
                    if (!fl) continue;
                    if (GATED) {   // rows 0-63: gate, rows 64-127: up, same features
                        tma_load_2d_e(wdst, &p.tw[0], fb, kb * BK + c * BOX, tc.o0, e);
                        tma_load_2d_e(wdst + (BM / 2) * BOX, &p.tw[1], fb, kb * BK + c * BOX, tc.o0, e);
                    } else {
                        tma_load_2d_e(wdst, wmap, fb, kb * BK + c * BOX, tc.o0, e);
                    }
                }
            }
        }
        // make sure no copy of ours is still landing when the CTA exits
        for (int j = kbg - NST < 0 ? 0 : kbg - NST; j < kbg; ++j)
            mbar_wait(bar_full + 8 * (j % NST), (j / NST) & 1, 20000000ull);
    } else if (warp == 1) {
        // -------------------------------------- MMA issuer (leader CTA only)
        // The whole warp runs the loop in step (waits, indices, descriptors)
        // and one elected lane issues: the values stay warp-uniform, so the
        // MMAs take their operands from uniform registers (an issue loop in
        // one divergent lane cost about 84 cycles an MMA).
        if (leader) {
            const uint32_t e = elect_one();
            constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
            // the loop keeps its indices incremental: ring slot s and A stage
            // ar with their phases
            int nfill = 0, s = 0, ar = 0;
            uint32_t sph = 0, aph = 0;
            for (int lt = 0; lt < ucnt && ok; ++lt) {
                const bool fl = fills(lt);
                // resident weights: the A stages are released after the last
                // unit that uses this widening
                const bool last_use = !res || lt + 1 == ucnt || fills(lt + 1);
                // TPA == 1: units alternate between the two accumulators;
                // TPA == 2: a unit's two token tiles use both
                const int b = TPA == 2 ? 0 : (lt & 1);
                const uint32_t ph = TPA == 2 ? (lt & 1) : ((lt >> 1) & 1);
                if (!__all_sync(0xFFFFFFFFu, mbar_wait_cluster(bar_accempty + 8 * b, ph ^ 1))) { ok = false; break; }
                tc_fence_after();
                const uint32_t dcol = tbase + (TPA == 2 ? 0 : b) * BN;
                int kb0 = 0;   // stages issued for both token tiles before the main loop
                if (TPA == 2) {
                    // Token tile 0's MMAs for the first widened stages start
                    // while the epilogue still drains tile 1 (it drains tile 0
                    // first and releases each accumulator on its own barrier);
                    // each accumulator keeps its own MMA order.
                    const int P = nkb < NA ? nkb : NA;
                    int ss = s, aa = ar;
                    uint32_t aph2 = aph;
                    for (int kb = 0; kb < P && ok; ++kb) {
                        if (!__all_sync(0xFFFFFFFFu, mbar_wait_cluster(bar_afull + 8 * aa, aph2))) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t d0 = smem_desc_sw128(sb + L::X_OFF + ss * L::XBYTES);
                        const uint32_t a0 = tbase + L::A_COL + 64 * aa;
#pragma unroll
                        for (int j = 0; j < BK / 16; ++j)
                            mma_ts_pair_e(dcol, a0 + 8 * j, d0 + (uint64_t)(((j >> 2) * L::XBOX + (j & 3) * 32) >> 4),
                                        idesc, j == 0 ? (uint32_t)(kb != 0) : 1u, e);
                        if (++ss == NST) ss = 0;
                        if (++aa == NA) { aa = 0; aph2 ^= 1u; }
                    }
                    if (!ok) break;
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait_cluster(bar_accempty + 8, ph ^ 1))) { ok = false; break; }
                    tc_fence_after();
                    for (int kb = 0; kb < P; ++kb) {   // tile 1 for the same stages, then release them
                        const uint64_t d0 = smem_desc_sw128(sb + L::X_OFF + s * L::XBYTES);
                        const uint32_t a0 = tbase + L::A_COL + 64 * ar;
#pragma unroll
                        for (int j = 0; j < BK / 16; ++j)
                            mma_ts_pair_e(dcol + BN, a0 + 8 * j,
                                        d0 + (uint64_t)((L::XTILE + (j >> 2) * L::XBOX + (j & 3) * 32) >> 4), idesc,
                                        j == 0 ? (uint32_t)(kb != 0) : 1u, e);
                        mma_commit_pair_e(bar_empty + 8 * s, 0x3, e);
                        mma_commit_pair_e(bar_aempty + 8 * ar, 0x3, e);
                        if (++s == NST) { s = 0; sph ^= 1u; }
                        if (++ar == NA) { ar = 0; aph ^= 1u; }
                    }
                    kb0 = P;
                }
                for (int kb = kb0; kb < nkb; ++kb) {
                    const int a = res ? kb : ar;
                    // resident weights: both CTAs' stages s have landed (our
                    // copies, and the peer's as relayed by its warp 1)
                    if (res && !__all_sync(0xFFFFFFFFu, mbar_wait_cluster(bar_full + 8 * s, sph))) {
                        ok = false;
                        break;
                    }
                    // both CTAs' converters have widened stage a, which they
                    // only do once their own TMA stage s has landed
                    if (fl && !__all_sync(0xFFFFFFFFu, mbar_wait_cluster(bar_afull + 8 * a, res ? (nfill & 1) : aph))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors: the stage's base plus constant offsets (the
                    // start-address field cannot carry: shared memory < 256 KB)
                    const uint64_t d0 = smem_desc_sw128(sb + L::X_OFF + s * L::XBYTES);
                    const uint32_t a0 = tbase + L::A_COL + 64 * a;
                    const uint32_t acc0 = kb != 0;
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j)
#pragma unroll
                        for (int tt = 0; tt < TPA; ++tt)
                            mma_ts_pair_e(dcol + tt * BN, a0 + 8 * j,
                                        d0 + (uint64_t)((tt * L::XTILE + (j >> 2) * L::XBOX + (j & 3) * 32) >> 4),
                                        idesc, j == 0 ? acc0 : 1u, e);
                    mma_commit_pair_e(bar_empty + 8 * s, 0x3, e);
                    if (last_use) mma_commit_pair_e(bar_aempty + 8 * a, 0x3, e);
                    if (++s == NST) { s = 0; sph ^= 1u; }
                    if (!res && ++ar == NA) { ar = 0; aph ^= 1u; }
                }
                if (fl) ++nfill;
                if (ok) mma_commit_pair_e(bar_accfull + 8 * b, 0x3, e);
            }
            // every MMA issued above has completed once this fires
            mma_commit_pair_e(bar_done, 0x1, e);
            mbar_wait(bar_done, 0, 20000000ull);
        } else if (res) {
            // the peer's relay: each of its stages has landed
            const uint32_t e = elect_one();
            int kbg = 0;
            for (int i = 0; i < ucnt && ok; ++i)
                for (int kb = 0; kb < nkb; ++kb, ++kbg) {
                    const int s = kbg % NST;
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_full + 8 * s, (kbg / NST) & 1))) {
                        ok = false;
                        break;
                    }
                    if (e) mbar_arrive_cluster_relaxed(full_ldr + 8 * s);
                }
        }
    } else if (warp < 10) {
        // -------------------------------- widen int8 -> bf16 into TMEM (A)
        const int q = warp & 3;                        // TMEM lane quadrant
        const int h = (warp - 2) >> 2;                 // which 64 of the 128 K columns (TMA box)
        const int row = 32 * q + lane;                 // TMEM lane = row of the MMA tile
        // gated: each lane quadrant holds 16 gate rows (lanes 0-15) and the
        // same 16 features' up rows (lanes 16-31), so that one epilogue warp
        // has both halves of its features; srow is the row in the loaded
        // weight tile (gate rows 0-63, up rows 64-127)
        const bool upper = GATED && (lane & 16);
        const int srow = GATED ? (upper ? BM / 2 : 0) + 16 * q + (lane & 15) : row;
        const int frow = GATED ? 16 * q + (lane & 15) : row;    // feature offset in the tile
        const uint32_t tl = (uint32_t)(32 * q) << 16;
        int kbg = 0, nfill = 0;
        const bool helper = helpers && h == 0;         // warps 2-5 also drain (see gated_drain)
        const uint32_t hstg = sb + L::HSTG_OFF + (uint32_t)((warp - 2) & 3) * 4096u;
        int hslot = 0;
        // two-tile units: warps 2-5 drain part of each unit's second tile (see help2_drain)
        const bool helper2 = L::HELP2 && h == 0;
        const uint32_t hstg2 = sb + L::HSTG_OFF + (uint32_t)((warp - 2) & 3) * 2048u;
        for (int i = 0; i < ucnt && ok; ++i) {
            if (!fills(i)) {                            // resident weights: nothing to widen
                kbg += nkb;
                if (helper) ok = gated_drain(i, 2, 4, hstg, hslot);
                continue;
            }
            const int u = unit_at(i);
            // the 32-element block formats: this row's f16 block scales (the
            // item is uniform over the warp: a warp's 32 rows share it)
            const uint16_t *bsr = nullptr;
            const float *colp = nullptr;              // q8_2f: the column field (all rows)
            bool blk = false;
            {
                const TileCoord tc = tile_coord<GATED>(p, u, rank);
                const int o = tc.o0 + frow;
                const uint16_t *b = upper ? p.it[tc.zi].bsc2 : p.it[tc.zi].bsc;
                colp = upper ? p.it[tc.zi].col2 : p.it[tc.zi].col;
                blk = b != nullptr;
                if (blk && o < p.it[tc.zi].n) bsr = b + (long long)o * p.kb32;
            }
            for (int kb = 0; kb < nkb; ++kb, ++kbg) {
                // two-tile units: the previous unit's second tile, once this
                // unit's leading stages are widened (the first tile's MMAs
                // take them while its second tile drains); the next stage's
                // A slot is only released after that drain
                if (helper2 && i > 0 && kb == (NA < nkb ? NA : nkb)) {
                    ok = help2_drain(i - 1, hstg2, hslot);
                    if (!ok) break;
                }
                const int s = kbg % NST, a = res ? kb : kbg % NA;
                // blocks 4 kb + 2 h and the next one (issued before the waits)
                uint32_t dd = 0;
                const int j0 = kb * 4 + h * 2;
                if (bsr && j0 < p.kb32) dd = *reinterpret_cast<const uint32_t *>(bsr + j0);
                const uint32_t apar = res ? (nfill & 1) ^ 1 : ((kbg / NA) & 1) ^ 1;
                // A stage a free first: then the MMAs of chunk kbg - nkb (resident
                // weights) or kbg - NA are done, so the ring has passed the
                // previous use of this chunk's slot and the parity wait on its
                // full barrier cannot match a phase two behind (the converters
                // skip the units that widen nothing)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_aempty + 8 * a, apar) &&
                                                 mbar_wait(bar_full + 8 * s, (kbg / NST) & 1));
                if (!ok) break;
                tc_fence_after();
                const uint8_t *wrow = smem + L::W_OFF + s * L::WBYTES + h * L::WBOX + srow * 64;
                const int sw = (srow >> 1) & 3;
                uint32_t r[32];
                if (colp) {
                    // column field of K = kb*128 + h*64 + 16c + e, staged with the
                    // weight tile (zero past k: the weight reads zeros there too)
                    const int k0 = kb * BK + h * BOX;
                    const float *cs = reinterpret_cast<const float *>(smem + L::COL_OFF + s * L::COL_BYTES) +
                                      (upper ? BK : 0) + h * BOX;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(wrow + ((c ^ sw) << 4));
                        float4 cv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            cv[e] = k0 + 16 * c + 4 * e < p.k
                                        ? *reinterpret_cast<const float4 *>(cs + 16 * c + 4 * e)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                        widen4_col(v.x, cv[0], r[8 * c + 0], r[8 * c + 1]);
                        widen4_col(v.y, cv[1], r[8 * c + 2], r[8 * c + 3]);
                        widen4_col(v.z, cv[2], r[8 * c + 4], r[8 * c + 5]);
                        widen4_col(v.w, cv[3], r[8 * c + 6], r[8 * c + 7]);
                    }
                } else if (blk) {
                    const float d2[2] = {__half2float(__ushort_as_half((unsigned short)(dd & 0xFFFFu))),
                                         __half2float(__ushort_as_half((unsigned short)(dd >> 16)))};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {       // chunks 0-1: block j0, 2-3: block j0 + 1
                        const uint4 v = *reinterpret_cast<const uint4 *>(wrow + ((c ^ sw) << 4));
                        const float d = d2[c >> 1];
                        widen4_scaled(v.x, d, r[8 * c + 0], r[8 * c + 1]);
                        widen4_scaled(v.y, d, r[8 * c + 2], r[8 * c + 3]);
                        widen4_scaled(v.z, d, r[8 * c + 4], r[8 * c + 5]);
                        widen4_scaled(v.w, d, r[8 * c + 6], r[8 * c + 7]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(wrow + ((c ^ sw) << 4));
                        widen4(v.x, r[8 * c + 0], r[8 * c + 1]);
                        widen4(v.y, r[8 * c + 2], r[8 * c + 3]);
                        widen4(v.z, r[8 * c + 4], r[8 * c + 5]);
                        widen4(v.w, r[8 * c + 6], r[8 * c + 7]);
                    }
                }
                tmem_st32(tbase + tl + L::A_COL + 64 * a + 32 * h, r);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(afull_ldr + 8 * a);
            }
            ++nfill;
            if (helper && ok) ok = gated_drain(i, 2, 4, hstg, hslot);
            if (helper2 && ok && i > 0 && nkb <= NA) ok = help2_drain(i - 1, hstg2, hslot);
        }
        if (helper2 && ok && ucnt > 0) ok = help2_drain(ucnt - 1, hstg2, hslot);
        if (helper || helper2) {
            // the stores must be complete before the CTA's shared memory goes away
            bulk_wait_all();
            __syncwarp();
        }
    } else {
        // ----------------------------------------------------------- epilogue
        // Lane = output feature: each 32 (features) x 32 (tokens) block is
        // scaled in registers, written to a staging tile in the output's own
        // layout (token rows, features contiguous) and sent out with one TMA
        // tensor store - or a TMA reduce-add when the residual is y itself.
        const int q = warp & 3;
        const int row = 32 * q + lane;
        // gated: lanes 0-15 hold the gate rows and lanes 16-31 the up rows of
        // the warp's 16 features (the converters' interleaved layout)
        const bool upper = GATED && (lane & 16);
        const int frow = GATED ? 16 * q + (lane & 15) : row;
        const uint32_t tl = (uint32_t)(32 * q) << 16;
        int lt = 0;
        // this warp's staging (a shared-memory address): a ring of output
        // blocks (gated 32 tokens x 16 features bf16, 1 KB; else 32 x 32, f32
        // 4 KB or bf16 2 KB) in two halves.  A token tile's blocks go out in
        // chunks of half the ring: each chunk is written, made visible to the
        // async proxy by one fence, and sent by one TMA store a block (one
        // bulk group a chunk; gated, one a store); the next chunk takes the
        // other half once the groups before the previous chunk have finished
        // reading.  One fence a chunk instead of one a block is what keeps the
        // short-K GEMMs' drain short.
        const uint32_t stg = sb + L::STG_OFF + (warp - 10) * L::STG_WARP;
        int half = 0, slot_bytes = 0;   // the next chunk's half, the ring's block size
        // gated: the ring position (blocks so far)
        int gslot = 0;
        if (helpers) {
            // blocks 0-1 of each token tile here, 2-3 by converter warps 2-5
            int hs = 0;
            for (; lt < ucnt && ok; ++lt) ok = gated_drain(lt, 0, 2, stg, hs);
        }
        for (; lt < ucnt && ok; ++lt) {
            const int u = unit_at(lt);
            const int b = TPA == 2 ? 0 : (lt & 1);
            const uint32_t ph = TPA == 2 ? (lt & 1) : ((lt >> 1) & 1);
            // this tile's row scale and bias before the wait: their load
            // latency overlaps the mainloop
            const TileCoord tc = tile_coord<GATED>(p, u, rank);
            const int o = tc.o0 + frow;
            const bool ov = o < p.it[tc.zi].n;
            const float *scale = upper ? p.it[tc.zi].scale2 : p.it[tc.zi].scale;
            const float *bias = upper ? p.it[tc.zi].bias2 : p.it[tc.zi].bias;
            const float sc = ov ? (scale ? scale[o] : 1.f) : 0.f;
            const float bi = (ov && bias) ? bias[o] : 0.f;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_accfull + 8 * b, ph));
            if (!ok) break;
            tc_fence_after();
            const int act = p.it[tc.zi].act;
            const int n = p.it[tc.zi].n;
            const void *ymap = &p.ty[tc.zi];
            const long long ldr = p.it[tc.zi].ldr;
            const bool f32out = p.it[tc.zi].ydt == TE_F32;
            const float *__restrict__ rbase = p.it[tc.zi].resid;
            const bool inplace = rbase != nullptr && rbase == p.it[tc.zi].y;
            // Drains blocks [0, cn) of one token tile (accumulator column acol,
            // tokens t0..) in chunks; the block size is a compile-time
            // constant of each output form (BYTES: 1024 gated, 4096 staged
            // f32, 2048 bf16), so a chunk's blocks unroll.  Items of one launch
            // may differ in block size: a change of size first lets every
            // store finish reading.
            auto drain_tile = [&](auto bytes_c, int acol, int t0, int cn, int fo) {
                constexpr int BYTES = decltype(bytes_c)::value;
                constexpr int NB = L::STG_WARP / BYTES;
                constexpr int BSZ = NB >= 2 ? NB / 2 : 1;       // blocks a chunk
                for (int c0 = 0; c0 < cn; c0 += BSZ) {
                    const bool resize = BYTES != slot_bytes;
                    if (resize) {
                        half = 0;
                        slot_bytes = BYTES;
                    }
                    // lane i stores block i of each chunk, one bulk group a
                    // chunk (empty when the chunk is short)
                    if (resize) bulk_wait_read_n<0>();   // every lane: earlier sizes' stores too
                    else if (lane < BSZ) {
                        if (NB < 2) bulk_wait_read_n<0>();
                        else bulk_wait_read_n<1>();
                    }
                    __syncwarp();
                    const uint32_t base = stg + (uint32_t)(half * (NB / 2) * BYTES);
                    if (NB >= 2) half ^= 1;
#pragma unroll
                    for (int i = 0; i < BSZ; ++i) {
                        const int c = c0 + i;
                        if (c >= cn) break;                         // warp-uniform
                        const uint32_t so = base + (uint32_t)(i * BYTES);
                        uint32_t v[32];
                        tmem_ld32(tbase + tl + acol + 32 * c, v);
                        tmem_wait_ld();
                        {
                            // v[] becomes the output values in place (f32 bits)
                            // s*acc + b in f32 pairs (two tokens an instruction)
                            {
                                const uint64_t sc2 = f2_pack(sc, sc), bi2 = f2_pack(bi, bi);
#pragma unroll
                                for (int j = 0; j < 32; j += 2) {
                                    float a, b2;
                                    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), sc2, bi2),
                                              a, b2);
                                    v[j] = __float_as_uint(a);
                                    v[j + 1] = __float_as_uint(b2);
                                }
                            }
                            if (act) {   // the ungated MLP: act(bf16(s*acc + b)), no residual
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    v[j] = __float_as_uint(apply_act_tanh(round_bf16(__uint_as_float(v[j])), act - 1));
                            }
                            if constexpr (BYTES == 4096) {
                                float *ostg_f = reinterpret_cast<float *>(smem + (so - sb));
#pragma unroll
                                for (int j = 0; j < 32; ++j) ostg_f[j * 32 + lane] = __uint_as_float(v[j]);
                                if (rbase && !inplace) {
                                    // a residual other than y (not used by the
                                    // block): added to the f32 staging from
                                    // global memory, then narrowed in place if
                                    // y is bf16.  Row j's bf16 bytes only cover
                                    // f32 rows <= j, which were read before.
                                    __syncwarp();
                                    const int tb = t0 + 32 * c;
                                    const float *rr = rbase + (long long)tb * ldr + o;
                                    const int jn = p.m - tb < 32 ? p.m - tb : 32;
#pragma unroll 1
                                    for (int j = 0; j < jn; ++j)
                                        if (ov) ostg_f[j * 32 + lane] += rr[(long long)j * ldr];
                                    if (!f32out) {
                                        uint16_t *ostg_h = reinterpret_cast<uint16_t *>(smem + (so - sb));
#pragma unroll 1
                                        for (int j = 0; j < 32; ++j) {
                                            __syncwarp();
                                            const float y = ostg_f[j * 32 + lane];
                                            __syncwarp();
                                            ostg_h[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
                                        }
                                    }
                                }
                            } else {
                                uint16_t *ostg_h = reinterpret_cast<uint16_t *>(smem + (so - sb));
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    ostg_h[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
                            }
                        }
                    }
                    // the chunk's writes, visible to the TMA engine, then its stores
                    fence_async_smem();
                    __syncwarp();
                    if (lane < BSZ) {
                        if (c0 + lane < cn) {
                            const uint32_t so = base + (uint32_t)(lane * BYTES);
                            if (!GATED && inplace)
                                tma_reduce_add_2d(ymap, so, fo, t0 + 32 * (c0 + lane));
                            else
                                tma_store_2d(ymap, so, fo, t0 + 32 * (c0 + lane));
                        }
                        bulk_commit();
                    }
                }
            };
            // f32 outputs where a warp's staging ring holds only one 32-token
            // block (4 KB): 16-token halves (2 KB; the f32 maps' box is 16
            // rows there), double-buffered, so that one half's store reads
            // while the next half is written (a whole block would wait for
            // its predecessor's store every time)
            auto drain_f32_halves = [&](int acol, int t0, int cn, int fo) {
                constexpr int HB = 2048;
                const uint64_t sc2 = f2_pack(sc, sc), bi2 = f2_pack(bi, bi);
                auto half_out = [&](const uint32_t (&v)[32], int h, int tb) {
                    const bool resize = slot_bytes != HB + 1;   // HB + 1: this form's mark
                    if (resize) {
                        half = 0;
                        slot_bytes = HB + 1;
                        bulk_wait_read_n<0>();                   // every lane: other forms' stores
                    } else if (lane == 0) {
                        bulk_wait_read_n<1>();                   // the other half may still be read
                    }
                    __syncwarp();
                    const uint32_t so = stg + (uint32_t)(half * HB);
                    half ^= 1;
                    float *ostg = reinterpret_cast<float *>(smem + (so - sb));
#pragma unroll
                    for (int j = 0; j < 16; ++j) ostg[j * 32 + lane] = __uint_as_float(v[16 * h + j]);
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (inplace)
                            tma_reduce_add_2d(ymap, so, fo, tb);
                        else
                            tma_store_2d(ymap, so, fo, tb);
                        bulk_commit();
                    }
                };
                for (int c = 0; c < cn; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tbase + tl + acol + 32 * c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        float a, b2;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), sc2, bi2), a,
                                  b2);
                        v[j] = __float_as_uint(a);
                        v[j + 1] = __float_as_uint(b2);
                    }
                    if (act) {   // the ungated MLP with an f32 output: act(bf16(s*acc + b))
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            v[j] = __float_as_uint(apply_act_tanh(round_bf16(__uint_as_float(v[j])), act - 1));
                    }
                    const int tb = t0 + 32 * c;
                    half_out(v, 0, tb);
                    if (tb + 16 < p.m) half_out(v, 1, tb + 16);
                }
            };
            for (int tt = 0; tt < TPA; ++tt) {
            const int acol = (TPA == 2 ? tt : b) * BN;     // this token tile's accumulator
            const int t0 = (tc.t0 * TPA + tt) * BN;
            // the token tile's 32-token blocks (the last may be partial; a
            // second tile past m has none); a two-tile unit's second tile is
            // drained by converter warps 2-5 (see e_blocks2)
            const int cn0 = t0 >= p.m ? 0 : ((p.m - t0 + 31) / 32 < BN / 32 ? (p.m - t0 + 31) / 32 : BN / 32);
            const int cn = L::HELP2 && tt == 1 ? e_blocks2(tc.zi, cn0) : cn0;
            // this warp's first output feature: a warp whose features all lie
            // past n (a phantom tile) has nothing to drain
            const int fo = tc.o0 + (GATED ? 16 : 32) * q;
            if (fo < n) {
                if constexpr (GATED) {
                    // 1 KB blocks in chunks of half the ring (the whole token
                    // tile where the ring holds two), one bulk group a store.
                    // Before a chunk, all but the previous chunk's GBSZ groups
                    // have finished reading - after a chunk of fewer stores
                    // (a ragged last tile), all of them.
                    // one 32-token block: scale and bias, both halves rounded
                    // to bf16 (one conversion for the pair); gate lane l and up
                    // lane l + 16 swap half their tokens, so that lane l
                    // computes m = act(g) * u for tokens 0-15 and lane l + 16
                    // for tokens 16-31 of feature 16 q + l; the arithmetic in
                    // f32 pairs (two tokens an instruction, each rounded as
                    // the scalar form), the tanh one token at a time
                    auto gated_math = [&](auto act_c, const uint32_t (&v)[32], float (&yv)[16]) {
                        constexpr int ACT = decltype(act_c)::value;
                        const uint64_t sc2 = f2_pack(sc, sc), bi2 = f2_pack(bi, bi);
                        const uint64_t half2 = f2_pack(0.5f, 0.5f);
                        float gv[16], uv[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            float lo, hi;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[16 + j])), sc2, bi2),
                                      lo, hi);
                            const uint32_t b2 = pack_bf16x2(lo, hi);
                            lo = bf16_lo(b2);
                            hi = bf16_hi(b2);
                            // the gate lane sends its token 16 + j, the up lane its token j
                            const float got = __shfl_xor_sync(0xFFFFFFFFu, upper ? lo : hi, 16);
                            // operands selected first: one activation per lane, no branch
                            gv[j] = upper ? got : lo;
                            uv[j] = upper ? hi : got;
                        }
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            const uint64_t g2 = f2_pack(gv[j], gv[j + 1]);
                            // GELU-tanh: z = g (0.79788456 + 0.035677408 g^2); SiLU: z = g / 2
                            uint64_t z2;
                            if constexpr (ACT == TE_ACT_GELU_TANH)
                                z2 = f2_mul(g2, f2_fma(f2_pack(0.035677408f, 0.035677408f), f2_mul(g2, g2),
                                                       f2_pack(0.79788456f, 0.79788456f)));
                            else
                                z2 = f2_mul(half2, g2);
                            float z0, z1;
                            f2_unpack(z2, z0, z1);
                            const uint64_t h2 = f2_mul(half2, g2);
                            const uint64_t a2 = f2_fma(h2, f2_pack(hw_tanh(z0), hw_tanh(z1)), h2);
                            f2_unpack(f2_mul(a2, f2_pack(uv[j], uv[j + 1])), yv[j], yv[j + 1]);
                        }
                    };
                    constexpr int GNB = L::STG_WARP / 1024;
                    constexpr int GBSZ = GNB / 2 < BN / 32 ? GNB / 2 : BN / 32;
                    static_assert(GBSZ == 2 || GBSZ == 4, "a ring of 2 GBSZ blocks indexed by a mask");
                    const int jb = upper ? 16 : 0;
                    for (int c0 = 0; c0 < cn; c0 += GBSZ) {
                        const int ce = c0 + GBSZ < cn ? c0 + GBSZ : cn;
                        // lane i stores block i of each chunk, one bulk group
                        // a chunk (empty when the chunk is short): its group
                        // of the chunk before the previous, which used this
                        // half of the ring, has finished reading
                        if (lane < GBSZ) bulk_wait_read_n<1>();
                        __syncwarp();
                        for (int c = c0; c < ce; ++c) {
                            uint32_t v[32];
                            tmem_ld32(tbase + tl + acol + 32 * c, v);
                            tmem_wait_ld();
                            float yv[16];
                            if (act == TE_ACT_GELU_TANH)
                                gated_math(std::integral_constant<int, TE_ACT_GELU_TANH>{}, v, yv);
                            else
                                gated_math(std::integral_constant<int, TE_ACT_SILU>{}, v, yv);
                            const uint32_t so = stg + (uint32_t)(((gslot + c) & (2 * GBSZ - 1)) * 1024);
                            uint16_t *ostg_h = reinterpret_cast<uint16_t *>(smem + (so - sb));
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                ostg_h[(jb + j) * 16 + (lane & 15)] = __bfloat16_as_ushort(__float2bfloat16_rn(yv[j]));
                        }
                        fence_async_smem();
                        __syncwarp();
                        if (lane < GBSZ) {
                            const int c = c0 + lane;
                            if (c < ce)
                                tma_store_2d(ymap, stg + (uint32_t)(((gslot + c) & (2 * GBSZ - 1)) * 1024), fo,
                                             t0 + 32 * c);
                            bulk_commit();
                        }
                    }
                    // chunk k of the tile used ring blocks gslot + k GBSZ + i
                    gslot += (cn + GBSZ - 1) / GBSZ * GBSZ;
                } else if (f32out || (rbase && !inplace)) {   // a residual other than y is added in f32
                    if (L::STG_WARP == 4096 && !(rbase && !inplace))
                        drain_f32_halves(acol, t0, cn, fo);
                    else
                        drain_tile(std::integral_constant<int, 4096>{}, acol, t0, cn, fo);
                } else {
                    drain_tile(std::integral_constant<int, 2048>{}, acol, t0, cn, fo);
                }
            }
            if (TPA == 2) {
                // this token tile's accumulator may take the next unit's MMAs
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(accempty_ldr + 8 * tt);
            }
            }
            if (TPA == 1) {
                // this accumulator may take the next tile's MMAs
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(accempty_ldr + 8 * b);
            }
        }
        // the stores must be complete before the CTA's shared memory goes away
        // (each storing lane waits for its own bulk groups)
        bulk_wait_all();
        __syncwarp();
    }
    if (!ok && s_skip == 0) atomicExch(&g_gemm_err, 1);
    tc_fence_before();
    __syncthreads();
    // the leader's MMAs write both CTAs' TMEM: both wait for them before freeing it
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tbase, L::TMEM_COLS);
    }
    // the peer may still arrive on our barriers until it is done too
    cluster_sync();
}

// ---------------------------------------------------------- MMA ceiling
// The 2-SM MMA of q8_gemm_kernel (kind::f16, A in TMEM, B in shared memory in
// the activation stage's layout, M = 256, N = BN, K = 16) issued back to back
// by the converged leader warp, 8 a stage as in the GEMM's main loop, with no
// loads, no waits and no epilogue: the rate this pipeline reaches when its
// operands are always ready.  The operands' values do not matter (B zeros, A
// whatever TMEM holds); only the time is read.
template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1) mma_peak_kernel(int stages) {
    constexpr int XBOX = BN / 2 * BOX * 2;        // one 64-wide box of this CTA's token half
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar_done = sb + 2 * XBOX;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + 2 * XBOX + 8);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 2 * XBOX / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(bar_done, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc_pair(smem_u32(tmem_slot), 512);
    fence_async_smem();        // the zeros, visible to the tensor core
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    if (cluster_rank() == 0 && warp == 0) {
        const uint32_t e = elect_one();
        constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
        const uint64_t d0 = smem_desc_sw128(sb);
        const uint32_t a0 = tbase + 256;          // one A stage after the accumulator (BN <= 256)
        for (int st = 0; st < stages; ++st) {
#pragma unroll
            for (int j = 0; j < BK / 16; ++j)
                mma_ts_pair_e(tbase, a0 + 8 * j, d0 + (uint64_t)(((j >> 2) * XBOX + (j & 3) * 32) >> 4), idesc,
                              (st | j) != 0, e);
        }
        mma_commit_pair_e(bar_done, 0x3, e);
    }
    // both CTAs: the leader's MMAs, which write both CTAs' TMEM, are done
    if (!mbar_wait(bar_done, 0) && threadIdx.x == 0) atomicExch(&g_gemm_err, 1);
    tc_fence_before();
    cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tbase, 512);
    }
}

int sm_count();

template <int BN>
te_status mma_peak_launch(int stages, float *ms, cudaStream_t stream) {
    constexpr int smem = 2 * (BN / 2 * BOX * 2) + 16 + 1024;
    const int clusters = sm_count() / 2;
    cudaEvent_t e0, e1;
    cudaError_t e = cudaEventCreate(&e0);
    if (e != cudaSuccess) return cuda_fail(e, "mma_peak: event");
    e = cudaEventCreate(&e1);
    if (e != cudaSuccess) {
        cudaEventDestroy(e0);
        return cuda_fail(e, "mma_peak: event");
    }
    e = cudaEventRecord(e0, stream);
    if (e == cudaSuccess) {
        mma_peak_kernel<BN><<<2 * clusters, 128, smem, stream>>>(stages);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaEventRecord(e1, stream);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return e == cudaSuccess ? TE_OK : cuda_fail(e, "mma_peak");
}

// ------------------------------------------------------------------ host side

int sm_count() {
    static int count[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!count[dev]) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c < 1)
            c = 148;
        count[dev] = c;
    }
    return count[dev];
}

// Long K (re-widened weights): the token-tile width and the token tiles per
// unit.  With two tiles a unit each widened weight stage feeds the MMAs of both,
// which halves the TMEM stores of the widened operand per flop (those stores
// contend with the MMAs for TMEM), at the price of an accumulator drain that
// is only partly overlapped.  The choice minimises the busiest cluster's time:
// whole waves of units times a unit's relative cost - a 192 x 2 unit takes
// about 1.65x a 192 x 1 unit (measured at K = 3840 and 10240; it loses at
// K <= 2048), a 128 x 2 unit about 1.4x (measured 1.33-1.48 at K = 2048 to
// 10240; at K = 768 the drain outweighs it).  The 128 x 2 unit pays where it
// saves a whole wave: the DiT out and down projections (2112 tokens: 62.0 ->
// 57.6 and 151.5 -> 134.3 us), the text stack's down projection.
struct LongKTile { int bn, tpa; };
constexpr double COST_128X2 = 1.4;
LongKTile long_k_tile(int m, int k, int ftiles) {
    const int clusters = sm_count() / 2;
    const long long fpairs = (ftiles + 1) / 2;
    auto t = [&](int tokens, double cost) {
        const long long units = fpairs * ((m + tokens - 1) / tokens);
        return (double)((units + clusters - 1) / clusters) * cost;
    };
    LongKTile best = {192, 1};
    double tb = t(192, 1.0);
    if (k >= 3072 && t(384, 1.65) < tb) { best = {192, 2}; tb = t(384, 1.65); }
    if (k >= 2048 && t(256, COST_128X2) < tb) best = {128, 2};
    return best;
}

// Token-tile width and whether the weights stay resident (every K stage in
// the TMEM A stages at once: K <= 256 at BN = 192, K <= 512 at 128 and 64).
// For 256 < K <= 512 the 128-wide tile with resident weights beats the
// 192-wide one that re-widens each stage for every token tile.
int pick_bn(int m, int k, int &res) {
    int bn = m >= 1024 ? 192 : (m > 64 ? 128 : 64);
    const int nkb = (k + BK - 1) / BK;
    if (bn == 192 && nkb > Layout<192, 1>::NA && nkb <= Layout<128, 1>::NA) bn = 128;
    const int na = bn == 192 ? Layout<192, 1>::NA : (bn == 128 ? Layout<128, 1>::NA : Layout<64, 1>::NA);
    res = nkb <= na ? 1 : 0;
    return bn;
}

// One launch's tile: width, token tiles a unit, resident weights.
struct TilePlan {
    int bn, tpa, res;
};
TilePlan tile_for(int m, int k, int ftiles) {
    TilePlan t;
    t.tpa = 1;
    t.bn = pick_bn(m, k, t.res);
    if (t.bn == 192 && !t.res) {
        const LongKTile lt = long_k_tile(m, k, ftiles);
        t.bn = lt.bn;
        t.tpa = lt.tpa;
    }
    return t;
}
double unit_cost(const TilePlan &t) {
    return t.tpa == 1 ? 1.0 : (t.bn == 192 ? 1.65 : COST_128X2);
}
double plan_time(int m, int ftiles, const TilePlan &t) {
    const int clusters = sm_count() / 2;
    const long long units = (long long)((ftiles + 1) / 2) * ((m + t.bn * t.tpa - 1) / (t.bn * t.tpa));
    return (double)((units + clusters - 1) / clusters) * unit_cost(t);
}

// The tile of a split's second launch: the fastest by the model among the
// long-K tiles (a one-tile unit costs about the same at 128 or 192 tokens: the
// per-stage cost does not depend on the width).
TilePlan tail_tile(int m, int k, int ftiles) {
    TilePlan best = tile_for(m, k, ftiles);
    if (best.res) return best;
    const TilePlan cands[4] = {{192, 1, 0}, {128, 1, 0}, {192, 2, 0}, {128, 2, 0}};
    double tb = plan_time(m, ftiles, best);
    for (const TilePlan &c : cands) {
        if ((c.tpa == 2 && c.bn == 192 && k < 3072) || (c.tpa == 2 && c.bn == 128 && k < 2048)) continue;
        const double tc = plan_time(m, ftiles, c);
        if (tc < tb) { best = c; tb = tc; }
    }
    return best;
}

// Long K with two 192-token tiles a unit: the last wave of units is often
// only partly filled (the DiT out and down projections at 8448 tokens: 330
// units on 76 clusters, 4.3 waves).  Splitting the rows into whole waves of
// the wide unit and one more launch for the rest, on narrower units, finishes
// sooner when the model says so (a launch costs about a tenth of a unit).
// Measured: c5 down 1633 -> 1774 and out 1532 -> 1570 TFLOP/s, DiT block
// q|k|v 1545 -> 1587; splits of 128 x 2 units (DiT block out and down, text
// stack down) measured slower, so they are not made.
// Returns the rows of the first launch, or m (no split).
int split_rows(int m, int k, int ftiles, const TilePlan &t) {
    if (t.res || t.tpa != 2 || t.bn != 192) return m;
    const int clusters = sm_count() / 2;
    const int fpairs = (ftiles + 1) / 2;
    const int per = t.bn * t.tpa;
    const long long units = (long long)fpairs * ((m + per - 1) / per);
    const long long waves = units / clusters;
    if (waves < 1) return m;
    const int k1 = (int)(waves * clusters / fpairs);   // token tiles of the whole waves
    const int m1 = k1 * per;
    if (k1 < 1 || m1 >= m) return m;
    const TilePlan t2 = tail_tile(m - m1, k, ftiles);
    const double split = plan_time(m1, ftiles, t) + plan_time(m - m1, ftiles, t2) + 0.1;
    return split < plan_time(m, ftiles, t) ? m1 : m;
}

template <int BN, bool GATED, int TPA>
te_status launch(Params &p, int ftiles, cudaStream_t stream) {
    const int smem = Layout<BN, TPA>::BYTES + 1024;
    // per instantiation and device: dynamic shared memory size, and how many
    // 2-CTA clusters can be resident at once (the persistent grid's size)
    static int max_clusters[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "q8_linear: cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(TE_EINVAL, "q8_linear: device %d out of range", dev);
    if (!max_clusters[dev]) {
        e = cudaFuncSetAttribute(q8_gemm_kernel<BN, GATED, TPA>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, "q8_linear: set shared memory size");
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * sm_count(), 1, 1);
        cfg.blockDim = dim3(NTHREADS, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, q8_gemm_kernel<BN, GATED, TPA>, &cfg);
        if (e != cudaSuccess || n < 1) n = sm_count() / 2;
        max_clusters[dev] = n;
    }
    p.ttiles = (p.m + TPA * BN - 1) / (TPA * BN);
    p.fpairs = (ftiles + 1) / 2;
    p.nunits = p.ttiles * p.fpairs;
    // token tiles per group: about XGROUP_BYTES of activation rows (resident
    // weights: one group, so a cluster's run keeps its feature pair)
    const long long xtile = (long long)TPA * BN * p.k * 2;
    const long long tg = p.res ? p.ttiles : XGROUP_BYTES / xtile;
    p.tgroup = tg < 1 ? 1 : (tg > p.ttiles ? p.ttiles : (int)tg);
    const int clusters = p.nunits < max_clusters[dev] ? p.nunits : max_clusters[dev];
    q8_gemm_kernel<BN, GATED, TPA><<<2 * clusters, NTHREADS, smem, stream>>>(p);
    e = cudaGetLastError();
    return e == cudaSuccess ? TE_OK : cuda_fail(e, "q8_linear launch");
}

}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

te_status make_map_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
                      uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                      CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(TE_ECUDA, "q8_linear: cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(TE_ECUDA, "q8_linear: cuTensorMapEncodeTiled failed (%d)", (int)r);
    return TE_OK;
}

int read_clear_gemm_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_err, sizeof(int)) != cudaSuccess) return -1;
    if (v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_gemm_err, &zero, sizeof(int));
    }
    return v;
}

}  // namespace tefwd

using namespace tefwd;

extern "C" te_status te_q8_linear(const void *x, int64_t ldx, int32_t m, int32_t k,
                                  const te_q8_item *items, int32_t z, te_stream stream) {
    if (!x || !items) return fail(TE_EINVAL, "q8_linear: NULL x or items");
    if (z < 1 || z > MAXZ) return fail(TE_ESHAPE, "q8_linear: z=%d (1..4)", z);
    if (m < 0 || k < 64 || k % 64) return fail(TE_ESHAPE, "q8_linear: m=%d k=%d (k %% 64 == 0)", m, k);
    if (ldx < k || ldx % 8) return fail(TE_ESHAPE, "q8_linear: ldx=%lld (>= k, multiple of 8)", (long long)ldx);
    if (!aligned16(x)) return fail(TE_EALIGN, "q8_linear: x not 16-byte aligned");
    Params p;
    memset(&p, 0, sizeof(p));
    p.z = z;
    p.m = m;
    p.k = k;
    p.kb32 = k / 32;
    int ftiles = 0;
    for (int i = 0; i < z; ++i) {
        const te_q8_item &src = items[i];
        if (!src.w.q || !src.y || (!src.w.scale && !src.w.block_scale))
            return fail(TE_EINVAL, "q8_linear: item %d has a NULL q, y or scale (NULL scale needs block scales)", i);
        if (src.w.block_scale && (reinterpret_cast<uintptr_t>(src.w.block_scale) & 3))
            return fail(TE_EALIGN, "q8_linear: item %d: block scales must be 4-byte aligned", i);
        if (src.w.col && src.w.block_scale)
            return fail(TE_EINVAL, "q8_linear: item %d: a column field and block scales together", i);
        if (src.w.col && !aligned16(src.w.col))
            return fail(TE_EALIGN, "q8_linear: item %d: the column field must be 16-byte aligned", i);
        if (src.w.k != k) return fail(TE_ESHAPE, "q8_linear: item %d has k=%d, x has %d", i, src.w.k, k);
        if (src.w.n < 32 || src.w.n % 32)
            return fail(TE_ESHAPE, "q8_linear: item %d n=%d (multiple of 32)", i, src.w.n);
        if (src.y_dtype != TE_F32 && src.y_dtype != TE_BF16)
            return fail(TE_EINVAL, "q8_linear: item %d bad y dtype", i);
        if (src.ldy < src.w.n) return fail(TE_ESHAPE, "q8_linear: item %d ldy < n", i);
        if ((src.ldy * (src.y_dtype == TE_F32 ? 4 : 2)) % 16)
            return fail(TE_EALIGN, "q8_linear: item %d: rows of y must be 16-byte aligned", i);
        if (!aligned16(src.w.q) || !aligned16(src.y) || (reinterpret_cast<uintptr_t>(src.w.scale) & 3) ||
            (src.w.bias && (reinterpret_cast<uintptr_t>(src.w.bias) & 3)))
            return fail(TE_EALIGN, "q8_linear: item %d: q and y must be 16-byte aligned", i);
        if (src.epilogue < TE_EPI_NONE || src.epilogue > TE_EPI_SILU)
            return fail(TE_EINVAL, "q8_linear: item %d bad epilogue %d", i, src.epilogue);
        if (src.epilogue != TE_EPI_NONE && src.residual)
            return fail(TE_EINVAL, "q8_linear: item %d: an epilogue activation takes no residual", i);
        if (src.residual) {
            if (src.ldr < src.w.n) return fail(TE_ESHAPE, "q8_linear: item %d ldr < n", i);
            if (!aligned16(src.residual) || src.ldr % 4)
                return fail(TE_EALIGN, "q8_linear: item %d: residual rows must be 16-byte aligned", i);
            if (src.residual == src.y && (src.ldr != src.ldy || src.y_dtype != TE_F32))
                return fail(TE_EINVAL, "q8_linear: item %d: in-place residual needs f32 y and ldr == ldy", i);
        }
        Item &d = p.it[i];
        d.scale = src.w.scale;
        d.bias = src.w.bias;
        d.bsc = src.w.block_scale;
        d.col = src.w.col;
        d.y = src.y;
        d.resid = src.residual;
        d.ldy = src.ldy;
        d.ldr = src.ldr;
        d.n = src.w.n;
        d.ydt = src.y_dtype;
        d.act = src.epilogue;
        d.tile0 = ftiles;
        d.ntiles = (src.w.n + BM - 1) / BM;
        ftiles += d.ntiles;
    }
    if (m == 0) return TE_OK;
    const TilePlan t1 = tile_for(m, k, ftiles);
    const int m1 = split_rows(m, k, ftiles, t1);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // rows [r0, r0 + mr) with tile t: the maps and item pointers start at row r0
    auto part = [&](int r0, int mr, const TilePlan &t) -> te_status {
        Params q = p;
        q.m = mr;
        q.res = t.res;
        const char *xb = static_cast<const char *>(x) + (size_t)r0 * ldx * 2;
        // each CTA of a cluster pair TMA-loads its own half of the token tile
        te_status st = make_map_2d(&q.tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xb, (uint64_t)k, (uint64_t)mr,
                                   (uint64_t)ldx * 2, BOX, t.bn / 2, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != TE_OK) return st;
        for (int i = 0; i < z; ++i) {
            const bool f32 = items[i].y_dtype == TE_F32;
            Item &d = q.it[i];
            d.y = static_cast<char *>(items[i].y) + (size_t)r0 * items[i].ldy * (f32 ? 4 : 2);
            if (items[i].residual) d.resid = items[i].residual + (size_t)r0 * items[i].ldr;
            st = make_map_2d(&q.tw[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, items[i].w.q, (uint64_t)k,
                             (uint64_t)items[i].w.n, (uint64_t)k, BOX, BM, CU_TENSOR_MAP_SWIZZLE_64B);
            if (st != TE_OK) return st;
            // f32 outputs without a separate residual go out in 16-token halves
            // where a warp's staging holds one 32-token f32 block (every tile
            // but the one-tile units at N <= 128): the kernel's own condition
            const bool halves = f32 && !(t.tpa == 1 && t.bn <= 128) &&
                                !(items[i].residual && items[i].residual != items[i].y);
            st = make_map_2d(&q.ty[i], f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                             d.y, (uint64_t)items[i].w.n, (uint64_t)mr, (uint64_t)items[i].ldy * (f32 ? 4 : 2), 32,
                             halves ? 16 : 32, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st != TE_OK) return st;
        }
        if (t.bn == 192) return t.tpa == 2 ? launch<192, false, 2>(q, ftiles, s) : launch<192, false, 1>(q, ftiles, s);
        if (t.bn == 128) return t.tpa == 2 ? launch<128, false, 2>(q, ftiles, s) : launch<128, false, 1>(q, ftiles, s);
        return launch<64, false, 1>(q, ftiles, s);
    };
    te_status st = part(0, m1, t1);
    if (st == TE_OK && m1 < m) st = part(m1, m - m1, tail_tile(m - m1, k, ftiles));
    return st;
}

extern "C" te_status te_q8_gated_linear(const void *x, int64_t ldx, int32_t m, int32_t k,
                                        const te_q8w *wg, const te_q8w *wu, int32_t act, void *out,
                                        int64_t ldm, te_stream stream) {
    if (!x || !wg || !wu || !out) return fail(TE_EINVAL, "q8_gated_linear: NULL x, wg, wu or out");
    if (act != TE_ACT_GELU_TANH && act != TE_ACT_SILU) return fail(TE_EINVAL, "q8_gated_linear: bad act");
    if (m < 0 || k < 64 || k % 64) return fail(TE_ESHAPE, "q8_gated_linear: m=%d k=%d (k %% 64 == 0)", m, k);
    if (ldx < k || ldx % 8) return fail(TE_ESHAPE, "q8_gated_linear: ldx=%lld (>= k, multiple of 8)", (long long)ldx);
    if (!wg->q || !wu->q || (!wg->scale && !wg->block_scale) || (!wu->scale && !wu->block_scale))
        return fail(TE_EINVAL, "q8_gated_linear: NULL q or scale (NULL scale needs block scales)");
    if ((reinterpret_cast<uintptr_t>(wg->block_scale) & 3) || (reinterpret_cast<uintptr_t>(wu->block_scale) & 3))
        return fail(TE_EALIGN, "q8_gated_linear: block scales must be 4-byte aligned");
    if ((wg->col && wg->block_scale) || (wu->col && wu->block_scale))
        return fail(TE_EINVAL, "q8_gated_linear: a column field and block scales together");
    if ((wg->col && !aligned16(wg->col)) || (wu->col && !aligned16(wu->col)))
        return fail(TE_EALIGN, "q8_gated_linear: the column field must be 16-byte aligned");
    if (wg->k != k || wu->k != k || wg->n != wu->n)
        return fail(TE_ESHAPE, "q8_gated_linear: wg [%d, %d] and wu [%d, %d] must both be [f, %d]", wg->n,
                    wg->k, wu->n, wu->k, k);
    const int f = wg->n;
    if (f < 32 || f % 32) return fail(TE_ESHAPE, "q8_gated_linear: f=%d (multiple of 32)", f);
    if (ldm < f || ldm % 8) return fail(TE_ESHAPE, "q8_gated_linear: ldm=%lld (>= f, multiple of 8)", (long long)ldm);
    if (!aligned16(x) || !aligned16(out) || !aligned16(wg->q) || !aligned16(wu->q) ||
        (reinterpret_cast<uintptr_t>(wg->scale) & 3) || (reinterpret_cast<uintptr_t>(wu->scale) & 3) ||
        (wg->bias && (reinterpret_cast<uintptr_t>(wg->bias) & 3)) ||
        (wu->bias && (reinterpret_cast<uintptr_t>(wu->bias) & 3)))
        return fail(TE_EALIGN, "q8_gated_linear: x, out and q must be 16-byte aligned");
    Params p;
    memset(&p, 0, sizeof(p));
    p.z = 1;
    p.m = m;
    p.k = k;
    p.kb32 = k / 32;
    Item &d = p.it[0];
    d.scale = wg->scale;
    d.bias = wg->bias;
    d.scale2 = wu->scale;
    d.bias2 = wu->bias;
    d.bsc = wg->block_scale;
    d.bsc2 = wu->block_scale;
    d.col = wg->col;
    d.col2 = wu->col;
    d.y = out;
    d.ldy = ldm;
    d.n = f;
    d.ydt = TE_BF16;
    d.act = act;
    d.tile0 = 0;
    d.ntiles = (f + BM / 2 - 1) / (BM / 2);
    if (m == 0) return TE_OK;
    const int ftiles = d.ntiles;
    const TilePlan t1 = tile_for(m, k, ftiles);
    const int m1 = split_rows(m, k, ftiles, t1);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // rows [r0, r0 + mr) with tile t (see te_q8_linear)
    auto part = [&](int r0, int mr, const TilePlan &t) -> te_status {
        Params q = p;
        q.m = mr;
        q.res = t.res;
        const char *xb = static_cast<const char *>(x) + (size_t)r0 * ldx * 2;
        char *ob = static_cast<char *>(out) + (size_t)r0 * ldm * 2;
        q.it[0].y = ob;
        te_status st = make_map_2d(&q.tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xb, (uint64_t)k, (uint64_t)mr,
                                   (uint64_t)ldx * 2, BOX, t.bn / 2, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != TE_OK) return st;
        if ((st = make_map_2d(&q.tw[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, wg->q, (uint64_t)k, (uint64_t)f,
                              (uint64_t)k, BOX, BM / 2, CU_TENSOR_MAP_SWIZZLE_64B)) != TE_OK)
            return st;
        if ((st = make_map_2d(&q.tw[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, wu->q, (uint64_t)k, (uint64_t)f,
                              (uint64_t)k, BOX, BM / 2, CU_TENSOR_MAP_SWIZZLE_64B)) != TE_OK)
            return st;
        // each epilogue warp stores 16 features x 32 tokens of a block
        if ((st = make_map_2d(&q.ty[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ob, (uint64_t)f, (uint64_t)mr,
                              (uint64_t)ldm * 2, 16, 32, CU_TENSOR_MAP_SWIZZLE_NONE)) != TE_OK)
            return st;
        if (t.bn == 192) return t.tpa == 2 ? launch<192, true, 2>(q, ftiles, s) : launch<192, true, 1>(q, ftiles, s);
        if (t.bn == 128) return t.tpa == 2 ? launch<128, true, 2>(q, ftiles, s) : launch<128, true, 1>(q, ftiles, s);
        return launch<64, true, 1>(q, ftiles, s);
    };
    te_status st = part(0, m1, t1);
    if (st == TE_OK && m1 < m) st = part(m1, m - m1, tail_tile(m - m1, k, ftiles));
    return st;
}

extern "C" te_status te_mma_peak(int32_t bn, int32_t stages, float *ms, te_stream stream) {
    if (!ms) return fail(TE_EINVAL, "mma_peak: NULL ms");
    if (stages < 1 || stages > (1 << 22)) return fail(TE_EINVAL, "mma_peak: stages=%d (1..4194304)", stages);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (bn) {
        case 64: return mma_peak_launch<64>(stages, ms, s);
        case 128: return mma_peak_launch<128>(stages, ms, s);
        case 192: return mma_peak_launch<192>(stages, ms, s);
        case 256: return mma_peak_launch<256>(stages, ms, s);
        default: return fail(TE_EINVAL, "mma_peak: bn=%d (64, 128, 192 or 256)", bn);
    }
}
