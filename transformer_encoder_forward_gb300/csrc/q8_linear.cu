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
// GB300 design (not the pages' 64x64x32 simdgroup tiling).  The tile computes
// the TRANSPOSED product Y^T[o, t] = W[o, :] . X[t, :] so that the 128 weight
// rows of a tile sit on the 128 TMEM lanes:
//   * warp 0 (one lane) streams K-slices of 64 with TMA: the bf16 activation
//     tile [BN tokens x 64] into 128-byte-swizzled shared memory (the MMA's B
//     operand) and the int8 weight tile [128 x 64] (64-byte swizzle);
//   * warps 2-5 widen the int8 tile to bf16 in registers (exact: |q| <= 127
//     fits bf16's 8-bit significand) and write it straight into TMEM with
//     tcgen05.st, where it is the MMA's A operand - the widened tile never
//     touches shared memory, leaving shared-memory bandwidth to the B reads;
//   * warp 1 (one lane) issues tcgen05.mma kind::f16 M=128 N=BN K=16 into an
//     f32 TMEM accumulator and releases each stage with tcgen05.commit;
//   * warps 2-5 then read the accumulator with tcgen05.ld: lane = output
//     feature o, so the row scale and bias are per-thread constants and each
//     store instruction writes 32 consecutive features of one token (one
//     128-byte line in f32).
// Every mbarrier wait is bounded (about 200 ms); a timeout sets an error word
// that te_check() reports, and the kernel still frees its TMEM.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace tefwd {
namespace {

constexpr int BM = 128;       // weight rows (output features) per tile = TMEM lanes
constexpr int BK = 64;        // K per pipeline stage
constexpr int NST = 4;        // pipeline stages
constexpr int MAXZ = 4;
constexpr int NTHREADS = 192;

struct Item {
    const float *scale;
    const float *bias;
    void *y;
    const float *resid;
    long long ldy, ldr;
    int n, ydt, tile0, pad;
};

struct Params {
    CUtensorMap tx;           // x: bf16 [m, k]
    CUtensorMap tw[MAXZ];     // q_i: int8 [n_i, k]
    Item it[MAXZ];
    int z, m, k;
};

__device__ int g_gemm_err;

template <int BN>
struct Layout {
    static constexpr int XBYTES = BN * BK * 2;          // activation stage
    static constexpr int WBYTES = BM * BK;              // int8 weight stage
    static constexpr int X_OFF = 0;
    static constexpr int W_OFF = NST * XBYTES;
    static constexpr int BAR_OFF = W_OFF + NST * WBYTES;
    // at most two CTAs per SM may hold TMEM at once (2 x 256 columns): the
    // smallest tile pads its shared memory so that a third cannot start
    static constexpr int USED = BAR_OFF + 8 * (3 * NST + 1) + 16;
    static constexpr int BYTES = (BN <= 64 && USED < 80 * 1024) ? 80 * 1024 : USED;
    static constexpr int TMEM_COLS = (BN + NST * 32 <= 256) ? 256 : 512;
    static_assert(BN + NST * 32 <= TMEM_COLS, "TMEM budget");
};

__device__ __forceinline__ int32_t sx8(uint32_t w, int byte) {
    return (int32_t)(w << (24 - 8 * byte)) >> 24;
}

template <int BN>
__global__ void __launch_bounds__(NTHREADS, 1) q8_gemm_kernel(const __grid_constant__ Params p) {
    using L = Layout<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar_full = sb + L::BAR_OFF;
    const uint32_t bar_afull = bar_full + 8 * NST;
    const uint32_t bar_empty = bar_afull + 8 * NST;
    const uint32_t bar_acc = bar_empty + 8 * NST;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * (3 * NST + 1));

    // once any CTA has given up a wait, the rest skip their work (the call
    // has failed; te_check reports it) instead of timing out one by one
    if (*reinterpret_cast<volatile int *>(&g_gemm_err) != 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ftile = blockIdx.y;
    int zi = 0;
    while (zi + 1 < p.z && ftile >= p.it[zi + 1].tile0) ++zi;
    const Item &it = p.it[zi];
    const int o0 = (ftile - it.tile0) * BM;
    const int t0 = blockIdx.x * BN;
    const int nkb = p.k / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_afull + 8 * s, 128);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_acc, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&p.tx);
            tma_prefetch_desc(&p.tw[zi]);
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % NST;
                const uint32_t ph = (kb / NST) & 1;
                if (!mbar_wait(bar_empty + 8 * s, ph ^ 1)) { ok = false; break; }
                mbar_arrive_expect_tx(bar_full + 8 * s, L::XBYTES + L::WBYTES);
                tma_load_2d(sb + L::X_OFF + s * L::XBYTES, &p.tx, bar_full + 8 * s, kb * BK, t0);
                tma_load_2d(sb + L::W_OFF + s * L::WBYTES, &p.tw[zi], bar_full + 8 * s, kb * BK, o0);
                issued = kb + 1;
            }
            // make sure no copy of ours is still landing when the CTA exits
            for (int kb = issued - NST < 0 ? 0 : issued - NST; kb < issued; ++kb)
                mbar_wait(bar_full + 8 * (kb % NST), (kb / NST) & 1, 20000000ull);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % NST;
                const uint32_t ph = (kb / NST) & 1;
                if (!mbar_wait(bar_full + 8 * s, ph) || !mbar_wait(bar_afull + 8 * s, ph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t xs = sb + L::X_OFF + s * L::XBYTES;
#pragma unroll
                for (int j = 0; j < BK / 16; ++j)
                    mma_ts_bf16(tbase, tbase + BN + 32 * s + 8 * j, smem_desc_sw128(xs + 32 * j),
                                idesc, (kb | j) != 0);
                mma_commit(bar_empty + 8 * s);
            }
            mma_commit(bar_acc);   // fires once every MMA issued above has completed
        }
    } else {
        // ---- widen int8 -> bf16 into TMEM (A operand), then the epilogue
        const int q = warp & 3;                       // TMEM lane quadrant of this warp
        const int row = 32 * q + lane;                // weight row within the tile
        const uint32_t tl = (uint32_t)(32 * q) << 16;
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % NST;
            const uint32_t ph = (kb / NST) & 1;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_full + 8 * s, ph));
            if (!ok) break;
            tc_fence_after();
            const uint8_t *wrow = smem + L::W_OFF + s * L::WBYTES + row * 64;
            uint32_t a[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 v = *reinterpret_cast<const uint4 *>(wrow + ((c ^ ((row >> 1) & 3)) << 4));
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a[c * 8 + e * 2 + 0] = pack_bf16x2((float)sx8(w4[e], 0), (float)sx8(w4[e], 1));
                    a[c * 8 + e * 2 + 1] = pack_bf16x2((float)sx8(w4[e], 2), (float)sx8(w4[e], 3));
                }
            }
            tmem_st32(tbase + tl + BN + 32 * s, a);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar_afull + 8 * s);
        }
        ok = __all_sync(0xFFFFFFFFu, ok && mbar_wait(bar_acc, 0));
        if (ok) {
            tc_fence_after();
            const int o = o0 + row;
            const bool ov = o < it.n;
            const float sc = ov ? it.scale[o] : 0.f;
            const float bi = (ov && it.bias) ? it.bias[o] : 0.f;
            for (int c = 0; c < BN / 32; ++c) {
                if (t0 + 32 * c >= p.m) break;        // warp-uniform
                uint32_t v[32];
                tmem_ld32(tbase + tl + 32 * c, v);
                tmem_wait_ld();
                if (ov) {
#pragma unroll 8
                    for (int j = 0; j < 32; ++j) {
                        const int t = t0 + 32 * c + j;
                        if (t >= p.m) break;
                        float y = __uint_as_float(v[j]) * sc + bi;
                        if (it.resid) y += it.resid[(long long)t * it.ldr + o];
                        if (it.ydt == TE_F32)
                            reinterpret_cast<float *>(it.y)[(long long)t * it.ldy + o] = y;
                        else
                            reinterpret_cast<__nv_bfloat16 *>(it.y)[(long long)t * it.ldy + o] =
                                __float2bfloat16_rn(y);
                    }
                }
                __syncwarp();
            }
        }
    }
    if (!ok) atomicExch(&g_gemm_err, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, L::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

template <int BN>
te_status launch(const Params &p, int ftiles, cudaStream_t stream) {
    const int smem = Layout<BN>::BYTES + 1024;
    static bool attr_done = false;   // per instantiation; benign race: same value
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(q8_gemm_kernel<BN>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return cuda_fail(e, "q8_linear: set shared memory size");
        attr_done = true;
    }
    const dim3 grid((p.m + BN - 1) / BN, ftiles);
    q8_gemm_kernel<BN><<<grid, NTHREADS, smem, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TE_OK : cuda_fail(e, "q8_linear launch");
}

}  // namespace

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
    int ftiles = 0;
    for (int i = 0; i < z; ++i) {
        const te_q8_item &src = items[i];
        if (!src.w.q || !src.w.scale || !src.y)
            return fail(TE_EINVAL, "q8_linear: item %d has a NULL q, scale or y", i);
        if (src.w.k != k) return fail(TE_ESHAPE, "q8_linear: item %d has k=%d, x has %d", i, src.w.k, k);
        if (src.w.n < 32 || src.w.n % 32)
            return fail(TE_ESHAPE, "q8_linear: item %d n=%d (multiple of 32)", i, src.w.n);
        if (src.y_dtype != TE_F32 && src.y_dtype != TE_BF16)
            return fail(TE_EINVAL, "q8_linear: item %d bad y dtype", i);
        if (src.ldy < src.w.n) return fail(TE_ESHAPE, "q8_linear: item %d ldy < n", i);
        if (!aligned16(src.w.q) || !aligned16(src.y) || (reinterpret_cast<uintptr_t>(src.w.scale) & 3) ||
            (src.w.bias && (reinterpret_cast<uintptr_t>(src.w.bias) & 3)))
            return fail(TE_EALIGN, "q8_linear: item %d: q and y must be 16-byte aligned", i);
        if (src.residual) {
            if (src.ldr < src.w.n) return fail(TE_ESHAPE, "q8_linear: item %d ldr < n", i);
            if ((reinterpret_cast<uintptr_t>(src.residual) & 3))
                return fail(TE_EALIGN, "q8_linear: item %d residual not 4-byte aligned", i);
            if (src.residual == src.y && (src.ldr != src.ldy || src.y_dtype != TE_F32))
                return fail(TE_EINVAL, "q8_linear: item %d: in-place residual needs f32 y and ldr == ldy", i);
        }
        Item &d = p.it[i];
        d.scale = src.w.scale;
        d.bias = src.w.bias;
        d.y = src.y;
        d.resid = src.residual;
        d.ldy = src.ldy;
        d.ldr = src.ldr;
        d.n = src.w.n;
        d.ydt = src.y_dtype;
        d.tile0 = ftiles;
        ftiles += (src.w.n + BM - 1) / BM;
    }
    if (m == 0) return TE_OK;
    const int bn = m >= 512 ? 256 : (m > 64 ? 128 : 64);
    te_status st = make_map_2d(&p.tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)k, (uint64_t)m,
                               (uint64_t)ldx * 2, BK, bn, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != TE_OK) return st;
    for (int i = 0; i < z; ++i) {
        st = make_map_2d(&p.tw[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, items[i].w.q, (uint64_t)k,
                         (uint64_t)items[i].w.n, (uint64_t)k, BK, BM, CU_TENSOR_MAP_SWIZZLE_64B);
        if (st != TE_OK) return st;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (bn == 256) return launch<256>(p, ftiles, s);
    if (bn == 128) return launch<128>(p, ftiles, s);
    return launch<64>(p, ftiles, s);
}
