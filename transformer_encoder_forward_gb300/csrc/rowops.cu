// Row operations of the encoder block: RMSNorm / LayerNorm, the residual add
// fused with the next norm, q/k norm + RoPE, the gate activation and the
// final-norm mean-pool.  Each is bound by HBM bandwidth: one warp owns a row
// (or a (row, head) pair), reads it once with 16-byte vector loads, keeps it
// in registers across the reductions and writes it once.
//
// Sources: "cortiq-engine 0.8.39 src/gpu_metal/egemma2.rs" (Prog::rms,
// Prog::add_norm, Prog::gelu, Prog::qkv, TextGpu::forward final norm + pool),
// "cortiq-engine 0.7.6 src/gpu_metal/zimage.rs" (Enc::rowop, Enc::block
// qk-norm + RoPE and SwiGLU), "cera 0.2.4 src/model/vision_encoder_gpu.rs"
// (VitGpuOps::layernorm / gelu / add).
#include <stdarg.h>
#include <string.h>

#include "common.cuh"

namespace tefwd {

// ------------------------------------------------------------ error reporting

static thread_local char g_msg[512] = "";

te_status fail(te_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

te_status cuda_fail(cudaError_t e, const char *what) {
    return fail(TE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

te_status check_cu(const int32_t *cu_host, const int32_t *cu_dev, int32_t nseq, int32_t *total,
                   int32_t *max_len) {
    if (!cu_host || !cu_dev) return fail(TE_EINVAL, "cu_seqlens: NULL host or device array");
    if (nseq < 1) return fail(TE_EINVAL, "cu_seqlens: nseq = %d, need >= 1", nseq);
    if ((reinterpret_cast<uintptr_t>(cu_dev) & 3u) != 0)
        return fail(TE_EALIGN, "cu_seqlens: device array not 4-byte aligned");
    if (cu_host[0] != 0) return fail(TE_EINVAL, "cu_seqlens: cu[0] = %d, need 0", cu_host[0]);
    int32_t mx = 0;
    for (int32_t s = 0; s < nseq; ++s) {
        const int64_t len = (int64_t)cu_host[s + 1] - cu_host[s];
        if (len < 1)
            return fail(TE_EINVAL, "cu_seqlens: sequence %d has length %lld (need >= 1)", s,
                        (long long)len);
        if (len > mx) mx = (int32_t)len;
    }
    *total = cu_host[nseq];
    *max_len = mx;
    return TE_OK;
}

__device__ int g_rowop_err;

// --------------------------------------------------------------- vector I/O

__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0];
    const float4 b = reinterpret_cast<const float4 *>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// The same load with the streaming (evict-first) cache hint: for rows read
// once, so that they do not push the per-feature vectors out of L1.
__device__ __forceinline__ void load8_stream(const float *p, float (&v)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void store8(float *p, const float (&v)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&v)[8]) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]); u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]); u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4 *>(p) = u;
}

// Normalises the warp's row held in v (NV chunks of 8 per lane, chunk i of
// lane l covers columns (i*32 + l)*8 ...) and writes w*v (+b) to y, times
// (1 + ms) when the adaLN scale ms is given.
template <typename Tout, int NV>
__device__ __forceinline__ void norm_store(float (&v)[NV][8], int lane, int d, int kind, float eps,
                                           const float *w, const float *b, const float *ms, Tout *y) {
    float inv, mean = 0.f;
    if (kind == TE_NORM_LN) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if ((i * 32 + lane) * 8 < d)
#pragma unroll
                for (int e = 0; e < 8; ++e) s += v[i][e];
        mean = warp_sum(s) / (float)d;
        float q = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if ((i * 32 + lane) * 8 < d)
#pragma unroll
                for (int e = 0; e < 8; ++e) q += (v[i][e] - mean) * (v[i][e] - mean);
        inv = rsqrtf(warp_sum(q) / (float)d + eps);
    } else {
        float q = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if ((i * 32 + lane) * 8 < d)
#pragma unroll
                for (int e = 0; e < 8; ++e) q += v[i][e] * v[i][e];
        inv = rsqrtf(warp_sum(q) / (float)d + eps);
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = (i * 32 + lane) * 8;
        if (c < d) {
            float wv[8], o[8];
            load8(w + c, wv);
            if (b) {
                float bv[8];
                load8(b + c, bv);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = (v[i][e] - mean) * inv * wv[e] + bv[e];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = (v[i][e] - mean) * inv * wv[e];
            }
            if (ms) {
                float sv[8];
                load8(ms + c, sv);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] *= 1.f + sv[e];
            }
            store8(y + c, o);
        }
    }
}

// ------------------------------------------------------------------ rownorm

template <typename Tin, typename Tout, int NV>
__global__ void __launch_bounds__(256) rownorm_kernel(const Tin *__restrict__ x, long long ldx,
                                                      const float *__restrict__ w,
                                                      const float *__restrict__ b,
                                                      const float *__restrict__ ms, int kind,
                                                      float eps, float pre, Tout *y, long long ldy,
                                                      int t, int d) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= t) return;
    float v[NV][8];
    const Tin *xr = x + (long long)row * ldx;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = (i * 32 + lane) * 8;
        if (c < d) {
            load8(xr + c, v[i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[i][e] *= pre;
        }
    }
    norm_store<Tout, NV>(v, lane, d, kind, eps, w, kind == TE_NORM_LN ? b : nullptr, ms,
                         y + (long long)row * ldy);
}

// ----------------------------------------------------------------- add_norm

template <typename Tout, int NV, bool MOD>
__global__ void __launch_bounds__(256) add_norm_kernel(float *h, const float *__restrict__ t,
                                                       const float *__restrict__ w_post,
                                                       const float *__restrict__ gate,
                                                       float post, const float *__restrict__ w_next,
                                                       const float *__restrict__ b_next,
                                                       const float *__restrict__ ms, int kind,
                                                       float eps, Tout *a, int rows, int d) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float v[NV][8];
    float *hr = h + (long long)row * d;
    const float *tr = t ? t + (long long)row * d : nullptr;
    if (tr) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = (i * 32 + lane) * 8;
            if (c < d) load8(tr + c, v[i]);
        }
    }
    float inv_t = 1.f;
    if (tr && w_post) {
        float q = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if ((i * 32 + lane) * 8 < d)
#pragma unroll
                for (int e = 0; e < 8; ++e) q += v[i][e] * v[i][e];
        inv_t = rsqrtf(warp_sum(q) / (float)d + eps);
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = (i * 32 + lane) * 8;
        if (c < d) {
            float hv[8];
            load8(hr + c, hv);
            if (MOD && tr && gate) {            // adaLN gate on the branch
                float gv[8];
                load8(gate + c, gv);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] *= gv[e];
            }
            if (tr && w_post) {
                float wv[8];
                load8(w_post + c, wv);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] = (hv[e] + v[i][e] * inv_t * wv[e]) * post;
            } else if (tr) {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] = hv[e] + v[i][e];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] = hv[e];
            }
            if (tr) store8(hr + c, v[i]);
        }
    }
    if (w_next)
        norm_store<Tout, NV>(v, lane, d, kind, eps, w_next, kind == TE_NORM_LN ? b_next : nullptr,
                             MOD ? ms : nullptr, a + (long long)row * d);
}

// Wide rows: WPR warps per row (d > 1024: 8, one row per 256-thread CTA;
// 512 < d <= 1024: 4, two rows a CTA, one 8-column chunk a thread).
// Each thread holds at most NV 8-column chunks of t and of h, all loaded up
// front (more bytes in flight per SM than one warp per row allows); the row
// reductions go through shared memory.  Eight warps a row (2 chunks a thread,
// ~50 registers, five CTAs an SM) keep more rows in flight than four warps
// (4 chunks, two CTAs an SM): d = 3840 6110 -> 6520 GB/s, with adaLN 5010 ->
// 5815 GB/s.
template <int WPR>
__device__ __forceinline__ float row4_sum(float x, float (*red)[WPR], int slot, int wr, int lane) {
    x = warp_sum(x);
    if (lane == 0) red[slot][wr] = x;
    __syncthreads();
    float s = red[slot][0] + red[slot][1];
    if (WPR >= 4) s += red[slot][2] + red[slot][3];
    if (WPR == 8) s += (red[slot][4] + red[slot][5]) + (red[slot][6] + red[slot][7]);
    __syncthreads();
    return s;
}

template <typename Tout, int NV, bool MOD, int WPR = 4>
__global__ void __launch_bounds__(256) add_norm_wide_kernel(float *h, const float *__restrict__ t,
                                                            const float *__restrict__ w_post,
                                                            const float *__restrict__ gate,
                                                            float post,
                                                            const float *__restrict__ w_next,
                                                            const float *__restrict__ b_next,
                                                            const float *__restrict__ ms, int kind,
                                                            float eps, Tout *a, int rows, int d) {
    constexpr int TPR = 32 * WPR;               // threads a row
    __shared__ float red[256 / TPR][WPR];
    const int slot = threadIdx.x / TPR, tid = threadIdx.x % TPR;
    const int wr = tid >> 5, lane = tid & 31;
    const int row = blockIdx.x * (256 / TPR) + slot;
    const bool active = row < rows;            // inactive threads still join the barriers
    float *hr = h + (long long)(active ? row : 0) * d;
    const float *tr = t ? t + (long long)(active ? row : 0) * d : nullptr;
    float tv[NV][8], hv[NV][8];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = (i * TPR + tid) * 8;
        if (active && c < d) {
            // adaLN form: its gate and scale vectors compete with the rows for L1
            if (MOD) {
                if (tr) load8_stream(tr + c, tv[i]);
                load8_stream(hr + c, hv[i]);
            } else {
                if (tr) load8(tr + c, tv[i]);
                load8(hr + c, hv[i]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) tv[i][e] = hv[i][e] = 0.f;
        }
    }
    if (tr) {
        float inv_t = 1.f;
        if (w_post) {
            float q = 0.f;
#pragma unroll
            for (int i = 0; i < NV; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) q += tv[i][e] * tv[i][e];
            inv_t = rsqrtf(row4_sum<WPR>(q, red, slot, wr, lane) / (float)d + eps);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = (i * TPR + tid) * 8;
            if (active && c < d) {
                if (MOD && gate) {              // adaLN gate on the branch
                    float gv[8];
                    load8(gate + c, gv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) tv[i][e] *= gv[e];
                }
                if (w_post) {
                    float wv[8];
                    load8(w_post + c, wv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) hv[i][e] = (hv[i][e] + tv[i][e] * inv_t * wv[e]) * post;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) hv[i][e] += tv[i][e];
                }
                store8(hr + c, hv[i]);
            }
        }
    }
    if (!w_next) return;                       // uniform across the CTA
    float mean = 0.f;
    if (kind == TE_NORM_LN) {
        float s1 = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) s1 += hv[i][e];
        mean = row4_sum<WPR>(s1, red, slot, wr, lane) / (float)d;
    }
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = (i * TPR + tid) * 8;
        if (c < d)
#pragma unroll
            for (int e = 0; e < 8; ++e) q += (hv[i][e] - mean) * (hv[i][e] - mean);
    }
    const float inv = rsqrtf(row4_sum<WPR>(q, red, slot, wr, lane) / (float)d + eps);
    const float *bn = kind == TE_NORM_LN ? b_next : nullptr;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = (i * TPR + tid) * 8;
        if (active && c < d) {
            float wv[8], o[8];
            load8(w_next + c, wv);
            if (bn) {
                float bv[8];
                load8(bn + c, bv);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = (hv[i][e] - mean) * inv * wv[e] + bv[e];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = (hv[i][e] - mean) * inv * wv[e];
            }
            if (MOD && ms) {
                float sv[8];
                load8(ms + c, sv);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] *= 1.f + sv[e];
            }
            store8(a + (long long)row * d + c, o);
        }
    }
}

// ------------------------------------------------------ bounded-wait check

// Waits on an mbarrier that nothing arrives at, with the bounded wait every
// pipeline kernel uses, but a short limit; when the wait gives up it records
// error 1 in the row-op error word, exactly as a stuck pipeline would.
__global__ void wait_timeout_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, limit_ns)) atomicExch(&g_rowop_err, 1);
}

// ---------------------------------------------------------------- cast bf16

// Grid-stride over 8-column chunks: 32 bytes in, 16 bytes out.
__global__ void __launch_bounds__(256) cast_bf16_kernel(const float *__restrict__ x, long long ldx,
                                                        __nv_bfloat16 *__restrict__ y, long long ldy,
                                                        int rows, int chunks) {
    const long long total = (long long)rows * chunks;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / chunks;
        const int c = (int)(i - r * chunks) * 8;
        float v[8];
        load8(x + r * ldx + c, v);
        store8(y + r * ldy + c, v);
    }
}

// ------------------------------------------------------------- qk prep + RoPE

// One warp per (packed row, group of 4 * 32 / (HD / 8) heads).  A head of HD
// channels spans HD/8 lanes, so the per-head RMS is a reduction over an
// aligned lane group.  Each lane owns both members of its RoPE pairs: 4
// channels of the first half of its section and the matching 4 of the second
// half (two 8-byte loads), so the rotation needs no exchange between lanes
// (without RoPE the two 4-channel pieces are simply adjacent).  The warp issues
// all loads of its group before any arithmetic (4 or 6 heads per lane in
// flight, chosen so that the heads split into whole groups: 60 heads of 128
// into five groups of 12; a loop of load -> norm -> store per head pair waited
// a full memory latency per iteration).
// heads per lane in flight: 4 or 6, chosen per launch so that the head
// count splits into whole groups where it can

__device__ __forceinline__ void unpack4(uint2 r, float (&v)[4]) {
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x); v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
}

template <int HD, bool VN, int QK_U>
__global__ void __launch_bounds__(256) qk_prep_kernel(__nv_bfloat16 *qkv, long long ld, int q_off,
                                                      int k_off, int v_off, int nq, int nkv, int nv,
                                                      const float *__restrict__ qn,
                                                      const float *__restrict__ kn, float eps,
                                                      const float *__restrict__ cosb,
                                                      const float *__restrict__ sinb,
                                                      const int *__restrict__ pos, int table_rows,
                                                      int sec, float q_mul, int rows) {
    constexpr int LPH = HD / 8;                 // lanes per head
    constexpr int HPI = 32 / LPH;               // heads per load slot
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int hl = lane / LPH;                  // head slot of this lane in a load slot
    const int j = lane % LPH;                   // lane within its head
    // this lane's channels: c1..c1+3 and c2..c2+3 (c2 = c1 + half of the section)
    const int secl = sec ? sec : 8;             // section (8: no RoPE, adjacent pieces)
    const int half = secl >> 1;
    const int lps = secl / 8;                   // lanes per section
    const int sct = j / lps, jj = j - sct * lps;
    const int c1 = sct * secl + 4 * jj, c2 = c1 + half;
    const int nh = nq + nkv + nv;               // q heads, k heads, then (v-norm) v heads
    const int hbase = blockIdx.y * (HPI * QK_U);
    float4 cv = make_float4(0.f, 0.f, 0.f, 0.f), sv = cv;
    if (sec) {
        long long prow = pos ? pos[row] : row;
        if (prow < 0 || prow >= table_rows) {
            atomicExch(&g_rowop_err, 2);
            prow = 0;
        }
        // pair index of c1 within its section: table column sct*half + 4*jj
        cv = *reinterpret_cast<const float4 *>(cosb + prow * (HD / 2) + sct * half + 4 * jj);
        sv = *reinterpret_cast<const float4 *>(sinb + prow * (HD / 2) + sct * half + 4 * jj);
    }
    uint2 r1[QK_U], r2[QK_U];
#pragma unroll
    for (int u = 0; u < QK_U; ++u) {           // every load of the group first
        const int hh = hbase + u * HPI + hl;
        if (hh < nh) {
            const int col = hh < nq ? q_off + hh * HD
                                    : (!VN || hh < nq + nkv ? k_off + (hh - nq) * HD : v_off + (hh - nq - nkv) * HD);
            const __nv_bfloat16 *p = qkv + row * ld + col;
            r1[u] = *reinterpret_cast<const uint2 *>(p + c1);
            r2[u] = *reinterpret_cast<const uint2 *>(p + c2);
        } else {
            r1[u] = r2[u] = make_uint2(0u, 0u);
        }
    }
#pragma unroll
    for (int u = 0; u < QK_U; ++u) {
        const int hh = hbase + u * HPI + hl;
        const bool active = hh < nh;            // lane groups past the last head idle
        const bool isq = hh < nq;
        const bool isv = VN && hh >= nq + nkv;  // v heads: RMS norm without weight, no RoPE
        float a[4], b[4];
        unpack4(r1[u], a);
        unpack4(r2[u], b);
        const float *nw = isq ? qn : kn;
        if (qn || VN) {                         // uniform: qn and kn are both given or both NULL
            float q = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) q = fmaf(a[e], a[e], fmaf(b[e], b[e], q));
#pragma unroll
            for (int o = 1; o < LPH; o <<= 1) q += __shfl_xor_sync(0xFFFFFFFFu, q, o);
            const float inv = rsqrtf(q / (float)HD + eps);
            if (VN && active && isv) {
#pragma unroll
                for (int e = 0; e < 4; ++e) { a[e] *= inv; b[e] *= inv; }
            } else if (active && qn) {
                const float4 w1 = *reinterpret_cast<const float4 *>(nw + c1);
                const float4 w2 = *reinterpret_cast<const float4 *>(nw + c2);
                a[0] *= inv * w1.x; a[1] *= inv * w1.y; a[2] *= inv * w1.z; a[3] *= inv * w1.w;
                b[0] *= inv * w2.x; b[1] *= inv * w2.y; b[2] *= inv * w2.z; b[3] *= inv * w2.w;
            }
        }
        if (sec && !(VN && isv)) {              // rotate-half: (a, b) -> (a c - b s, b c + a s)
            const float cc[4] = {cv.x, cv.y, cv.z, cv.w}, ss[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x1 = a[e], x2 = b[e];
                a[e] = fmaf(x1, cc[e], -x2 * ss[e]);
                b[e] = fmaf(x2, cc[e], x1 * ss[e]);
            }
        }
        if (active) {
            const float mul = isq ? q_mul : 1.f;
            const int col = isq ? q_off + hh * HD
                                : (VN && isv ? v_off + (hh - nq - nkv) * HD : k_off + (hh - nq) * HD);
            __nv_bfloat16 *p = qkv + row * ld + col;
            *reinterpret_cast<uint2 *>(p + c1) = make_uint2(pack_bf16x2(a[0] * mul, a[1] * mul),
                                                            pack_bf16x2(a[2] * mul, a[3] * mul));
            *reinterpret_cast<uint2 *>(p + c2) = make_uint2(pack_bf16x2(b[0] * mul, b[1] * mul),
                                                            pack_bf16x2(b[2] * mul, b[3] * mul));
        }
    }
}

// ---------------------------------------------------------------- gate_act

__global__ void __launch_bounds__(256) gate_act_kernel(const __nv_bfloat16 *__restrict__ gu,
                                                       long long ld, int u_off, int act,
                                                       __nv_bfloat16 *__restrict__ m,
                                                       long long ldm, int rows, int f) {
    const int per_row = f >> 3;
    const long long total = (long long)rows * per_row;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long row = idx / per_row;
        const int c = (int)(idx - row * per_row) * 8;
        float g[8], o[8];
        load8(gu + row * ld + c, g);
        if (u_off >= 0) {
            float u[8];
            load8(gu + row * ld + u_off + c, u);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = apply_act(g[e], act) * u[e];
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = apply_act(g[e], act);
        }
        store8(m + row * ldm + c, o);
    }
}

// --------------------------------------------------------------- pool_mean

// One CTA per sequence; 8 warps take rows round-robin, each keeps column
// partial sums in registers; the partials are combined in a fixed order, so
// the result does not depend on scheduling.
template <int NV>
__global__ void __launch_bounds__(256) pool_kernel(const float *__restrict__ x, int d,
                                                   const int *__restrict__ cu,
                                                   const float *__restrict__ w, float eps,
                                                   float *__restrict__ out) {
    extern __shared__ float part[];   // [d]
    const int s = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = cu[s], r1 = cu[s + 1];
    float acc[NV][8];
#pragma unroll
    for (int i = 0; i < NV; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
    for (int r = r0 + warp; r < r1; r += 8) {
        const float *xr = x + (long long)r * d;
        float inv = 1.f;
        if (w) {   // first pass: the row's RMS (the second pass re-reads it from L1)
            float q = 0.f;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = (i * 32 + lane) * 8;
                if (c < d) {
                    float v[8];
                    load8(xr + c, v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) q += v[e] * v[e];
                }
            }
            inv = rsqrtf(warp_sum(q) / (float)d + eps);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = (i * 32 + lane) * 8;
            if (c < d) {
                float v[8];
                load8(xr + c, v);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[i][e] += v[e] * inv;
            }
        }
    }
    for (int ww = 0; ww < 8; ++ww) {
        if (warp == ww) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c = (i * 32 + lane) * 8;
                if (c < d)
#pragma unroll
                    for (int e = 0; e < 8; ++e) part[c + e] = (ww ? part[c + e] : 0.f) + acc[i][e];
            }
        }
        __syncthreads();
    }
    const float scale = 1.f / (float)(r1 - r0);
    for (int c = threadIdx.x; c < d; c += blockDim.x)
        out[(long long)s * d + c] = part[c] * scale * (w ? w[c] : 1.f);
}

// --------------------------------------------------------------- dispatch

static int nv_for(int d) {
    const int chunks = (d + 255) / 256;   // per-lane chunks of 8
    if (chunks <= 1) return 1;
    if (chunks <= 2) return 2;
    if (chunks <= 4) return 4;
    if (chunks <= 8) return 8;
    return 16;
}

#define TE_NV_SWITCH(nv, ...)                       \
    switch (nv) {                                   \
    case 1: { constexpr int NV = 1; __VA_ARGS__; } break;   \
    case 2: { constexpr int NV = 2; __VA_ARGS__; } break;   \
    case 4: { constexpr int NV = 4; __VA_ARGS__; } break;   \
    case 8: { constexpr int NV = 8; __VA_ARGS__; } break;   \
    default: { constexpr int NV = 16; __VA_ARGS__; } break; \
    }

static te_status launched(const char *what) {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TE_OK : cuda_fail(e, what);
}

static bool dtype_ok(int32_t dt) { return dt == TE_F32 || dt == TE_BF16; }

}  // namespace tefwd

using namespace tefwd;

extern "C" {

te_status te_rownorm_mod(const void *x, int32_t xdt, int64_t ldx, const float *w, const float *b,
                         const float *ms, int32_t kind, float eps, float pre, void *y, int32_t ydt,
                         int64_t ldy, int32_t t, int32_t d, te_stream stream) {
    if (!x || !w || !y) return fail(TE_EINVAL, "rownorm: NULL x, w or y");
    if (!dtype_ok(xdt) || !dtype_ok(ydt)) return fail(TE_EINVAL, "rownorm: bad dtype");
    if (kind != TE_NORM_RMS && kind != TE_NORM_LN) return fail(TE_EINVAL, "rownorm: bad kind");
    if (t < 0 || d < 8 || d > 4096 || d % 8) return fail(TE_ESHAPE, "rownorm: t=%d d=%d (d %% 8 == 0, 8..4096)", t, d);
    if (ldx < d || ldy < d) return fail(TE_ESHAPE, "rownorm: leading dimension below d");
    if (!aligned16(x) || !aligned16(y) || !aligned16(w) || (b && !aligned16(b)) || (ms && !aligned16(ms)) ||
        (ldx * (xdt == TE_F32 ? 4 : 2)) % 16 || (ldy * (ydt == TE_F32 ? 4 : 2)) % 16)
        return fail(TE_EALIGN, "rownorm: pointers and rows must be 16-byte aligned");
    if (x == y && (xdt != ydt || ldx != ldy))
        return fail(TE_EINVAL, "rownorm: in place needs equal dtype and leading dimension");
    if (t == 0) return TE_OK;
    const dim3 grid((t + 7) / 8);
    TE_NV_SWITCH(nv_for(d), {
        if (xdt == TE_F32 && ydt == TE_BF16)
            rownorm_kernel<float, __nv_bfloat16, NV><<<grid, 256, 0, stream>>>(
                (const float *)x, ldx, w, b, ms, kind, eps, pre, (__nv_bfloat16 *)y, ldy, t, d);
        else if (xdt == TE_F32 && ydt == TE_F32)
            rownorm_kernel<float, float, NV><<<grid, 256, 0, stream>>>(
                (const float *)x, ldx, w, b, ms, kind, eps, pre, (float *)y, ldy, t, d);
        else if (xdt == TE_BF16 && ydt == TE_BF16)
            rownorm_kernel<__nv_bfloat16, __nv_bfloat16, NV><<<grid, 256, 0, stream>>>(
                (const __nv_bfloat16 *)x, ldx, w, b, ms, kind, eps, pre, (__nv_bfloat16 *)y, ldy, t, d);
        else
            rownorm_kernel<__nv_bfloat16, float, NV><<<grid, 256, 0, stream>>>(
                (const __nv_bfloat16 *)x, ldx, w, b, ms, kind, eps, pre, (float *)y, ldy, t, d);
    })
    return launched("rownorm launch");
}

te_status te_rownorm(const void *x, int32_t xdt, int64_t ldx, const float *w, const float *b,
                     int32_t kind, float eps, float pre, void *y, int32_t ydt, int64_t ldy,
                     int32_t t, int32_t d, te_stream stream) {
    return te_rownorm_mod(x, xdt, ldx, w, b, nullptr, kind, eps, pre, y, ydt, ldy, t, d, stream);
}

te_status te_add_norm_mod(float *h, const float *t, const float *w_post, const float *gate, float post,
                          const float *w_next, const float *b_next, const float *ms, int32_t kind,
                          float eps, void *a, int32_t adt, int32_t rows, int32_t d, te_stream stream) {
    if (!h) return fail(TE_EINVAL, "add_norm: NULL h");
    if (w_post && !t) return fail(TE_EINVAL, "add_norm: w_post given without t");
    if (gate && !t) return fail(TE_EINVAL, "add_norm: gate given without t");
    if (w_next && !a) return fail(TE_EINVAL, "add_norm: w_next given without a");
    if (ms && !w_next) return fail(TE_EINVAL, "add_norm: scale given without w_next");
    if (w_next && !dtype_ok(adt)) return fail(TE_EINVAL, "add_norm: bad dtype");
    if (kind != TE_NORM_RMS && kind != TE_NORM_LN) return fail(TE_EINVAL, "add_norm: bad kind");
    if (rows < 0 || d < 8 || d > 4096 || d % 8) return fail(TE_ESHAPE, "add_norm: rows=%d d=%d (d %% 8 == 0, 8..4096)", rows, d);
    if (!aligned16(h) || (t && !aligned16(t)) || (w_post && !aligned16(w_post)) ||
        (w_next && !aligned16(w_next)) || (b_next && !aligned16(b_next)) || (a && !aligned16(a)) ||
        (gate && !aligned16(gate)) || (ms && !aligned16(ms)))
        return fail(TE_EALIGN, "add_norm: pointers must be 16-byte aligned");
    if (rows == 0) return TE_OK;
    // the adaLN loads only in their own instantiation: the unmodulated kernel
    // keeps its registers (and occupancy)
    const bool mod = gate || ms;
    if (d > 512 && d <= 1024) {
        // four warps a row, one 8-column chunk a thread: at d = 768 this beats
        // the one-warp-a-row kernel (more loads in flight a row); at d <= 512
        // the one-warp kernel stays ahead, so narrow rows keep it.  Both
        // forms take the same kernel, so identity adaLN vectors stay a no-op
        // to the bit.
        const dim3 g2((rows + 1) / 2);
        if (adt == TE_F32) {
            if (mod)
                add_norm_wide_kernel<float, 1, true, 4><<<g2, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (float *)a, rows, d);
            else
                add_norm_wide_kernel<float, 1, false, 4><<<g2, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (float *)a, rows, d);
        } else {
            if (mod)
                add_norm_wide_kernel<__nv_bfloat16, 1, true, 4><<<g2, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (__nv_bfloat16 *)a, rows, d);
            else
                add_norm_wide_kernel<__nv_bfloat16, 1, false, 4><<<g2, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (__nv_bfloat16 *)a, rows, d);
        }
        return launched("add_norm launch");
    }
    if (d > 1024) {
        // eight warps per row (d <= 4096: at most 2 chunks of 8 per thread)
        const dim3 grid2(rows);
        if (adt == TE_F32) {
            if (mod)
                add_norm_wide_kernel<float, 2, true, 8><<<grid2, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (float *)a, rows, d);
            else
                add_norm_wide_kernel<float, 2, false, 8><<<grid2, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (float *)a, rows, d);
        } else {
            if (mod)
                add_norm_wide_kernel<__nv_bfloat16, 2, true, 8><<<grid2, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (__nv_bfloat16 *)a, rows, d);
            else
                add_norm_wide_kernel<__nv_bfloat16, 2, false, 8><<<grid2, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (__nv_bfloat16 *)a, rows, d);
        }
        return launched("add_norm launch");
    }
    const dim3 grid((rows + 7) / 8);
    TE_NV_SWITCH(nv_for(d), {
        if (adt == TE_F32) {
            if (mod)
                add_norm_kernel<float, NV, true><<<grid, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (float *)a, rows, d);
            else
                add_norm_kernel<float, NV, false><<<grid, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (float *)a, rows, d);
        } else {
            if (mod)
                add_norm_kernel<__nv_bfloat16, NV, true><<<grid, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (__nv_bfloat16 *)a, rows, d);
            else
                add_norm_kernel<__nv_bfloat16, NV, false><<<grid, 256, 0, stream>>>(
                    h, t, w_post, gate, post, w_next, b_next, ms, kind, eps, (__nv_bfloat16 *)a, rows, d);
        }
    })
    return launched("add_norm launch");
}

te_status te_add_norm(float *h, const float *t, const float *w_post, float post,
                      const float *w_next, const float *b_next, int32_t kind, float eps, void *a,
                      int32_t adt, int32_t rows, int32_t d, te_stream stream) {
    return te_add_norm_mod(h, t, w_post, nullptr, post, w_next, b_next, nullptr, kind, eps, a, adt, rows, d,
                           stream);
}

te_status te_qkv_prep_rope(void *qkv, int64_t ld, int32_t q_off, int32_t k_off, int32_t v_off,
                           int32_t nq, int32_t nkv, int32_t hd, const float *qn, const float *kn,
                           int32_t v_norm, float eps, const float *cos, const float *sin,
                           const int32_t *pos, int32_t table_rows, int32_t sec, float q_mul,
                           int32_t rows, te_stream stream) {
    if (!qkv) return fail(TE_EINVAL, "qk_prep_rope: NULL qkv");
    if (hd != 64 && hd != 128) return fail(TE_ESHAPE, "qk_prep_rope: hd=%d (64 or 128)", hd);
    if (nq < 0 || nkv < 0 || rows < 0 || q_off < 0 || k_off < 0 || (v_norm && v_off < 0))
        return fail(TE_ESHAPE, "qk_prep_rope: negative size or offset");
    if ((int64_t)q_off + (int64_t)nq * hd > ld || (int64_t)k_off + (int64_t)nkv * hd > ld ||
        (v_norm && (int64_t)v_off + (int64_t)nkv * hd > ld))
        return fail(TE_ESHAPE, "qk_prep_rope: heads run past the row (ld=%lld)", (long long)ld);
    if (sec != 0 && sec != hd && sec != hd / 2)
        return fail(TE_ESHAPE, "qk_prep_rope: sec=%d (0, hd or hd/2)", sec);
    if (sec && (!cos || !sin || table_rows < 1))
        return fail(TE_EINVAL, "qk_prep_rope: RoPE needs cos, sin and table_rows >= 1");
    if (sec && !pos && table_rows < rows)
        return fail(TE_ESHAPE, "qk_prep_rope: table has %d rows, need %d (pos == NULL)", table_rows, rows);
    if (!aligned16(qkv) || (ld * 2) % 16 || (q_off * 2) % 16 || (k_off * 2) % 16 ||
        (v_norm && (v_off * 2) % 16) || (qn && !aligned16(qn)) || (kn && !aligned16(kn)) ||
        (cos && !aligned16(cos)) || (sin && !aligned16(sin)))
        return fail(TE_EALIGN, "qk_prep_rope: qkv rows, head offsets and tables must be 16-byte aligned");
    if ((qn == nullptr) != (kn == nullptr))
        return fail(TE_EINVAL, "qk_prep_rope: give both qn and kn or neither");
    const int nv = v_norm ? nkv : 0;
    if (rows == 0 || nq + nkv + nv == 0) return TE_OK;
    // 6 heads a lane in flight when that splits the heads into whole groups and
    // 4 would not (hd 128: 60 heads; v-norm at hd 64: 24), else 4
    const int nh = nq + nkv + nv, hpi = 32 / (hd / 8);
    const int qu = (nh % (6 * hpi) == 0 && nh % (4 * hpi) != 0) || (hd == 128 && nh % (4 * hpi) != 0) ? 6 : 4;
    const int heads_per_warp = hpi * qu;
    const dim3 grid((unsigned)(((long long)rows + 7) / 8), (unsigned)((nh + heads_per_warp - 1) / heads_per_warp));
    auto go = [&](auto kern) {
        kern<<<grid, 256, 0, stream>>>((__nv_bfloat16 *)qkv, ld, q_off, k_off, v_off, nq, nkv, nv, qn, kn, eps,
                                       cos, sin, pos, table_rows, sec, q_mul, rows);
    };
    // the v-norm heads in their own instantiation: the q/k pass keeps its code
    if (hd == 64) {
        if (qu == 6) nv ? go(qk_prep_kernel<64, true, 6>) : go(qk_prep_kernel<64, false, 6>);
        else nv ? go(qk_prep_kernel<64, true, 4>) : go(qk_prep_kernel<64, false, 4>);
    } else {
        if (qu == 6) nv ? go(qk_prep_kernel<128, true, 6>) : go(qk_prep_kernel<128, false, 6>);
        else nv ? go(qk_prep_kernel<128, true, 4>) : go(qk_prep_kernel<128, false, 4>);
    }
    return launched("qk_prep_rope launch");
}

te_status te_qk_prep_rope(void *qkv, int64_t ld, int32_t q_off, int32_t k_off, int32_t nq,
                          int32_t nkv, int32_t hd, const float *qn, const float *kn, float eps,
                          const float *cos, const float *sin, const int32_t *pos,
                          int32_t table_rows, int32_t sec, float q_mul, int32_t rows,
                          te_stream stream) {
    return te_qkv_prep_rope(qkv, ld, q_off, k_off, 0, nq, nkv, hd, qn, kn, 0, eps, cos, sin, pos,
                            table_rows, sec, q_mul, rows, stream);
}

te_status te_selftest_wait_timeout(int32_t limit_us, te_stream stream) {
    if (limit_us < 1 || limit_us > 1000000) return fail(TE_EINVAL, "selftest: limit_us=%d (1..1000000)", limit_us);
    wait_timeout_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_us * 1000ull);
    return launched("selftest launch");
}

te_status te_cast_bf16(const float *x, int64_t ldx, void *y, int64_t ldy, int32_t rows, int32_t d,
                       te_stream stream) {
    if (!x || !y) return fail(TE_EINVAL, "cast_bf16: NULL x or y");
    if (rows < 0 || d < 8 || d % 8 || ldx < d || ldy < d) return fail(TE_ESHAPE, "cast_bf16: rows=%d d=%d", rows, d);
    if (!aligned16(x) || !aligned16(y) || ldx % 4 || ldy % 8)
        return fail(TE_EALIGN, "cast_bf16: rows must be 16-byte aligned");
    if (rows == 0) return TE_OK;
    const long long total = (long long)rows * (d / 8);
    const long long want = (total + 255) / 256;
    const unsigned blocks = (unsigned)(want < 152 * 16 ? want : 152 * 16);
    cast_bf16_kernel<<<blocks, 256, 0, stream>>>(x, ldx, (__nv_bfloat16 *)y, ldy, rows, d / 8);
    return launched("cast_bf16 launch");
}

te_status te_gate_act(const void *gu, int64_t ld, int32_t u_off, int32_t act, void *m,
                      int64_t ldm, int32_t rows, int32_t f, te_stream stream) {
    if (!gu || !m) return fail(TE_EINVAL, "gate_act: NULL gu or m");
    if (act != TE_ACT_GELU_TANH && act != TE_ACT_SILU) return fail(TE_EINVAL, "gate_act: bad act");
    if (rows < 0 || f < 8 || f % 8) return fail(TE_ESHAPE, "gate_act: rows=%d f=%d (f %% 8 == 0)", rows, f);
    if (ld < f || (u_off >= 0 && (int64_t)u_off + f > ld) || ldm < f)
        return fail(TE_ESHAPE, "gate_act: columns run past the row");
    if (!aligned16(gu) || !aligned16(m) || (ld * 2) % 16 || (ldm * 2) % 16 ||
        (u_off >= 0 && (u_off * 2) % 16))
        return fail(TE_EALIGN, "gate_act: rows and u_off must be 16-byte aligned");
    if (rows == 0) return TE_OK;
    const long long total = (long long)rows * (f / 8);
    const long long want = (total + 255) / 256;
    const unsigned blocks = (unsigned)(want < 152 * 16 ? want : 152 * 16);
    gate_act_kernel<<<blocks, 256, 0, stream>>>((const __nv_bfloat16 *)gu, ld, u_off, act,
                                                (__nv_bfloat16 *)m, ldm, rows, f);
    return launched("gate_act launch");
}

te_status te_pool_mean(const float *x, int32_t d, const int32_t *cu_host, const int32_t *cu_dev,
                       int32_t nseq, const float *w_final, float eps, float *out,
                       te_stream stream) {
    if (!x || !out) return fail(TE_EINVAL, "pool_mean: NULL x or out");
    if (d < 8 || d > 4096 || d % 8) return fail(TE_ESHAPE, "pool_mean: d=%d (d %% 8 == 0, 8..4096)", d);
    int32_t total = 0, mx = 0;
    te_status st = check_cu(cu_host, cu_dev, nseq, &total, &mx);
    if (st != TE_OK) return st;
    if (!aligned16(x) || !aligned16(out) || (w_final && !aligned16(w_final)))
        return fail(TE_EALIGN, "pool_mean: pointers must be 16-byte aligned");
    TE_NV_SWITCH(nv_for(d), {
        pool_kernel<NV><<<nseq, 256, d * sizeof(float), stream>>>(x, d, cu_dev, w_final, eps, out);
    })
    return launched("pool_mean launch");
}

te_status te_check(te_stream stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "te_check: stream");
    int rowop = 0;
    e = cudaMemcpyFromSymbol(&rowop, g_rowop_err, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "te_check: read error word");
    if (rowop) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_rowop_err, &zero, sizeof(int));
    }
    const int gemm = read_clear_gemm_error();
    const int attn = read_clear_attn_error();
    if (gemm < 0 || attn < 0) return fail(TE_ECUDA, "te_check: could not read device error words");
    if (rowop || gemm || attn)
        return fail(TE_EDEVICE, "device error words: rowops=%d gemm=%d attn=%d "
                    "(2 = RoPE table index out of range, 1 = bounded wait gave up)", rowop, gemm, attn);
    return TE_OK;
}

const char *te_last_error(void) { return g_msg; }

const char *te_version(void) { return "tefwd 0.1.0 (sm_103a)"; }

}  // extern "C"
