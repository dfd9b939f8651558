// Unpacking of the 32-element block weight formats into the q8 GEMM's
// operands: int8 q [n, k] and f16 block scales [n, k/32].
//
// Source: "cera 0.2.4 src/model/vision_encoder_gpu.rs" - the test quantisers
// (q8_0_weight: 34 bytes a block, f16 scale then 32 int8; q4_0_weight: 18
// bytes a block, f16 scale then 16 bytes whose low nibbles are elements 0-15
// and high nibbles elements 16-31, each stored with an offset of 8) and
// upload_weight (the packed bytes are kept and decoded by the GEMM).
//
// Here the decode happens once, when the weights are loaded: the GEMM then
// reads int8 through TMA exactly as for q8_row and applies the block scale
// while widening (q8_linear.cu).  One thread per block; integer work, exact.
#include "common.cuh"

namespace tefwd {
namespace {

// Bytes b0..b15 (as 4 words) of one block's 16 or 32 payload bytes -> int8 q.
__global__ void q8_0_unpack_kernel(const uint8_t *__restrict__ packed, long long nblocks,
                                   int8_t *__restrict__ q, uint16_t *__restrict__ bs) {
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint16_t *src = reinterpret_cast<const uint16_t *>(packed + b * 34);   // 2-byte aligned
    bs[b] = src[0];
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (uint32_t)src[1 + 2 * i] | ((uint32_t)src[2 + 2 * i] << 16);
    uint4 *dst = reinterpret_cast<uint4 *>(q + b * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

__global__ void q4_0_unpack_kernel(const uint8_t *__restrict__ packed, long long nblocks,
                                   int8_t *__restrict__ q, uint16_t *__restrict__ bs) {
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint16_t *src = reinterpret_cast<const uint16_t *>(packed + b * 18);   // 2-byte aligned
    bs[b] = src[0];
    uint8_t by[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint16_t v = src[1 + i];
        by[2 * i] = (uint8_t)(v & 0xFFu);
        by[2 * i + 1] = (uint8_t)(v >> 8);
    }
    uint32_t lo[4], hi[4];   // elements 0-15 from the low nibbles, 16-31 from the high
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        lo[j] = hi[j] = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint8_t v = by[4 * j + e];
            lo[j] |= (uint32_t)(uint8_t)((int)(v & 15) - 8) << (8 * e);
            hi[j] |= (uint32_t)(uint8_t)((int)(v >> 4) - 8) << (8 * e);
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(q + b * 32);
    dst[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    dst[1] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
}

te_status check_unpack(const void *packed, int32_t n, int32_t k, const int8_t *q, const uint16_t *bs,
                       const char *what) {
    if (!packed || !q || !bs) return fail(TE_EINVAL, "%s: NULL packed, q or block_scale", what);
    if (n < 0 || k < 32 || k % 32) return fail(TE_ESHAPE, "%s: n=%d k=%d (k %% 32 == 0)", what, n, k);
    if ((reinterpret_cast<uintptr_t>(packed) & 1) || !aligned16(q) || (reinterpret_cast<uintptr_t>(bs) & 3))
        return fail(TE_EALIGN, "%s: packed 2-byte, q 16-byte, block_scale 4-byte aligned", what);
    return TE_OK;
}

}  // namespace
}  // namespace tefwd

using namespace tefwd;

extern "C" te_status te_q8_0_unpack(const void *packed, int32_t n, int32_t k, int8_t *q,
                                    uint16_t *block_scale, te_stream stream) {
    te_status st = check_unpack(packed, n, k, q, block_scale, "q8_0_unpack");
    if (st != TE_OK) return st;
    const long long nb = (long long)n * (k / 32);
    if (nb == 0) return TE_OK;
    q8_0_unpack_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(packed), nb, q, block_scale);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TE_OK : cuda_fail(e, "q8_0_unpack launch");
}

extern "C" te_status te_q4_0_unpack(const void *packed, int32_t n, int32_t k, int8_t *q,
                                    uint16_t *block_scale, te_stream stream) {
    te_status st = check_unpack(packed, n, k, q, block_scale, "q4_0_unpack");
    if (st != TE_OK) return st;
    const long long nb = (long long)n * (k / 32);
    if (nb == 0) return TE_OK;
    q4_0_unpack_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(packed), nb, q, block_scale);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TE_OK : cuda_fail(e, "q4_0_unpack launch");
}
