// te_encoder_block_fwd_static: the encoder block without a caller-provided
// workspace, for callers that cannot allocate device memory.
//
// The block needs scratch for its intermediates (the q|k|v panel, the
// attention output, the projection output, the gate|up panel and the FFN
// hidden).  te_encoder_block_fwd takes that scratch from the caller.  Some
// callers cannot provide it: a host application that has already handed all
// device memory to its own allocator and forbids plug-ins from calling
// cudaMalloc, or a latency-critical path that must never allocate.  This entry
// point uses instead one fixed array in device memory that belongs to the
// library: it is created when the library's device code is loaded, every GPU
// that loads the library holds it until the process exits, and it is never
// allocated or freed by a call.
#include <mutex>

#include "common.cuh"

namespace tefwd {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)32 << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_block_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_block_scratch on the current device.  Host code only
// holds a host-side stand-in for the array's name, so the address is looked
// up once per device with that device current, and cached.
te_status scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "block_static: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(TE_EINVAL, "block_static: device %d beyond the supported %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_block_scratch);
        if (e != cudaSuccess || !p)
            return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                             "block_static: cudaGetSymbolAddress(scratch)");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return TE_OK;
}

}  // namespace
}  // namespace tefwd

using namespace tefwd;

extern "C" te_status te_encoder_block_fwd_static(const te_block_desc *desc, float *x, void *a,
                                                 const int32_t *cu_host, const int32_t *cu_dev,
                                                 int32_t nseq, te_stream stream) {
    if (!desc) return fail(TE_EINVAL, "block_static: NULL descriptor");
    int32_t t = 0, max_len = 0;
    te_status st = check_cu(cu_host, cu_dev, nseq, &t, &max_len);
    if (st != TE_OK) return st;
    const size_t need = te_encoder_block_workspace(desc, t);
    if (need > kStaticScratchBytes)
        return fail(TE_EWORKSPACE,
                    "block_static: %d rows need %zu bytes of scratch, the static array holds %zu; "
                    "use te_encoder_block_fwd with a workspace", t, need, kStaticScratchBytes);
    void *scratch = nullptr;
    if ((st = scratch_address(&scratch)) != TE_OK) return st;
    return te_encoder_block_fwd(desc, x, a, cu_host, cu_dev, nseq, scratch, kStaticScratchBytes,
                                stream);
}
