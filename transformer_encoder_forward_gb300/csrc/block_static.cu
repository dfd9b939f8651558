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

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_block_scratch[TE_STATIC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// The driver's cuCtxGetCurrent, looked up once (the library links only the
// runtime): it names the context a cached address belongs to.
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    });
    return fn;
}

std::mutex g_scratch_mu;
struct ScratchEntry {
    void *addr;
    CUcontext ctx;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Device address of g_block_scratch on the current device.  Host code only
// holds a host-side stand-in for the array's name, so the address is looked
// up with the device current and cached per device, together with the
// context it belongs to: a destroyed and recreated context (cudaDeviceReset)
// reloads the module, and the address is then looked up again.
te_status scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "block_static: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(TE_EINVAL, "block_static: device %d beyond the supported %d", dev, kMaxDevices);
    CtxGetCurrentFn get = ctx_get_current();
    auto current = [&]() {
        CUcontext c = nullptr;
        if (get && get(&c) != CUDA_SUCCESS) c = nullptr;
        return c;
    };
    const CUcontext ctx = current();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry &ent = g_scratch[dev];
    if (!ent.addr || !ctx || ent.ctx != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_block_scratch);
        if (e != cudaSuccess || !p)
            return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                             "block_static: cudaGetSymbolAddress(scratch)");
        ent.addr = p;
        ent.ctx = current();   // the lookup made the device's context current if none was
    }
    *out = ent.addr;
    return TE_OK;
}

}  // namespace
}  // namespace tefwd

using namespace tefwd;

extern "C" te_status te_encoder_block_fwd_static(const te_block_desc *desc, float *x, void *a,
                                                 const int32_t *cu_host, const int32_t *cu_dev,
                                                 int32_t nseq, te_stream stream) {
    te_status st = check_block_desc(desc);
    if (st != TE_OK) return st;
    int32_t t = 0, max_len = 0;
    if ((st = check_cu(cu_host, cu_dev, nseq, &t, &max_len)) != TE_OK) return st;
    const size_t need = te_encoder_block_workspace(desc, t);
    if (need > TE_STATIC_SCRATCH_BYTES)
        return fail(TE_EWORKSPACE,
                    "block_static: %d rows need %zu bytes of scratch, the static array holds %zu "
                    "(TE_STATIC_SCRATCH_BYTES); use te_encoder_block_fwd with a workspace",
                    t, need, (size_t)TE_STATIC_SCRATCH_BYTES);
    void *scratch = nullptr;
    if ((st = scratch_address(&scratch)) != TE_OK) return st;
    return te_encoder_block_fwd(desc, x, a, cu_host, cu_dev, nseq, scratch, TE_STATIC_SCRATCH_BYTES,
                                stream);
}
