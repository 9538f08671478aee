// noalloc.cu -- qlin_quantize_noalloc: the quantizer for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine): code that
// runs while a caching allocator holds its lock, a plug-in whose host
// framework owns all device memory, or a hot loop whose memory plan is fixed
// ahead of time.  qlin_quantize needs a caller-provided workspace for the
// per-tensor, per-column and percentile scopes (cross-block range statistics
// and histograms).  This entry point takes the same arguments minus the
// workspace and uses a fixed scratch array in the library's own device memory
// instead.
#include <mutex>

#include "qlin_common.cuh"
#include "qlin_internal.h"

namespace qlin {

// Fixed scratch: every GPU that loads the library holds this much device
// memory until the process exits.  It covers the percentile histograms
// (393,232 bytes) and the range statistics of up to 65,536 columns.
constexpr size_t kNoAllocScratchBytes = QLIN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device (host code only sees a
// host-side stand-in for the array's name).  Outside stream capture the
// address is looked up again on every call, so a context that was torn down
// and re-created (cudaDeviceReset) never receives a stale address; during a
// capture the address cached by an earlier call on that device is used.
static void* g_noalloc_ptr[256];
static std::mutex g_noalloc_mu;

static int noalloc_scratch(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return QLIN_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return QLIN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (cap == cudaStreamCaptureStatusNone || !g_noalloc_ptr[dev]) {
        if (cap != cudaStreamCaptureStatusNone) return QLIN_ERR_CUDA;  // first call must precede any capture
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QLIN_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return QLIN_OK;
}

}  // namespace qlin

extern "C" {

int qlin_quantize_noalloc(const void* x, qlin_dtype xt, int64_t rows, int64_t cols, int64_t ld, const float* smooth,
                          const qlin_qparams* p, void* q, void* s, int32_t* z, void* stream) {
    // the argument checks of qlin_quantize come first, so a bad argument
    // reports QLIN_ERR_ARG / QLIN_ERR_UNSUPPORTED exactly as there
    int rc = qlin::quantize_check(x, xt, rows, cols, ld, smooth, p, q, s, z);
    if (rc == qlin::QLIN_NOTHING_TO_DO) return QLIN_OK;
    if (rc != QLIN_OK) return rc;
    const size_t need = qlin::quantize_ws_bytes(rows, cols, p);
    if (need > qlin::kNoAllocScratchBytes) return QLIN_ERR_WORKSPACE;
    void* ws = nullptr;
    if (need > 0) {
        rc = qlin::noalloc_scratch((cudaStream_t)stream, &ws);
        if (rc != QLIN_OK) return rc;
    }
    return qlin_quantize(x, xt, rows, cols, ld, smooth, p, q, s, z, ws, need, stream);
}

}  // extern "C"
