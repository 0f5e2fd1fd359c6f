// bwd_noalloc.cu -- the attention backward for callers that cannot allocate.
//
// ring_attn_bwd needs a small device workspace (one fp32 per query row) and
// asks the caller for it.  Some callers have no way to provide one: a plugin
// that a host application hands only its input and output tensors, a runtime
// that reserves all device memory for its own pool up front and gives library
// code no allocator, or a latency-critical server that forbids any allocation
// after warm-up.  For them, ring_attn_bwd_noalloc takes the workspace from a
// fixed array compiled into this library instead, and calls no allocating
// routine (no cudaMalloc / cudaFree, nothing of torch's).
//
// The array: `g_bwd_noalloc_scratch` below, RA_BWD_NOALLOC_MAX_ROWS floats
// (4 MiB).  Every GPU that loads the library holds it until the process exits.
// In host code its name is only a host-side stand-in, so the entry point looks
// up its device address once per device, with that device current, through
// cudaGetSymbolAddress, and passes that address on.  That lookup happens inside
// the first call on each device.  Every call on a device shares the one array
// and leaves its contents behind; nothing in it needs to start at zero, since
// each call writes every row it later reads.  Calls whose work overlaps on the
// GPU (for example on two streams) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "ring_attn.h"

namespace {

constexpr unsigned long long kMaxRows = RA_BWD_NOALLOC_MAX_ROWS;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_bwd_noalloc_scratch[kMaxRows];

float* g_scratch_dev_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

// Device address of the array on the current device (looked up on first use).
ra_status scratch_on_current_device(float** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_dev_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_noalloc_scratch) != cudaSuccess) return RA_ERR_CUDA;
        g_scratch_dev_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_dev_ptr[dev];
    return RA_OK;
}

}  // namespace

extern "C" ra_status ring_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                           const void* out, const float* lse, const void* dout,
                                           void* dq, void* dk, void* dv, int B, int L, int H,
                                           int D, int P, int causal, ra_stream_t stream)
{
    if (B < 1 || L < 1 || H < 1) return RA_ERR_INVALID_ARG;
    const unsigned long long rows = static_cast<unsigned long long>(B) * L * H;
    if (rows > kMaxRows) return RA_ERR_INVALID_ARG;   // larger problems: use ring_attn_bwd
    float* scratch = nullptr;
    const ra_status st = scratch_on_current_device(&scratch);
    if (st != RA_OK) return st;
    return ring_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, scratch, kMaxRows * sizeof(float), B,
                         L, H, D, P, causal, stream);
}
