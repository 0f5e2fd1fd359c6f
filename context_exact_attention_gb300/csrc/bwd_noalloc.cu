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
// (4 MiB).  It comes into being on a device when the CUDA runtime loads this
// file's module there: at context creation when the process runs with
// CUDA_MODULE_LOADING=EAGER, otherwise (lazy loading, the default) on the first
// call on that device.  Its 4 MiB are then held until the process exits.  A
// caller that must not allocate after some point makes one call on each device
// before it (or runs with eager loading).
//
// In host code the array's name is only a host-side stand-in, so every call
// looks up its device address through cudaGetSymbolAddress with the device
// current, and passes that address on.  The lookup is repeated on each call (it
// is a table lookup once the module is loaded), so a device reset, after which
// the module may be loaded again at another address, leaves no stale pointer.
//
// Every call on a device shares the one array and leaves its contents behind;
// nothing in it needs to start at zero, since each call writes every row it later
// reads.  Calls whose work overlaps on the GPU (for example on two streams) race
// on the array: the caller must order them.
#include <cuda_runtime.h>

#include "ring_attn.h"

namespace {

constexpr unsigned long long kMaxRows = RA_BWD_NOALLOC_MAX_ROWS;

static __device__ __align__(256) float g_bwd_noalloc_scratch[kMaxRows];

}  // namespace

extern "C" ra_status ring_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                           const void* out, const float* lse, const void* dout,
                                           void* dq, void* dk, void* dv, int B, int L, int H,
                                           int D, int P, int causal, ra_stream_t stream)
{
    if (B < 1 || L < 1 || H < 1) return RA_ERR_INVALID_ARG;
    const unsigned long long rows = static_cast<unsigned long long>(B) * L * H;
    if (rows > kMaxRows) return RA_ERR_INVALID_ARG;   // larger problems: use ring_attn_bwd
    // device address of the array on the current device
    void* scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_bwd_noalloc_scratch) != cudaSuccess) return RA_ERR_CUDA;
    return ring_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, scratch, kMaxRows * sizeof(float), B,
                         L, H, D, P, causal, stream);
}
