// host_pipeline.cu -- ring_attn_fwd on host-resident tensors, with the host<->device
// copies overlapped with the attention.
//
// Attention is independent per head, so the heads are processed in groups of
// `heads_per_group`.  Each group moves through three stages on three kinds of
// streams, rotating through three device slots of the caller's workspace:
//
//   copy-in stream   : q, k, v of group g, host [B, L, H, D] column block of
//                      heads [g*hg, (g+1)*hg)  ->  slot g%3, dense [B, L, hg, D]
//                      (one 2-D copy per tensor: rows of hg*D elements; one stream,
//                      since concurrent host-to-device copies slow the copies back)
//   compute stream   : ring_attn_fwd on the slot (two streams alternate, so the
//                      tail of one group's launch overlaps the head of the next),
//                      then the slot's lse [B, L, hg] scattered into a device
//                      [B, L, H] buffer
//   copy-out stream  : out of group g  ->  host column block (2-D copy)
//
// and after the last group the whole lse goes back in one copy.  The slot of
// group g is reused by group g+3 once group g's output copy has finished.
//
// The streams and events are created once per device and kept for the life of
// the process.  Enqueueing holds a per-device mutex, so calls from several host
// threads interleave safely; each call's work is ordered after the caller's
// stream's earlier work, and the caller's stream waits for all of it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "ra_check.cuh"
#include "ra_internal.h"
#include "ring_attn.h"

namespace {

constexpr int kSlots = 3;
constexpr int kMaxDevices = 64;

struct Pipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr, comp[2] = {nullptr, nullptr};
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t ev_in[kSlots] = {}, ev_comp[kSlots] = {}, ev_free[kSlots] = {};
    std::mutex enqueue;
};

Pipe g_pipe[kMaxDevices];
std::mutex g_init;

ra_status pipe_for_current_device(Pipe** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_init);
    Pipe& p = g_pipe[dev];
    if (!p.ready) {
        const unsigned fl = cudaStreamNonBlocking;
        const unsigned ef = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&p.in, fl) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.out, fl) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.comp[0], fl) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.comp[1], fl) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.start, ef) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.done, ef) == cudaSuccess;
        for (int s = 0; ok && s < kSlots; ++s)
            ok = cudaEventCreateWithFlags(&p.ev_in[s], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.ev_comp[s], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.ev_free[s], ef) == cudaSuccess;
        if (!ok) return RA_ERR_CUDA;   // what was created stays owned by the process
        p.ready = true;
    }
    *out = &p;
    return RA_OK;
}

unsigned long long round256(unsigned long long x) { return (x + 255ull) & ~255ull; }

// Byte layout of the workspace: kSlots x {q, k, v, out, lse of one group}, then the
// full lse [B, L, H].
struct Layout {
    unsigned long long tile, lse_slot, slot, lse_full, total;
};

bool layout(int B, int L, int H, int D, int hg, Layout* lay)
{
    if (B < 1 || L < 1 || H < 1 || D < 1 || hg < 1 || hg > H || H % hg != 0) return false;
    const unsigned long long rows = static_cast<unsigned long long>(B) * L;
    if (rows * H * D >= (1ull << 40)) return false;
    lay->tile = round256(rows * hg * D * 2);
    lay->lse_slot = round256(rows * hg * 4);
    lay->slot = 4 * lay->tile + lay->lse_slot;
    lay->lse_full = round256(rows * H * 4);
    lay->total = kSlots * lay->slot + lay->lse_full;
    return true;
}

bool host_overlap(const void* a, unsigned long long na, const void* b, unsigned long long nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// dst[row * H + h0 + j] = src[row * hg + j] for j < hg
__global__ void __launch_bounds__(256)
    lse_scatter_kernel(const float* __restrict__ src, float* __restrict__ dst, long long rows,
                       int hg, int H, int h0, unsigned int* status)
{
    const long long n = rows * hg;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = i / hg;
        const long long d = row * H + h0 + (i - row * hg);
        if (ra::in_bounds(i, 1, n, status) && ra::in_bounds(d, 1, rows * H, status)) dst[d] = src[i];
    }
}

}  // namespace

extern "C" {

unsigned long long ring_attn_fwd_host_workspace_bytes(int B, int L, int H, int D,
                                                      int heads_per_group)
{
    Layout lay;
    return layout(B, L, H, D, heads_per_group, &lay) ? lay.total : 0ull;
}

ra_status ring_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                             void* out_host, float* lse_host, void* workspace,
                             unsigned long long workspace_bytes, int B, int L, int H, int D, int P,
                             int causal, int heads_per_group, ra_stream_t stream)
{
    if (!q_host || !k_host || !v_host || !out_host || !workspace) return RA_ERR_INVALID_ARG;
    if (P < 1) return RA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return RA_ERR_UNSUPPORTED;
    Layout lay;
    if (!layout(B, L, H, D, heads_per_group, &lay)) {
        if (B >= 1 && H >= 1 && heads_per_group >= 1 && heads_per_group <= H &&
            H % heads_per_group != 0)
            return RA_ERR_NOT_DIVISIBLE;
        return RA_ERR_INVALID_ARG;
    }
    if (L % P != 0) return RA_ERR_NOT_DIVISIBLE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return RA_ERR_MISALIGNED;
    if (workspace_bytes < lay.total) return RA_ERR_INVALID_ARG;
    const int hg = heads_per_group;
    const unsigned long long rows = static_cast<unsigned long long>(B) * L;
    const unsigned long long bytes = rows * H * D * 2;
    if (host_overlap(out_host, bytes, q_host, bytes) || host_overlap(out_host, bytes, k_host, bytes) ||
        host_overlap(out_host, bytes, v_host, bytes))
        return RA_ERR_INVALID_ARG;
    if (lse_host && (host_overlap(lse_host, rows * H * 4, out_host, bytes) ||
                     host_overlap(lse_host, rows * H * 4, q_host, bytes)))
        return RA_ERR_INVALID_ARG;

    Pipe* pp = nullptr;
    ra_status st = pipe_for_current_device(&pp);
    if (st != RA_OK) return st;
    Pipe& p = *pp;
    std::lock_guard<std::mutex> lock(p.enqueue);
    const cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);

    auto fail = [](cudaError_t e) { return e != cudaSuccess; };
    // everything below runs after the caller's earlier work on its stream
    if (fail(cudaEventRecord(p.start, user)) || fail(cudaStreamWaitEvent(p.in, p.start, 0)) ||
        fail(cudaStreamWaitEvent(p.out, p.start, 0)) ||
        fail(cudaStreamWaitEvent(p.comp[0], p.start, 0)) ||
        fail(cudaStreamWaitEvent(p.comp[1], p.start, 0)))
        return RA_ERR_CUDA;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* lse_full = reinterpret_cast<float*>(ws + kSlots * lay.slot);
    const size_t row_all = static_cast<size_t>(H) * D * 2;     // host row pitch, bytes
    const size_t row_grp = static_cast<size_t>(hg) * D * 2;    // one group's part of a row
    const int groups = H / hg;
    for (int g = 0; g < groups; ++g) {
        const int s = g % kSlots;
        uint8_t* slot = ws + s * lay.slot;
        void* dq = slot;
        void* dk = slot + lay.tile;
        void* dv = slot + 2 * lay.tile;
        void* dout = slot + 3 * lay.tile;
        float* dlse = reinterpret_cast<float*>(slot + 4 * lay.tile);
        const size_t off = static_cast<size_t>(g) * row_grp;
        // copy in (after the slot's previous group has been copied out)
        if (g >= kSlots && fail(cudaStreamWaitEvent(p.in, p.ev_free[s], 0))) return RA_ERR_CUDA;
        const void* src[3] = {q_host, k_host, v_host};
        void* dst[3] = {dq, dk, dv};
        for (int t = 0; t < 3; ++t)
            if (fail(cudaMemcpy2DAsync(dst[t], row_grp, static_cast<const uint8_t*>(src[t]) + off,
                                       row_all, row_grp, rows, cudaMemcpyHostToDevice, p.in)))
                return RA_ERR_CUDA;
        if (fail(cudaEventRecord(p.ev_in[s], p.in))) return RA_ERR_CUDA;
        // attention on the slot
        const cudaStream_t cs = p.comp[g & 1];
        if (fail(cudaStreamWaitEvent(cs, p.ev_in[s], 0))) return RA_ERR_CUDA;
        st = ring_attn_fwd(dq, dk, dv, dout, lse_host ? dlse : nullptr, B, L, hg, D, P, causal,
                           reinterpret_cast<ra_stream_t>(cs));
        if (st != RA_OK) return st;
        if (lse_host) {
            const long long n = static_cast<long long>(rows) * hg;
            const unsigned blocks = static_cast<unsigned>(n / 256 + 1 < 1024 ? n / 256 + 1 : 1024);
            unsigned int* status = nullptr;
            st = ra::current_status_word(&status);
            if (st != RA_OK) return st;
            lse_scatter_kernel<<<blocks, 256, 0, cs>>>(dlse, lse_full, static_cast<long long>(rows),
                                                       hg, H, g * hg, status);
            if (fail(cudaGetLastError())) return RA_ERR_CUDA;
        }
        if (fail(cudaEventRecord(p.ev_comp[s], cs))) return RA_ERR_CUDA;
        // copy out
        if (fail(cudaStreamWaitEvent(p.out, p.ev_comp[s], 0))) return RA_ERR_CUDA;
        if (fail(cudaMemcpy2DAsync(static_cast<uint8_t*>(out_host) + off, row_all, dout, row_grp,
                                   row_grp, rows, cudaMemcpyDeviceToHost, p.out)))
            return RA_ERR_CUDA;
        if (fail(cudaEventRecord(p.ev_free[s], p.out))) return RA_ERR_CUDA;
    }
    if (lse_host) {
        // the scatters ran on both compute streams: the copy-out stream has waited for
        // every group's ev_comp, so it follows all of them
        if (fail(cudaMemcpyAsync(lse_host, lse_full, rows * H * 4, cudaMemcpyDeviceToHost, p.out)))
            return RA_ERR_CUDA;
    }
    // the caller's stream follows the last copy out (and with it every earlier stage)
    if (fail(cudaEventRecord(p.done, p.out)) || fail(cudaStreamWaitEvent(user, p.done, 0)))
        return RA_ERR_CUDA;
    return RA_OK;
}

}  // extern "C"
