// ulysses.cu -- the Ulysses all-to-all as an on-device layout transpose
// ("序列并行与 Ring Attention", section 3.5): sequence-sharded
// [P][B][L/P][H][D] <-> head-sharded [P][B][L][H/P][D].
//
// For fixed (source rank r, batch b, position l, head group g) the H/P heads of
// group g form one contiguous run ("chunk") of Hg*D elements on both sides, so
// the transpose is a gather of contiguous chunks.  A warp takes four chunks at
// a time (index math once per chunk), its lanes stream each chunk's 16-byte
// vectors: all loads of the four chunks are issued before their stores, reads
// and writes are coalesced, and the data is touched once (streaming hints).
#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kBlock = 256;
constexpr int kBatch = 4;   // chunks in flight per warp

struct PermuteGeom {
    long long n_chunks;    // chunks in the whole buffer
    long long cv;          // 16-byte vectors per chunk (Hg * D * elem / 16)
    long long hv;          // vectors per position on the sequence side (H * D * elem / 16)
    long long B, L, Ls, P;
};

// Output chunk ch -> first vector of its source chunk.
//   dir 0 (seq -> head): ch = (g*B + b)*L + lg with lg = r*Ls + l;
//                        source = ((r*B + b)*Ls + l)*hv + g*cv.
//   dir 1 (head -> seq): ch = ((r*B + b)*Ls + l)*P + g;
//                        source = ((g*B + b)*L + r*Ls + l)*cv.
template <int kDir>
__device__ __forceinline__ long long source_chunk(long long ch, const PermuteGeom& g)
{
    if (kDir == 0) {
        const long long lg = ch % g.L;
        const long long gb = ch / g.L;
        const long long b = gb % g.B;
        const long long grp = gb / g.B;
        const long long r = lg / g.Ls, l = lg - r * g.Ls;
        return ((r * g.B + b) * g.Ls + l) * g.hv + grp * g.cv;
    } else {
        const long long grp = ch % g.P;
        const long long rbl = ch / g.P;
        const long long l = rbl % g.Ls;
        const long long rb = rbl / g.Ls;
        const long long b = rb % g.B;
        const long long r = rb / g.B;
        return ((grp * g.B + b) * g.L + r * g.Ls + l) * g.cv;
    }
}

template <int kDir>
__global__ void __launch_bounds__(kBlock)
    permute_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, PermuteGeom g)
{
    const int lane = threadIdx.x & 31;
    const long long warp_global = (static_cast<long long>(blockIdx.x) * kBlock + threadIdx.x) >> 5;
    const long long n_warps = (static_cast<long long>(gridDim.x) * kBlock) >> 5;
    for (long long ch0 = warp_global; ch0 < g.n_chunks; ch0 += kBatch * n_warps) {
        long long src[kBatch], dst[kBatch];
        bool live[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const long long ch = ch0 + u * n_warps;
            live[u] = ch < g.n_chunks;
            src[u] = live[u] ? source_chunk<kDir>(ch, g) : 0;
            dst[u] = ch * g.cv;
        }
        for (long long c = lane; c < g.cv; c += 32) {
            uint4 x[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (live[u]) x[u] = __ldcs(in + src[u] + c);
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (live[u]) __stcs(out + dst[u] + c, x[u]);
        }
    }
}

}  // namespace

cudaError_t launch_ulysses_permute(const void* in, void* out, int B, int L, int H, int D, int P,
                                   int elem_bytes, int dir, cudaStream_t stream)
{
    PermuteGeom g;
    g.B = B;
    g.L = L;
    g.P = P;
    g.Ls = L / P;
    g.cv = static_cast<long long>(H / P) * D * elem_bytes / 16;
    g.hv = static_cast<long long>(H) * D * elem_bytes / 16;
    g.n_chunks = static_cast<long long>(B) * L * P;   // B*L positions x P groups, either side
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long warps_needed = (g.n_chunks + kBatch - 1) / kBatch;
    long long blocks = (warps_needed * 32 + kBlock - 1) / kBlock;
    const long long cap = static_cast<long long>(sms) * 8;   // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (dir == 0)
        permute_kernel<0><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(
            static_cast<const uint4*>(in), static_cast<uint4*>(out), g);
    else
        permute_kernel<1><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(
            static_cast<const uint4*>(in), static_cast<uint4*>(out), g);
    return cudaGetLastError();
}

}  // namespace ra
