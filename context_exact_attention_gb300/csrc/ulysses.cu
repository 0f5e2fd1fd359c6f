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
// The grid is one resident wave (occupancy query); index math is 32-bit when
// the buffer has fewer than 2^31 vectors.
#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kBlock = 256;
constexpr int kBatch = 4;   // chunks in flight per warp

template <typename I>
struct PermuteGeom {
    I n_chunks;    // chunks in the whole buffer
    I cv;          // 16-byte vectors per chunk (Hg * D * elem / 16)
    I hv;          // vectors per position on the sequence side (H * D * elem / 16)
    I B, L, Ls, P;
};

// Output chunk ch -> first vector of its source chunk.
//   dir 0 (seq -> head): ch = (g*B + b)*L + lg with lg = r*Ls + l;
//                        source = ((r*B + b)*Ls + l)*hv + g*cv.
//   dir 1 (head -> seq): ch = ((r*B + b)*Ls + l)*P + g;
//                        source = ((g*B + b)*L + r*Ls + l)*cv.
template <int kDir, typename I>
__device__ __forceinline__ I source_chunk(I ch, const PermuteGeom<I>& g)
{
    if (kDir == 0) {
        const I gb = ch / g.L;
        const I lg = ch - gb * g.L;
        const I grp = gb / g.B;
        const I b = gb - grp * g.B;
        const I r = lg / g.Ls, l = lg - r * g.Ls;
        return ((r * g.B + b) * g.Ls + l) * g.hv + grp * g.cv;
    } else {
        const I rbl = ch / g.P;
        const I grp = ch - rbl * g.P;
        const I rb = rbl / g.Ls;
        const I l = rbl - rb * g.Ls;
        const I r = rb / g.B;
        const I b = rb - r * g.B;
        return ((grp * g.B + b) * g.L + r * g.Ls + l) * g.cv;
    }
}

// I is the index type of vectors (32-bit when the whole buffer has < 2^31 vectors).
template <int kDir, typename I>
__global__ void __launch_bounds__(kBlock)
    permute_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, PermuteGeom<I> g)
{
    const int lane = threadIdx.x & 31;
    const I warp_global = static_cast<I>((blockIdx.x * kBlock + threadIdx.x) >> 5);
    const I n_warps = static_cast<I>((gridDim.x * kBlock) >> 5);
    for (I ch0 = warp_global; ch0 < g.n_chunks; ch0 += kBatch * n_warps) {
        I src[kBatch], dst[kBatch];
        bool live[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const I ch = ch0 + u * n_warps;
            live[u] = ch < g.n_chunks;
            src[u] = live[u] ? source_chunk<kDir>(ch, g) : I(0);
            dst[u] = ch * g.cv;
        }
        for (I c = lane; c < g.cv; c += 32) {
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

template <int kDir, typename I>
cudaError_t launch_typed(const void* in, void* out, int B, int L, int H, int D, int P,
                         int elem_bytes, cudaStream_t stream)
{
    PermuteGeom<I> g;
    g.B = B;
    g.L = L;
    g.P = P;
    g.Ls = L / P;
    g.cv = static_cast<I>(static_cast<long long>(H / P) * D * elem_bytes / 16);
    g.hv = static_cast<I>(static_cast<long long>(H) * D * elem_bytes / 16);
    g.n_chunks = static_cast<I>(static_cast<long long>(B) * L * P);
    int dev = 0, sms = 148, per_sm = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, permute_kernel<kDir, I>, kBlock, 0);
    const long long warps_needed = (static_cast<long long>(g.n_chunks) + kBatch - 1) / kBatch;
    long long blocks = (warps_needed * 32 + kBlock - 1) / kBlock;
    const long long cap = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);  // one resident wave
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    permute_kernel<kDir, I><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(
        static_cast<const uint4*>(in), static_cast<uint4*>(out), g);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ulysses_permute(const void* in, void* out, int B, int L, int H, int D, int P,
                                   int elem_bytes, int dir, cudaStream_t stream)
{
    const long long total_vec = static_cast<long long>(B) * L * H * D * elem_bytes / 16;
    const bool small = total_vec < (1ll << 30);   // headroom for the grid-stride steps
    if (dir == 0)
        return small ? launch_typed<0, int>(in, out, B, L, H, D, P, elem_bytes, stream)
                     : launch_typed<0, long long>(in, out, B, L, H, D, P, elem_bytes, stream);
    return small ? launch_typed<1, int>(in, out, B, L, H, D, P, elem_bytes, stream)
                 : launch_typed<1, long long>(in, out, B, L, H, D, P, elem_bytes, stream);
}

}  // namespace ra
