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
//
// The usual shapes (D and H/P up to 256, a run of H/P heads at most 32 KB) take a
// copy-engine path instead (permute_tma_kernel): for a fixed source rank r and batch
// b, R consecutive positions of head group g are one box {D, H/P, 1, R, 1} of a 5-D
// view {D, H/P, P, L/P, P*B} of the sequence-sharded buffer, and one contiguous run of
// R*H/P*D elements of the head-sharded buffer.  One thread per CTA streams such tiles
// through four shared-memory stages: a TMA tiled load and a 1-D bulk store (seq ->
// head), or a bulk load and a TMA tiled store (head -> seq).  The view's row dimension
// ends at L/P, so a ragged last box reads zeros past the shard and a store of it writes
// only the shard's rows.
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
    long long n_vec;        // 16-byte vectors in each buffer (the debug build's extent)
    unsigned int* status;
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
            live[u] = live[u] && in_bounds(src[u], g.cv, g.n_vec, g.status) &&
                      in_bounds(dst[u], g.cv, g.n_vec, g.status);
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
                         int elem_bytes, unsigned int* status, cudaStream_t stream)
{
    PermuteGeom<I> g;
    g.n_vec = static_cast<long long>(B) * L * H * D * elem_bytes / 16;
    g.status = status;
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

// -------------------------------------------------------- copy-engine path --

constexpr int kTStages = 4;
constexpr int kTStageMax = 32768;     // bytes of one stage (a tile of R rows)

struct TmaPermute {
    long long n_tiles;       // (P*B) * row blocks * P
    int n_rblk;              // row blocks per (r, b): ceil(Ls / R)
    int R;                   // rows per tile (the box's row extent)
    int P, B, Ls, L;
    int row_bytes;           // one position's run of H/P heads: H/P * D * elem
    int stage_bytes;         // R * row_bytes rounded up to 1024
    long long head_bytes;    // size of the head-sharded buffer (the debug build's extent)
    unsigned int* status;
    unsigned long long timeout_ns;
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2, int c3, int c4)
{
    asm volatile("cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
                 "r"(c4)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// every committed store group but the most recent one has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all_but_one()
{
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// dir 0 (seq -> head): tiled load from the 5-D view, bulk store to the head side.
// dir 1 (head -> seq): bulk load from the head side, tiled store to the 5-D view.
template <int kDir>
__global__ void __launch_bounds__(32, 1)
    permute_tma_kernel(const __grid_constant__ CUtensorMap seq_map, uint8_t* head, const TmaPermute p)
{
    extern __shared__ uint8_t smem_raw[];
    if (threadIdx.x != 0) return;   // one thread drives every copy of the CTA
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bars = sbase + kTStages * p.stage_bytes;
    int* abort_flag = reinterpret_cast<int*>(smem + kTStages * p.stage_bytes + 8 * kTStages);
    *abort_flag = 0;
    for (int s = 0; s < kTStages; ++s) mbar_init(bars + 8 * s, 1);
    fence_mbar_init();
    const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
    const uint64_t once = l2_policy_evict_first();

    // tile t = (rb * n_rblk + k) * P + g: neighbouring tiles read or write neighbouring
    // head groups of the same positions on the sequence side
    auto decode = [&](long long t, int& rb, int& g, int& l0, int& rows, size_t& off) {
        g = static_cast<int>(t % p.P);
        const long long rest = t / p.P;
        const int k = static_cast<int>(rest % p.n_rblk);
        rb = static_cast<int>(rest / p.n_rblk);
        l0 = k * p.R;
        rows = min(p.R, p.Ls - l0);
        const int r = rb / p.B, b = rb - r * p.B;
        off = ((static_cast<size_t>(g) * p.B + b) * p.L + static_cast<size_t>(r) * p.Ls + l0) *
              static_cast<size_t>(p.row_bytes);
    };
    auto tile_of = [&](long long j) { return static_cast<long long>(blockIdx.x) + j * gridDim.x; };
    auto load = [&](long long j) {
        int rb, g, l0, rows;
        size_t off;
        decode(tile_of(j), rb, g, l0, rows, off);
        const int s = static_cast<int>(j % kTStages);
        const uint32_t dst = sbase + s * p.stage_bytes;
        if constexpr (kDir == 0) {
            mbar_arrive_expect_tx(bars + 8 * s, static_cast<uint32_t>(p.R * p.row_bytes));
            tma_load_5d(dst, &seq_map, bars + 8 * s, 0, 0, g, l0, rb, once);
        } else if (in_bounds(static_cast<long long>(off), static_cast<long long>(rows) * p.row_bytes,
                             p.head_bytes, p.status)) {
            mbar_arrive_expect_tx(bars + 8 * s, static_cast<uint32_t>(rows * p.row_bytes));
            bulk_load(dst, head + off, static_cast<uint32_t>(rows * p.row_bytes), bars + 8 * s, once);
        } else {
            mbar_arrive(bars + 8 * s);     // skipped copy: complete the phase without data
        }
    };
    long long n_mine = 0;                       // tiles of this CTA
    if (blockIdx.x < p.n_tiles) n_mine = (p.n_tiles - 1 - blockIdx.x) / gridDim.x + 1;
    long long issued = 0;
    for (; issued < n_mine && issued < kTStages; ++issued) load(issued);
    long long j = 0;
    for (; j < n_mine; ++j) {
        const int s = static_cast<int>(j % kTStages);
        if (!mbar_wait(bars + 8 * s, static_cast<uint32_t>((j / kTStages) & 1), wc)) break;
        int rb, g, l0, rows;
        size_t off;
        decode(tile_of(j), rb, g, l0, rows, off);
        const uint32_t src = sbase + s * p.stage_bytes;
        if constexpr (kDir == 0) {
            if (in_bounds(static_cast<long long>(off), static_cast<long long>(rows) * p.row_bytes,
                          p.head_bytes, p.status))
                bulk_store(head + off, src, static_cast<uint32_t>(rows * p.row_bytes));
        } else
            tma_store_5d(&seq_map, src, 0, 0, g, l0, rb);
        bulk_commit();
        // the previous tile's stage is free once its store has read it: refill it
        if (j >= 1 && issued < n_mine) {
            bulk_wait_read_all_but_one();
            load(issued);
            ++issued;
        }
    }
    // loads still in flight (only after a timed-out wait, from tile j on) land before
    // the CTA leaves
    for (long long x = j; x < issued; ++x)
        mbar_wait_drain(bars + 8 * static_cast<int>(x % kTStages), static_cast<uint32_t>((x / kTStages) & 1), wc);
    bulk_wait_all();
}

}  // namespace

bool ulysses_permute_tma_fits(int H, int D, int P, int elem_bytes)
{
    const long long hg = H / P;
    return D <= 256 && hg <= 256 && hg * D * elem_bytes <= kTStageMax;
}

int ulysses_permute_tma_rows(int L, int H, int D, int P, int elem_bytes)
{
    const int row_bytes = H / P * D * elem_bytes;
    int R = kTStageMax / row_bytes;
    if (R > 256) R = 256;
    if (R > L / P) R = L / P;
    return R < 1 ? 1 : R;
}

cudaError_t launch_ulysses_permute_tma(const CUtensorMap& seq_map, void* head_side, int B, int L,
                                       int H, int D, int P, int elem_bytes, int dir, int R,
                                       unsigned int* status, unsigned long long timeout_ns,
                                       cudaStream_t stream)
{
    TmaPermute p;
    p.P = P;
    p.B = B;
    p.L = L;
    p.Ls = L / P;
    p.R = R;
    p.n_rblk = (p.Ls + R - 1) / R;
    p.row_bytes = H / P * D * elem_bytes;
    p.stage_bytes = (R * p.row_bytes + 1023) & ~1023;
    p.n_tiles = static_cast<long long>(P) * B * p.n_rblk * P;
    p.head_bytes = static_cast<long long>(B) * L * H * D * elem_bytes;
    p.status = status;
    p.timeout_ns = timeout_ns;
    constexpr int kSmemMax = kTStages * kTStageMax + 1024 + 8 * kTStages + 16;
    const int smem = kTStages * p.stage_bytes + 1024 + 8 * kTStages + 16;
    // shared-memory limit set, per direction and device
    static std::atomic<int> configured[2][kMaxDevices];
    int dev = 0, sms = 148;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    auto kern = dir == 0 ? permute_tma_kernel<0> : permute_tma_kernel<1>;
    e = smem_limit_once(configured[dir ? 1 : 0], dev, kern, kSmemMax);
    if (e != cudaSuccess) return e;
    long long grid = p.n_tiles < sms ? p.n_tiles : sms;
    if (grid < 1) grid = 1;
    kern<<<static_cast<unsigned>(grid), 32, smem, stream>>>(seq_map, static_cast<uint8_t*>(head_side), p);
    return cudaGetLastError();
}

cudaError_t launch_ulysses_permute(const void* in, void* out, int B, int L, int H, int D, int P,
                                   int elem_bytes, int dir, unsigned int* status, cudaStream_t stream)
{
    const long long total_vec = static_cast<long long>(B) * L * H * D * elem_bytes / 16;
    const bool small = total_vec < (1ll << 30);   // headroom for the grid-stride steps
    if (dir == 0)
        return small ? launch_typed<0, int>(in, out, B, L, H, D, P, elem_bytes, status, stream)
                     : launch_typed<0, long long>(in, out, B, L, H, D, P, elem_bytes, status, stream);
    return small ? launch_typed<1, int>(in, out, B, L, H, D, P, elem_bytes, status, stream)
                 : launch_typed<1, long long>(in, out, B, L, H, D, P, elem_bytes, status, stream);
}

}  // namespace ra
