// attn_f32.cu -- fp32 exact attention over P virtual ring shards on the SIMT
// cores, for results at fp32 tolerance (tensor-core tf32 would not meet it).
//
// Same operation and schedule as the bf16 kernel ("序列并行与 Ring Attention",
// sections 3.1-3.4): the queries of shard r meet shard (r - t) mod P at step t,
// wholly-future shards are skipped under causal masking, and the online-softmax
// recurrence of section 3.2 runs over blocks of 32 keys with natural-base
// exponentials (expf, full precision).
//
// One warp owns one query row.  Lane j scores key j of the current 32-key
// block (query row broadcast from shared memory), the block max and sum are
// warp reductions, and lane d accumulates output columns d, d+32, ...
#include <cmath>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxD = 256;

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Global position of local row i of a shard: contiguous shards, or zigzag (shard
// r holds chunks r and 2P-1-r of 2P chunks of Ls/2 positions).
__device__ __forceinline__ int position_of(int shard, int i, int P, int Ls, int zig)
{
    if (!zig) return shard * Ls + i;
    const int c = Ls / 2;
    return i < c ? shard * c + i : (2 * P - 1 - shard) * c + (i - c);
}

__global__ void __launch_bounds__(kWarps * 32, 1)
    ring_attn_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                         const float* __restrict__ v, float* __restrict__ out,
                         float* __restrict__ lse, int* __restrict__ trace, int B, int L, int H,
                         int Hkv, int D, int P, int causal, int zig, const int* cu_seqlens,
                         int n_seqs, float scale, unsigned int* status)
{
    // extents of q/out and k/v (elements) for the debug build's index checks
    const long long q_elems = static_cast<long long>(B) * L * H * D;
    const long long kv_elems = static_cast<long long>(B) * L * Hkv * D;
    __shared__ float qs[kWarps][kMaxD];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long row_id = static_cast<long long>(blockIdx.x) * kWarps + warp;  // (b, h, i)
    const long long n_rows = static_cast<long long>(B) * H * L;
    if (row_id >= n_rows) return;                     // whole warp leaves together
    const int i = static_cast<int>(row_id % L);       // query position
    const long long bh = row_id / L;
    const int h = static_cast<int>(bh % H);
    const int b = static_cast<int>(bh / H);
    const int Ls = L / P;
    const int r = i / Ls;
    const int q_pos = position_of(r, i - r * Ls, P, Ls, zig);
    // visible key positions [lo, hi]: everything (or up to the query, causal), or for
    // packed sequences the query's own sequence (up to the query, causal)
    int lo = 0, hi = causal ? q_pos : L - 1;
    if (cu_seqlens != nullptr) {
        int a = 0, bb = n_seqs;
        while (bb - a > 1) {
            const int mid = (a + bb) >> 1;
            if (checked_ldg(cu_seqlens, mid, n_seqs + 1, status) <= q_pos) a = mid;
            else bb = mid;
        }
        lo = checked_ldg(cu_seqlens, a, n_seqs + 1, status);
        hi = causal ? q_pos : checked_ldg(cu_seqlens, a + 1, n_seqs + 1, status) - 1;
    }
    const size_t row_stride = static_cast<size_t>(H) * D;   // between consecutive positions
    const long long qoff = (static_cast<long long>(b) * L + i) * row_stride + static_cast<long long>(h) * D;
    for (int d = lane; d < D; d += 32) qs[warp][d] = in_bounds(qoff + d, 1, q_elems, status) ? q[qoff + d] : 0.f;
    __syncwarp();

    // the shard's last row meets every shard the shard visits, in either layout
    const bool tracing = trace != nullptr && b == 0 && h == 0 && i == r * Ls + Ls - 1;
    float m = -INFINITY, l = 0.f;
    float acc[kMaxD / 32];
#pragma unroll
    for (int c = 0; c < kMaxD / 32; ++c) acc[c] = 0.f;

    // key/value rows: Hkv heads per position; query head h reads head h / (H / Hkv)
    const size_t kv_stride = static_cast<size_t>(Hkv) * D;
    const int hk = h / (H / Hkv);
    const float* kb = k + static_cast<size_t>(b) * L * kv_stride + static_cast<size_t>(hk) * D;
    const float* vb = v + static_cast<size_t>(b) * L * kv_stride + static_cast<size_t>(hk) * D;

    for (int t = 0; t < P; ++t) {
        int s = r - t;
        if (s < 0) s += P;
        // whole shard outside the visible keys of this query: skipped
        const bool skip = cu_seqlens != nullptr ? (s * Ls > hi || s * Ls + Ls - 1 < lo)
                                                : (causal && position_of(s, 0, P, Ls, zig) > q_pos);
        if (tracing && lane == 0 && in_bounds(r * P + t, 1, static_cast<long long>(P) * P, status))
            trace[r * P + t] = skip ? -1 : s;
        if (skip) continue;
        const int j_begin = s * Ls;
        const int j_end = j_begin + Ls;
        for (int j0 = j_begin; j0 < j_end; j0 += 32) {
            const int j = j0 + lane;
            float sc = -INFINITY;
            const int kpos = position_of(s, j - j_begin, P, Ls, zig);
            const long long koff = (kb - k) + static_cast<long long>(j) * kv_stride;
            if (j < j_end && kpos >= lo && kpos <= hi && in_bounds(koff, D, kv_elems, status)) {
                const float* krow = k + koff;
                float dot = 0.f;
                for (int d = 0; d < D; d += 4) {
                    const float4 kk = *reinterpret_cast<const float4*>(krow + d);
                    dot = fmaf(qs[warp][d], kk.x, dot);
                    dot = fmaf(qs[warp][d + 1], kk.y, dot);
                    dot = fmaf(qs[warp][d + 2], kk.z, dot);
                    dot = fmaf(qs[warp][d + 3], kk.w, dot);
                }
                sc = dot * scale;
            }
            const float m_new = fmaxf(m, warp_max(sc));
            const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
            const float pj = (sc == -INFINITY) ? 0.f : expf(sc - m_new);
            l = l * alpha + warp_sum(pj);
            const int n_here = min(32, j_end - j0);
#pragma unroll
            for (int c = 0; c < kMaxD / 32; ++c) acc[c] *= alpha;
            for (int jj = 0; jj < n_here; ++jj) {
                const float pw = __shfl_sync(0xffffffffu, pj, jj);
                const long long voff = (vb - v) + static_cast<long long>(j0 + jj) * kv_stride;
                if (!in_bounds(voff, D, kv_elems, status)) continue;
                const float* vrow = v + voff;
#pragma unroll
                for (int c = 0; c < kMaxD / 32; ++c) {
                    const int d = lane + 32 * c;
                    if (d < D) acc[c] = fmaf(pw, vrow[d], acc[c]);
                }
            }
            m = m_new;
        }
    }
    const float inv_l = l > 0.f ? 1.f / l : 0.f;          // a row that saw no key: 0
#pragma unroll
    for (int c = 0; c < kMaxD / 32; ++c) {
        const int d = lane + 32 * c;
        if (d < D && in_bounds(qoff + d, 1, q_elems, status)) out[qoff + d] = acc[c] * inv_l;
    }
    const long long lidx = (static_cast<long long>(b) * L + i) * H + h;
    if (lse != nullptr && lane == 0 && in_bounds(lidx, 1, q_elems / D, status))
        lse[lidx] = l > 0.f ? m + logf(l) : -INFINITY;
}

}  // namespace

cudaError_t launch_attn_f32(const AttnArgs& a)
{
    const long long rows = static_cast<long long>(a.B) * a.H * a.L;
    const long long blocks = (rows + kWarps - 1) / kWarps;
    if (blocks <= 0 || blocks > 0x7fffffffLL || a.D > kMaxD) return cudaErrorInvalidConfiguration;
    ring_attn_f32_kernel<<<static_cast<unsigned>(blocks), kWarps * 32, 0, a.stream>>>(
        static_cast<const float*>(a.q), static_cast<const float*>(a.k),
        static_cast<const float*>(a.v), static_cast<float*>(a.out), a.lse, a.trace, a.B, a.L,
        a.H, a.Hkv, a.D, a.P, a.causal, a.zigzag, a.cu_seqlens, a.n_seqs,
        1.0f / sqrtf(static_cast<float>(a.D)), a.status);
    return cudaGetLastError();
}

}  // namespace ra
