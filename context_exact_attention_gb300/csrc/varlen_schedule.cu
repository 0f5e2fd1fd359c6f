// varlen_schedule.cu -- heaviest-first unit orders for the packed-sequence kernels
// (ring_attn_varlen_schedule).
//
// With packed sequences ("序列并行与 Ring Attention", section 6.5) a query sees only
// keys of its own sequence, so a query tile's work is the number of key tiles between
// its sequence's start and its last query (causal) or its sequence's end; a key tile's
// work in the backward is the number of query tiles that see it.  That grows with the
// tile's offset inside its sequence, not with its global position, so the position
// order the kernels use for the other layouts does not put heavy units first.  This
// kernel counts every unit's tiles from cu_seqlens and writes the units in descending
// work (ties: ascending natural index), which the kernels then read by block index.
//
// One CTA per unit kind: all threads count (two binary searches over cu_seqlens per
// unit), then a counting sort over work values -- histogram in shared memory, a
// descending exclusive scan and a stable scatter by one warp (__match_any_sync ranks
// the lanes of equal bins in lane order, so the order is deterministic).
#include "ra_check.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kThreads = 1024;
constexpr int kMaxBins = 4096;        // work values beyond this share bins (long sequences)
constexpr int kSmemWork = 8192;       // units whose counts stay in shared memory
constexpr int kTileRows = 128;

// First and last position of the sequence holding pos: the largest g with
// cu[g] <= pos.  Bounded for any contents of cu.
__device__ void seq_span(const int* cu, int n_seqs, int pos, int& first, int& last,
                         unsigned int* status)
{
    int a = 0, b = n_seqs - 1;
    while (a < b) {
        const int m = (a + b + 1) >> 1;
        if (checked_ldg(cu, m, n_seqs + 1, status) <= pos) a = m;
        else b = m - 1;
    }
    first = checked_ldg(cu, a, n_seqs + 1, status);
    last = checked_ldg(cu, a + 1, n_seqs + 1, status) - 1;
}

// 128-row tiles (each within one shard of Ls rows) holding a position in [lo, hi].
__device__ int tiles_in(int lo, int hi, int Ls, int L)
{
    lo = max(lo, 0);
    hi = min(hi, L - 1);
    if (lo > hi) return 0;
    int n = 0;
    for (int s = lo / Ls; s <= hi / Ls; ++s) {
        const int base = s * Ls;
        const int a = max(lo, base) - base, b = min(hi, base + Ls - 1) - base;
        n += b / kTileRows - a / kTileRows + 1;
    }
    return n;
}

__device__ __forceinline__ int bin_of(int w, int nb, int max_work)
{
    w = min(max(w, 0), max_work);
    if (nb == max_work + 1) return w;
    return static_cast<int>(static_cast<long long>(w) * nb / (max_work + 1));
}

__global__ void __launch_bounds__(kThreads, 1)
    varlen_schedule_kernel(const int* __restrict__ cu, int n_seqs, int L, int P, int causal,
                           int* __restrict__ sched, VarlenSchedLayout lay, unsigned int* status)
{
    __shared__ int bins[kMaxBins];
    __shared__ int work_s[kSmemWork];
    const int lane = threadIdx.x & 31;
    const int Ls = L / P;
    const int max_work = P * static_cast<int>(lay.n_t);
    // the persistent kernels' work counters start at zero
    if (blockIdx.x == 0 && threadIdx.x < kCounters &&
        in_bounds(lay.counters + threadIdx.x, 1, lay.total, status))
        sched[lay.counters + threadIdx.x] = 0;
    const int nb = min(max_work + 1, kMaxBins);
    {
        // kind 0: forward query-tile pairs; 1: backward key tiles; 2: backward query tiles
        const int kind = blockIdx.x;
        const int per = static_cast<int>(kind == 0 ? lay.n_pair : lay.n_t);   // units per shard
        const int rows = kind == 0 ? 2 * kTileRows : kTileRows;
        const int U = P * per;
        const long long off = kind == 0 ? lay.fwd : kind == 1 ? lay.bwd_k : lay.bwd_q;
        int* order = sched + off;
        // each kind's scratch sits as far past the scratch base as its order past the first
        const bool in_smem = U <= kSmemWork;
        int* work = in_smem ? work_s : sched + lay.scratch + off;
        // the debug build checks every global index against the schedule array
        auto work_ok = [&](int u) {
            return in_smem || in_bounds(lay.scratch + off + u, 1, lay.total, status);
        };
        for (int i = threadIdx.x; i < nb; i += kThreads) bins[i] = 0;
        __syncthreads();
        for (int u = threadIdx.x; u < U; u += kThreads) {
            const int s = u / per, i = u - s * per;
            const int a = s * Ls + i * rows;
            const int b = min(s * Ls + Ls - 1, a + rows - 1);
            int fa, la, fb, lb;
            seq_span(cu, n_seqs, a, fa, la, status);
            seq_span(cu, n_seqs, b, fb, lb, status);
            int lo, hi;
            if (kind == 1) {        // the queries that see some key of the tile
                lo = causal ? a : fa;
                hi = lb;
            } else {                // the keys some query of the tile (pair) sees
                lo = fa;
                hi = causal ? b : lb;
            }
            const int w = tiles_in(lo, hi, Ls, L);
            if (work_ok(u)) work[u] = w;
            atomicAdd(&bins[bin_of(w, nb, max_work)], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // bins[x] := number of units in bins above x (descending exclusive scan)
            int carry = 0;
            for (int top = nb - 1; top >= 0; top -= 32) {
                const int i = top - lane;
                const int v = i >= 0 ? bins[i] : 0;
                int x = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (i >= 0) bins[i] = carry + x - v;
                carry += __shfl_sync(0xffffffffu, x, 31);
            }
            __syncwarp();
            // stable scatter, 32 units at a time in index order
            for (int base = 0; base < U; base += 32) {
                const int u = base + lane;
                const bool act = u < U;
                const int key = act ? bin_of(work_ok(u) ? work[u] : 0, nb, max_work) : -1 - lane;
                const unsigned peers = __match_any_sync(0xffffffffu, key);
                const int rank = __popc(peers & ((1u << lane) - 1u));
                if (act && in_bounds(bins[key] + rank, 1, U, status))   // inside this order
                    order[bins[key] + rank] = u;
                __syncwarp();
                if (act && rank == 0) bins[key] += __popc(peers);
                __syncwarp();
            }
        }
    }
}

}  // namespace

cudaError_t launch_varlen_schedule(const int* cu_seqlens, int n_seqs, int L, int P, int causal,
                                   int* schedule, unsigned int* status, cudaStream_t stream)
{
    const VarlenSchedLayout lay = varlen_sched_layout(L, P);
    varlen_schedule_kernel<<<3, kThreads, 0, stream>>>(cu_seqlens, n_seqs, L, P, causal ? 1 : 0,
                                                       schedule, lay, status);
    return cudaGetLastError();
}

}  // namespace ra
