// attn_bwd_sm103.cu -- backward of the exact ring-attention forward (bf16 in,
// fp32 accumulate) on the sm_103a tensor cores.
//
// What it computes: with S = Q K^T / sqrt(D), P = softmax(S) (causal: keys at
// later global positions excluded) and the upstream gradient dO,
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - Dvec),  Dvec_i = sum_d dO_id O_id,
//   dQ = dS K / sqrt(D),  dK = dS^T Q / sqrt(D),
// recomputing P from the forward's row statistics (lse) instead of storing it:
// the backward that "序列并行与 Ring Attention" describes in sections 3.3 and
// 6.2, where each K/V block meets every query shard around the ring and its
// dK, dV return to the shard that owns it.  On one device the K/V-owner side is
// one CTA per 128-key block that walks the query shards in ring order
// (r = (s + t) mod P, skipping r < s under causal masking) and writes dK, dV
// once; the query side (dQ) is one CTA per 128-row query tile walking the K/V
// shards in the forward's order.  No atomics: results are deterministic.  The same
// kernels serve the zigzag shard layout and packed variable-length sequences
// (template parameter kMode; see "shard layouts" below): only the walk over tiles
// and the visibility masks change.
//
// Kernels (warp 0 TMA producer, warp 1 MMA issuer; warp-uniform schedules with one
// elected lane issuing).  dK/dV kernel, 640 threads: warps 2-3 the per-query statistics,
// warps 4-19 the elementwise step, four warps per TMEM lane quarter each taking 32 of the
// 128 query columns of its rows.  dQ kernel, 384 threads: warps 4-11 the elementwise step,
// two warps per lane quarter taking 64 key columns each.  Each warp writes its bf16
// results inside the fp32 columns it read; the MMA issuers address the bf16 operand
// accordingly:
//   bwd_rowdot_kernel   Dvec = rowsum(dO o O), fp32 workspace [B, L, H]
//   bwd_dkdv_kernel<D, kMode>  TMEM: S^T [0,128), dP^T [128,256), dV, dK (D columns each)
//       S^T = K Q^T, dP^T = V dO^T (SS); P^T, dS^T (bf16) written over them, the pairs
//       of query columns [16 k, 16 k + 16) in columns [16 k, 16 k + 8);
//       dV += P^T dO, dK += dS^T Q (A from TMEM, B = dO / Q as MN-major SMEM).
//       Tensor-pipe order per block: dV(n) S^T(n+1) dK(n) dP^T(n+1), so that
//       P^T(n) is computed while dP^T(n) runs, dS^T(n) while dV(n) and S^T(n+1) run.
//   bwd_dq_kernel<D, kMode>    TMEM: S, then dS, alternating between [0,128) and [128,256) by
//       block parity; dP in [256,384); dQ (D columns) at 384.  S = Q K^T, dP = dO V^T
//       (SS); dS (bf16) written over S; dQ += dS K.  Tensor-pipe order per block:
//       S(n+1) dP(n+1) dQ(n), so block n+1's elementwise step overlaps dQ(n).
//   Elementwise arithmetic runs on packed fp32 pairs (f32x2 fma/add/mul); the causal
//   and ragged-tail mask is applied only in the blocks that need one.
#include <cuda_bf16.h>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kRows = 128;     // rows per tile (TMEM lanes), both queries and keys
constexpr int kThreads = 384;   // dQ kernel: warps 0-1 producer, MMA issuer; 4-11 elementwise
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

template <int D>
struct BwdLayout {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTileBytes = kRows * D * 2;
    static constexpr uint64_t kTileU = kTileBytes >> 4;
};

struct BwdParams {
    const float* lse;        // [B, L, H] natural log
    const float* dvec;       // [B, L, H]
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    unsigned int* status;
    unsigned long long timeout_ns;
    int B, L, H, P, Ls, causal;
    int Hkv, group;          // key/value heads; query heads per key/value head (H / Hkv)
    int n_t;                 // 128-row tiles per shard
    float scale_log2;        // log2(e) / sqrt(D)
    float scale;             // 1 / sqrt(D)
    const int* cu_seqlens;   // packed sequences: starts of n_seqs sequences, then L
    int n_seqs;
    const int* sched_k;      // packed sequences: key tiles heaviest first (s * n_t + kt), or null
    const int* sched_q;      // packed sequences: query tiles heaviest first (r * n_t + qt), or null
    // extents for the debug build's index checks: dq (and q, dout), dk and dv, lse and
    // dvec, each schedule order
    long long q_elems, kv_elems, row_elems;
    int sched_elems;
    // persistent grids (packed sequences with a schedule): the kernel's work counter in the
    // schedule array (zeroed before the launch), its index there and the array's size
    int* claim;
    long long claim_index, claim_extent;
    int n_units;     // work units of the launch
};

// ------------------------------------------------------- shard layouts --
//
// kMode 0: contiguous shards (shard x holds positions [x Ls, (x+1) Ls)), with the
// closed-form schedules below.  kMode 1: zigzag shards ("序列并行与 Ring Attention",
// section 3.4: 2P chunks of Ls/2 positions, shard x holds chunk x, then chunk 2P-1-x;
// causal).  kMode 2: packed sequences over contiguous shards (section 6.5: a query sees
// only keys of its own sequence).  Modes 1 and 2 walk the ring with PosWalk.

constexpr int kFar = 1 << 30;    // a position bound that never binds

__device__ __forceinline__ int layout_position(int x, int i, int Ls, int P, bool zig)
{
    if (!zig) return x * Ls + i;
    const int c = Ls >> 1;
    return i < c ? x * c + i : (2 * P - 1 - x) * c + (i - c);
}

// First and last position of the packed sequence that holds position pos
// (cu: n_seqs starts, then the total; cu[a] <= pos < cu[a+1] for exactly one
// non-empty sequence a).
__device__ __forceinline__ void seq_range(const int* cu, int n_seqs, int pos, int& first, int& last,
                                          unsigned int* status)
{
    int a = 0, b = n_seqs;
    while (b - a > 1) {
        const int mid = (a + b) >> 1;
        if (checked_ldg(cu, mid, n_seqs + 1, status) <= pos) a = mid;
        else b = mid;
    }
    first = checked_ldg(cu, a, n_seqs + 1, status);
    last = checked_ldg(cu, a + 1, n_seqs + 1, status) - 1;
}

// Ring walk over the 128-row tiles that hold positions in [lo, hi]: at step t the
// shard x = (own + dir t) mod P (dir = -1: the queries of shard `own` meet K/V shard
// (own - t) mod P, the forward's order; dir = +1: the keys of shard `own` meet query
// shard (own + t) mod P, the owner's side of the same exchange), and of shard x the
// tiles whose positions intersect [lo, hi] -- one run of tiles in a contiguous shard,
// one run in each chunk of a zigzag shard (chunks are whole tiles).  Every role of a
// CTA walks the same sequence, each with its own copy, in order.
struct PosWalk {
    int own, dir, P, Ls, n_half, zig, lo, hi;
    int t, x, idx, first_a, cnt_a, first_b, cnt_b;
    __device__ __forceinline__ void init(int own_, int dir_, int P_, int Ls_, int zig_, int lo_,
                                         int hi_)
    {
        own = own_;
        dir = dir_;
        P = P_;
        Ls = Ls_;
        zig = zig_;
        n_half = (Ls_ >> 1) / kRows;
        lo = lo_;
        hi = hi_;
    }
    __device__ __forceinline__ void run(int base, int len, int& first, int& cnt) const
    {
        const int a = max(lo, base), b = min(hi, base + len - 1);
        if (a > b) {
            first = 0;
            cnt = 0;
        } else {
            first = (a - base) / kRows;
            cnt = (b - base) / kRows - first + 1;
        }
    }
    __device__ __forceinline__ void enter()
    {
        x = own + dir * t;
        if (x >= P) x -= P;
        if (x < 0) x += P;
        first_b = 0;
        cnt_b = 0;
        if (!zig) {
            run(x * Ls, Ls, first_a, cnt_a);
        } else {
            const int c = Ls >> 1;
            run(x * c, c, first_a, cnt_a);
            run((2 * P - 1 - x) * c, c, first_b, cnt_b);
        }
        idx = 0;
    }
    __device__ __forceinline__ void settle()
    {
        while (t < P && idx >= cnt_a + cnt_b) {
            ++t;
            if (t < P) enter();
        }
    }
    __device__ __forceinline__ int total()
    {
        int n = 0;
        for (t = 0; t < P; ++t) {
            enter();
            n += cnt_a + cnt_b;
        }
        return n;
    }
    // n = 0, 1, 2, ... in order
    __device__ __forceinline__ void at(int n)
    {
        if (n == 0) {
            t = 0;
            enter();
        } else {
            ++idx;
        }
        settle();
    }
    // tile within shard x
    __device__ __forceinline__ int tile() const
    {
        return idx < cnt_a ? first_a + idx : n_half + first_b + (idx - cnt_a);
    }
};

// The g-th 128-row tile in global position order of the zigzag layout (2P chunks of n_t/2
// tiles; chunk j < P is the first half of shard j, chunk j >= P the second half of shard
// 2P-1-j): its shard and its tile within the shard.
__device__ __forceinline__ void zigzag_tile_at(int g, int P, int n_t, int& shard, int& tile)
{
    const int per_chunk = n_t >> 1;
    const int chunk = g / per_chunk, within = g - chunk * per_chunk;
    if (chunk < P) {
        shard = chunk;
        tile = within;
    } else {
        shard = 2 * P - 1 - chunk;
        tile = per_chunk + within;
    }
}

// Zero rows [row0, row0 + n) of a [B, L, heads, D] bf16 tensor's head `head` (gradients of
// a tile that no pair reaches: possible only with malformed sequence boundaries).
template <int D>
__device__ void zero_tile_rows(__nv_bfloat16* t, int b, int L, int heads, int head, int row0, int n,
                               long long extent, unsigned int* status)
{
    constexpr int kVec = D / 8;     // 16-byte vectors per row
    for (int i = threadIdx.x; i < n * kVec; i += blockDim.x) {
        const int row = row0 + i / kVec;
        const long long idx =
            ((static_cast<long long>(b) * L + row) * heads + head) * D + (i % kVec) * 8;
        if (in_bounds(idx, 8, extent, status))
            *reinterpret_cast<uint4*>(t + idx) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// ------------------------------------------------------------------ row dot --

// Output staging of the elementwise warps' epilogues.  A warp holds 32 rows of kCols
// bf16 columns, one row per lane; written straight to global memory every store
// instruction would touch 32 rows.  Each lane first writes its row's 16-byte chunks
// (four per call, starting at chunk `first`) to a 32-row staging slice, chunk j at slot
// j ^ (row mod chunks) so that neither the row-wise writes nor the chunk-wise reads
// conflict on banks; store_staged_rows then stores whole row pieces per instruction.
template <int kCols>
__device__ __forceinline__ void stage_row_chunks(uint8_t* stage, int lane, int first,
                                                 const uint32_t (&pk)[16])
{
    constexpr int kChunks = kCols / 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int slot = (first + j) ^ (lane & (kChunks - 1));
        *reinterpret_cast<uint4*>(stage + lane * (2 * kCols) + slot * 16) =
            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    }
}

// Rows 0..31 of the slice to base + off0 + row * stride (elements), rows < n_valid only;
// extent: elements of the tensor at base (checked in the debug build).
template <int kCols>
__device__ __forceinline__ void store_staged_rows(const uint8_t* stage, int lane, __nv_bfloat16* base,
                                                  long long off0, long long stride, int n_valid,
                                                  long long extent, unsigned int* status)
{
    constexpr int kChunks = kCols / 8;
    constexpr int kRowsPerStore = 32 / kChunks;
    const int sub = lane / kChunks, cc = lane % kChunks;
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
        const int rr = k * kRowsPerStore + sub;
        const uint4 val = *reinterpret_cast<const uint4*>(stage + rr * (2 * kCols) +
                                                          ((cc ^ (rr & (kChunks - 1))) * 16));
        const long long idx = off0 + rr * stride + cc * 8;
        if (rr < n_valid && in_bounds(idx, 8, extent, status))
            *reinterpret_cast<uint4*>(base + idx) = val;
    }
}

// Dvec[row] = sum_d dO[row, d] * O[row, d] for every (b, l, h) row; a group of
// D/8 lanes takes one row, one 16-byte vector each.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_rowdot_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                      float* __restrict__ dvec, long long rows, unsigned int* status)
{
    constexpr int kLanes = D / 8;
    constexpr int kRowsPerWarp = 32 / kLanes;
    const int lane = threadIdx.x & 31;
    const int sub = lane % kLanes;
    const long long warp_global = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) >> 5;
    const long long n_warps = (static_cast<long long>(gridDim.x) * 256) >> 5;
    for (long long base = warp_global * kRowsPerWarp; base < rows; base += n_warps * kRowsPerWarp) {
        const long long row = base + lane / kLanes;
        float acc = 0.f;
        if (row < rows && in_bounds(row * kLanes + sub, 1, rows * kLanes, status)) {
            const uint4 a = o[row * kLanes + sub];
            const uint4 g = dout[row * kLanes + sub];
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
            const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 fa = __bfloat1622float2(a2[i]);
                const float2 fg = __bfloat1622float2(g2[i]);
                acc = fmaf(fa.x, fg.x, acc);
                acc = fmaf(fa.y, fg.y, acc);
            }
        }
#pragma unroll
        for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (row < rows && sub == 0 && in_bounds(row, 1, rows, status)) dvec[row] = acc;
    }
}

// ------------------------------------------------------------------ dK, dV --

constexpr int kQStages = 3;          // Q is read last by dK, late in a block: three stages
// dK/dV kernel: 20 warps -- 0 producer, 1 MMA issuer, 2-3 statistics, 4-19 elementwise, four
// warps per TMEM lane quarter, each taking 32 of the 128 query columns of its rows
constexpr int kKVParts = 4;
constexpr int kKVCols = kRows / kKVParts;
constexpr int kKVThreads = (4 + 4 * kKVParts) * 32;
constexpr int kMaxSmem = 232448;     // opt-in shared memory limit of one block (227 KiB)
// Byte offset, within the 256-byte barrier area of either kernel, of the per-stage tile
// records (int2: layout position of the tile's first row, number of valid rows) that the
// loading warps publish with each stage, so the elementwise warps need no schedule walk.
// Layout of the 256-byte barrier area of both backward kernels: the barriers, the TMEM
// address and abort flag, from kInfoOff the per-stage tile records (int2: layout position of
// the tile's first row, number of valid rows) that the loading warps publish with each stage
// so the elementwise warps need no schedule walk, and from kRingOff the two slots of a
// persistent grid's unit ring.
constexpr int kInfoOff = 184;
constexpr int kRingOff = 208;
constexpr int kRingInts = 6;

enum : int {
    kKVFull = 0,
    kQFull = 1,        // +stage (3): Q tile (TMA) and its -lse statistics (warp 2)
    kQEmpty = 4,       // +stage: released after dK, the last reader of Q
    kKVDOFull = 7,     // +stage (2): dO tile and its -Dvec statistics (warp 3)
    kKVDOEmpty = 9,    // +stage: released after dK too (the dS^T step reads -Dvec)
    kKVSFull = 11,     // S^T ready
    kKVDPFull = 12,    // dP^T ready
    kKVPFull = 13,     // P^T written (all elementwise threads)
    kKVDSFull = 14,    // dS^T written
    kKVOFull = 15,     // dK, dV final
    kKVDone = 16,
    kKVUnitFull = 17,  // +slot: persistent grids, the producer published a unit
    kKVUnitEmpty = 19, // +slot: every consumer warp has read it
    kKVKVEmpty = 21,   // persistent grids: the unit's last S^T and dP^T finished
    kKVBars = 22
};
constexpr int kKVUnitReaders = 1 + 2 + 4 * kKVParts;   // MMA, statistics, elementwise warps

// Shared memory of the dK/dV kernel from a 1024-aligned base: K, V, three Q stages, two dO
// stages, the statistics (128 fp32 per stage), barriers.  The allocation adds what is left
// of the 227 KiB limit for aligning the base; the kernel checks that this was enough.
template <int D>
struct KVSmem {
    static constexpr int T = kRows * D * 2;
    static constexpr int kK = 0, kV = T, kQ = 2 * T, kDO = (2 + kQStages) * T;
    static constexpr int kNlse = (4 + kQStages) * T;
    static constexpr int kNdvec = kNlse + kQStages * kRows * 4;
    static constexpr int kBar = kNdvec + 2 * kRows * 4;
    static constexpr int kNeed = kBar + 256;
    static constexpr int kAlloc = kNeed + 1023 < kMaxSmem ? kNeed + 1023 : kMaxSmem;
    static_assert(kNeed <= kMaxSmem, "dK/dV shared memory layout exceeds the limit");
    static_assert(kKVBars * 8 + 8 <= kInfoOff && kInfoOff + 8 * kQStages <= kRingOff &&
                      kRingOff + 2 * kRingInts * 4 <= 256,
                  "barrier area");
};

// A dK/dV work unit: one 128-key tile of one (batch, key/value head) and the query tiles
// it meets.  With grouped heads the unit's keys meet the queries of every query head of
// its group (h = hk * group + g), one head after the other, and dK, dV accumulate over
// all of them.
template <int kMode>
struct KVUnit {
    int bh, b, hk, s, kt, key0;
    int q_begin, n_first, n_head, n_blocks;
    PosWalk walk;

    // unit g of the call: heaviest key tile first (low shard, low tile), two (b, key/value
    // head) pairs interleaved (unit_of_block)
    __device__ __forceinline__ void decode(int g, const BwdParams& p)
    {
        const int units_per_bh = p.P * p.n_t;
        int u;
        unit_of_block(g, p.B * p.Hkv, units_per_bh, bh, u);
        s = u / p.n_t;                // shard owning these keys
        kt = u - s * p.n_t;           // key tile within the shard
        if constexpr (kMode == 1) {
            // zigzag: a key tile's work falls with its global position (it meets every
            // later query), so heaviest first is position order: unit u is the u-th tile by
            // position
            zigzag_tile_at(u, p.P, p.n_t, s, kt);
        }
        if constexpr (kMode == 2) {
            // packed sequences: a precomputed heaviest-first order, if given (entries
            // outside the unit range are ignored)
            if (p.sched_k != nullptr) {
                const int x = checked_ldg(p.sched_k, u, p.sched_elems, p.status);
                if (static_cast<unsigned>(x) < static_cast<unsigned>(units_per_bh)) {
                    s = x / p.n_t;
                    kt = x - s * p.n_t;
                }
            }
        }
    }
    // zigzag shards and packed sequences: the query positions [lo, hi] some key of the
    // tile is visible to (causal: from the tile's first key position on; packed: within
    // the sequences of its first and last key)
    __device__ __forceinline__ void bounds(const BwdParams& p, int& lo, int& hi) const
    {
        constexpr bool kZig = kMode == 1;
        const int kp0 = layout_position(s, kt * kRows, p.Ls, p.P, kZig);
        lo = kp0;
        hi = kFar;
        if constexpr (kMode == 2) {
            const int kp1 = s * p.Ls + min(p.Ls - 1, kt * kRows + kRows - 1);
            int f0, l0, f1, l1;
            seq_range(p.cu_seqlens, p.n_seqs, kp0, f0, l0, p.status);
            seq_range(p.cu_seqlens, p.n_seqs, kp1, f1, l1, p.status);
            lo = p.causal ? kp0 : f0;
            hi = l1;
        }
    }
    // the rest, from the decoded tile (lo, hi: the bounds above, modes 1 and 2)
    __device__ __forceinline__ void finish(const BwdParams& p, int lo, int hi)
    {
        b = bh / p.Hkv;
        hk = bh - b * p.Hkv;
        key0 = s * p.Ls + kt * kRows;
        // ring schedule from the owner's side: query shard r = (s + t) mod P at step t;
        // step 0 is the own shard (causal: query tiles from the diagonal on)
        q_begin = p.causal ? kt : 0;
        n_first = p.n_t - q_begin;
        n_head = n_first + (p.causal ? (p.P - 1 - s) : (p.P - 1)) * p.n_t;
        if constexpr (kMode != 0) {
            // the query tiles holding those positions, walked in the same ring order
            walk.init(s, +1, p.P, p.Ls, kMode == 1 ? 1 : 0, lo, hi);
            n_head = walk.total();
        } else {
            (void)lo;
            (void)hi;
        }
        n_blocks = n_head * p.group;
    }
    __device__ __forceinline__ void setup(int g, const BwdParams& p)
    {
        decode(g, p);
        int lo = 0, hi = 0;
        if constexpr (kMode != 0) bounds(p, lo, hi);
        finish(p, lo, hi);
    }
    // block n: query head h, query shard r, query tile qt (modes 1 and 2: n = 0, 1, ... in
    // order; the walk restarts for each query head of the group)
    __device__ __forceinline__ void block(int n, const BwdParams& p, int& r, int& qt, int& h)
    {
        if constexpr (kMode != 0) {
            const int g = p.group == 1 ? 0 : n / n_head;
            walk.at(n - g * n_head);
            r = walk.x;
            qt = walk.tile();
            h = hk * p.group + g;
            return;
        }
        const int g = p.group == 1 ? 0 : n / n_head;
        h = hk * p.group + g;
        n -= g * n_head;
        if (n < n_first) {
            r = s;
            qt = q_begin + n;
            return;
        }
        const int m = n - n_first;
        const int t = 1 + m / p.n_t;
        qt = m - (t - 1) * p.n_t;
        r = s + t;
        if (r >= p.P) r -= p.P;
    }
};

// kPersist: 0 one CTA per key tile (the grid lists the units); 2 one CTA per SM that
// takes units dynamically (packed sequences with a schedule): the producer warp claims
// each next unit from a counter in the schedule array (zeroed before the launch) and hands
// it, decoded, to the other warps through a two-slot ring in shared memory.  A persistent
// CTA loads the next unit's K and V as soon as the current unit's last S^T and dP^T (their
// last readers) have finished, and keeps streaming Q and dO stages across units (barrier
// phases count blocks and units from the CTA's start); its epilogue stores dK and dV from
// registers, since the Q stages it would stage them in are already refilling.
template <int D, int kMode, int kPersist>
__global__ void __launch_bounds__(kKVThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q,
                    const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_do, const BwdParams p)
{
    using Lay = BwdLayout<D>;
    using Sm = KVSmem<D>;
    constexpr int T = Lay::kTileBytes;
    constexpr int kK = Sm::kK, kV = Sm::kV, kQ = Sm::kQ, kDO = Sm::kDO, kBar = Sm::kBar;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    if (pad + Sm::kNeed > static_cast<uint32_t>(Sm::kAlloc)) {
        // the dynamic shared memory base leaves too little room to align the tiles
        if (threadIdx.x == 0) atomicOr(p.status, RA_STATUS_LAYOUT);
        return;
    }
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBar + kKVBars * 8);
    int* abort_flag = reinterpret_cast<int*>(smem + kBar + kKVBars * 8 + 4);
    // per Q stage: first query position and valid query rows (written by warp 2)
    int2* qinfo = reinterpret_cast<int2*>(smem + kBar + kInfoOff);
    // dynamic grids: two ring slots of a decoded unit (unit, shard, tile, lo, hi, n_head)
    volatile int* unit_slot = reinterpret_cast<volatile int*>(smem + kBar + kRingOff);
    auto bar = [&](int i) -> uint32_t { return sbase + kBar + 8u * i; };
    // per-query statistics, negated for the packed adds: -lse log2(e) with the Q stage,
    // -Dvec with the dO stage
    auto stats_nlse2 = [&](int qs) { return reinterpret_cast<float*>(smem + Sm::kNlse + qs * 512); };
    auto stats_ndvec = [&](int ds) { return reinterpret_cast<float*>(smem + Sm::kNdvec + ds * 512); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool kZig = kMode == 1;
    WaitCtx wc{abort_flag, p.status, p.timeout_ns};

    // The i-th unit of this CTA, set up in V (-1: no more).  Dynamic grids: the consumers'
    // side of the ring (the producer publishes below).
    auto consume_unit = [&](int i, KVUnit<kMode>& V) -> int {
        if constexpr (kPersist == 0) {
            if (i > 0) return -1;
            V.setup(static_cast<int>(blockIdx.x), p);
            return static_cast<int>(blockIdx.x);
        }
        const int slot = i & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kKVUnitFull + slot), (i >> 1) & 1, wc)))
            return -1;
        volatile int* e = unit_slot + kRingInts * slot;
        const int g = e[0];
        if (g >= 0) {
            int u;
            unit_of_block(g, p.B * p.Hkv, p.P * p.n_t, V.bh, u);
            V.s = e[1];
            V.kt = e[2];
            V.finish(p, e[3], e[4]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kKVUnitEmpty + slot));
        return g;
    };
    // an empty walk (only with malformed sequence boundaries): zero gradient rows
    auto zero_rows = [&](const KVUnit<kMode>& V) {
        const int n = min(kRows, p.Ls - V.kt * kRows);
        zero_tile_rows<D>(p.dk, V.b, p.L, p.Hkv, V.hk, V.key0, n, p.kv_elems, p.status);
        zero_tile_rows<D>(p.dv, V.b, p.L, p.Hkv, V.hk, V.key0, n, p.kv_elems, p.status);
    };

    KVUnit<kMode> first;
    int g_first = -1;
    if constexpr (kPersist == 0) {
        g_first = consume_unit(0, first);
        if (first.n_head == 0) {          // every key of a tile sees at least its own query
            zero_rows(first);
            return;
        }
    }

    if (threadIdx.x == 0) {
        mbar_init(bar(kKVFull), 1);
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(bar(kQFull + i), 1 + 32);
            mbar_init(bar(kQEmpty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kKVDOFull + i), 1 + 32);
            mbar_init(bar(kKVDOEmpty + i), 1);
            mbar_init(bar(kKVUnitFull + i), 1);
            mbar_init(bar(kKVUnitEmpty + i), kKVUnitReaders);
        }
        mbar_init(bar(kKVSFull), 1);
        mbar_init(bar(kKVDPFull), 1);
        mbar_init(bar(kKVPFull), kKVParts * kRows);
        mbar_init(bar(kKVDSFull), kKVParts * kRows);
        mbar_init(bar(kKVOFull), 1);
        mbar_init(bar(kKVDone), 1);
        mbar_init(bar(kKVKVEmpty), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        const bool leader = elect_one();
        const uint64_t keep = l2_policy_evict_last();
        if (leader) {
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_do);
        }
        // dynamic grids: claim the i-th unit, decode it and publish it (-1: done)
        auto publish_unit = [&](int i, KVUnit<kMode>& U) -> int {
            const int slot = i & 1;
            int g = -1;
            if (leader && in_bounds(p.claim_index, 1, p.claim_extent, p.status))
                g = atomicAdd(p.claim, 1);
            g = __shfl_sync(0xffffffffu, g, __ffs(__ballot_sync(0xffffffffu, leader)) - 1);
            if (g < 0 || g >= p.n_units) g = -1;
            int lo = 0, hi = 0;
            if (g >= 0) {
                U.decode(g, p);
                if constexpr (kMode != 0) U.bounds(p, lo, hi);
                U.finish(p, lo, hi);
            }
            if (i >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar(kKVUnitEmpty + slot),
                                                             ((i - 2) >> 1) & 1, wc)))
                return -1;
            if (leader) {
                volatile int* e = unit_slot + kRingInts * slot;
                e[0] = g;
                e[1] = U.s;
                e[2] = U.kt;
                e[3] = lo;
                e[4] = hi;
                mbar_arrive(bar(kKVUnitFull + slot));
            }
            __syncwarp();
            return g;
        };
        uint32_t N = 0;       // query blocks loaded by this CTA so far
        int un = 0;           // units with a non-empty walk so far
        int last_q[kQStages] = {-1, -1, -1}, last_do[2] = {-1, -1};
        bool ok = true;
        for (int i = 0; ok; ++i) {
            KVUnit<kMode> U;
            int g;
            if constexpr (kPersist == 2) g = publish_unit(i, U);
            else {
                g = i == 0 ? g_first : -1;
                U = first;
            }
            if (g < 0) break;
            if (U.n_head == 0) continue;
            // K and V of the tile: refilled once the previous unit's last S^T and dP^T (their
            // last readers) have finished
            if (un > 0 && !(ok = __all_sync(0xffffffffu,
                                            mbar_wait(bar(kKVKVEmpty), (un - 1) & 1, wc))))
                break;
            if (leader) {
                mbar_arrive_expect_tx(bar(kKVFull), 2 * T);
                for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                    tma_load_4d(sbase + kK + bx * 16384, &tmap_k, bar(kKVFull), bx * 64, U.hk, U.key0,
                                U.b, keep);
                    tma_load_4d(sbase + kV + bx * 16384, &tmap_v, bar(kKVFull), bx * 64, U.hk, U.key0,
                                U.b, keep);
                }
            }
            __syncwarp();
            for (int n = 0; n < U.n_blocks; ++n) {
                int r, qt, h;
                U.block(n, p, r, qt, h);
                const uint32_t Nn = N + n;
                const int qs = Nn % kQStages, ds = Nn & 1;
                const int qrow = r * p.Ls + qt * kRows;
                // Q first: its stage frees a block earlier than the dO stage, and S^T needs it first
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kQEmpty + qs), ((Nn / kQStages) & 1) ^ 1, wc))))
                    break;
                if (leader) {
                    mbar_arrive_expect_tx(bar(kQFull + qs), T);
                    for (int bx = 0; bx < Lay::kBoxes; ++bx)
                        tma_load_4d(sbase + kQ + qs * T + bx * 16384, &tmap_q, bar(kQFull + qs), bx * 64,
                                    h, qrow, U.b, keep);
                }
                last_q[qs] = static_cast<int>(Nn);
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kKVDOEmpty + ds), ((Nn >> 1) & 1) ^ 1, wc))))
                    break;
                if (leader) {
                    mbar_arrive_expect_tx(bar(kKVDOFull + ds), T);
                    for (int bx = 0; bx < Lay::kBoxes; ++bx)
                        tma_load_4d(sbase + kDO + ds * T + bx * 16384, &tmap_do, bar(kKVDOFull + ds),
                                    bx * 64, h, qrow, U.b, keep);
                }
                last_do[ds] = static_cast<int>(Nn);
            }
            N += U.n_blocks;
            ++un;
        }
        if (un > 0) mbar_wait_drain(bar(kKVFull), (un - 1) & 1, wc);
        for (int i = 0; i < kQStages; ++i)
            if (last_q[i] >= 0) mbar_wait_drain(bar(kQFull + i), (last_q[i] / kQStages) & 1, wc);
        for (int i = 0; i < 2; ++i)
            if (last_do[i] >= 0) mbar_wait_drain(bar(kKVDOFull + i), (last_do[i] >> 1) & 1, wc);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        const bool leader = elect_one();
        constexpr uint32_t kIdescS = idesc_bf16_f32(kRows, kRows, false);
        constexpr uint32_t kIdescAcc = idesc_bf16_f32(kRows, D, true);
        const uint64_t dK_A = sdesc_sw128(sbase + kK, 16, 1024);     // K as K-major A
        const uint64_t dV_A = sdesc_sw128(sbase + kV, 16, 1024);     // V as K-major A
        const uint64_t dQ_B = sdesc_sw128(sbase + kQ, 16, 1024);     // Q as K-major B
        const uint64_t dDO_B = sdesc_sw128(sbase + kDO, 16, 1024);   // dO as K-major B
        const uint64_t dQ_MN = sdesc_sw128(sbase + kQ, 16384, 1024); // Q as MN-major B
        const uint64_t dDO_MN = sdesc_sw128(sbase + kDO, 16384, 1024);
        auto ss = [&](uint32_t dcol, uint64_t a0, uint64_t b0) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint64_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                mma_ss(tmem + dcol, a0 + off, b0 + off, kIdescS, k > 0 ? 1u : 0u);
            }
        };
        // A operand in TMEM: the bf16 pairs of query columns [16 k, 16 k + 16) sit in
        // columns [acol + 16 k, acol + 16 k + 8), inside the fp32 columns they replace
        auto ts = [&](uint32_t dcol, uint32_t acol, uint64_t b0, bool acc) {
#pragma unroll
            for (int k = 0; k < kRows / 16; ++k)
                mma_ts(tmem + dcol, tmem + acol + 16 * k, b0 + ((k * 2048) >> 4), kIdescAcc,
                       (acc || k > 0) ? 1u : 0u);
        };
        auto wait_q = [&](uint32_t n) {
            return __all_sync(0xffffffffu,
                              mbar_wait(bar(kQFull + n % kQStages), (n / kQStages) & 1, wc));
        };
        auto wait_do = [&](uint32_t n) {
            return __all_sync(0xffffffffu, mbar_wait(bar(kKVDOFull + (n & 1)), (n >> 1) & 1, wc));
        };
        // Tensor-pipe order: S(0) dP(0) | dV(0) S(1) dK(0) dP(1) | dV(1) S(2) dK(1) dP(2) | ...
        // so P^T(n) is computed while dP^T(n) runs and dS^T(n) while dV(n), S(n+1) run.
        // Each product overwrites TMEM only after the products reading it were issued.
        uint32_t N = 0;
        int un = 0;
        bool ok = true;
        for (int i = 0; ok; ++i) {
            int n_blocks;
            if (kPersist == 0) {
                if (i > 0) break;
                n_blocks = first.n_blocks;
            } else {
                KVUnit<kMode> U;
                if (consume_unit(i, U) < 0) break;
                n_blocks = U.n_blocks;
            }
            if (n_blocks == 0) continue;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kKVFull), un & 1, wc)) && wait_q(N);
            if (ok) {
                tc_fence_after();
                if (leader) {
                    ss(0, dK_A, dQ_B + (N % kQStages) * Lay::kTileU);          // S^T = K Q^T
                    tc_commit(bar(kKVSFull));
                }
                __syncwarp();
            }
            if (ok && (ok = wait_do(N))) {
                tc_fence_after();
                if (leader) {
                    ss(128, dV_A, dDO_B + (N & 1) * Lay::kTileU);              // dP^T = V dO^T
                    tc_commit(bar(kKVDPFull));
                    // persistent grids: the unit's last readers of K and V have been issued
                    if (kPersist != 0 && n_blocks == 1) tc_commit(bar(kKVKVEmpty));
                }
                __syncwarp();
            }
            for (int n = 0; ok && n < n_blocks; ++n) {
                const uint32_t Nn = N + n;
                const int st = Nn & 1;
                const bool more = n + 1 < n_blocks;
                // P^T(n) written and (if another block follows) Q(n+1) loaded: dV(n), S^T(n+1)
                const int q1 = (Nn + 1) % kQStages;
                ok = more ? mbar_wait2(bar(kKVPFull), Nn & 1, bar(kQFull + q1), ((Nn + 1) / kQStages) & 1, wc)
                          : mbar_wait(bar(kKVPFull), Nn & 1, wc);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                tc_fence_after();
                if (leader) {
                    ts(256, 0, dDO_MN + st * Lay::kTileU, n > 0);                   // dV += P^T dO
                    if (more) {
                        ss(0, dK_A, dQ_B + q1 * Lay::kTileU);
                        tc_commit(bar(kKVSFull));
                    }
                }
                __syncwarp();
                // dS^T(n) written and dO(n+1) loaded: dK(n), dP^T(n+1)
                ok = more ? mbar_wait2(bar(kKVDSFull), Nn & 1, bar(kKVDOFull + (st ^ 1)), ((Nn + 1) >> 1) & 1, wc)
                          : mbar_wait(bar(kKVDSFull), Nn & 1, wc);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                tc_fence_after();
                if (leader) {
                    ts(256 + D, 128, dQ_MN + (Nn % kQStages) * Lay::kTileU, n > 0);  // dK += dS^T Q
                    tc_commit(bar(kQEmpty + Nn % kQStages));
                    tc_commit(bar(kKVDOEmpty + st));
                    if (!more) tc_commit(bar(kKVOFull));
                    if (more) {
                        ss(128, dV_A, dDO_B + (st ^ 1) * Lay::kTileU);
                        tc_commit(bar(kKVDPFull));
                        if (kPersist != 0 && n + 2 == n_blocks) tc_commit(bar(kKVKVEmpty));
                    }
                }
                __syncwarp();
            }
            N += n_blocks;
            ++un;
        }
        if (leader) tc_commit(bar(kKVDone));
        __syncwarp();
        mbar_wait_drain(bar(kKVDone), 0, wc);
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------------ statistics
        // Warp 2 writes -lse log2(e) into the Q stage, warp 3 -Dvec into the dO stage, each
        // lane four query rows; within a unit the global loads of a block are issued before
        // waiting for its stage, so their latency overlaps the wait.
        const bool is_lse = warp == 2;
        const float* src = is_lse ? p.lse : p.dvec;
        const float mul = is_lse ? -kLog2e : -1.f;
        uint32_t N = 0;
        bool ok = true;
        for (int i = 0; ok; ++i) {
            KVUnit<kMode> U;
            if constexpr (kPersist == 0) {
                if (i > 0) break;
                U = first;
            } else {
                if (consume_unit(i, U) < 0) break;
            }
            const int n_blocks = U.n_blocks;
            if (n_blocks == 0) continue;
            auto fetch = [&](int n, float (&v)[4], int2& info) {
                int r, qt, h;
                U.block(n, p, r, qt, h);
                const int qrow = r * p.Ls + qt * kRows;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = lane + 32 * j;
                    const long long idx = (static_cast<long long>(U.b) * p.L + qrow + c) * p.H + h;
                    v[j] = (qt * kRows + c < p.Ls && in_bounds(idx, 1, p.row_elems, p.status))
                               ? src[idx] * mul : 0.f;
                }
                info = make_int2(layout_position(r, qt * kRows, p.Ls, p.P, kZig),
                                 min(kRows, p.Ls - qt * kRows));
            };
            float v[4];
            int2 info;
            fetch(0, v, info);
            for (int n = 0; n < n_blocks; ++n) {
                const uint32_t Nn = N + n;
                float nxt[4] = {0.f, 0.f, 0.f, 0.f};
                int2 nxt_info = info;
                if (n + 1 < n_blocks) fetch(n + 1, nxt, nxt_info);
                float* dst;
                uint32_t full;
                if (is_lse) {
                    const int qs = Nn % kQStages;
                    ok = mbar_wait(bar(kQEmpty + qs), ((Nn / kQStages) & 1) ^ 1, wc);
                    dst = stats_nlse2(qs);
                    full = bar(kQFull + qs);
                } else {
                    const int ds = Nn & 1;
                    ok = mbar_wait(bar(kKVDOEmpty + ds), ((Nn >> 1) & 1) ^ 1, wc);
                    dst = stats_ndvec(ds);
                    full = bar(kKVDOFull + ds);
                }
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
#pragma unroll
                for (int j = 0; j < 4; ++j) dst[lane + 32 * j] = v[j];
                if (is_lse && lane == 0) qinfo[Nn % kQStages] = info;
                mbar_arrive(full);
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = nxt[j];
                info = nxt_info;
            }
            N += n_blocks;
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------ elementwise
        const int quarter = warp & 3;
        const int part = (warp - 4) >> 2;                 // query columns [32 part, 32 part + 32)
        const int row = quarter * 32 + lane;              // key row of the tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + kKVCols * part;        // S^T, then P^T
        const uint32_t tP = tmem + lane_off + 128 + kKVCols * part;  // dP^T, then dS^T
        const uint64_t sl2 = f2pack(p.scale_log2, p.scale_log2);
        // this thread's key row of unit V and the positions of the queries that see it,
        // [vis_lo, vis_hi]
        struct KeyRow {
            int key_local;
            bool key_valid;
            int vis_lo, vis_hi;
        };
        auto key_row = [&](const KVUnit<kMode>& V) {
            KeyRow k;
            k.key_local = V.kt * kRows + row;             // within shard s
            k.key_valid = k.key_local < p.Ls;
            k.vis_lo = 0;
            k.vis_hi = kFar;
            if (k.key_valid) {
                const int kp = layout_position(V.s, k.key_local, p.Ls, p.P, kZig);
                if (p.causal || kZig) k.vis_lo = kp;
                if constexpr (kMode == 2) {
                    int f, l;
                    seq_range(p.cu_seqlens, p.n_seqs, kp, f, l, p.status);
                    if (!p.causal) k.vis_lo = f;
                    k.vis_hi = l;
                }
            }
            return k;
        };
        auto get_unit = [&](int i, KVUnit<kMode>& V) -> int {
            if constexpr (kPersist == 0) {
                V = first;
                return i == 0 ? g_first : -1;
            }
            return consume_unit(i, V);
        };
        uint32_t N = 0;
        int un = 0;
        bool ok = true;
        KVUnit<kMode> U;
        int g = get_unit(0, U);
        KeyRow kr = key_row(U);
        for (int i = 0; ok && g >= 0; ++i) {
            const int n_blocks = U.n_blocks;
            // what the epilogue needs of this unit
            const int b = U.b, hk = U.hk, s = U.s, kt = U.kt;
            if (n_blocks > 0) {
                for (int n = 0; n < n_blocks; ++n) {
                    const uint32_t Nn = N + n;
                    const int st = Nn & 1;
                    ok = mbar_wait(bar(kKVSFull), Nn & 1, wc);
                    ok = ok && mbar_wait(bar(kQFull + Nn % kQStages), (Nn / kQStages) & 1, wc);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    // visible query columns [lo, hi] of this tile for this key row (a query
                    // tile holds consecutive positions in every layout)
                    const int2 qi = qinfo[Nn % kQStages];
                    int lo = max(0, kr.vis_lo - qi.x);
                    const int hi = min(qi.y - 1, kr.vis_hi - qi.x);
                    if (!kr.key_valid) lo = kRows;
                    const bool masked = __any_sync(0xffffffffu, lo > 0 || hi < kRows - 1);
                    const float* nl2 = stats_nlse2(Nn % kQStages) + kKVCols * part;
                    const float* ndv = stats_ndvec(st) + kKVCols * part;
                    // P^T = exp2(S^T scale log2(e) - lse log2(e)); kept in fp32 for dS^T.  The
                    // bf16 pairs of the warp's two 16-query chunks go to the first 8 of each
                    // chunk's 16 fp32 columns (the layout the MMA issuer reads them in).
                    uint64_t pp[16];
                    {
                        uint32_t sr[32];
                        tmem_ld32(tS, sr);
                        uint32_t pk[16];
#pragma unroll
                        for (int i2 = 0; i2 < 8; ++i2) {
                            const ulonglong2 nl = *reinterpret_cast<const ulonglong2*>(nl2 + 4 * i2);
                            const uint64_t x0 = ffma2(f2pack(u2f(sr[4 * i2]), u2f(sr[4 * i2 + 1])), sl2, nl.x);
                            const uint64_t x1 = ffma2(f2pack(u2f(sr[4 * i2 + 2]), u2f(sr[4 * i2 + 3])), sl2, nl.y);
                            float a0, a1, a2, a3;
                            f2unpack(x0, a0, a1);
                            f2unpack(x1, a2, a3);
                            float e[4] = {ex2(a0), ex2(a1), ex2(a2), ex2(a3)};
                            if (masked) {
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const int c = kKVCols * part + 4 * i2 + j;
                                    e[j] = (c >= lo && c <= hi) ? e[j] : 0.f;
                                }
                            }
                            pp[2 * i2] = f2pack(e[0], e[1]);
                            pp[2 * i2 + 1] = f2pack(e[2], e[3]);
                            pk[2 * i2] = pack_bf16x2(e[0], e[1]);
                            pk[2 * i2 + 1] = pack_bf16x2(e[2], e[3]);
                        }
                        tmem_st8x2(tS, tS + 16, pk);
                    }
                    tc_fence_before();
                    mbar_arrive(bar(kKVPFull));
                    // dS^T = P^T (dP^T - Dvec)
                    ok = mbar_wait(bar(kKVDPFull), Nn & 1, wc);
                    ok = ok && mbar_wait(bar(kKVDOFull + st), (Nn >> 1) & 1, wc);    // -Dvec statistics
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc_fence_after();
                    {
                        uint32_t dr[32];
                        tmem_ld32(tP, dr);
                        uint32_t pk[16];
#pragma unroll
                        for (int i2 = 0; i2 < 8; ++i2) {
                            const ulonglong2 nd = *reinterpret_cast<const ulonglong2*>(ndv + 4 * i2);
                            const uint64_t d0 = fadd2(f2pack(u2f(dr[4 * i2]), u2f(dr[4 * i2 + 1])), nd.x);
                            const uint64_t d1 = fadd2(f2pack(u2f(dr[4 * i2 + 2]), u2f(dr[4 * i2 + 3])), nd.y);
                            float g0, g1, g2, g3;
                            f2unpack(fmul2(pp[2 * i2], d0), g0, g1);
                            f2unpack(fmul2(pp[2 * i2 + 1], d1), g2, g3);
                            pk[2 * i2] = pack_bf16x2(g0, g1);
                            pk[2 * i2 + 1] = pack_bf16x2(g2, g3);
                        }
                        tmem_st8x2(tP, tP + 16, pk);
                    }
                    tc_fence_before();
                    mbar_arrive(bar(kKVDSFull));
                }
                if (!ok) break;
            }
            // persistent grids: the next unit and this thread's key row of it are set up
            // while this unit's last dK runs (the packed sequences' binary search included)
            const bool empty = n_blocks == 0;
            const KVUnit<kMode> cur_for_zero = U;
            int g_next = -1;
            if constexpr (kPersist != 0) {
                g_next = get_unit(i + 1, U);
                if (g_next >= 0) kr = key_row(U);
            }
            if (empty) {
                // an empty walk (only with malformed sequence boundaries): zero rows,
                // written by the first quarter's warps
                if (kPersist != 0 && part == 0) {
                    const int krow = kt * kRows + row;
                    if (krow < p.Ls) {
                        const long long off =
                            ((static_cast<long long>(b) * p.L + s * p.Ls + krow) * p.Hkv + hk) * D;
                        for (int c = 0; c < D; c += 8)
                            if (in_bounds(off + c, 8, p.kv_elems, p.status)) {
                                *reinterpret_cast<uint4*>(p.dk + off + c) = make_uint4(0u, 0u, 0u, 0u);
                                *reinterpret_cast<uint4*>(p.dv + off + c) = make_uint4(0u, 0u, 0u, 0u);
                            }
                    }
                }
                (void)cur_for_zero;
                g = g_next;
                continue;
            }
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kKVOFull), un & 1, wc));
            if (!ok) break;
            tc_fence_after();
            // parts 0-1 write the two column halves of dV, parts 2-3 those of dK
            const int which = part >> 1;
            const int col0 = (part & 1) * (D / 2);
            const uint32_t tA = tmem + lane_off + 256 + which * D + col0;
            const float mul = which ? p.scale : 1.f;
            const int krow0 = kt * kRows + quarter * 32;      // within shard s
            const long long off0 =
                ((static_cast<long long>(b) * p.L + s * p.Ls + krow0) * p.Hkv + hk) * D + col0;
            __nv_bfloat16* gdst = which ? p.dk : p.dv;
            if constexpr (kPersist == 0) {
                // the warp's 32 rows of D/2 columns leave through its slice of the Q stages (no
                // product reads them any more), so that each store covers whole row halves
                uint8_t* stage = smem + kQ + (warp - 4) * 32 * D;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tA + 32 * c, o);
                    uint32_t pk[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2)
                        pk[i2] = pack_bf16x2(u2f(o[2 * i2]) * mul, u2f(o[2 * i2 + 1]) * mul);
                    stage_row_chunks<D / 2>(stage, lane, 4 * c, pk);
                }
                __syncwarp();
                store_staged_rows<D / 2>(stage, lane, gdst, off0, static_cast<long long>(p.Hkv) * D,
                                         p.Ls - krow0, p.kv_elems, p.status);
            } else {
                // persistent grids: the Q stages are refilling, so each thread stores its row
                const long long roff = off0 + static_cast<long long>(lane) * p.Hkv * D;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tA + 32 * c, o);
                    uint32_t pk[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2)
                        pk[i2] = pack_bf16x2(u2f(o[2 * i2]) * mul, u2f(o[2 * i2 + 1]) * mul);
                    if (krow0 + lane < p.Ls) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (in_bounds(roff + 32 * c + 8 * j, 8, p.kv_elems, p.status))
                                *reinterpret_cast<uint4*>(gdst + roff + 32 * c + 8 * j) =
                                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
            }
            // this warp's reads of dK, dV are complete before the next unit's first dV
            // product (gated on its P^T, which this warp writes later) overwrites them
            N += n_blocks;
            ++un;
            g = g_next;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------- dQ --

enum : int {
    kQDFull = 0,     // Q and dO of the tile
    kDKFull = 1,     // +stage (three K stages: K is read last by dQ, late in a block)
    kDKEmpty = 4,    // +stage
    kDVFull = 7,     // +stage (two V stages)
    kDVEmpty = 9,    // +stage
    kDSFull = 11,    // +(block parity): S ready
    kDDSFull = 13,   // +(block parity): dS written
    kDOFull = 15,    // dQ final
    kDDone = 16,
    kDPFull = 17,    // dP ready
    kDUnitFull = 18, // +slot: persistent grids, the producer published a unit
    kDUnitEmpty = 20,// +slot: every consumer warp has read it
    kDQDEmpty = 22,  // persistent grids: the unit's last S and dP (readers of Q, dO) finished
    kDBars = 23
};
constexpr int kKStages = 3;
// the dQ kernel's barrier area is 512 bytes (its shared memory has room): barriers, TMEM
// address and abort flag, per-K-stage tile records, the persistent grids' unit ring
constexpr int kDBarArea = 512;
constexpr int kDInfoOff = 256;
constexpr int kDRingOff = 288;
constexpr int kDUnitReaders = 1 + 8;    // the MMA warp and the eight elementwise warps

// A dQ work unit: one 128-row query tile of one (batch, head) and the K/V tiles it meets.
template <int kMode>
struct QUnit {
    int bh, b, h, hk, r, qt, q_local0, q0, n_first, n_blocks;
    PosWalk walk;

    // unit g of the call: heaviest query tile first (last shard, last tile), two (b, h)
    // pairs interleaved (unit_of_block)
    __device__ __forceinline__ void decode(int g, const BwdParams& p)
    {
        const int units_per_bh = p.P * p.n_t;
        int u;
        unit_of_block(g, p.B * p.H, units_per_bh, bh, u);
        r = p.P - 1 - u / p.n_t;
        qt = p.n_t - 1 - (u - (u / p.n_t) * p.n_t);
        if constexpr (kMode == 1) {
            // zigzag: a query tile's work grows with its global position, so heaviest
            // first is descending position order
            zigzag_tile_at(p.P * p.n_t - 1 - u, p.P, p.n_t, r, qt);
        }
        if constexpr (kMode == 2) {
            if (p.sched_q != nullptr) {
                const int x = checked_ldg(p.sched_q, u, p.sched_elems, p.status);
                if (static_cast<unsigned>(x) < static_cast<unsigned>(units_per_bh)) {
                    r = x / p.n_t;
                    qt = x - r * p.n_t;
                }
            }
        }
    }
    // zigzag shards and packed sequences: the key positions [lo, hi] some query of the
    // tile sees (causal: up to its last query; packed: within the sequences of its first
    // and last query)
    __device__ __forceinline__ void bounds(const BwdParams& p, int& lo, int& hi) const
    {
        constexpr bool kZig = kMode == 1;
        const int ql = qt * kRows;
        const int q_last = min(p.Ls - 1, ql + kRows - 1);
        const int qp0 = layout_position(r, ql, p.Ls, p.P, kZig);
        const int qp1 = layout_position(r, q_last, p.Ls, p.P, kZig);
        lo = 0;
        hi = qp1;
        if constexpr (kMode == 2) {
            int f0, l0, f1, l1;
            seq_range(p.cu_seqlens, p.n_seqs, qp0, f0, l0, p.status);
            seq_range(p.cu_seqlens, p.n_seqs, qp1, f1, l1, p.status);
            lo = f0;
            if (!p.causal) hi = l1;
        }
    }
    __device__ __forceinline__ void finish(const BwdParams& p, int lo, int hi)
    {
        b = bh / p.H;
        h = bh - b * p.H;
        hk = h / p.group;                       // key/value head of this query head
        q_local0 = qt * kRows;
        q0 = r * p.Ls + q_local0;
        // the forward's ring order: K/V shard (r - t) mod P at step t, future shards skipped
        if (p.causal) {
            const int q_last = min(p.Ls - 1, q_local0 + kRows - 1);
            n_first = min(p.n_t, q_last / kRows + 1);
            n_blocks = n_first + r * p.n_t;
        } else {
            n_first = p.n_t;
            n_blocks = p.P * p.n_t;
        }
        if constexpr (kMode != 0) {
            // the K/V tiles holding those positions, in the same ring order
            walk.init(r, -1, p.P, p.Ls, kMode == 1 ? 1 : 0, lo, hi);
            n_blocks = walk.total();
        } else {
            (void)lo;
            (void)hi;
        }
    }
    __device__ __forceinline__ void setup(int g, const BwdParams& p)
    {
        decode(g, p);
        int lo = 0, hi = 0;
        if constexpr (kMode != 0) bounds(p, lo, hi);
        finish(p, lo, hi);
    }
    // block n (in order 0, 1, 2, ... for modes 1 and 2): K/V shard s, tile kt
    __device__ __forceinline__ void block(int n, const BwdParams& p, int& s, int& kt)
    {
        if constexpr (kMode != 0) {
            walk.at(n);
            s = walk.x;
            kt = walk.tile();
            return;
        }
        if (n < n_first) {
            s = r;
            kt = n;
            return;
        }
        const int m = n - n_first;
        const int t = 1 + m / p.n_t;
        kt = m - (t - 1) * p.n_t;
        s = r - t;
        if (s < 0) s += p.P;
    }
};

// kPersist: 0 one CTA per query tile; 2 one CTA per SM taking units dynamically (packed
// sequences with a schedule), as the dK/dV kernel: the next unit's Q and dO load once the
// current unit's last S and dP (their last readers) have finished, K/V stages stream on
// across units, and the epilogue stores dQ from registers.
template <int D, int kMode, int kPersist>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_do, const BwdParams p)
{
    using Lay = BwdLayout<D>;
    constexpr int T = Lay::kTileBytes;
    constexpr int kQ = 0, kDO = T, kK = 2 * T, kV = (2 + kKStages) * T, kBar = (4 + kKStages) * T;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBar + kDBars * 8);
    int* abort_flag = reinterpret_cast<int*>(smem + kBar + kDBars * 8 + 4);
    // per K stage: first key position and valid key rows (written by the producer)
    int2* kinfo = reinterpret_cast<int2*>(smem + kBar + kDInfoOff);
    volatile int* unit_slot = reinterpret_cast<volatile int*>(smem + kBar + kDRingOff);
    static_assert(kDBars * 8 + 8 <= kDInfoOff && kDInfoOff + 8 * kKStages <= kDRingOff &&
                      kDRingOff + 2 * kRingInts * 4 <= kDBarArea,
                  "barrier area");
    auto bar = [&](int i) -> uint32_t { return sbase + kBar + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool kZig = kMode == 1;
    WaitCtx wc{abort_flag, p.status, p.timeout_ns};

    // The i-th unit of this CTA, set up in V (-1: no more); dynamic grids read the ring.
    auto consume_unit = [&](int i, QUnit<kMode>& V) -> int {
        if constexpr (kPersist == 0) {
            if (i > 0) return -1;
            V.setup(static_cast<int>(blockIdx.x), p);
            return static_cast<int>(blockIdx.x);
        }
        const int slot = i & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kDUnitFull + slot), (i >> 1) & 1, wc)))
            return -1;
        volatile int* e = unit_slot + kRingInts * slot;
        const int g = e[0];
        if (g >= 0) {
            int u;
            unit_of_block(g, p.B * p.H, p.P * p.n_t, V.bh, u);
            V.r = e[1];
            V.qt = e[2];
            V.finish(p, e[3], e[4]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kDUnitEmpty + slot));
        return g;
    };

    QUnit<kMode> first;
    int g_first = -1;
    if constexpr (kPersist == 0) {
        g_first = consume_unit(0, first);
        if (first.n_blocks == 0) {        // every query of a tile sees at least its own key
            zero_tile_rows<D>(p.dq, first.b, p.L, p.H, first.h, first.q0,
                              min(kRows, p.Ls - first.q_local0), p.q_elems, p.status);
            return;
        }
    }

    if (threadIdx.x == 0) {
        mbar_init(bar(kQDFull), 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(bar(kDKFull + i), 1);
            mbar_init(bar(kDKEmpty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kDVFull + i), 1);
            mbar_init(bar(kDVEmpty + i), 1);
            mbar_init(bar(kDSFull + i), 1);
            mbar_init(bar(kDDSFull + i), 2 * kRows);
            mbar_init(bar(kDUnitFull + i), 1);
            mbar_init(bar(kDUnitEmpty + i), kDUnitReaders);
        }
        mbar_init(bar(kDOFull), 1);
        mbar_init(bar(kDDone), 1);
        mbar_init(bar(kDPFull), 1);
        mbar_init(bar(kDQDEmpty), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        const bool leader = elect_one();
        const uint64_t keep = l2_policy_evict_last();
        const uint64_t once = l2_policy_evict_first();
        if (leader) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        auto publish_unit = [&](int i, QUnit<kMode>& U) -> int {
            const int slot = i & 1;
            int g = -1;
            if (leader && in_bounds(p.claim_index, 1, p.claim_extent, p.status))
                g = atomicAdd(p.claim, 1);
            g = __shfl_sync(0xffffffffu, g, __ffs(__ballot_sync(0xffffffffu, leader)) - 1);
            if (g < 0 || g >= p.n_units) g = -1;
            int lo = 0, hi = 0;
            if (g >= 0) {
                U.decode(g, p);
                if constexpr (kMode != 0) U.bounds(p, lo, hi);
                U.finish(p, lo, hi);
            }
            if (i >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar(kDUnitEmpty + slot),
                                                             ((i - 2) >> 1) & 1, wc)))
                return -1;
            if (leader) {
                volatile int* e = unit_slot + kRingInts * slot;
                e[0] = g;
                e[1] = U.r;
                e[2] = U.qt;
                e[3] = lo;
                e[4] = hi;
                mbar_arrive(bar(kDUnitFull + slot));
            }
            __syncwarp();
            return g;
        };
        uint32_t N = 0;       // K/V blocks loaded by this CTA so far
        int un = 0;           // units with a non-empty walk so far
        int last_k[kKStages] = {-1, -1, -1}, last_v[2] = {-1, -1};
        bool ok = true;
        for (int i = 0; ok; ++i) {
            QUnit<kMode> U;
            int g;
            if constexpr (kPersist == 2) g = publish_unit(i, U);
            else {
                g = i == 0 ? g_first : -1;
                U = first;
            }
            if (g < 0) break;
            if (U.n_blocks == 0) continue;
            // Q and dO of the tile: refilled once the previous unit's last S and dP (their
            // last readers) have finished
            if (un > 0 && !(ok = __all_sync(0xffffffffu,
                                            mbar_wait(bar(kDQDEmpty), (un - 1) & 1, wc))))
                break;
            if (leader) {
                mbar_arrive_expect_tx(bar(kQDFull), 2 * T);
                for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                    tma_load_4d(sbase + kQ + bx * 16384, &tmap_q, bar(kQDFull), bx * 64, U.h, U.q0,
                                U.b, once);
                    tma_load_4d(sbase + kDO + bx * 16384, &tmap_do, bar(kQDFull), bx * 64, U.h, U.q0,
                                U.b, once);
                }
            }
            __syncwarp();
            for (int n = 0; n < U.n_blocks; ++n) {
                int s, kt;
                U.block(n, p, s, kt);
                const uint32_t Nn = N + n;
                const int st = Nn & 1;
                const uint32_t ph = (Nn >> 1) & 1;
                const int kst = Nn % kKStages;
                const uint32_t kph = (Nn / kKStages) & 1;
                const int row = s * p.Ls + kt * kRows;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kDKEmpty + kst), kph ^ 1, wc)))) break;
                if (leader) {
                    kinfo[kst] = make_int2(layout_position(s, kt * kRows, p.Ls, p.P, kZig),
                                           min(kRows, p.Ls - kt * kRows));
                    mbar_arrive_expect_tx(bar(kDKFull + kst), T);
                    for (int bx = 0; bx < Lay::kBoxes; ++bx)
                        tma_load_4d(sbase + kK + kst * T + bx * 16384, &tmap_k, bar(kDKFull + kst),
                                    bx * 64, U.hk, row, U.b, keep);
                }
                last_k[kst] = static_cast<int>(Nn);
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kDVEmpty + st), ph ^ 1, wc)))) break;
                if (leader) {
                    mbar_arrive_expect_tx(bar(kDVFull + st), T);
                    for (int bx = 0; bx < Lay::kBoxes; ++bx)
                        tma_load_4d(sbase + kV + st * T + bx * 16384, &tmap_v, bar(kDVFull + st),
                                    bx * 64, U.hk, row, U.b, keep);
                }
                last_v[st] = static_cast<int>(Nn);
            }
            N += U.n_blocks;
            ++un;
        }
        if (un > 0) mbar_wait_drain(bar(kQDFull), (un - 1) & 1, wc);
        for (int st = 0; st < kKStages; ++st)
            if (last_k[st] >= 0) mbar_wait_drain(bar(kDKFull + st), (last_k[st] / kKStages) & 1, wc);
        for (int st = 0; st < 2; ++st)
            if (last_v[st] >= 0) mbar_wait_drain(bar(kDVFull + st), (last_v[st] >> 1) & 1, wc);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        const bool leader = elect_one();
        constexpr uint32_t kIdescS = idesc_bf16_f32(kRows, kRows, false);
        constexpr uint32_t kIdescAcc = idesc_bf16_f32(kRows, D, true);
        const uint64_t dQ_A = sdesc_sw128(sbase + kQ, 16, 1024);
        const uint64_t dDO_A = sdesc_sw128(sbase + kDO, 16, 1024);
        const uint64_t dK_B = sdesc_sw128(sbase + kK, 16, 1024);      // K as K-major B
        const uint64_t dV_B = sdesc_sw128(sbase + kV, 16, 1024);      // V as K-major B
        const uint64_t dK_MN = sdesc_sw128(sbase + kK, 16384, 1024);  // K as MN-major B
        auto ss = [&](uint32_t dcol, uint64_t a0, uint64_t b0) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint64_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                mma_ss(tmem + dcol, a0 + off, b0 + off, kIdescS, k > 0 ? 1u : 0u);
            }
        };
        // TMEM: S, then dS, alternate between columns [0,128) and [128,256) by block parity;
        // dP always in [256,384); dQ in [384, 384 + D).  Per block the issuer waits twice:
        // for K(n+1) and V(n+1), then queues S(n+1); for dS(n), then queues dP(n+1) and
        // dQ(n).  Tensor-pipe order S(n+1) dP(n+1) dQ(n): block n+1's P is computed while
        // dP(n+1) and dQ(n) run.  Why each product may overwrite what it does:
        //  - S(n+1) goes over dS(n-1), which dQ(n-1) (issued before it) consumed;
        //  - dP(n+1) goes over dP(n), which every elementwise thread read before writing
        //    dS(n) (for a persistent grid's next unit too: the issuer left the unit's loop
        //    only after the last dS was written).
        // No barrier phase can be produced twice ahead of its consumer: S and dS use one
        // barrier per block parity, S(n+2)/dP(n+2) are queued only after dS(n+1) was
        // consumed, and dP has one barrier whose next phase follows dS of this block.
        // Block parities count on across a persistent CTA's units.
        constexpr uint32_t kDPCol = 256, kDQCol = 384;
        auto wait_kv = [&](uint32_t n) {
            return __all_sync(0xffffffffu,
                              mbar_wait2(bar(kDKFull + n % kKStages), (n / kKStages) & 1,
                                         bar(kDVFull + (n & 1)), (n >> 1) & 1, wc));
        };
        auto issue_s = [&](uint32_t n) {     // S(n) = Q K_n^T
            ss(128u * (n & 1), dQ_A, dK_B + (n % kKStages) * Lay::kTileU);
            tc_commit(bar(kDSFull + (n & 1)));
        };
        auto issue_dp = [&](uint32_t n) {    // dP(n) = dO V_n^T
            ss(kDPCol, dDO_A, dV_B + (n & 1) * Lay::kTileU);
            tc_commit(bar(kDPFull));
            tc_commit(bar(kDVEmpty + (n & 1)));
        };
        uint32_t N = 0;
        int un = 0;
        bool ok = true;
        for (int i = 0; ok; ++i) {
            int n_blocks;
            if (kPersist == 0) {
                if (i > 0) break;
                n_blocks = first.n_blocks;
            } else {
                QUnit<kMode> U;
                if (consume_unit(i, U) < 0) break;
                n_blocks = U.n_blocks;
            }
            if (n_blocks == 0) continue;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kQDFull), un & 1, wc)) && wait_kv(N);
            if (!ok) break;
            tc_fence_after();
            if (leader) {
                issue_s(N);
                issue_dp(N);
                // persistent grids: the unit's last readers of Q and dO have been issued
                if (kPersist != 0 && n_blocks == 1) tc_commit(bar(kDQDEmpty));
            }
            __syncwarp();
            for (int n = 0; ok && n < n_blocks; ++n) {
                const uint32_t Nn = N + n;
                const bool more = n + 1 < n_blocks;
                if (more) {
                    if (!(ok = wait_kv(Nn + 1))) break;
                    tc_fence_after();
                    if (leader) issue_s(Nn + 1);
                    __syncwarp();
                }
                if (!(ok = __all_sync(0xffffffffu,
                                      mbar_wait(bar(kDDSFull + (Nn & 1)), (Nn >> 1) & 1, wc))))
                    break;
                tc_fence_after();
                if (leader) {
                    if (more) {
                        issue_dp(Nn + 1);
                        if (kPersist != 0 && n + 2 == n_blocks) tc_commit(bar(kDQDEmpty));
                    }
                    const uint64_t b0 = dK_MN + (Nn % kKStages) * Lay::kTileU;
                    const uint32_t a0 = tmem + 128u * (Nn & 1);
                    // dQ += dS K; dS of keys [64 h, 64 h + 64) sits in columns [64 h, 64 h + 32)
#pragma unroll
                    for (int k = 0; k < kRows / 16; ++k)
                        mma_ts(tmem + kDQCol, a0 + 64 * (k >> 2) + (k & 3) * 8, b0 + ((k * 2048) >> 4),
                               kIdescAcc, (n > 0 || k > 0) ? 1u : 0u);
                    tc_commit(bar(kDKEmpty + Nn % kKStages));
                    if (!more) tc_commit(bar(kDOFull));
                }
                __syncwarp();
            }
            N += n_blocks;
            ++un;
        }
        if (leader) tc_commit(bar(kDDone));
        __syncwarp();
        mbar_wait_drain(bar(kDDone), 0, wc);
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------ elementwise
        const int quarter = warp & 3;
        const int half = (warp - 4) >> 2;                   // key columns [64 half, 64 half + 64)
        const int row = quarter * 32 + lane;                // query row of the tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint64_t sl2 = f2pack(p.scale_log2, p.scale_log2);
        const uint32_t tP = tmem + lane_off + 256 + 64 * half;                  // dP
        // this thread's query row of unit V: its statistics and the positions of the keys
        // it sees, [vis_lo, vis_hi]
        struct QRow {
            bool row_valid;
            float nl2, ndv;
            int vis_lo, vis_hi;
        };
        auto query_row = [&](const QUnit<kMode>& V) {
            QRow w;
            const int row_local = V.q_local0 + row;
            w.row_valid = row_local < p.Ls;
            const long long sidx = (static_cast<long long>(V.b) * p.L + V.q0 + row) * p.H + V.h;
            const bool stats_ok = w.row_valid && in_bounds(sidx, 1, p.row_elems, p.status);
            w.nl2 = stats_ok ? -p.lse[sidx] * kLog2e : 0.f;
            w.ndv = stats_ok ? -p.dvec[sidx] : 0.f;
            w.vis_lo = 0;
            w.vis_hi = kFar;
            if (w.row_valid) {
                const int qp = layout_position(V.r, row_local, p.Ls, p.P, kZig);
                if (p.causal || kZig) w.vis_hi = qp;
                if constexpr (kMode == 2) {
                    int f, l;
                    seq_range(p.cu_seqlens, p.n_seqs, qp, f, l, p.status);
                    w.vis_lo = f;
                    if (!p.causal) w.vis_hi = l;
                }
            }
            return w;
        };
        auto get_unit = [&](int i, QUnit<kMode>& V) -> int {
            if constexpr (kPersist == 0) {
                V = first;
                return i == 0 ? g_first : -1;
            }
            return consume_unit(i, V);
        };
        uint32_t N = 0;
        int un = 0;
        bool ok = true;
        QUnit<kMode> U;
        int g = get_unit(0, U);
        QRow qr = query_row(U);
        for (int i = 0; ok && g >= 0; ++i) {
            const int n_blocks = U.n_blocks;
            const uint64_t nl2x2 = f2pack(qr.nl2, qr.nl2);
            const uint64_t ndvx2 = f2pack(qr.ndv, qr.ndv);
            for (int n = 0; n < n_blocks; ++n) {
                const uint32_t Nn = N + n;
                // S(n), and the K stage of block n for its record: that stage is refilled
                // only after dQ(n), which waits for this warp's dS(n)
                ok = __all_sync(0xffffffffu, mbar_wait2(bar(kDSFull + (Nn & 1)), (Nn >> 1) & 1,
                                                        bar(kDKFull + Nn % kKStages), (Nn / kKStages) & 1, wc));
                if (!ok) break;
                tc_fence_after();
                // visible key columns [lo, lim] (a K/V tile holds consecutive positions in
                // every layout)
                const int2 ki = kinfo[Nn % kKStages];
                int lim = min(ki.y - 1, qr.vis_hi - ki.x);
                const int lo = qr.vis_lo - ki.x;
                if (!qr.row_valid) lim = -1;
                const bool masked = __any_sync(0xffffffffu, lim < kRows - 1 || lo > 0);
                const uint32_t tS = tmem + lane_off + 128u * (Nn & 1) + 64 * half;  // S, then dS
                // P = exp2(S scale log2(e) - lse log2(e)) of this warp's 64 columns, in fp32
                uint64_t pp[32];
                {
                    uint32_t sr[64];
                    tmem_ld64(tS, sr);
#pragma unroll
                    for (int i2 = 0; i2 < 32; ++i2) {
                        float a0, a1;
                        f2unpack(ffma2(f2pack(u2f(sr[2 * i2]), u2f(sr[2 * i2 + 1])), sl2, nl2x2), a0, a1);
                        float e0 = ex2(a0), e1 = ex2(a1);
                        if (masked) {
                            const int c = 64 * half + 2 * i2;
                            e0 = (c <= lim && c >= lo) ? e0 : 0.f;
                            e1 = (c + 1 <= lim && c + 1 >= lo) ? e1 : 0.f;
                        }
                        pp[i2] = f2pack(e0, e1);
                    }
                }
                // dS = P (dP - Dvec), bf16, written over this warp's S columns
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kDPFull), Nn & 1, wc)))) break;
                tc_fence_after();
                {
                    uint32_t dr[64];
                    tmem_ld64(tP, dr);
                    uint32_t pk[32];
#pragma unroll
                    for (int i2 = 0; i2 < 32; ++i2) {
                        const uint64_t d = fadd2(f2pack(u2f(dr[2 * i2]), u2f(dr[2 * i2 + 1])), ndvx2);
                        float g0, g1;
                        f2unpack(fmul2(pp[i2], d), g0, g1);
                        pk[i2] = pack_bf16x2(g0, g1);
                    }
                    // 64 keys as bf16 pairs: 32 columns inside the ones already read
                    tmem_st32(tS, pk);
                }
                tc_fence_before();
                mbar_arrive(bar(kDDSFull + (Nn & 1)));
            }
            if (!ok) break;
            // what the epilogue needs of this unit
            const bool empty = n_blocks == 0;
            const int b = U.b, h = U.h, r = U.r, q_local0 = U.q_local0;
            // persistent grids: the next unit and this thread's row of it (statistics loads
            // and the packed sequences' binary search) are set up while this unit's last dQ
            // runs
            int g_next = -1;
            if constexpr (kPersist != 0) {
                g_next = get_unit(i + 1, U);
                if (g_next >= 0) qr = query_row(U);
            }
            const int qrow0 = q_local0 + quarter * 32;        // within shard r
            if (empty) {
                // an empty walk (only with malformed sequence boundaries): zero rows, written
                // by the first half's warps
                if (kPersist != 0 && half == 0 && qrow0 + lane < p.Ls) {
                    const long long off =
                        ((static_cast<long long>(b) * p.L + r * p.Ls + qrow0 + lane) * p.H + h) * D;
                    for (int c = 0; c < D; c += 8)
                        if (in_bounds(off + c, 8, p.q_elems, p.status))
                            *reinterpret_cast<uint4*>(p.dq + off + c) = make_uint4(0u, 0u, 0u, 0u);
                }
                g = g_next;
                continue;
            }
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kDOFull), un & 1, wc));
            if (!ok) break;
            tc_fence_after();
            const long long off0 =
                ((static_cast<long long>(b) * p.L + r * p.Ls + qrow0) * p.H + h) * D + half * (D / 2);
            if constexpr (kPersist == 0) {
                // each half writes half of the D output columns, through the warp's slice of
                // the K stages (no product reads them any more) so that stores cover row halves
                uint8_t* stage = smem + kK + (warp - 4) * 32 * D;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    const int col = half * (D / 2) + 32 * c;
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + 384 + col, o);
                    uint32_t pk[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2)
                        pk[i2] = pack_bf16x2(u2f(o[2 * i2]) * p.scale, u2f(o[2 * i2 + 1]) * p.scale);
                    stage_row_chunks<D / 2>(stage, lane, 4 * c, pk);
                }
                __syncwarp();
                store_staged_rows<D / 2>(stage, lane, p.dq, off0, static_cast<long long>(p.H) * D,
                                         p.Ls - qrow0, p.q_elems, p.status);
            } else {
                // persistent grids: the K stages are refilling, so each thread stores its row
                const long long roff = off0 + static_cast<long long>(lane) * p.H * D;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    const int col = half * (D / 2) + 32 * c;
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + 384 + col, o);
                    uint32_t pk[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2)
                        pk[i2] = pack_bf16x2(u2f(o[2 * i2]) * p.scale, u2f(o[2 * i2 + 1]) * p.scale);
                    if (qrow0 + lane < p.Ls) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (in_bounds(roff + 32 * c + 8 * j, 8, p.q_elems, p.status))
                                *reinterpret_cast<uint4*>(p.dq + roff + 32 * c + 8 * j) =
                                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
            }
            // this warp's reads of dQ are complete before the next unit's first dQ product
            // (gated on its dS, which this warp writes later) overwrites it
            N += n_blocks;
            ++un;
            g = g_next;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------ dQ on pairs of SMs --
//
// bwd_dq_pair_kernel: the dQ kernel's products issued for a pair of SMs
// (tcgen05.mma.cta_group::2, M = 256), contiguous (kMode 0) or zigzag (kMode 1) shards,
// head dim 128.  A cluster of two CTAs takes two consecutive query tiles of one shard of
// one (batch, head) -- (2j, 2j + 1) of a contiguous shard, or of one chunk of a zigzag
// shard, where a chunk of an odd number of tiles leaves its last pair one tile -- and CTA
// rank c holds the pair's tile c: its Q and dO, and its rows of S/dS, dP and dQ in TMEM.
// Of every K/V block each CTA stages half, so a product reads half of its B operand from
// each SM's shared memory:
//   S = Q K^T (N = keys):    K keys [64 c, 64 c + 64), all head-dim columns;
//   dP = dO V^T (N = keys):  V keys [64 c, 64 c + 64);
//   dQ += dS K (N = D):      K head-dim columns [64 c, 64 c + 64) of all 128 keys.
// Per block and CTA that is 6 KiB + 4 KiB + 2 KiB of operand reads per 16-deep step
// instead of 8 + 8 + 4, and 48 instead of 64 KiB of K/V staging.  The pair walks the
// union of its tiles' key blocks (causal: the later tile's, one diagonal block more than
// the earlier tile needs, which is all masked for it, so its dS rows are 0; a CTA without
// a tile masks every row and stores nothing).  The even CTA's MMA
// warp issues every product; the even CTA's barriers count both CTAs' TMA bytes and both
// CTAs' dS (one arrival per elementwise warp); every commit goes to the same barrier of
// both CTAs.  Bounded waits and the exit handshake as in the pair forward.
template <int D, int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    bwd_dq_pair_kernel(const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_k64,
                       const __grid_constant__ CUtensorMap tmap_v64,
                       const __grid_constant__ CUtensorMap tmap_do, const BwdParams p)
{
    static_assert(D == 128, "pair dQ kernel: head dim 128");
    static_assert(kMode == 0 || kMode == 1, "pair dQ kernel: contiguous or zigzag shards");
    constexpr bool kZig = kMode == 1;
    constexpr int T = kRows * D * 2;        // one 128-row tile, 32 KiB
    constexpr int H2 = T / 2;               // one CTA's half of a K or V block
    constexpr int kQ = 0, kDO = T, kK = 2 * T, kV = 5 * T, kBar = 6 * T;
    // per K stage: keys half (two 64-column boxes of 64 rows), then the head-dim half (one
    // 64-column box of 128 rows); per V stage: keys half
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBar + kDBars * 8);
    int* abort_flag = reinterpret_cast<int*>(smem + kBar + kDBars * 8 + 4);
    static_assert(kDBars * 8 + 8 <= kDBarArea, "barrier area");
    auto bar = [&](int i) -> uint32_t { return sbase + kBar + 8u * i; };
    const uint32_t rank = cluster_ctarank();
    const bool lead = rank == 0;
    auto lead_bar = [&](int i) -> uint32_t { return mapa_shared(bar(i), 0); };
    constexpr uint16_t kBoth = 3;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work unit: a pair of query tiles, heaviest first (contiguous: last shard, last
    // pair; zigzag: descending global position), two (batch, head) pairs interleaved
    int bh, u, r, qt;
    bool tile_valid = true;             // zigzag: this CTA has a tile of the pair's chunk
    PosWalk zwalk;                      // zigzag: the pair's ring walk over positions
    int n_first = p.n_t, n_blocks = p.P * p.n_t;
    if constexpr (kZig) {
        const int per_chunk = p.n_t >> 1;
        const int npc = (per_chunk + 1) >> 1;
        unit_of_block(static_cast<int>(blockIdx.x >> 1), p.B * p.H, 2 * p.P * npc, bh, u);
        const int g = 2 * p.P * npc - 1 - u;
        const int chunk = g / npc, within = g - chunk * npc;
        const int base = chunk < p.P ? 0 : per_chunk;
        r = chunk < p.P ? chunk : 2 * p.P - 1 - chunk;
        tile_valid = 2 * within + static_cast<int>(rank) < per_chunk;
        qt = base + 2 * within + static_cast<int>(rank);
        // the K/V tiles holding positions up to the pair's last query, in the forward's
        // ring order (zigzag is causal)
        const int last_t = base + min(2 * within + 1, per_chunk - 1);
        zwalk.init(r, -1, p.P, p.Ls, 1, 0,
                   layout_position(r, last_t * kRows + kRows - 1, p.Ls, p.P, true));
        n_blocks = zwalk.total();
    } else {
        const int n_pair = (p.n_t + 1) / 2;
        unit_of_block(static_cast<int>(blockIdx.x >> 1), p.B * p.H, p.P * n_pair, bh, u);
        r = p.P - 1 - u / n_pair;
        const int pj = n_pair - 1 - (u - (u / n_pair) * n_pair);
        qt = 2 * pj + static_cast<int>(rank);
        // the pair's ring walk: K/V shard (r - t) mod P at step t, future shards skipped;
        // of the diagonal shard the tiles up to the pair's last query
        if (p.causal) {
            const int q_last = min(p.Ls - 1, (2 * pj + 1) * kRows + kRows - 1);
            n_first = min(p.n_t, q_last / kRows + 1);
            n_blocks = n_first + r * p.n_t;
        }
    }
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int hk = h / p.group;
    const int q_local0 = qt * kRows;
    const int q0 = r * p.Ls + q_local0;
    // walked in order: block n + 1 from block n (contiguous: the diagonal shard's first
    // n_first tiles, then whole shards r - 1, r - 2, ... mod P; zigzag: the position walk)
    struct Walk {
        int s, kt;
        PosWalk pw;
        __device__ __forceinline__ void start(int r, const PosWalk& z)
        {
            if constexpr (kZig) {
                pw = z;
                pw.at(0);
                s = pw.x;
                kt = pw.tile();
            } else {
                s = r;
                kt = 0;
            }
        }
        __device__ __forceinline__ void next(int n, int n_first, int n_t, int P)
        {
            if constexpr (kZig) {
                pw.at(n + 1);
                s = pw.x;
                kt = pw.tile();
            } else if (++kt == (n + 1 == n_first ? n_first : n_t)) {
                kt = 0;
                s = s == 0 ? P - 1 : s - 1;
            }
        }
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(kQDFull), 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(bar(kDKFull + i), 1);
            mbar_init(bar(kDKEmpty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kDVFull + i), 1);
            mbar_init(bar(kDVEmpty + i), 1);
            mbar_init(bar(kDSFull + i), 1);
            mbar_init(bar(kDDSFull + i), 2 * 8);   // one arrival per elementwise warp, both CTAs
        }
        mbar_init(bar(kDOFull), 1);
        mbar_init(bar(kDDone), 1);
        mbar_init(bar(kDPFull), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(tmem_slot), 512);
        tmem_relinquish_pair();
        tc_fence_before();
    }
    // both CTAs' barriers exist and the pair's TMEM is allocated before either CTA signals
    // the other
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------ producer (both CTAs)
        const bool leader = elect_one();
        const uint64_t keep = l2_policy_evict_last();
        const uint64_t once = l2_policy_evict_first();
        if (leader) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_k64);
            tma_prefetch_desc(&tmap_v64);
            // this CTA's Q and dO tiles, counted on the even CTA's barrier
            if (lead) mbar_arrive_expect_tx(bar(kQDFull), 4 * T);
            for (int bx = 0; bx < 2; ++bx) {
                tma_load_4d_pair(sbase + kQ + bx * 16384, &tmap_q, lead_bar(kQDFull), bx * 64, h, q0,
                                 b, once);
                tma_load_4d_pair(sbase + kDO + bx * 16384, &tmap_do, lead_bar(kQDFull), bx * 64, h,
                                 q0, b, once);
            }
        }
        int last_k[kKStages] = {-1, -1, -1}, last_v[2] = {-1, -1};
        Walk w;
        w.start(r, zwalk);
        for (int n = 0; n < n_blocks; w.next(n, n_first, p.n_t, p.P), ++n) {
            const int s = w.s, kt = w.kt;
            const int st = n & 1;
            const uint32_t ph = (n >> 1) & 1;
            const int kst = n % kKStages;
            const uint32_t kph = (n / kKStages) & 1;
            const int row = s * p.Ls + kt * kRows;               // first key of the block
            const int krow = row + 64 * static_cast<int>(rank);  // this CTA's keys
            if (!__all_sync(0xffffffffu, mbar_wait(bar(kDKEmpty + kst), kph ^ 1, wc))) break;
            if (leader) {
                if (lead) mbar_arrive_expect_tx(bar(kDKFull + kst), 2 * (H2 + H2));
                const uint32_t base = sbase + kK + kst * T;
                for (int bx = 0; bx < 2; ++bx)
                    tma_load_4d_pair(base + bx * 8192, &tmap_k64, lead_bar(kDKFull + kst), bx * 64, hk,
                                     krow, b, keep);
                tma_load_4d_pair(base + H2, &tmap_k, lead_bar(kDKFull + kst), 64 * static_cast<int>(rank),
                                 hk, row, b, keep);
            }
            last_k[kst] = n;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(kDVEmpty + st), ph ^ 1, wc))) break;
            if (leader) {
                if (lead) mbar_arrive_expect_tx(bar(kDVFull + st), 2 * H2);
                for (int bx = 0; bx < 2; ++bx)
                    tma_load_4d_pair(sbase + kV + st * H2 + bx * 8192, &tmap_v64, lead_bar(kDVFull + st),
                                     bx * 64, hk, krow, b, keep);
            }
            last_v[st] = n;
        }
        // the even CTA's barriers count both CTAs' copies: it waits for all of them to land
        // (the odd CTA leaves only after the cluster-wide barrier that follows)
        if (lead) {
            mbar_wait_drain(bar(kQDFull), 0, wc);
            for (int st = 0; st < kKStages; ++st)
                if (last_k[st] >= 0) mbar_wait_drain(bar(kDKFull + st), (last_k[st] / kKStages) & 1, wc);
            for (int st = 0; st < 2; ++st)
                if (last_v[st] >= 0) mbar_wait_drain(bar(kDVFull + st), (last_v[st] >> 1) & 1, wc);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer (even CTA)
        if (lead) {
            const bool leader = elect_one();
            constexpr uint32_t kIdescS = idesc_bf16_f32(2 * kRows, kRows, false);
            constexpr uint32_t kIdescAcc = idesc_bf16_f32(2 * kRows, D, true);
            // Q, dO (A, K-major): 128 rows per 64-column box (16 KiB); K, V keys half (B,
            // K-major): 64 keys per box (8 KiB); K head-dim half (B, MN-major): one
            // 64-column box of 128 keys, 8 keys per 1024-byte swizzle atom, 16-key steps
            // 2 KiB apart
            const uint64_t dQ_A = sdesc_sw128(sbase + kQ, 16, 1024);
            const uint64_t dDO_A = sdesc_sw128(sbase + kDO, 16, 1024);
            const uint64_t dK_B = sdesc_sw128(sbase + kK, 16, 1024);
            const uint64_t dV_B = sdesc_sw128(sbase + kV, 16, 1024);
            const uint64_t dK_MN = sdesc_sw128(sbase + kK + H2, 16384, 1024);
            constexpr uint64_t kTU = static_cast<uint64_t>(T) >> 4, kHU = static_cast<uint64_t>(H2) >> 4;
            auto ss = [&](uint32_t dcol, uint64_t a0, uint64_t b0) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t oa = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                    const uint64_t ob = ((k >> 2) * 8192 + (k & 3) * 32) >> 4;
                    mma_ss_pair(tmem + dcol, a0 + oa, b0 + ob, kIdescS, k > 0 ? 1u : 0u);
                }
            };
            // TMEM columns as in the single-SM dQ kernel: S, then dS, alternate between
            // [0,128) and [128,256) by block parity; dP in [256,384); dQ in [384,512).  The
            // issue order and the reasons each product may overwrite what it does are the
            // single-SM kernel's.
            constexpr uint32_t kDPCol = 256, kDQCol = 384;
            auto wait_kv = [&](uint32_t n) {
                return __all_sync(0xffffffffu,
                                  mbar_wait2(bar(kDKFull + n % kKStages), (n / kKStages) & 1,
                                             bar(kDVFull + (n & 1)), (n >> 1) & 1, wc));
            };
            auto issue_s = [&](uint32_t n) {     // S(n) = Q K_n^T
                ss(128u * (n & 1), dQ_A, dK_B + (n % kKStages) * kTU);
                tc_commit_pair(bar(kDSFull + (n & 1)), kBoth);
            };
            auto issue_dp = [&](uint32_t n) {    // dP(n) = dO V_n^T
                ss(kDPCol, dDO_A, dV_B + (n & 1) * kHU);
                tc_commit_pair(bar(kDPFull), kBoth);
                tc_commit_pair(bar(kDVEmpty + (n & 1)), kBoth);
            };
            bool ok = n_blocks > 0 &&
                      __all_sync(0xffffffffu, mbar_wait(bar(kQDFull), 0, wc)) && wait_kv(0);
            if (ok) {
                tc_fence_after();
                if (leader) {
                    issue_s(0);
                    issue_dp(0);
                }
                __syncwarp();
            }
            for (int n = 0; ok && n < n_blocks; ++n) {
                const uint32_t Nn = n;
                const bool more = n + 1 < n_blocks;
                if (more) {
                    if (!(ok = wait_kv(Nn + 1))) break;
                    tc_fence_after();
                    if (leader) issue_s(Nn + 1);
                    __syncwarp();
                }
                if (!(ok = __all_sync(0xffffffffu,
                                      mbar_wait(bar(kDDSFull + (Nn & 1)), (Nn >> 1) & 1, wc))))
                    break;
                tc_fence_after();
                if (leader) {
                    if (more) issue_dp(Nn + 1);
                    const uint64_t b0 = dK_MN + (Nn % kKStages) * kTU;
                    const uint32_t a0 = tmem + 128u * (Nn & 1);
                    // dQ += dS K; dS of keys [64 x, 64 x + 64) sits in columns [64 x, 64 x + 32)
#pragma unroll
                    for (int k = 0; k < kRows / 16; ++k)
                        mma_ts_pair(tmem + kDQCol, a0 + 64 * (k >> 2) + (k & 3) * 8,
                                    b0 + ((k * 2048) >> 4), kIdescAcc, (n > 0 || k > 0) ? 1u : 0u);
                    tc_commit_pair(bar(kDKEmpty + Nn % kKStages), kBoth);
                    if (!more) tc_commit_pair(bar(kDOFull), kBoth);
                }
                __syncwarp();
            }
            // every product the pair issued has finished before either CTA frees TMEM: the
            // even CTA's issuer waits for them here; the odd CTA's issuer goes to the cluster
            // barrier below without spinning through the kernel (the even one arrives there
            // only after this wait) and then sees the same commit's arrival on its own barrier
            if (leader) tc_commit_pair(bar(kDDone), kBoth);
            __syncwarp();
            mbar_wait_drain(bar(kDDone), 0, wc);
            __syncwarp();
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------ elementwise (both CTAs)
        const int quarter = warp & 3;
        const int half = (warp - 4) >> 2;                   // key columns [64 half, 64 half + 64)
        const int row = quarter * 32 + lane;                // query row of this CTA's tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint64_t sl2 = f2pack(p.scale_log2, p.scale_log2);
        const uint32_t tP = tmem + lane_off + 256 + 64 * half;                  // dP
        const int row_local = q_local0 + row;
        const bool row_valid = kZig ? tile_valid : row_local < p.Ls;
        const long long sidx = (static_cast<long long>(b) * p.L + q0 + row) * p.H + h;
        const bool stats_ok = row_valid && in_bounds(sidx, 1, p.row_elems, p.status);
        const float nl2 = stats_ok ? -p.lse[sidx] * kLog2e : 0.f;
        const float ndv = stats_ok ? -p.dvec[sidx] : 0.f;
        // causal bound: the row's global position (zigzag positions, chunks of whole tiles)
        const int vis_hi = kZig       ? layout_position(r, row_local, p.Ls, p.P, true)
                           : p.causal ? r * p.Ls + row_local
                                      : kFar;
        const uint64_t nl2x2 = f2pack(nl2, nl2), ndvx2 = f2pack(ndv, ndv);
        bool ok = true;
        Walk w;
        w.start(r, zwalk);
        for (int n = 0; n < n_blocks; w.next(n, n_first, p.n_t, p.P), ++n) {
            const uint32_t Nn = n;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kDSFull + (Nn & 1)), (Nn >> 1) & 1, wc));
            if (!ok) break;
            tc_fence_after();
            // visible key columns [0, lim] of the block
            const int s = w.s, kt = w.kt;
            const int kp0 = kZig ? layout_position(s, kt * kRows, p.Ls, p.P, true) : s * p.Ls + kt * kRows;
            int lim = min(min(kRows, p.Ls - kt * kRows) - 1, vis_hi - kp0);
            if (!row_valid) lim = -1;
            const bool masked = __any_sync(0xffffffffu, lim < kRows - 1);
            const uint32_t tS = tmem + lane_off + 128u * (Nn & 1) + 64 * half;  // S, then dS
            // P = exp2(S scale log2(e) - lse log2(e)) of this warp's 64 columns, in fp32
            uint64_t pp[32];
            {
                uint32_t sr[64];
                tmem_ld64(tS, sr);
#pragma unroll
                for (int i2 = 0; i2 < 32; ++i2) {
                    float a0, a1;
                    f2unpack(ffma2(f2pack(u2f(sr[2 * i2]), u2f(sr[2 * i2 + 1])), sl2, nl2x2), a0, a1);
                    float e0 = ex2(a0), e1 = ex2(a1);
                    if (masked) {
                        const int c = 64 * half + 2 * i2;
                        e0 = c <= lim ? e0 : 0.f;
                        e1 = c + 1 <= lim ? e1 : 0.f;
                    }
                    pp[i2] = f2pack(e0, e1);
                }
            }
            // dS = P (dP - Dvec), bf16, written over this warp's S columns
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kDPFull), Nn & 1, wc)))) break;
            tc_fence_after();
            {
                uint32_t dr[64];
                tmem_ld64(tP, dr);
                uint32_t pk[32];
#pragma unroll
                for (int i2 = 0; i2 < 32; ++i2) {
                    const uint64_t d = fadd2(f2pack(u2f(dr[2 * i2]), u2f(dr[2 * i2 + 1])), ndvx2);
                    float g0, g1;
                    f2unpack(fmul2(pp[i2], d), g0, g1);
                    pk[i2] = pack_bf16x2(g0, g1);
                }
                tmem_st32(tS, pk);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(lead_bar(kDDSFull + (Nn & 1)));
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(kDOFull), 0, wc));
        if (ok) {
            tc_fence_after();
            // each half writes half of the D output columns of this CTA's rows, through the
            // warp's slice of the K stages (no product reads them any more) so that stores
            // cover row halves
            const int qrow0 = q_local0 + quarter * 32;         // within shard r
            const long long off0 =
                ((static_cast<long long>(b) * p.L + r * p.Ls + qrow0) * p.H + h) * D + half * (D / 2);
            uint8_t* stage = smem + kK + (warp - 4) * 32 * D;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                const int col = half * (D / 2) + 32 * c;
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + 384 + col, o);
                uint32_t pk[16];
#pragma unroll
                for (int i2 = 0; i2 < 16; ++i2)
                    pk[i2] = pack_bf16x2(u2f(o[2 * i2]) * p.scale, u2f(o[2 * i2 + 1]) * p.scale);
                stage_row_chunks<D / 2>(stage, lane, 4 * c, pk);
            }
            __syncwarp();
            store_staged_rows<D / 2>(stage, lane, p.dq, off0, static_cast<long long>(p.H) * D,
                                     tile_valid ? p.Ls - qrow0 : 0, p.q_elems, p.status);
        }
    }

    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        if (!lead) mbar_wait_drain(bar(kDDone), 0, wc);
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

template <int D, int kMode, int kPersist>
cudaError_t launch_bwd_d(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap* tk64,
                         const CUtensorMap* tv64)
{
    using Lay = BwdLayout<D>;
    constexpr int kSmemKV = KVSmem<D>::kAlloc;
    constexpr int kSmemQ = (4 + kKStages) * Lay::kTileBytes + kDBarArea + 1024;
    static_assert(kSmemQ <= kMaxSmem, "dQ shared memory layout exceeds the limit");
    static std::atomic<int> configured_kv[kMaxDevices], configured_q[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = smem_limit_once(configured_kv, dev, bwd_dkdv_kernel<D, kMode, kPersist>, kSmemKV);
    if (e != cudaSuccess) return e;
    e = smem_limit_once(configured_q, dev, bwd_dq_kernel<D, kMode, kPersist>, kSmemQ);
    if (e != cudaSuccess) return e;
    // Dvec = rowsum(dO o O) into the workspace
    const long long rows = static_cast<long long>(a.B) * a.L * a.H;
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (rows * (D / 8) + 255) / 256;
    if (blocks > static_cast<long long>(sms) * 8) blocks = static_cast<long long>(sms) * 8;
    if (blocks < 1) blocks = 1;
    bwd_rowdot_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
        static_cast<const uint4*>(a.out), static_cast<const uint4*>(a.dout), a.dvec, rows, a.status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    BwdParams p;
    p.lse = a.lse;
    p.dvec = a.dvec;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.B = a.B;
    p.L = a.L;
    p.H = a.H;
    p.Hkv = a.Hkv;
    p.group = a.H / a.Hkv;
    p.P = a.P;
    p.Ls = a.L / a.P;
    p.causal = a.causal;
    p.n_t = (p.Ls + kRows - 1) / kRows;
    p.scale = 1.0f / sqrtf(static_cast<float>(D));
    p.scale_log2 = kLog2e * p.scale;
    p.cu_seqlens = a.cu_seqlens;
    p.n_seqs = a.n_seqs;
    p.sched_k = p.sched_q = nullptr;
    p.q_elems = static_cast<long long>(a.B) * a.L * a.H * D;
    p.kv_elems = static_cast<long long>(a.B) * a.L * a.Hkv * D;
    p.row_elems = static_cast<long long>(a.B) * a.L * a.H;
    p.sched_elems = a.P * p.n_t;
    p.claim = nullptr;
    p.claim_index = 0;
    p.claim_extent = 0;
    VarlenSchedLayout lay{};
    if (a.schedule != nullptr) {
        lay = varlen_sched_layout(a.L, a.P);
        p.sched_k = a.schedule + lay.bwd_k;
        p.sched_q = a.schedule + lay.bwd_q;
    }
    // dK/dV: one unit per key tile of each key/value head; dQ: per query tile of each head
    const long long units_kv = static_cast<long long>(a.B) * a.Hkv * a.P * p.n_t;
    const long long units_q = static_cast<long long>(a.B) * a.H * a.P * p.n_t;
    if (units_q <= 0 || units_q > 0x7fffffffLL || units_kv <= 0) return cudaErrorInvalidConfiguration;
    long long grid_kv = units_kv, grid_q = units_q;
    BwdParams pk = p, pq = p;
    pk.n_units = static_cast<int>(units_kv);
    pq.n_units = static_cast<int>(units_q);
    if constexpr (kPersist == 2) {
        // one CTA per SM claiming units from the schedule array's counters (entries 2 and
        // 4 of the counters; both zeroed here, in stream order)
        if (grid_kv > sms) grid_kv = sms;
        if (grid_q > sms) grid_q = sms;
        int* ctr = const_cast<int*>(a.schedule) + lay.counters;
        e = cudaMemsetAsync(ctr + 2, 0, 4 * sizeof(int), a.stream);
        if (e != cudaSuccess) return e;
        pk.claim = ctr + 2;
        pk.claim_index = lay.counters + 2;
        pq.claim = ctr + 4;
        pq.claim_index = lay.counters + 4;
        pk.claim_extent = pq.claim_extent = lay.total;
    }
    bwd_dkdv_kernel<D, kMode, kPersist>
        <<<static_cast<unsigned>(grid_kv), kKVThreads, kSmemKV, a.stream>>>(tq, tk, tv, tdo, pk);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if constexpr (D == 128 && (kMode == 0 || kMode == 1) && kPersist == 0) {
        if (tk64 != nullptr && tv64 != nullptr) {
            // dQ on pairs of SMs: one cluster per pair of query tiles (zigzag: per pair
            // within a chunk, a chunk of an odd number of tiles ending in a lone tile)
            constexpr int kSmemPair = 6 * Lay::kTileBytes + kDBarArea + 1024;
            static_assert(kSmemPair <= kMaxSmem, "pair dQ shared memory layout exceeds the limit");
            static std::atomic<int> configured_pair[kMaxDevices];
            e = smem_limit_once(configured_pair, dev, bwd_dq_pair_kernel<D, kMode>, kSmemPair);
            if (e != cudaSuccess) return e;
            const int pairs_per_shard = kMode == 1 ? 2 * ((p.n_t / 2 + 1) / 2) : (p.n_t + 1) / 2;
            const long long pairs = static_cast<long long>(a.B) * a.H * a.P * pairs_per_shard;
            if (2 * pairs > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
            bwd_dq_pair_kernel<D, kMode><<<static_cast<unsigned>(2 * pairs), kThreads, kSmemPair, a.stream>>>(
                tq, tk, *tk64, *tv64, tdo, pq);
            return cudaGetLastError();
        }
    }
    (void)tk64;
    (void)tv64;
    bwd_dq_kernel<D, kMode, kPersist>
        <<<static_cast<unsigned>(grid_q), kThreads, kSmemQ, a.stream>>>(tq, tk, tv, tdo, pq);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_layout(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap* tk64,
                              const CUtensorMap* tv64)
{
    // packed sequences with a schedule: persistent grids that claim units heaviest first;
    // the other layouts keep one CTA per tile (the block scheduler balances their
    // heaviest-first order)
    if (a.cu_seqlens != nullptr) {
        if (a.schedule != nullptr) return launch_bwd_d<D, 2, 2>(a, tq, tk, tv, tdo, nullptr, nullptr);
        return launch_bwd_d<D, 2, 0>(a, tq, tk, tv, tdo, nullptr, nullptr);
    }
    if (a.zigzag) return launch_bwd_d<D, 1, 0>(a, tq, tk, tv, tdo, tk64, tv64);
    return launch_bwd_d<D, 0, 0>(a, tq, tk, tv, tdo, tk64, tv64);
}

}  // namespace

bool bwd_dq_pair_applies(const BwdArgs& a)
{
    // head dim 128 over contiguous or zigzag shards (plain and grouped heads)
    return a.D == 128 && a.cu_seqlens == nullptr;
}

cudaError_t launch_attn_bwd_bf16(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo,
                                 const CUtensorMap* tk64, const CUtensorMap* tv64)
{
    if (a.D == 64) return launch_bwd_layout<64>(a, tq, tk, tv, tdo, nullptr, nullptr);
    if (a.D == 128) return launch_bwd_layout<128>(a, tq, tk, tv, tdo, tk64, tv64);
    return cudaErrorInvalidValue;
}

}  // namespace ra
