// attn_bf16_sm103.cu -- exact attention forward over P virtual ring shards,
// bf16 in / fp32 accumulate, on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes ("序列并行与 Ring Attention"): O = softmax(Q K^T / sqrt(D)) V
// (section 3.1) by the online-softmax recurrence of section 3.2 (running max m,
// denominator l, unnormalised sum u, rescale alpha = exp(m_t - m_{t+1}),
// o = u / l), visiting K/V in the ring order of section 3.3 (the queries of
// shard r meet shard (r - t) mod P at step t) and, under causal masking,
// skipping shards wholly in the future and masking the diagonal shard by
// global position (section 3.4).
//
// One CTA owns two 128-row query tiles of one shard of one (batch, head) and
// walks that shard's K/V blocks (128 keys each) in ring order.  Warp roles:
//   warp 0      TMA producer: Q tiles once, then K and V blocks through two
//               2-deep shared-memory rings (the next block loads while the
//               current one is used: the ring's double buffer, section 6.3).
//   warp 1      MMA issuer: S_t = Q_t K^T into TMEM, then O_t += P_t V with P_t
//               read from TMEM.
//   Both run their schedule warp-wide, so addresses and descriptors stay
//   warp-uniform, and one elected lane issues each TMA / tcgen05 instruction
//   (a lone-lane issuer pays register-to-uniform moves on every MMA and
//   cannot keep the tensor pipe fed).
//   warps 4-7   softmax of query tile 0; warps 8-11 softmax of query tile 1.
//               One thread per query row (TMEM lane): row max, exp2, row sum,
//               P packed to bf16 back into TMEM over S in two 64-key halves
//               (each half released to the MMA issuer on its own barrier, so the
//               first half's P V overlaps the second half's exponentials), O
//               rescale when needed.
// The two tiles ping-pong: while one tile's softmax runs, the tensor core
// computes the other tile's P V and next S.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
//
// The reference max used in the exponentials is raised only when a row's max
// grows by more than 2^8 (in base-2 units); otherwise the old one is kept.
// Any common reference leaves u / l unchanged (section 3.2: old numerator and
// denominator are scaled together), so the result stays exact; it only bounds
// p by 256, well inside fp32 and bf16 range.
#include <cuda_bf16.h>

#include <type_traits>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kRows = 128;    // query rows per tile = TMEM lanes
constexpr int kKeys = 128;    // keys per K/V block
constexpr int kTiles = 2;     // query tiles per CTA
constexpr int kThreads = 384;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

// kOwnStage: the output leaves through a staging buffer of its own (persistent grids,
// where the query buffers are refilled for the next unit while the output is written)
// instead of through the tile's query buffer.  Either way a warp stages 32 rows of D/2
// columns at a time.
template <int D, bool kOwnStage = false>
struct Layout {
    static constexpr int kBoxes = D / 64;              // 64-element (128-byte) swizzle boxes
    static constexpr int kTileBytes = kRows * D * 2;   // one Q, K or V tile
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTiles * kTileBytes;
    static constexpr int kV = kK + 2 * kTileBytes;
    static constexpr int kStage = kV + 2 * kTileBytes; // 8 warps x 32 rows x D/2 bf16
    static constexpr int kBar = kStage + (kOwnStage ? kTileBytes : 0);
    static constexpr int kSmem = kBar + 256 + 1024;    // barriers + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    __device__ static constexpr uint32_t col_s(int tq) { return 128u * tq; }
    __device__ static constexpr uint32_t col_o(int tq)
    {
        return 256u + static_cast<uint32_t>(D) * tq;
    }
};

// Barrier slots (8 bytes each) after the tiles.
enum : int {
    kBarQ = 0,
    kBarKFull = 1,   // +stage
    kBarKEmpty = 3,  // +stage
    kBarVFull = 5,   // +stage
    kBarVEmpty = 7,  // +stage
    kBarSFull = 9,   // +tile
    kBarPFull = 11,  // +2*tile +half: P columns of keys [0,64) and [64,128)
    kBarOFull = 15,  // +tile
    kBarDone = 17,
    kBarQ1 = 18,     // query tile 1 (tile 0 on kBarQ), so that tile 0's first S starts earlier
    kBarUnitFull = 19,   // +slot: dynamic grids, the producer published a unit
    kBarUnitEmpty = 21,  // +slot: every consumer warp has read it
    kBarQEmpty = 23,     // +tile: persistent grids, the unit's last Q K^T of the tile finished
    kBarCount = 25
};
constexpr int kUnitReaders = 1 + 8;   // the MMA warp and the eight softmax warps

struct Params {
    __nv_bfloat16* out;
    float* lse;
    int* trace;
    unsigned int* status;
    unsigned long long timeout_ns;
    int B, L, H, P, Ls, causal;
    int zigzag;      // shard r holds chunks r and 2P-1-r of 2P chunks (causal only)
    const int* cu_seqlens;   // packed sequences: starts of n_seqs sequences, then L
    int n_seqs;
    const int* schedule;     // packed sequences: units heaviest first (r * n_pair + pair), or null
    int group;       // query heads per key/value head
    int u_B, u_H, u_Ls;  // Ulysses head groups (kMode 3): batch, heads, shard rows of the sources
    int n_kt;        // K/V blocks per shard
    int n_pair;      // query-tile pairs per shard
    float scale_log2;
    long long out_elems, lse_elems;   // extents for the debug build's index checks
    int sched_elems;                  // entries of the schedule's forward order
    int* claim;      // dynamic grids: the work counter (zeroed before the launch)
    long long claim_index, claim_extent;   // its index in the schedule array, for the checks
    int n_units;     // work units of the whole call: B * H * P * n_pair
};

// Global position of local row i of shard `shard`.  Contiguous layout: shard r
// holds positions [r Ls, (r+1) Ls).  Zigzag layout ("序列并行与 Ring Attention",
// section 3.4: each rank holds an early and a late part so causal work is even):
// with 2P chunks of c = Ls/2 positions, shard r holds chunk r, then chunk 2P-1-r.
__device__ __forceinline__ int position(int shard, int i, int P, int Ls, int zig)
{
    if (!zig) return shard * Ls + i;
    const int c = Ls >> 1;
    return i < c ? shard * c + i : (2 * P - 1 - shard) * c + (i - c);
}

// Ring walk of one CTA: at step t = 0..P-1 the queries of shard r meet shard
// s = (r - t) mod P (section 3.3).  Of shard s only the key tiles whose first key
// position does not exceed the CTA's last query position are visited (all of
// them without causal masking): in the contiguous layout that is all of a past
// shard, a prefix of the diagonal one and none of a future one (section 3.4's
// whole-block skip); in the zigzag layout a prefix of each of the shard's two
// chunks.  Every role walks the same sequence.
struct RingWalk {
    int r, P, n_kt, Ls, zig, causal, maxq;
    int t, s, idx, cnt_a, cnt_b;
    __device__ __forceinline__ int prefix(int first_pos, int n) const
    {
        if (!causal) return n;
        if (maxq < first_pos) return 0;
        return min(n, (maxq - first_pos) / kKeys + 1);
    }
    __device__ __forceinline__ void enter()
    {
        s = r - t;
        if (s < 0) s += P;
        if (!zig) {
            cnt_a = prefix(s * Ls, n_kt);
            cnt_b = 0;
        } else {
            const int c = Ls >> 1, nh = n_kt >> 1;
            cnt_a = prefix(s * c, nh);
            cnt_b = prefix((2 * P - 1 - s) * c, nh);
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
    __device__ __forceinline__ void begin()
    {
        t = 0;
        enter();
        settle();
    }
    __device__ __forceinline__ void next()
    {
        ++idx;
        settle();
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
    // key tile within shard s, and the position of its first key
    __device__ __forceinline__ int kt() const { return idx < cnt_a ? idx : (n_kt >> 1) + (idx - cnt_a); }
    __device__ __forceinline__ int pos0() const { return position(s, kt() * kKeys, P, Ls, zig); }
};

// The contiguous layout's schedule in closed form (same sequence as RingWalk
// gives for it): step 0 is the own shard r (under causal masking only the tiles
// up to the diagonal), then shards r-1, r-2, ... (causal: down to 0; otherwise
// all of them, wrapping around).
struct ContigSched {
    int r, P, n_kt, Ls, n_first, n_blocks;
    int s, kt_, t;
    __device__ __forceinline__ void init(int r_, int P_, int n_kt_, int Ls_, int causal, int q_last)
    {
        r = r_;
        P = P_;
        n_kt = n_kt_;
        Ls = Ls_;
        if (causal) {
            n_first = min(n_kt, q_last / kKeys + 1);
            n_blocks = n_first + r * n_kt;
        } else {
            n_first = n_kt;
            n_blocks = P * n_kt;
        }
    }
    // block n, walked in order (at(n) must see n = 0, 1, 2, ...): the diagonal shard's
    // first n_first tiles, then whole shards r - 1, r - 2, ... mod P
    __device__ __forceinline__ void at(int n)
    {
        if (n == 0) {
            t = 0;
            s = r;
            kt_ = 0;
            return;
        }
        if (++kt_ == (t == 0 ? n_first : n_kt)) {
            kt_ = 0;
            ++t;
            s = s == 0 ? P - 1 : s - 1;
        }
    }
    __device__ __forceinline__ int kt() const { return kt_; }
    __device__ __forceinline__ bool first_of_shard() const { return kt_ == 0; }
    __device__ __forceinline__ int pos0() const { return s * Ls + kt_ * kKeys; }
};

// The zigzag layout's schedule, walked in order (at(n) must see n = 0, 1, 2, ...).
struct ZigzagSched {
    RingWalk w;
    int n_blocks, s, t;
    __device__ __forceinline__ void init(int r_, int P_, int n_kt_, int Ls_, int causal, int maxq)
    {
        w.r = r_;
        w.P = P_;
        w.n_kt = n_kt_;
        w.Ls = Ls_;
        w.zig = 1;
        w.causal = causal;
        w.maxq = maxq;
        n_blocks = w.total();
    }
    __device__ __forceinline__ void at(int n)
    {
        if (n == 0) w.begin();
        else w.next();
        s = w.s;
        t = w.t;
    }
    __device__ __forceinline__ int kt() const { return w.kt(); }
    __device__ __forceinline__ bool first_of_shard() const { return w.idx == 0; }
    __device__ __forceinline__ int pos0() const { return w.pos0(); }
};

// Packed sequences: sequence g covers positions [cu[g], cu[g+1]); a query sees
// only keys of its own sequence (and, causal, not after itself).  Returns the
// first and last visible key position of the query at `pos`.
__device__ __forceinline__ void seq_bounds(const int* cu, int n_seqs, int pos, int causal, int& lo,
                                           int& hi, unsigned int* status)
{
    int a = 0, b = n_seqs;                       // invariant: cu[a] <= pos < cu[b]
    while (b - a > 1) {
        const int mid = (a + b) >> 1;
        if (checked_ldg(cu, mid, n_seqs + 1, status) <= pos) a = mid;
        else b = mid;
    }
    lo = checked_ldg(cu, a, n_seqs + 1, status);
    hi = causal ? pos : checked_ldg(cu, a + 1, n_seqs + 1, status) - 1;
}

// Packed-sequence schedule: ring order as always; of shard s the key tiles that
// intersect the CTA's visible position range [lo, hi] (a contiguous run of tiles,
// possibly none).
struct VarlenSched {
    int r, P, n_kt, Ls, lo, hi;
    int n_blocks, s, t, idx, k_first, k_count;
    __device__ __forceinline__ void enter()
    {
        s = r - t;
        if (s < 0) s += P;
        const int base = s * Ls;
        const int a = max(lo, base), b = min(hi, base + Ls - 1);
        if (a > b) {
            k_first = 0;
            k_count = 0;
        } else {
            k_first = (a - base) / kKeys;
            k_count = (b - base) / kKeys - k_first + 1;
        }
        idx = 0;
    }
    __device__ __forceinline__ void init(int r_, int P_, int n_kt_, int Ls_, int lo_, int hi_)
    {
        r = r_;
        P = P_;
        n_kt = n_kt_;
        Ls = Ls_;
        lo = lo_;
        hi = hi_;
        n_blocks = 0;
        for (t = 0; t < P; ++t) {
            enter();
            n_blocks += k_count;
        }
    }
    __device__ __forceinline__ void at(int n)
    {
        if (n == 0) {
            t = 0;
            enter();
        } else {
            ++idx;
        }
        while (idx >= k_count && t < P) {
            ++t;
            if (t < P) enter();
        }
    }
    __device__ __forceinline__ int kt() const { return k_first + idx; }
    __device__ __forceinline__ bool first_of_shard() const { return idx == 0; }
    __device__ __forceinline__ int pos0() const { return s * Ls + kt() * kKeys; }
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// One work unit: two 128-row query tiles of one shard of one (batch, head), and the walk
// over the K/V blocks they meet.
template <int kMode>
struct Unit {
    int bh, b, h, hk;
    int r, pair;
    int bo, h_src, hk_src;       // indices in the source tensors (kMode 3)
    int q0_local, q0;            // first query row of the pair: within shard r, global
    int n_blocks;
    typename std::conditional<kMode == 1, ZigzagSched,
                              typename std::conditional<kMode == 2, VarlenSched,
                                                        ContigSched>::type>::type walk;

    // Unit g of the call's order: heaviest (shard, pair) first within each (batch, head),
    // two (batch, head) pairs interleaved (zigzag shards: by global position); packed
    // sequences take the schedule's order.
    __device__ __forceinline__ void setup(int g, const Params& p)
    {
        decode(g, p);
        int lo = 0, hi = 0;
        if constexpr (kMode == 2) pair_bounds(p, lo, hi);
        finish(p, lo, hi);
    }
    // (batch, head), shard and pair of unit g
    __device__ __forceinline__ void decode(int g, const Params& p)
    {
        const int units_per_bh = p.P * p.n_pair;
        int u;
        if constexpr (kMode == 2) unit_of_claim_varlen(g, p.B * p.H, units_per_bh, bh, u);
        else unit_of_block(g, p.B * p.H, units_per_bh, bh, u);
        r = p.P - 1 - u / p.n_pair;
        pair = p.n_pair - 1 - (u - (u / p.n_pair) * p.n_pair);
        if constexpr (kMode == 1) {
            // zigzag shards whose chunks hold whole pairs: descending global position (a
            // pair's work grows with its position, not its shard); other shapes keep the
            // order above
            const int per_chunk = p.n_kt >> 1;          // tiles per chunk
            if ((per_chunk & 1) == 0) {
                const int ppc = per_chunk >> 1;         // pairs per chunk
                const int gp = units_per_bh - 1 - u;    // position order of the pair
                const int chunk = gp / ppc, within = gp - chunk * ppc;
                r = chunk < p.P ? chunk : 2 * p.P - 1 - chunk;
                pair = (chunk < p.P ? 0 : ppc) + within;
            }
        }
        if constexpr (kMode == 2) {
            // packed sequences: work follows the offset inside a sequence, not the position;
            // a precomputed order (entries outside the unit range are ignored) puts the
            // heaviest units first
            if (p.schedule != nullptr) {
                const int x = checked_ldg(p.schedule, u, p.sched_elems, p.status);
                if (static_cast<unsigned>(x) < static_cast<unsigned>(units_per_bh)) {
                    r = x / p.n_pair;
                    pair = x - r * p.n_pair;
                }
            }
        }
    }
    // packed sequences: the positions the pair's queries see, from the first row's sequence
    // start to the last row's (causal) position or sequence end
    __device__ __forceinline__ void pair_bounds(const Params& p, int& lo, int& hi) const
    {
        const int ql = pair * (kTiles * kRows);
        const int last = min(p.Ls - 1, ql + kTiles * kRows - 1);
        int lo0, hi0, lo1, hi1;
        seq_bounds(p.cu_seqlens, p.n_seqs, r * p.Ls + ql, p.causal, lo0, hi0, p.status);
        seq_bounds(p.cu_seqlens, p.n_seqs, r * p.Ls + last, p.causal, lo1, hi1, p.status);
        lo = lo0;
        hi = hi1;
    }
    // everything else, from the decoded unit (lo, hi: packed sequences' pair bounds)
    __device__ __forceinline__ void finish(const Params& p, int lo, int hi)
    {
        b = bh / p.H;
        h = bh - b * p.H;
        hk = h / p.group;                       // key/value head of this query head
        bo = b;
        h_src = h;
        hk_src = hk;
        if constexpr (kMode == 3) {
            const int gg = b / p.u_B;
            bo = b - gg * p.u_B;
            h_src = gg * p.H + h;
            hk_src = h_src / p.group;
        }
        q0_local = pair * (kTiles * kRows);
        q0 = r * p.Ls + q0_local;
        const int last = min(p.Ls - 1, q0_local + kTiles * kRows - 1);
        if constexpr (kMode == 2) {
            walk.init(r, p.P, p.n_kt, p.Ls, lo, hi);
        } else if constexpr (kMode == 1) {
            // last query position of the pair (positions rise within each chunk, and the
            // late chunk lies after the early one)
            const int mid = min(p.Ls - 1, q0_local + kRows - 1);
            walk.init(r, p.P, p.n_kt, p.Ls, p.causal,
                      max(position(r, last, p.P, p.Ls, 1), position(r, mid, p.P, p.Ls, 1)));
        } else {
            walk.init(r, p.P, p.n_kt, p.Ls, p.causal, last);
            (void)lo;
            (void)hi;
        }
        n_blocks = walk.n_blocks;
    }
};

// kMode: 0 contiguous shards, 1 zigzag shards, 2 packed sequences (contiguous shards),
// 3 Ulysses head groups read from and written to the sequence-sharded buffers (the
// all-to-all of "序列并行与 Ring Attention" section 3.5 done by the tensor maps' addressing:
// batch b of the kernel is head group g = b / u_B of batch b % u_B, its head h is source
// head g*H + h, and position l sits in source shard l / u_Ls at row l % u_Ls).
//
// kPersist: how CTAs get their work units.
//   0  one CTA per unit: the grid lists the units and the block scheduler hands them to
//      SMs as SMs free up;
//   1  one CTA per SM, static: CTA c runs units c, c + G, c + 2G, ... of the G-CTA grid
//      (used when all units are equal: calls without causal masking);
//   2  one CTA per SM, dynamic: the producer warp claims each next unit from a counter in
//      global memory (packed sequences with a schedule: the counter sits in the caller's
//      schedule array and is zeroed before the launch) and hands it to the other warps
//      through a two-slot ring of unit indices in shared memory.
// A persistent CTA overlaps consecutive units: the producer loads the next unit's query
// tiles as soon as the current unit's last products of each tile have finished and its
// K/V blocks as ring stages free up; the issuer starts the next unit's first products
// while the softmax warps write the previous output, which leaves through a staging
// buffer of its own (the query buffers are already being refilled).  Barrier phases run
// on across units: blocks and units are counted from the CTA's start.  A unit with an
// empty walk (possible only with malformed sequence boundaries) writes 0 and -inf and
// touches no barrier.
template <int D, int kMode, int kPersist>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attn_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q,
                          const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const Params p)
{
    using Lay = Layout<D, kPersist != 0>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kBar + kBarCount * 8);
    int* abort_flag = reinterpret_cast<int*>(smem + Lay::kBar + kBarCount * 8 + 4);
    // dynamic grids: two ring slots of (unit, shard, pair, walk bounds lo and hi, number
    // of K/V blocks), everything the other warps need to run the unit without loads
    constexpr int kSlotInts = 6;
    volatile int* unit_slot = reinterpret_cast<volatile int*>(smem + Lay::kBar + kBarCount * 8 + 8);
    auto bar = [&](int i) -> uint32_t { return sbase + Lay::kBar + 8u * i; };
    static_assert(kBarCount * 8 + 8 + 2 * kSlotInts * 4 <= 256, "barrier area");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool kZig = kMode == 1;
    constexpr bool kVarlen = kMode == 2;

    // The i-th unit of this CTA, set up in V (returns -1: no more).  Dynamic grids: the
    // consumers' side of the ring; the producer publishes (publish_unit below).
    WaitCtx wc{abort_flag, p.status, p.timeout_ns};
    auto consume_unit = [&](int i, Unit<kMode>& V) -> int {
        if constexpr (kPersist != 2) {
            const long long g = blockIdx.x + static_cast<long long>(i) * gridDim.x;
            if (g >= p.n_units || (kPersist == 0 && i > 0)) return -1;
            V.setup(static_cast<int>(g), p);
            return static_cast<int>(g);
        }
        const int slot = i & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarUnitFull + slot), (i >> 1) & 1, wc)))
            return -1;
        volatile int* e = unit_slot + kSlotInts * slot;
        const int g = e[0];
        if (g >= 0) {
            int u;
            if constexpr (kMode == 2) unit_of_claim_varlen(g, p.B * p.H, p.P * p.n_pair, V.bh, u);
            else unit_of_block(g, p.B * p.H, p.P * p.n_pair, V.bh, u);
            V.r = e[1];
            V.pair = e[2];
            V.finish(p, e[3], e[4]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarUnitEmpty + slot));
        return g;
    };

    Unit<kMode> first;
    const int g_first = kPersist == 2 ? -1 : consume_unit(0, first);

    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQ), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarKFull + i), 1);
            mbar_init(bar(kBarKEmpty + i), 1);
            mbar_init(bar(kBarVFull + i), 1);
            mbar_init(bar(kBarVEmpty + i), 1);
            mbar_init(bar(kBarSFull + i), 1);
            mbar_init(bar(kBarPFull + 2 * i), kRows);
            mbar_init(bar(kBarPFull + 2 * i + 1), kRows);
            mbar_init(bar(kBarOFull + i), 1);
            mbar_init(bar(kBarUnitFull + i), 1);
            mbar_init(bar(kBarUnitEmpty + i), kUnitReaders);
            mbar_init(bar(kBarQEmpty + i), 1);
        }
        mbar_init(bar(kBarDone), 1);
        mbar_init(bar(kBarQ1), 1);
        *abort_flag = 0;
        fence_mbar_init();
        if constexpr (kPersist == 0) {
            // Start the loads the first products need (Q0 and K0 for tile 0's first S,
            // then Q1) before the TMEM allocation and the block-wide barrier: every CTA of
            // a wave starts by loading at once, so the sooner they are queued the better.
            // The producer loop below issues V0 and everything after it.
            const Unit<kMode>& U = first;
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            const uint64_t once = l2_policy_evict_first();
            auto load_q = [&](int tq, uint32_t full) {
                mbar_arrive_expect_tx(bar(full), Lay::kTileBytes);
                for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                    const uint32_t dst = sbase + Lay::kQ + tq * Lay::kTileBytes + bx * 16384;
                    const int row = U.q0 + tq * kRows;
                    if constexpr (kMode == 3)
                        tma_load_5d(dst, &tmap_q, bar(full), bx * 64, U.h_src, row % p.u_Ls, U.bo,
                                    row / p.u_Ls, once);
                    else
                        tma_load_4d(dst, &tmap_q, bar(full), bx * 64, U.h, row, U.b, once);
                }
            };
            load_q(0, kBarQ);
            if (U.n_blocks > 0) {
                Unit<kMode> W = U;
                W.walk.at(0);
                const int row = W.walk.s * p.Ls + W.walk.kt() * kKeys;
                const uint64_t keep = l2_policy_evict_last();
                mbar_arrive_expect_tx(bar(kBarKFull + 0), Lay::kTileBytes);
                for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                    const uint32_t dst = sbase + Lay::kK + bx * 16384;
                    if constexpr (kMode == 3)
                        tma_load_5d(dst, &tmap_k, bar(kBarKFull + 0), bx * 64, U.hk_src,
                                    row % p.u_Ls, U.bo, row / p.u_Ls, keep);
                    else
                        tma_load_4d(dst, &tmap_k, bar(kBarKFull + 0), bx * 64, U.hk, row, U.b, keep);
                }
            }
            load_q(1, kBarQ1);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), Lay::kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // The whole warp runs the loop (warp-uniform values); one elected lane issues.
        const bool leader = elect_one();
        if (leader) {
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        const uint64_t keep = l2_policy_evict_last();    // K/V: read by every tile pair of the head
        const uint64_t once = l2_policy_evict_first();
        // Dynamic grids: claim the i-th unit, set it up, and publish it with its number of
        // K/V blocks to the other warps (-1: done)
        auto publish_unit = [&](int i, Unit<kMode>& U) -> int {
            const int slot = i & 1;
            int g = -1;
            if (leader && in_bounds(p.claim_index, 1, p.claim_extent, p.status))
                g = atomicAdd(p.claim, 1);
            g = __shfl_sync(0xffffffffu, g, __ffs(__ballot_sync(0xffffffffu, leader)) - 1);
            if (g < 0 || g >= p.n_units) g = -1;
            int lo = 0, hi = 0;
            if (g >= 0) {
                U.decode(g, p);
                if constexpr (kMode == 2) U.pair_bounds(p, lo, hi);
                U.finish(p, lo, hi);
            }
            if (i >= 2 &&
                !__all_sync(0xffffffffu, mbar_wait(bar(kBarUnitEmpty + slot), ((i - 2) >> 1) & 1, wc)))
                return -1;
            if (leader) {
                volatile int* e = unit_slot + kSlotInts * slot;
                e[0] = g;
                e[1] = U.r;
                e[2] = U.pair;
                e[3] = lo;
                e[4] = hi;
                e[5] = g >= 0 ? U.n_blocks : 0;
                mbar_arrive(bar(kBarUnitFull + slot));
            }
            __syncwarp();
            return g;
        };
        uint32_t N = 0;       // K/V blocks loaded by this CTA so far
        int qn = 0;           // units with a non-empty walk so far (query barrier phases)
        int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};   // last block loaded per stage
        bool ok = true;
        for (int i = 0; ok; ++i) {
            Unit<kMode> U;
            int g;
            if (kPersist == 2) g = publish_unit(i, U);
            else if (i == 0) {
                g = g_first;
                U = first;
            } else {
                g = consume_unit(i, U);
            }
            if (g < 0) break;
            if (U.n_blocks == 0) continue;
            // the shard's last query pair meets every shard the shard visits, in either layout
            const bool tracing = p.trace != nullptr && U.bh == 0 && U.pair == p.n_pair - 1;
            if (tracing && leader)
                for (int t = 0; t < p.P; ++t)
                    if (in_bounds(U.r * p.P + t, 1, p.P * p.P, p.status)) p.trace[U.r * p.P + t] = -1;
            if constexpr (kPersist != 0) {
                // query tiles: reloaded once the previous unit's last Q K^T of the tile (the
                // last reader of its buffer) has finished, a block before its last P V
                for (int tq = 0; tq < kTiles; ++tq) {
                    if (qn > 0 &&
                        !(ok = __all_sync(0xffffffffu,
                                          mbar_wait(bar(kBarQEmpty + tq), (qn - 1) & 1, wc))))
                        break;
                    if (leader) {
                        const uint32_t full = tq == 0 ? bar(kBarQ) : bar(kBarQ1);
                        mbar_arrive_expect_tx(full, Lay::kTileBytes);
                        for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                            const uint32_t dst = sbase + Lay::kQ + tq * Lay::kTileBytes + bx * 16384;
                            const int row = U.q0 + tq * kRows;
                            if constexpr (kMode == 3)
                                tma_load_5d(dst, &tmap_q, full, bx * 64, U.h_src, row % p.u_Ls, U.bo,
                                            row / p.u_Ls, once);
                            else
                                tma_load_4d(dst, &tmap_q, full, bx * 64, U.h, row, U.b, once);
                        }
                    }
                    __syncwarp();
                }
                if (!ok) break;
            }
            for (int n = 0; n < U.n_blocks; ++n) {
                U.walk.at(n);
                if (tracing && U.walk.first_of_shard() && leader &&
                    in_bounds(U.r * p.P + U.walk.t, 1, p.P * p.P, p.status))
                    p.trace[U.r * p.P + U.walk.t] = U.walk.s;
                const uint32_t Nn = N + n;
                const int st = Nn & 1;
                const uint32_t ph = (Nn >> 1) & 1;
                const int row = U.walk.s * p.Ls + U.walk.kt() * kKeys;   // physical row of the tile
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarKEmpty + st), ph ^ 1, wc)))) break;
                // (classic grids: thread 0 issued the first K block before the block-wide barrier)
                if (leader && (kPersist != 0 || n > 0)) {
                    mbar_arrive_expect_tx(bar(kBarKFull + st), Lay::kTileBytes);
                    for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                        const uint32_t dst = sbase + Lay::kK + st * Lay::kTileBytes + bx * 16384;
                        if constexpr (kMode == 3)
                            tma_load_5d(dst, &tmap_k, bar(kBarKFull + st), bx * 64, U.hk_src,
                                        row % p.u_Ls, U.bo, row / p.u_Ls, keep);
                        else
                            tma_load_4d(dst, &tmap_k, bar(kBarKFull + st), bx * 64, U.hk, row, U.b,
                                        keep);
                    }
                }
                last_k[st] = static_cast<int>(Nn);
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarVEmpty + st), ph ^ 1, wc)))) break;
                if (leader) {
                    mbar_arrive_expect_tx(bar(kBarVFull + st), Lay::kTileBytes);
                    for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                        const uint32_t dst = sbase + Lay::kV + st * Lay::kTileBytes + bx * 16384;
                        if constexpr (kMode == 3)
                            tma_load_5d(dst, &tmap_v, bar(kBarVFull + st), bx * 64, U.hk_src,
                                        row % p.u_Ls, U.bo, row / p.u_Ls, keep);
                        else
                            tma_load_4d(dst, &tmap_v, bar(kBarVFull + st), bx * 64, U.hk, row, U.b,
                                        keep);
                    }
                }
                last_v[st] = static_cast<int>(Nn);
            }
            N += U.n_blocks;
            ++qn;
        }
        // let this CTA's own copies land before anyone leaves
        if (qn > 0) {
            mbar_wait_drain(bar(kBarQ), (qn - 1) & 1, wc);
            mbar_wait_drain(bar(kBarQ1), (qn - 1) & 1, wc);
        } else if constexpr (kPersist == 0) {
            // classic grid, empty walk: thread 0 still loaded both query tiles
            mbar_wait_drain(bar(kBarQ), 0, wc);
            mbar_wait_drain(bar(kBarQ1), 0, wc);
        }
        if constexpr (kPersist == 0) {
            if (first.n_blocks > 0 && last_k[0] < 0) mbar_wait_drain(bar(kBarKFull + 0), 0, wc);
        }
        for (int st = 0; st < 2; ++st) {
            if (last_k[st] >= 0) mbar_wait_drain(bar(kBarKFull + st), (last_k[st] >> 1) & 1, wc);
            if (last_v[st] >= 0) mbar_wait_drain(bar(kBarVFull + st), (last_v[st] >> 1) & 1, wc);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        // The whole warp runs the loop so that descriptors stay warp-uniform; one
        // elected lane issues the tcgen05 instructions.
        const bool leader = elect_one();
        constexpr uint32_t kIdescQK = idesc_bf16_f32(kRows, kKeys, false);
        constexpr uint32_t kIdescPV = idesc_bf16_f32(kRows, D, true);
        constexpr uint64_t kTileU = Lay::kTileBytes >> 4;   // descriptor address unit: 16 bytes
        // S_tq = Q_tq K^T: both operands K-major (head dim contiguous), 128-byte swizzled
        // rows of 64 elements, 8-row atoms 1024 bytes apart; 16-element K steps advance
        // 32 bytes inside a swizzle row, then jump to the next 64-wide box (16 KiB).
        const uint64_t dq = sdesc_sw128(sbase + Lay::kQ, 16, 1024);
        const uint64_t dk = sdesc_sw128(sbase + Lay::kK, 16, 1024);
        // V is the MN-major B operand (head dim contiguous): 8 key rows of 128 bytes per
        // swizzle atom (stride 1024), the second 64-wide box 16 KiB further (leading
        // offset); 16-key steps advance 2 KiB.
        const uint64_t dv = sdesc_sw128(sbase + Lay::kV, 16384, 1024);
        auto issue_qk = [&](int tq, int st) {
            const uint32_t d_t = tmem + Lay::col_s(tq);
            const uint64_t a0 = dq + tq * kTileU, b0 = dk + st * kTileU;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint64_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                mma_ss(d_t, a0 + off, b0 + off, kIdescQK, k > 0 ? 1u : 0u);
            }
        };
        // O_tq += P_tq V for keys [64 half, 64 half + 64): P (bf16 pairs) sits in TMEM
        // over S_tq, 32 columns per half.
        auto issue_pv = [&](int tq, int st, int half, bool acc) {
            const uint32_t d_t = tmem + Lay::col_o(tq);
            const uint32_t pa = tmem + Lay::col_s(tq) + 32 * half;
            const uint64_t b0 = dv + st * kTileU + ((half * 64 * 128) >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_ts(d_t, pa + k * 8, b0 + ((k * 2048) >> 4), kIdescPV, (acc || k > 0) ? 1u : 0u);
        };
        auto wait_all = [&](int idx, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar(idx), parity, wc));
        };

        uint32_t N = 0;       // K/V blocks consumed by this CTA so far
        int qn = 0;           // units with a non-empty walk so far
        bool ok = true;
        for (int i = 0; ok; ++i) {
            int n_blocks;
            if (i == 0 && kPersist != 2) {
                if (g_first < 0) break;
                n_blocks = first.n_blocks;
            } else {
                Unit<kMode> U;
                if (consume_unit(i, U) < 0) break;
                n_blocks = U.n_blocks;
            }
            // an empty walk (possible only with malformed sequence boundaries) issues nothing
            if (n_blocks == 0) continue;
            const uint32_t qpar = qn & 1;
            const int st0 = N & 1;
            const uint32_t ph0 = (N >> 1) & 1;
            ok = wait_all(kBarQ, qpar) && wait_all(kBarKFull + st0, ph0);
            if (!ok) break;
            // persistent grids: after the unit's last Q K^T of a tile its query buffer may be
            // refilled for the next unit
            const bool last_qk0 = kPersist != 0 && n_blocks == 1;
            tc_fence_after();
            if (leader) {
                issue_qk(0, st0);
                tc_commit(bar(kBarSFull + 0));
                if (last_qk0) tc_commit(bar(kBarQEmpty + 0));
            }
            __syncwarp();
            if (!(ok = wait_all(kBarQ1, qpar))) break;
            tc_fence_after();
            if (leader) {
                issue_qk(1, st0);
                tc_commit(bar(kBarSFull + 1));
                tc_commit(bar(kBarKEmpty + st0));
                if (last_qk0) tc_commit(bar(kBarQEmpty + 1));
            }
            __syncwarp();
            for (int n = 0; ok && n < n_blocks; ++n) {
                const uint32_t Nn = N + n;
                const int st = Nn & 1;
                const uint32_t ph = (Nn >> 1) & 1;
                const bool more = n + 1 < n_blocks;
                const int st1 = (Nn + 1) & 1;
                const uint32_t ph1 = ((Nn + 1) >> 1) & 1;
                // Each wait between MMA batches costs the tensor pipe ~100 cycles even when the
                // barrier is already complete, so barriers that gate the same batch are checked
                // together: V and the first P half of tile 0, then its second P half and the
                // next K block.
                if (!(ok = __all_sync(0xffffffffu, mbar_wait2(bar(kBarVFull + st), ph,
                                                              bar(kBarPFull + 0), Nn & 1, wc))))
                    break;
                tc_fence_after();
                if (leader) issue_pv(0, st, 0, n > 0);
                __syncwarp();
                ok = more ? mbar_wait2(bar(kBarPFull + 1), Nn & 1, bar(kBarKFull + st1), ph1, wc)
                          : mbar_wait(bar(kBarPFull + 1), Nn & 1, wc);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                const bool last_qk = kPersist != 0 && n + 2 == n_blocks;
                tc_fence_after();
                if (leader) {
                    issue_pv(0, st, 1, true);
                    if (!more) tc_commit(bar(kBarOFull + 0));
                    if (more) {
                        issue_qk(0, st1);
                        tc_commit(bar(kBarSFull + 0));
                        if (last_qk) tc_commit(bar(kBarQEmpty + 0));
                    }
                }
                __syncwarp();
                if (!(ok = wait_all(kBarPFull + 2, Nn & 1))) break;
                tc_fence_after();
                if (leader) issue_pv(1, st, 0, n > 0);
                __syncwarp();
                if (!(ok = wait_all(kBarPFull + 3, Nn & 1))) break;
                tc_fence_after();
                if (leader) {
                    issue_pv(1, st, 1, true);
                    tc_commit(bar(kBarVEmpty + st));
                    if (!more) tc_commit(bar(kBarOFull + 1));
                    if (more) {
                        issue_qk(1, st1);
                        tc_commit(bar(kBarSFull + 1));
                        tc_commit(bar(kBarKEmpty + st1));
                        if (last_qk) tc_commit(bar(kBarQEmpty + 1));
                    }
                }
                __syncwarp();
            }
            N += n_blocks;
            ++qn;
        }
        // every MMA this CTA issued has finished before TMEM is released
        if (leader) tc_commit(bar(kBarDone));
        __syncwarp();
        mbar_wait_drain(bar(kBarDone), 0, wc);
        __syncwarp();
    } else if (warp >= 4) {
        // ----------------------------------------------------------- softmax
        const int tq = (warp - 4) >> 2;
        const int quarter = warp & 3;                 // TMEM lane quarter of this warp
        const int row = quarter * 32 + lane;          // row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + Lay::col_s(tq);
        const uint32_t tO = tmem + lane_off + Lay::col_o(tq);
        const float sl2 = p.scale_log2;
        uint32_t N = 0;       // K/V blocks of the units this CTA has run
        int qn = 0;           // units with a non-empty walk so far
        bool ok = true;
        // the i-th unit with this thread's row: global position and (packed sequences) the
        // visible key positions [seq_lo, seq_hi]
        struct Row {
            int row_local, row_pos, seq_lo, seq_hi;
        };
        auto row_of = [&](const Unit<kMode>& V) {
            Row w;
            w.row_local = V.q0_local + tq * kRows + row;   // within shard r
            w.row_pos = position(V.r, w.row_local, p.P, p.Ls, kZig ? 1 : 0);
            w.seq_lo = 0;
            w.seq_hi = 0;
            if constexpr (kVarlen) {
                if (w.row_local < p.Ls)
                    seq_bounds(p.cu_seqlens, p.n_seqs, w.row_pos, p.causal, w.seq_lo, w.seq_hi,
                               p.status);
                else w.seq_hi = -1;
            }
            return w;
        };
        auto get_unit = [&](int i, Unit<kMode>& V) -> int {
            if (i == 0 && kPersist != 2) {
                V = first;
                return g_first;
            }
            return consume_unit(i, V);
        };
        Unit<kMode> U;
        int g = get_unit(0, U);
        Row R = row_of(U);
        for (int i = 0; ok && g >= 0; ++i) {
            const int n_blocks = U.n_blocks;
            const int row_local = R.row_local, row_pos = R.row_pos;
            const int seq_lo = R.seq_lo, seq_hi = R.seq_hi;

            float m = -INFINITY;   // running max of scaled scores, base-2 units
            float l = 0.f;         // running denominator, relative to m
            for (int n = 0; n < n_blocks; ++n) {
                U.walk.at(n);
                const uint32_t Nn = N + n;
                ok = mbar_wait(bar(kBarSFull + tq), Nn & 1, wc);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();

                uint32_t sraw[128];
                tmem_ld128(tS, sraw);
                float sv[128];
#pragma unroll
                for (int c = 0; c < 128; ++c) sv[c] = u2f(sraw[c]);

                // visible columns: inside the shard, and under causal masking key
                // position <= query position (global positions)
                int lim = min(kKeys - 1, p.Ls - U.walk.kt() * kKeys - 1);
                int lo_lim = 0;
                if constexpr (kVarlen) {
                    lim = min(lim, seq_hi - U.walk.pos0());
                    lo_lim = seq_lo - U.walk.pos0();
                } else if (p.causal) {
                    lim = min(lim, row_pos - U.walk.pos0());
                }
                if (lim < kKeys - 1 || lo_lim > 0) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) sv[c] = (c > lim || c < lo_lim) ? -INFINITY : sv[c];
                }

                float mx0 = fmaxf(sv[0], sv[1]), mx1 = fmaxf(sv[2], sv[3]);
                float mx2 = fmaxf(sv[4], sv[5]), mx3 = fmaxf(sv[6], sv[7]);
#pragma unroll
                for (int c = 8; c < 128; c += 8) {
                    mx0 = fmax3(mx0, sv[c], sv[c + 1]);
                    mx1 = fmax3(mx1, sv[c + 2], sv[c + 3]);
                    mx2 = fmax3(mx2, sv[c + 4], sv[c + 5]);
                    mx3 = fmax3(mx3, sv[c + 6], sv[c + 7]);
                }
                const float m_blk = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
                const float m_new = fmaxf(m, m_blk);
                const bool raise = m_new > m + kRescaleThreshold;   // always on the first finite block
                const float m_ref = raise ? m_new : m;
                const float alpha = raise ? ex2(m - m_ref) : 1.f;    // ex2(-inf) = 0
                const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;

                // p = 2^(s * scale*log2(e) - m_ref) for column pairs (packed fp32 FMA and
                // adds), packed to bf16 pairs and written over S as the A operand of P V,
                // in two halves of 64 keys so that the first half's P V overlaps the
                // second half's exponentials.
                const uint64_t scale2 = f2pack(sl2, sl2), negm2 = f2pack(neg_m, neg_m);
                uint64_t sum_a = 0, sum_b = 0;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i2 = 0; i2 < 32; ++i2) {
                        const int c = 64 * half + 2 * i2;
                        float x0, x1;
                        f2unpack(ffma2(f2pack(sv[c], sv[c + 1]), scale2, negm2), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        if (i2 & 1) sum_b = fadd2(sum_b, f2pack(p0, p1));
                        else sum_a = fadd2(sum_a, f2pack(p0, p1));
                        pk[i2] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(tS + 32 * half, pk);
                    // O was last written by P V of the previous block, which finished
                    // before this block's S (same issuing thread, in order); it is rescaled
                    // before this block's first P V can start accumulating into it.
                    if (half == 0 && n > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tO + 32 * c, o);
#pragma unroll
                            for (int i2 = 0; i2 < 32; ++i2) o[i2] = f2u(u2f(o[i2]) * alpha);
                            tmem_st32(tO + 32 * c, o);
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(bar(kBarPFull + 2 * tq + half));
                }
                float sa0, sa1;
                f2unpack(fadd2(sum_a, sum_b), sa0, sa1);
                l = l * alpha + (sa0 + sa1);
                m = m_ref;
            }
            if (!ok) break;

            // what the epilogue needs of this unit: index of (row, head) among the output's
            // rows of D elements for this warp's first row (the warp's 32 rows lie in one tile,
            // so `ostride` apart)
            const bool empty = n_blocks == 0;
            const bool valid = row_local < p.Ls;
            const int x0 = U.q0_local + tq * kRows + quarter * 32;   // within shard r
            const int g0 = U.r * p.Ls + x0;
            size_t orow0 = (static_cast<size_t>(U.b) * p.L + g0) * p.H + U.h;
            size_t ostride = p.H;
            if constexpr (kMode == 3) {
                const int rs = g0 / p.u_Ls;
                orow0 = (static_cast<size_t>(rs * p.u_B + U.bo) * p.u_Ls + (g0 - rs * p.u_Ls)) *
                            p.u_H + U.h_src;
                ostride = p.u_H;
            }

            // persistent grids: the next unit and this thread's row of it are set up while
            // this unit's last P V runs (the packed sequences' binary search included)
            int g_next = -1;
            if constexpr (kPersist != 0) {
                g_next = get_unit(i + 1, U);
                if (g_next >= 0) R = row_of(U);
            }

            // An empty walk leaves O unwritten: its rows saw no key and get 0 and -inf.
            // Classic grids stage the output in the tile's query buffer, whose load must then
            // have landed; persistent grids stage it in a buffer of their own.
            if (!empty) ok = mbar_wait(bar(kBarOFull + tq), qn & 1, wc);
            else if constexpr (kPersist == 0) ok = mbar_wait(bar(tq == 0 ? kBarQ : kBarQ1), 0, wc);
            if (!(ok = __all_sync(0xffffffffu, ok))) break;
            if (!empty) tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;        // a row that saw no key: 0
            // The rows go out through a 32-row staging slice of the warp (the tile's query
            // buffer, free once O is final -- the tile's last Q K^T finished before its last
            // P V -- or the persistent grids' own buffer), half of the columns at a time, so
            // that every global store covers whole row halves instead of one 16-byte piece
            // of 32 rows.  A thread writes its row's 16-byte chunk c at slot c ^ (row mod
            // kChunks): conflict-free for both the row-wise writes and the chunk-wise reads.
            constexpr int kHalfCols = D / 2;
            constexpr int kChunks = kHalfCols / 8;             // 16-byte chunks per staged row
            constexpr int kRowsPerStore = 32 / kChunks;        // rows one warp store covers
            uint8_t* stage = kPersist != 0
                                 ? smem + Lay::kStage + (warp - 4) * 32 * (2 * kHalfCols)
                                 : smem + Lay::kQ + tq * Lay::kTileBytes + quarter * 32 * (2 * D);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int c = 0; c < kHalfCols / 32; ++c) {
                    uint32_t o[32] = {};
                    if (!empty) tmem_ld32(tO + hh * kHalfCols + 32 * c, o);
                    uint32_t pk[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2)
                        pk[i2] = pack_bf16x2(u2f(o[2 * i2]) * inv_l, u2f(o[2 * i2 + 1]) * inv_l);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int slot = (4 * c + j) ^ (lane & (kChunks - 1));
                        *reinterpret_cast<uint4*>(stage + lane * (2 * kHalfCols) + slot * 16) =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
                __syncwarp();
                {
                    const int sub = lane / kChunks, cc = lane % kChunks;
#pragma unroll
                    for (int k = 0; k < 32 / kRowsPerStore; ++k) {
                        const int rr = k * kRowsPerStore + sub;         // row within the warp's 32
                        const uint4 val = *reinterpret_cast<const uint4*>(
                            stage + rr * (2 * kHalfCols) + ((cc ^ (rr & (kChunks - 1))) * 16));
                        const long long idx =
                            static_cast<long long>(orow0 + rr * ostride) * D + hh * kHalfCols + cc * 8;
                        if (x0 + rr < p.Ls && in_bounds(idx, 8, p.out_elems, p.status))
                            *reinterpret_cast<uint4*>(p.out + idx) = val;
                    }
                }
                __syncwarp();
            }
            if (valid && p.lse != nullptr &&
                in_bounds(static_cast<long long>(orow0 + lane * ostride), 1, p.lse_elems, p.status))
                p.lse[orow0 + lane * ostride] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
            if (!empty) {
                // this warp's reads of O are complete before the next unit's first P V
                // (gated on its P, which this warp writes later) overwrites it
                N += n_blocks;
                ++qn;
            }
            g = g_next;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

// ------------------------------------------------------------------ pair of SMs --
//
// ring_attn_bf16_pair_kernel: the same computation with the products issued for a pair of
// SMs (tcgen05.mma.cta_group::2, M = 256).  A cluster of two CTAs takes four consecutive
// 128-row query tiles of one shard of one (batch, head): CTA rank c holds tiles 2c and
// 2c + 1 (its "tile 0" and "tile 1"), and the pair's products for tile slot a cover the
// two CTAs' tile a together.  Each CTA loads half of every K/V block: keys [64 c, 64 c + 64)
// of K (the B operand of Q K^T, split along N = keys) and head-dim columns [64 c, 64 c + 64)
// of V (the B operand of P V, split along N = D), so a product reads 6 KiB of shared memory
// per SM per 16-deep step instead of 8 (Q K^T) and 2 instead of 4 (P V) -- the tensor
// core's shared-memory read pipe, which holds single-SM products to ~71 cycles, stops
// being the limit (a stream of these products issues at the nominal 64 cycles).
// The even CTA's MMA warp issues everything; its barriers count both CTAs' TMA bytes and
// both CTAs' P (one arrival per softmax warp, the odd CTA's through its cluster address),
// and every commit is multicast to the same barrier of both CTAs.  S and O of a CTA's rows
// live in its own TMEM, so the softmax warps work exactly as in the single-SM kernel.
// Head dim 128 only.
template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    ring_attn_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmap_q,
                               const __grid_constant__ CUtensorMap tmap_k,
                               const __grid_constant__ CUtensorMap tmap_v, const Params p)
{
    constexpr int D = 128;
    constexpr int kTileBytes = kRows * D * 2;          // one Q tile, 32 KiB
    constexpr int kHalfBytes = kTileBytes / 2;         // one CTA's half of a K or V block
    constexpr int kQOff = 0;
    constexpr int kKOff = kQOff + kTiles * kTileBytes;
    constexpr int kVOff = kKOff + 2 * kHalfBytes;
    constexpr int kBarOff = kVOff + 2 * kHalfBytes;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kBarCount * 8);
    int* abort_flag = reinterpret_cast<int*>(smem + kBarOff + kBarCount * 8 + 4);
    auto bar = [&](int i) -> uint32_t { return sbase + kBarOff + 8u * i; };
    const uint32_t rank = cluster_ctarank();
    const bool lead = rank == 0;
    // the even CTA's copy of a barrier (cluster address)
    auto lead_bar = [&](int i) -> uint32_t { return mapa_shared(bar(i), 0); };
    constexpr uint16_t kBoth = 3;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work unit: a quad of query tiles, heaviest first, two (batch, head) pairs
    // interleaved.  Contiguous shards: last shard, last quad first.  Zigzag shards whose
    // chunks hold whole quads: descending global position (chunk 2P - 1, the late half of
    // shard 0, first), since there a quad's work grows with its position, not its shard;
    // other zigzag shapes keep the contiguous order.
    const int n_quad = (p.n_pair + 1) / 2;
    const int units_per_bh = p.P * n_quad;
    int bh, u;
    unit_of_block(static_cast<int>(blockIdx.x >> 1), p.B * p.H, units_per_bh, bh, u);
    int r = p.P - 1 - u / n_quad;
    int quad = n_quad - 1 - (u - (u / n_quad) * n_quad);
    if constexpr (kMode == 1) {
        const int per_chunk = p.n_kt >> 1;              // tiles per chunk
        if ((per_chunk & 3) == 0) {
            const int qpc = per_chunk >> 2;             // quads per chunk
            const int g = units_per_bh - 1 - u;         // position order of the quad
            const int chunk = g / qpc, within = g - chunk * qpc;
            r = chunk < p.P ? chunk : 2 * p.P - 1 - chunk;
            quad = (chunk < p.P ? 0 : qpc) + within;
        }
    }
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int hk = h / p.group;
    int bo = b, h_src = h, hk_src = hk;
    if constexpr (kMode == 3) {
        const int g = b / p.u_B;
        bo = b - g * p.u_B;
        h_src = g * p.H + h;
        hk_src = h_src / p.group;
    }
    const int quad0 = quad * (4 * kRows);                  // first query row of the quad
    const int q0_local = quad0 + static_cast<int>(rank) * (kTiles * kRows);   // this CTA's
    // the quad's walk: contiguous shards see up to the quad's last row; zigzag shards up to
    // the largest position among the quad's four tiles (their last rows: positions rise
    // within each chunk, and the late chunk lies after the early one), walked in order
    typename std::conditional<kMode == 1, ZigzagSched, ContigSched>::type walk;
    if constexpr (kMode == 1) {
        int maxq = 0;
        for (int k = 0; k < 4; ++k)
            maxq = max(maxq, position(r, min(p.Ls - 1, quad0 + k * kRows + kRows - 1), p.P, p.Ls, 1));
        walk.init(r, p.P, p.n_kt, p.Ls, p.causal, maxq);
    } else {
        walk.init(r, p.P, p.n_kt, p.Ls, p.causal, min(p.Ls - 1, quad0 + 4 * kRows - 1));
    }
    const int n_blocks = walk.n_blocks;

    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQ), 1);
        mbar_init(bar(kBarQ1), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarKFull + i), 1);
            mbar_init(bar(kBarKEmpty + i), 1);
            mbar_init(bar(kBarVFull + i), 1);
            mbar_init(bar(kBarVEmpty + i), 1);
            mbar_init(bar(kBarSFull + i), 1);
            // one arrival per softmax warp of the tile, in both CTAs
            mbar_init(bar(kBarPFull + 2 * i), 2 * (kRows / 32));
            mbar_init(bar(kBarPFull + 2 * i + 1), 2 * (kRows / 32));
            mbar_init(bar(kBarOFull + i), 1);
        }
        mbar_init(bar(kBarDone), 1);
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
        // ------------------------------------------------------ TMA producer (both CTAs)
        const bool leader = elect_one();
        if (leader) {
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        const uint64_t keep = l2_policy_evict_last();
        const uint64_t once = l2_policy_evict_first();
        const bool tracing = p.trace != nullptr && lead && bh == 0 && quad == n_quad - 1;
        if (tracing && leader)
            for (int t = 0; t < p.P; ++t)
                if (in_bounds(r * p.P + t, 1, p.P * p.P, p.status)) p.trace[r * p.P + t] = -1;
        if (leader) {
            // this CTA's two query tiles, counted on the even CTA's barriers
            for (int tq = 0; tq < kTiles; ++tq) {
                const int full = tq == 0 ? kBarQ : kBarQ1;
                if (lead) mbar_arrive_expect_tx(bar(full), 2 * kTileBytes);
                for (int bx = 0; bx < 2; ++bx) {
                    const uint32_t dst = sbase + kQOff + tq * kTileBytes + bx * 16384;
                    const int row = r * p.Ls + q0_local + tq * kRows;
                    if constexpr (kMode == 3)
                        tma_load_5d_pair(dst, &tmap_q, lead_bar(full), bx * 64, h_src, row % p.u_Ls,
                                         bo, row / p.u_Ls, once);
                    else
                        tma_load_4d_pair(dst, &tmap_q, lead_bar(full), bx * 64, h, row, b, once);
                }
            }
        }
        int last[2] = {-1, -1};
        for (int n = 0; n < n_blocks; ++n) {
            walk.at(n);
            if (tracing && walk.first_of_shard() && leader &&
                in_bounds(r * p.P + walk.t, 1, p.P * p.P, p.status))
                p.trace[r * p.P + walk.t] = walk.s;
            const int st = n & 1;
            const uint32_t ph = (n >> 1) & 1;
            const int row = walk.s * p.Ls + walk.kt() * kKeys;   // first key of the block
            // K: keys [64 rank, 64 rank + 64) of the block, both 64-column boxes
            if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarKEmpty + st), ph ^ 1, wc))) break;
            if (leader) {
                if (lead) mbar_arrive_expect_tx(bar(kBarKFull + st), 2 * kHalfBytes);
                const int krow = row + 64 * static_cast<int>(rank);
                for (int bx = 0; bx < 2; ++bx) {
                    const uint32_t dst = sbase + kKOff + st * kHalfBytes + bx * 8192;
                    if constexpr (kMode == 3)
                        tma_load_5d_pair(dst, &tmap_k, lead_bar(kBarKFull + st), bx * 64, hk_src,
                                         krow % p.u_Ls, bo, krow / p.u_Ls, keep);
                    else
                        tma_load_4d_pair(dst, &tmap_k, lead_bar(kBarKFull + st), bx * 64, hk, krow, b,
                                         keep);
                }
            }
            // V: head-dim columns [64 rank, 64 rank + 64) of the block's 128 keys (one box)
            if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarVEmpty + st), ph ^ 1, wc))) break;
            if (leader) {
                if (lead) mbar_arrive_expect_tx(bar(kBarVFull + st), 2 * kHalfBytes);
                const uint32_t dst = sbase + kVOff + st * kHalfBytes;
                if constexpr (kMode == 3)
                    tma_load_5d_pair(dst, &tmap_v, lead_bar(kBarVFull + st), 64 * rank, hk_src,
                                     row % p.u_Ls, bo, row / p.u_Ls, keep);
                else
                    tma_load_4d_pair(dst, &tmap_v, lead_bar(kBarVFull + st), 64 * rank, hk, row, b,
                                     keep);
            }
            last[st] = n;
        }
        // the even CTA's barriers count both CTAs' copies: it waits for all of them to land
        // (the odd CTA leaves only after the cluster-wide barrier that follows)
        if (lead) {
            mbar_wait_drain(bar(kBarQ), 0, wc);
            mbar_wait_drain(bar(kBarQ1), 0, wc);
            for (int st = 0; st < 2; ++st)
                if (last[st] >= 0) {
                    mbar_wait_drain(bar(kBarKFull + st), (last[st] >> 1) & 1, wc);
                    mbar_wait_drain(bar(kBarVFull + st), (last[st] >> 1) & 1, wc);
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer (even CTA)
        if (lead) {
            const bool leader = elect_one();
            constexpr uint32_t kIdescQK = idesc_bf16_f32(2 * kRows, kKeys, false);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(2 * kRows, D, true);
            constexpr uint64_t kTileU = kTileBytes >> 4;
            constexpr uint64_t kHalfU = kHalfBytes >> 4;
            // Q (A, K-major): 128 rows per 64-column box (16 KiB); K half (B, K-major): 64
            // keys per box (8 KiB); V half (B, MN-major): one 64-column box of 128 keys, 8
            // keys per 1024-byte swizzle atom, 16-key steps 2 KiB apart
            const uint64_t dq = sdesc_sw128(sbase + kQOff, 16, 1024);
            const uint64_t dk = sdesc_sw128(sbase + kKOff, 16, 1024);
            const uint64_t dv = sdesc_sw128(sbase + kVOff, 16384, 1024);
            auto issue_qk = [&](int tq, int st) {
                const uint32_t d_t = tmem + Layout<D>::col_s(tq);
                const uint64_t a0 = dq + tq * kTileU, b0 = dk + st * kHalfU;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t oa = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                    const uint64_t ob = ((k >> 2) * 8192 + (k & 3) * 32) >> 4;
                    mma_ss_pair(d_t, a0 + oa, b0 + ob, kIdescQK, k > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int tq, int st, int half, bool acc) {
                const uint32_t d_t = tmem + Layout<D>::col_o(tq);
                const uint32_t pa = tmem + Layout<D>::col_s(tq) + 32 * half;
                const uint64_t b0 = dv + st * kHalfU + ((half * 64 * 128) >> 4);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ts_pair(d_t, pa + k * 8, b0 + ((k * 2048) >> 4), kIdescPV,
                                (acc || k > 0) ? 1u : 0u);
            };
            auto wait_all = [&](int idx, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar(idx), parity, wc));
            };
            bool ok = n_blocks > 0 && wait_all(kBarQ, 0) && wait_all(kBarKFull + 0, 0);
            if (ok) {
                tc_fence_after();
                if (leader) {
                    issue_qk(0, 0);
                    tc_commit_pair(bar(kBarSFull + 0), kBoth);
                }
                __syncwarp();
            }
            if (ok && (ok = wait_all(kBarQ1, 0))) {
                tc_fence_after();
                if (leader) {
                    issue_qk(1, 0);
                    tc_commit_pair(bar(kBarSFull + 1), kBoth);
                    tc_commit_pair(bar(kBarKEmpty + 0), kBoth);
                }
                __syncwarp();
            }
            for (int n = 0; ok && n < n_blocks; ++n) {
                const int st = n & 1;
                const uint32_t ph = (n >> 1) & 1;
                const bool more = n + 1 < n_blocks;
                const int st1 = (n + 1) & 1;
                const uint32_t ph1 = ((n + 1) >> 1) & 1;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait2(bar(kBarPFull + 0), n & 1,
                                                              bar(kBarVFull + st), ph, wc))))
                    break;
                tc_fence_after();
                if (leader) issue_pv(0, st, 0, n > 0);
                __syncwarp();
                ok = more ? mbar_wait2(bar(kBarPFull + 1), n & 1, bar(kBarKFull + st1), ph1, wc)
                          : mbar_wait(bar(kBarPFull + 1), n & 1, wc);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                tc_fence_after();
                if (leader) {
                    issue_pv(0, st, 1, true);
                    if (!more) tc_commit_pair(bar(kBarOFull + 0), kBoth);
                    if (more) {
                        issue_qk(0, st1);
                        tc_commit_pair(bar(kBarSFull + 0), kBoth);
                    }
                }
                __syncwarp();
                if (!(ok = wait_all(kBarPFull + 2, n & 1))) break;
                tc_fence_after();
                if (leader) issue_pv(1, st, 0, n > 0);
                __syncwarp();
                if (!(ok = wait_all(kBarPFull + 3, n & 1))) break;
                tc_fence_after();
                if (leader) {
                    issue_pv(1, st, 1, true);
                    tc_commit_pair(bar(kBarVEmpty + st), kBoth);
                    if (!more) tc_commit_pair(bar(kBarOFull + 1), kBoth);
                    if (more) {
                        issue_qk(1, st1);
                        tc_commit_pair(bar(kBarSFull + 1), kBoth);
                        tc_commit_pair(bar(kBarKEmpty + st1), kBoth);
                    }
                }
                __syncwarp();
            }
            // every product the pair issued has finished before either CTA frees TMEM: the
            // even CTA's issuer waits for them here; the odd CTA's issuer goes to the cluster
            // barrier below without spinning through the kernel (the even one arrives there
            // only after this wait) and then sees the same commit's arrival on its own barrier
            if (leader) tc_commit_pair(bar(kBarDone), kBoth);
            __syncwarp();
            mbar_wait_drain(bar(kBarDone), 0, wc);
            __syncwarp();
        }
    } else if (warp >= 4) {
        // ----------------------------------------------------------- softmax (both CTAs)
        const int tq = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + Layout<D>::col_s(tq);
        const uint32_t tO = tmem + lane_off + Layout<D>::col_o(tq);
        const int row_local = q0_local + tq * kRows + row;   // within shard r
        const int row_pos = position(r, row_local, p.P, p.Ls, kMode == 1 ? 1 : 0);
        const float sl2 = p.scale_log2;
        // P ready: one arrival per warp of either CTA, after the warp's TMEM stores
        const uint32_t pfull0 = lead_bar(kBarPFull + 2 * tq);      // half 1: the next word

        float m = -INFINITY;
        float l = 0.f;
        bool ok = true;
        for (int n = 0; n < n_blocks; ++n) {
            walk.at(n);
            ok = mbar_wait(bar(kBarSFull + tq), n & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();

            uint32_t sraw[128];
            tmem_ld128(tS, sraw);
            float sv[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) sv[c] = u2f(sraw[c]);
            int lim = min(kKeys - 1, p.Ls - walk.kt() * kKeys - 1);
            if (p.causal) lim = min(lim, row_pos - walk.pos0());
            if (lim < kKeys - 1) {
#pragma unroll
                for (int c = 0; c < 128; ++c) sv[c] = c > lim ? -INFINITY : sv[c];
            }
            float mx0 = fmaxf(sv[0], sv[1]), mx1 = fmaxf(sv[2], sv[3]);
            float mx2 = fmaxf(sv[4], sv[5]), mx3 = fmaxf(sv[6], sv[7]);
#pragma unroll
            for (int c = 8; c < 128; c += 8) {
                mx0 = fmax3(mx0, sv[c], sv[c + 1]);
                mx1 = fmax3(mx1, sv[c + 2], sv[c + 3]);
                mx2 = fmax3(mx2, sv[c + 4], sv[c + 5]);
                mx3 = fmax3(mx3, sv[c + 6], sv[c + 7]);
            }
            const float m_blk = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
            const float m_new = fmaxf(m, m_blk);
            const bool raise = m_new > m + kRescaleThreshold;
            const float m_ref = raise ? m_new : m;
            const float alpha = raise ? ex2(m - m_ref) : 1.f;
            const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
            const uint64_t scale2 = f2pack(sl2, sl2), negm2 = f2pack(neg_m, neg_m);
            uint64_t sum_a = 0, sum_b = 0;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int i2 = 0; i2 < 32; ++i2) {
                    const int c = 64 * half + 2 * i2;
                    float x0, x1;
                    f2unpack(ffma2(f2pack(sv[c], sv[c + 1]), scale2, negm2), x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    if (i2 & 1) sum_b = fadd2(sum_b, f2pack(p0, p1));
                    else sum_a = fadd2(sum_a, f2pack(p0, p1));
                    pk[i2] = pack_bf16x2(p0, p1);
                }
                tmem_st32(tS + 32 * half, pk);
                if (half == 0 && n > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32 * c, o);
#pragma unroll
                        for (int i2 = 0; i2 < 32; ++i2) o[i2] = f2u(u2f(o[i2]) * alpha);
                        tmem_st32(tO + 32 * c, o);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(pfull0 + 8 * half);
            }
            float sa0, sa1;
            f2unpack(fadd2(sum_a, sum_b), sa0, sa1);
            l = l * alpha + (sa0 + sa1);
            m = m_ref;
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarOFull + tq), 0, wc));
        if (ok) {
            tc_fence_after();
            const bool valid = row_local < p.Ls;
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const int x0 = q0_local + tq * kRows + quarter * 32;
            const int g0 = r * p.Ls + x0;
            size_t orow0 = (static_cast<size_t>(b) * p.L + g0) * p.H + h;
            size_t ostride = p.H;
            if constexpr (kMode == 3) {
                const int rs = g0 / p.u_Ls;
                orow0 = (static_cast<size_t>(rs * p.u_B + bo) * p.u_Ls + (g0 - rs * p.u_Ls)) * p.u_H +
                        h_src;
                ostride = p.u_H;
            }
            // staged through the warp's 32-row slice of this CTA's query tile (free: the
            // tile's last Q K^T finished before its last P V)
            constexpr int kHalfCols = D / 2;
            constexpr int kChunks = kHalfCols / 8;
            constexpr int kRowsPerStore = 32 / kChunks;
            uint8_t* stage = smem + kQOff + tq * kTileBytes + quarter * 32 * (2 * D);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int c = 0; c < kHalfCols / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + hh * kHalfCols + 32 * c, o);
                    uint32_t pk[16];
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2)
                        pk[i2] = pack_bf16x2(u2f(o[2 * i2]) * inv_l, u2f(o[2 * i2 + 1]) * inv_l);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int slot = (4 * c + j) ^ (lane & (kChunks - 1));
                        *reinterpret_cast<uint4*>(stage + lane * (2 * kHalfCols) + slot * 16) =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
                __syncwarp();
                {
                    const int sub = lane / kChunks, cc = lane % kChunks;
#pragma unroll
                    for (int k = 0; k < 32 / kRowsPerStore; ++k) {
                        const int rr = k * kRowsPerStore + sub;
                        const uint4 val = *reinterpret_cast<const uint4*>(
                            stage + rr * (2 * kHalfCols) + ((cc ^ (rr & (kChunks - 1))) * 16));
                        const long long idx =
                            static_cast<long long>(orow0 + rr * ostride) * D + hh * kHalfCols + cc * 8;
                        if (x0 + rr < p.Ls && in_bounds(idx, 8, p.out_elems, p.status))
                            *reinterpret_cast<uint4*>(p.out + idx) = val;
                    }
                }
                __syncwarp();
            }
            if (valid && p.lse != nullptr &&
                in_bounds(static_cast<long long>(orow0 + lane * ostride), 1, p.lse_elems, p.status))
                p.lse[orow0 + lane * ostride] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        }
    }

    // neither CTA frees TMEM or leaves while the other may still read its shared memory
    // or signal its barriers
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        if (!lead) mbar_wait_drain(bar(kBarDone), 0, wc);
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

template <int kMode>
cudaError_t launch_pair(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv)
{
    constexpr int D = 128;
    constexpr int kSmem = kTiles * kRows * D * 2 + 4 * (kRows * D) + 256 + 1024;
    static std::atomic<int> configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = smem_limit_once(configured, dev, ring_attn_bf16_pair_kernel<kMode>, kSmem);
    if (e != cudaSuccess) return e;
    Params p{};
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.lse = a.lse;
    p.trace = a.trace;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.B = a.B;
    p.L = a.L;
    p.H = a.H;
    p.P = a.P;
    p.Ls = a.L / a.P;
    p.causal = a.causal;
    p.zigzag = a.zigzag;
    p.group = a.H / a.Hkv;
    p.u_B = a.u_B;
    p.u_H = a.u_H;
    p.u_Ls = a.u_P > 0 ? a.L / a.u_P : 0;
    p.n_kt = (p.Ls + kKeys - 1) / kKeys;
    p.n_pair = (p.n_kt + kTiles - 1) / kTiles;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    p.out_elems = static_cast<long long>(a.B) * a.L * a.H * D;
    p.lse_elems = static_cast<long long>(a.B) * a.L * a.H;
    const long long quads = static_cast<long long>(a.B) * a.H * a.P * ((p.n_pair + 1) / 2);
    if (quads <= 0 || 2 * quads > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    p.n_units = static_cast<int>(quads);
    ring_attn_bf16_pair_kernel<kMode>
        <<<static_cast<unsigned>(2 * quads), kThreads, kSmem, a.stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

template <int D, int kMode, int kPersist>
cudaError_t launch_d(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv)
{
    using Lay = Layout<D, kPersist != 0>;
    static std::atomic<int> configured[kMaxDevices];  // shared-memory limit set, per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = smem_limit_once(configured, dev, ring_attn_bf16_kernel<D, kMode, kPersist>, Lay::kSmem);
    if (e != cudaSuccess) return e;
    Params p;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.lse = a.lse;
    p.trace = a.trace;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.B = a.B;
    p.L = a.L;
    p.H = a.H;
    p.P = a.P;
    p.Ls = a.L / a.P;
    p.causal = a.causal;
    p.zigzag = a.zigzag;
    p.cu_seqlens = a.cu_seqlens;
    p.n_seqs = a.n_seqs;
    p.schedule = a.schedule != nullptr ? a.schedule + varlen_sched_layout(a.L, a.P).fwd : nullptr;
    p.group = a.H / a.Hkv;
    p.u_B = a.u_B;
    p.u_H = a.u_H;
    p.u_Ls = a.u_P > 0 ? a.L / a.u_P : 0;
    p.n_kt = (p.Ls + kKeys - 1) / kKeys;
    p.n_pair = (p.n_kt + kTiles - 1) / kTiles;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    // the kernel's B and H count head-group batches and heads; the element count of out
    // and lse is the same in the Ulysses view
    p.out_elems = static_cast<long long>(a.B) * a.L * a.H * D;
    p.lse_elems = static_cast<long long>(a.B) * a.L * a.H;
    p.sched_elems = static_cast<int>(a.P * p.n_pair);
    p.claim = nullptr;
    p.claim_index = 0;
    p.claim_extent = 0;
    const long long units = static_cast<long long>(a.B) * a.H * a.P * p.n_pair;
    if (units <= 0 || units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    p.n_units = static_cast<int>(units);
    long long grid = units;
    if constexpr (kPersist != 0) {
        int sms = 148;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (grid > sms) grid = sms;
    }
    if constexpr (kPersist == 2) {
        // the work counter at the end of the caller's schedule array, zeroed in stream order
        const VarlenSchedLayout lay = varlen_sched_layout(a.L, a.P);
        p.claim_index = lay.counters;
        p.claim_extent = lay.total;
        p.claim = const_cast<int*>(a.schedule) + lay.counters;
        e = cudaMemsetAsync(p.claim, 0, sizeof(int), a.stream);
        if (e != cudaSuccess) return e;
    }
    ring_attn_bf16_kernel<D, kMode, kPersist>
        <<<static_cast<unsigned>(grid), kThreads, Lay::kSmem, a.stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

template <int D, int kMode>
cudaError_t launch_mode(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv)
{
    // persistent grids where they pay: calls whose units are all equal (no causal
    // masking) run a static round-robin; packed sequences with a schedule claim units
    // dynamically through the schedule array's counter; everything else (causal
    // contiguous or zigzag shards, whose heaviest-first unit order the block scheduler
    // balances) keeps one CTA per unit
    if constexpr (kMode == 2) {
        if (a.schedule != nullptr) return launch_d<D, kMode, 2>(a, tq, tk, tv);
    } else if constexpr (kMode == 0 || kMode == 3) {
        if (!a.causal) return launch_d<D, kMode, 1>(a, tq, tk, tv);
    }
    return launch_d<D, kMode, 0>(a, tq, tk, tv);
}

}  // namespace

bool attn_bf16_pair_applies(const AttnArgs& a)
{
    // Head dim 128, contiguous or zigzag shards or Ulysses head groups, and key walks of
    // at least 64 blocks: a pair halves each SM's K/V staging and operand reads, which
    // pays on long walks (3-4 % faster at 32k-128k keys, equal on causal 32k; 3 % at the
    // power cap, where the lighter traffic leaves the clock higher), while the pair's
    // fixed costs (cluster barriers, paired TMEM allocation, the lock-step of two CTAs)
    // made 4096-key walks about 3 % slower than the single-SM kernel.
    return a.D == 128 && a.cu_seqlens == nullptr && a.L >= 8192;
}

cudaError_t launch_attn_bf16(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                             const CUtensorMap& tv)
{
    if (attn_bf16_pair_applies(a)) {
        if (a.u_P > 0) return launch_pair<3>(a, tq, tk, tv);
        return a.zigzag ? launch_pair<1>(a, tq, tk, tv) : launch_pair<0>(a, tq, tk, tv);
    }
    if (a.u_P > 0) {
        if (a.D == 64) return launch_mode<64, 3>(a, tq, tk, tv);
        if (a.D == 128) return launch_mode<128, 3>(a, tq, tk, tv);
    } else if (a.cu_seqlens != nullptr) {
        if (a.D == 64) return launch_mode<64, 2>(a, tq, tk, tv);
        if (a.D == 128) return launch_mode<128, 2>(a, tq, tk, tv);
    } else if (a.zigzag) {
        if (a.D == 64) return launch_mode<64, 1>(a, tq, tk, tv);
        if (a.D == 128) return launch_mode<128, 1>(a, tq, tk, tv);
    } else {
        if (a.D == 64) return launch_mode<64, 0>(a, tq, tk, tv);
        if (a.D == 128) return launch_mode<128, 0>(a, tq, tk, tv);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ra
