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
// shards in the forward's order.  No atomics: results are deterministic.
//
// Kernels (256 threads: warp 0 TMA producer, warp 1 MMA issuer, warps 4-7 one
// thread per TMEM lane for the elementwise step; warp-uniform schedules with one
// elected lane issuing):
//   bwd_rowdot_kernel   Dvec = rowsum(dO o O), fp32 workspace [B, L, H]
//   bwd_dkdv_kernel<D>  TMEM: S^T [0,128), dP^T [128,256), dV, dK (D columns each)
//       S^T = K Q^T, dP^T = V dO^T (SS); P^T, dS^T (bf16) written over them;
//       dV += P^T dO, dK += dS^T Q (A from TMEM, B = dO / Q as MN-major SMEM).
//   bwd_dq_kernel<D>    TMEM: S [0,128), dP [128,256), dQ (D columns)
//       S = Q K^T, dP = dO V^T (SS); dS (bf16) written over S; dQ += dS K.
#include <cuda_bf16.h>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kRows = 128;     // rows per tile (TMEM lanes), both queries and keys
constexpr int kThreads = 256;
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
    int n_t;                 // 128-row tiles per shard
    float scale_log2;        // log2(e) / sqrt(D)
    float scale;             // 1 / sqrt(D)
};

// ------------------------------------------------------------------ row dot --

// Dvec[row] = sum_d dO[row, d] * O[row, d] for every (b, l, h) row; a group of
// D/8 lanes takes one row, one 16-byte vector each.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_rowdot_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                      float* __restrict__ dvec, long long rows)
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
        if (row < rows) {
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
        if (row < rows && sub == 0) dvec[row] = acc;
    }
}

// ------------------------------------------------------------------ dK, dV --

enum : int {
    kKVFull = 0,
    kQFull = 1,      // +stage: Q, dO tiles (TMA) and the stats (32 producer lanes)
    kQEmpty = 3,     // +stage
    kKVSFull = 5,    // S^T, dP^T ready
    kKVPFull = 6,    // P^T, dS^T written
    kKVOFull = 7,    // dK, dV final
    kKVDone = 8,
    kKVBars = 9
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q,
                    const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_do, const BwdParams p)
{
    using Lay = BwdLayout<D>;
    constexpr int T = Lay::kTileBytes;
    constexpr int kK = 0, kV = T, kQ = 2 * T, kDO = 4 * T, kStats = 6 * T;   // stats: 2 x 1 KiB
    constexpr int kBar = kStats + 2048;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBar + kKVBars * 8);
    int* abort_flag = reinterpret_cast<int*>(smem + kBar + kKVBars * 8 + 4);
    auto bar = [&](int i) -> uint32_t { return sbase + kBar + 8u * i; };
    auto stats_lse2 = [&](int st) { return reinterpret_cast<float*>(smem + kStats + st * 1024); };
    auto stats_dvec = [&](int st) { return reinterpret_cast<float*>(smem + kStats + st * 1024 + 512); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // unit: (b, h) outer; inside, heaviest key tile first (low shard, low tile)
    const int units_per_bh = p.P * p.n_t;
    const int bh = blockIdx.x / units_per_bh;
    const int u = blockIdx.x - bh * units_per_bh;
    const int s = u / p.n_t;          // shard owning these keys
    const int kt = u - s * p.n_t;     // key tile within the shard
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int key0 = s * p.Ls + kt * kRows;
    // ring schedule from the owner's side: query shard r = (s + t) mod P at step t;
    // step 0 is the own shard (causal: query tiles from the diagonal on)
    const int q_begin = p.causal ? kt : 0;
    const int n_first = p.n_t - q_begin;
    const int n_blocks = n_first + (p.causal ? (p.P - 1 - s) : (p.P - 1)) * p.n_t;
    auto block = [&](int n, int& r, int& qt) {
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
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(kKVFull), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kQFull + i), 1 + 32);
            mbar_init(bar(kQEmpty + i), 1);
        }
        mbar_init(bar(kKVSFull), 1);
        mbar_init(bar(kKVPFull), kRows);
        mbar_init(bar(kKVOFull), 1);
        mbar_init(bar(kKVDone), 1);
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
    const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------ producer
        const bool leader = elect_one();
        const uint64_t keep = l2_policy_evict_last();
        if (leader) {
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_do);
            mbar_arrive_expect_tx(bar(kKVFull), 2 * T);
            for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                tma_load_4d(sbase + kK + bx * 16384, &tmap_k, bar(kKVFull), bx * 64, h, key0, b, keep);
                tma_load_4d(sbase + kV + bx * 16384, &tmap_v, bar(kKVFull), bx * 64, h, key0, b, keep);
            }
        }
        int last[2] = {-1, -1};
        for (int n = 0; n < n_blocks; ++n) {
            int r, qt;
            block(n, r, qt);
            const int st = n & 1;
            const uint32_t ph = (n >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(kQEmpty + st), ph ^ 1, wc))) break;
            const int qrow = r * p.Ls + qt * kRows;
            if (leader) {
                mbar_arrive_expect_tx(bar(kQFull + st), 2 * T);
                for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                    tma_load_4d(sbase + kQ + st * T + bx * 16384, &tmap_q, bar(kQFull + st), bx * 64,
                                h, qrow, b, keep);
                    tma_load_4d(sbase + kDO + st * T + bx * 16384, &tmap_do, bar(kQFull + st), bx * 64,
                                h, qrow, b, keep);
                }
            }
            // per-query statistics of this tile: lse in base-2 units, Dvec
            float* l2 = stats_lse2(st);
            float* dvs = stats_dvec(st);
            for (int c = lane; c < kRows; c += 32) {
                const int q_local = qt * kRows + c;
                const bool valid = q_local < p.Ls;
                const size_t idx = (static_cast<size_t>(b) * p.L + qrow + c) * p.H + h;
                l2[c] = valid ? p.lse[idx] * kLog2e : 0.f;
                dvs[c] = valid ? p.dvec[idx] : 0.f;
            }
            mbar_arrive(bar(kQFull + st));
            last[st] = n;
        }
        mbar_wait_drain(bar(kKVFull), 0, wc);
        for (int st = 0; st < 2; ++st)
            if (last[st] >= 0) mbar_wait_drain(bar(kQFull + st), (last[st] >> 1) & 1, wc);
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
        auto ts = [&](uint32_t dcol, uint32_t acol, uint64_t b0, bool acc) {
#pragma unroll
            for (int k = 0; k < kRows / 16; ++k)
                mma_ts(tmem + dcol, tmem + acol + k * 8, b0 + ((k * 2048) >> 4), kIdescAcc,
                       (acc || k > 0) ? 1u : 0u);
        };
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(kKVFull), 0, wc));
        for (int n = 0; ok && n < n_blocks; ++n) {
            const int st = n & 1;
            const uint32_t ph = (n >> 1) & 1;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kQFull + st), ph, wc)))) break;
            tc_fence_after();
            if (leader) {
                ss(0, dK_A, dQ_B + st * Lay::kTileU);       // S^T = K Q^T
                ss(128, dV_A, dDO_B + st * Lay::kTileU);    // dP^T = V dO^T
                tc_commit(bar(kKVSFull));
            }
            __syncwarp();
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kKVPFull), n & 1, wc)))) break;
            tc_fence_after();
            if (leader) {
                ts(256, 0, dDO_MN + st * Lay::kTileU, n > 0);          // dV += P^T dO
                ts(256 + D, 128, dQ_MN + st * Lay::kTileU, n > 0);     // dK += dS^T Q
                tc_commit(bar(kQEmpty + st));
                if (n + 1 == n_blocks) tc_commit(bar(kKVOFull));
            }
            __syncwarp();
        }
        if (leader) tc_commit(bar(kKVDone));
        __syncwarp();
        mbar_wait_drain(bar(kKVDone), 0, wc);
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------ elementwise
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;              // key row of the tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off;              // S^T, then P^T
        const uint32_t tP = tmem + lane_off + 128;        // dP^T, then dS^T
        const int key_local = kt * kRows + row;           // within shard s
        const bool key_valid = key_local < p.Ls;
        const float sl2 = p.scale_log2;
        bool ok = true;
        for (int n = 0; n < n_blocks; ++n) {
            int r, qt;
            block(n, r, qt);
            const int st = n & 1;
            ok = mbar_wait(bar(kKVSFull), n & 1, wc);
            ok = ok && mbar_wait(bar(kQFull + st), (n >> 1) & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // visible query columns [lo, hi] of this tile for this key row
            const int hi = min(kRows - 1, p.Ls - qt * kRows - 1);
            int lo = 0;
            if (p.causal && r == s) lo = max(0, key_local - qt * kRows);
            if (!key_valid) lo = kRows;
            const float* l2 = stats_lse2(st);
            const float* dvs = stats_dvec(st);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t sr[64], dr[64];
                tmem_ld64(tS + 64 * half, sr);
                tmem_ld64(tP + 64 * half, dr);
                uint32_t pk_p[32], pk_ds[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = 64 * half + 4 * i;
                    const float4 lse4 = *reinterpret_cast<const float4*>(l2 + c);
                    const float4 dv4 = *reinterpret_cast<const float4*>(dvs + c);
                    const float la[4] = {lse4.x, lse4.y, lse4.z, lse4.w};
                    const float da[4] = {dv4.x, dv4.y, dv4.z, dv4.w};
                    float pv[4], dsv[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int cc = c + j;
                        const bool vis = cc >= lo && cc <= hi;
                        const float pr = vis ? ex2(fmaf(u2f(sr[4 * i + j]), sl2, -la[j])) : 0.f;
                        pv[j] = pr;
                        dsv[j] = pr * (u2f(dr[4 * i + j]) - da[j]);
                    }
                    pk_p[2 * i] = pack_bf16x2(pv[0], pv[1]);
                    pk_p[2 * i + 1] = pack_bf16x2(pv[2], pv[3]);
                    pk_ds[2 * i] = pack_bf16x2(dsv[0], dsv[1]);
                    pk_ds[2 * i + 1] = pack_bf16x2(dsv[2], dsv[3]);
                }
                tmem_st32(tS + 32 * half, pk_p);
                tmem_st32(tP + 32 * half, pk_ds);
            }
            tc_fence_before();
            mbar_arrive(bar(kKVPFull));
        }
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kKVOFull), 0, wc));
        }
        if (ok) {
            tc_fence_after();
            const size_t base = ((static_cast<size_t>(b) * p.L + key0 + row) * p.H + h) * D;
#pragma unroll
            for (int which = 0; which < 2; ++which) {       // 0: dV, 1: dK
                const uint32_t tA = tmem + lane_off + 256 + which * D;
                const float mul = which ? p.scale : 1.f;
                __nv_bfloat16* dst = (which ? p.dk : p.dv) + base;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tA + 32 * c, o);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(u2f(o[2 * i]) * mul, u2f(o[2 * i + 1]) * mul);
                    if (key_valid) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
            }
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
    kDKFull = 1,     // +stage
    kDKEmpty = 3,    // +stage
    kDVFull = 5,     // +stage
    kDVEmpty = 7,    // +stage
    kDSFull = 9,     // S, dP ready
    kDDSFull = 10,   // dS written
    kDOFull = 11,    // dQ final
    kDDone = 12,
    kDBars = 13
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_do, const BwdParams p)
{
    using Lay = BwdLayout<D>;
    constexpr int T = Lay::kTileBytes;
    constexpr int kQ = 0, kDO = T, kK = 2 * T, kV = 4 * T, kBar = 6 * T;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBar + kDBars * 8);
    int* abort_flag = reinterpret_cast<int*>(smem + kBar + kDBars * 8 + 4);
    auto bar = [&](int i) -> uint32_t { return sbase + kBar + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // unit: (b, h) outer; inside, heaviest query tile first (last shard, last tile)
    const int units_per_bh = p.P * p.n_t;
    const int bh = blockIdx.x / units_per_bh;
    const int u = blockIdx.x - bh * units_per_bh;
    const int r = p.P - 1 - u / p.n_t;
    const int qt = p.n_t - 1 - (u - (u / p.n_t) * p.n_t);
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int q_local0 = qt * kRows;
    const int q0 = r * p.Ls + q_local0;
    // the forward's ring order: K/V shard (r - t) mod P at step t, future shards skipped
    int n_first, n_blocks;
    if (p.causal) {
        const int q_last = min(p.Ls - 1, q_local0 + kRows - 1);
        n_first = min(p.n_t, q_last / kRows + 1);
        n_blocks = n_first + r * p.n_t;
    } else {
        n_first = p.n_t;
        n_blocks = p.P * p.n_t;
    }
    auto block = [&](int n, int& s, int& kt) {
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
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(kQDFull), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kDKFull + i), 1);
            mbar_init(bar(kDKEmpty + i), 1);
            mbar_init(bar(kDVFull + i), 1);
            mbar_init(bar(kDVEmpty + i), 1);
        }
        mbar_init(bar(kDSFull), 1);
        mbar_init(bar(kDDSFull), kRows);
        mbar_init(bar(kDOFull), 1);
        mbar_init(bar(kDDone), 1);
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
    const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------ producer
        const bool leader = elect_one();
        const uint64_t keep = l2_policy_evict_last();
        const uint64_t once = l2_policy_evict_first();
        if (leader) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            mbar_arrive_expect_tx(bar(kQDFull), 2 * T);
            for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                tma_load_4d(sbase + kQ + bx * 16384, &tmap_q, bar(kQDFull), bx * 64, h, q0, b, once);
                tma_load_4d(sbase + kDO + bx * 16384, &tmap_do, bar(kQDFull), bx * 64, h, q0, b, once);
            }
        }
        int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
        for (int n = 0; n < n_blocks; ++n) {
            int s, kt;
            block(n, s, kt);
            const int st = n & 1;
            const uint32_t ph = (n >> 1) & 1;
            const int row = s * p.Ls + kt * kRows;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(kDKEmpty + st), ph ^ 1, wc))) break;
            if (leader) {
                mbar_arrive_expect_tx(bar(kDKFull + st), T);
                for (int bx = 0; bx < Lay::kBoxes; ++bx)
                    tma_load_4d(sbase + kK + st * T + bx * 16384, &tmap_k, bar(kDKFull + st), bx * 64,
                                h, row, b, keep);
            }
            last_k[st] = n;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(kDVEmpty + st), ph ^ 1, wc))) break;
            if (leader) {
                mbar_arrive_expect_tx(bar(kDVFull + st), T);
                for (int bx = 0; bx < Lay::kBoxes; ++bx)
                    tma_load_4d(sbase + kV + st * T + bx * 16384, &tmap_v, bar(kDVFull + st), bx * 64,
                                h, row, b, keep);
            }
            last_v[st] = n;
        }
        mbar_wait_drain(bar(kQDFull), 0, wc);
        for (int st = 0; st < 2; ++st) {
            if (last_k[st] >= 0) mbar_wait_drain(bar(kDKFull + st), (last_k[st] >> 1) & 1, wc);
            if (last_v[st] >= 0) mbar_wait_drain(bar(kDVFull + st), (last_v[st] >> 1) & 1, wc);
        }
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
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(kQDFull), 0, wc));
        for (int n = 0; ok && n < n_blocks; ++n) {
            const int st = n & 1;
            const uint32_t ph = (n >> 1) & 1;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kDKFull + st), ph, wc) &&
                                                   mbar_wait(bar(kDVFull + st), ph, wc))))
                break;
            tc_fence_after();
            if (leader) {
                ss(0, dQ_A, dK_B + st * Lay::kTileU);      // S = Q K^T
                ss(128, dDO_A, dV_B + st * Lay::kTileU);   // dP = dO V^T
                tc_commit(bar(kDSFull));
                tc_commit(bar(kDVEmpty + st));
            }
            __syncwarp();
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(kDDSFull), n & 1, wc)))) break;
            tc_fence_after();
            if (leader) {
                const uint64_t b0 = dK_MN + st * Lay::kTileU;
#pragma unroll
                for (int k = 0; k < kRows / 16; ++k)             // dQ += dS K
                    mma_ts(tmem + 256, tmem + k * 8, b0 + ((k * 2048) >> 4), kIdescAcc,
                           (n > 0 || k > 0) ? 1u : 0u);
                tc_commit(bar(kDKEmpty + st));
                if (n + 1 == n_blocks) tc_commit(bar(kDOFull));
            }
            __syncwarp();
        }
        if (leader) tc_commit(bar(kDDone));
        __syncwarp();
        mbar_wait_drain(bar(kDDone), 0, wc);
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------ elementwise
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;                // query row of the tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off;                // S, then dS
        const uint32_t tP = tmem + lane_off + 128;          // dP
        const int row_local = q_local0 + row;
        const bool row_valid = row_local < p.Ls;
        const size_t sidx = (static_cast<size_t>(b) * p.L + q0 + row) * p.H + h;
        const float lse2 = row_valid ? p.lse[sidx] * kLog2e : 0.f;
        const float dvr = row_valid ? p.dvec[sidx] : 0.f;
        const float sl2 = p.scale_log2;
        bool ok = true;
        for (int n = 0; n < n_blocks; ++n) {
            int s, kt;
            block(n, s, kt);
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kDSFull), n & 1, wc));
            if (!ok) break;
            tc_fence_after();
            int lim = min(kRows - 1, p.Ls - kt * kRows - 1);
            if (p.causal && s == r) lim = min(lim, row_local - kt * kRows);
            if (!row_valid) lim = -1;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t sr[64], dr[64];
                tmem_ld64(tS + 64 * half, sr);
                tmem_ld64(tP + 64 * half, dr);
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = 64 * half + 2 * i;
                    const float p0 = (c <= lim) ? ex2(fmaf(u2f(sr[2 * i]), sl2, -lse2)) : 0.f;
                    const float p1 = (c + 1 <= lim) ? ex2(fmaf(u2f(sr[2 * i + 1]), sl2, -lse2)) : 0.f;
                    pk[i] = pack_bf16x2(p0 * (u2f(dr[2 * i]) - dvr), p1 * (u2f(dr[2 * i + 1]) - dvr));
                }
                tmem_st32(tS + 32 * half, pk);
            }
            tc_fence_before();
            mbar_arrive(bar(kDDSFull));
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(kDOFull), 0, wc));
        if (ok) {
            tc_fence_after();
            __nv_bfloat16* dst = p.dq + ((static_cast<size_t>(b) * p.L + q0 + row) * p.H + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + 256 + 32 * c, o);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(u2f(o[2 * i]) * p.scale, u2f(o[2 * i + 1]) * p.scale);
                if (row_valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo)
{
    using Lay = BwdLayout<D>;
    constexpr int kSmemKV = 6 * Lay::kTileBytes + 2048 + 256 + 1024;
    constexpr int kSmemQ = 6 * Lay::kTileBytes + 256 + 1024;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemKV);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemQ);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    // Dvec = rowsum(dO o O) into the workspace
    const long long rows = static_cast<long long>(a.B) * a.L * a.H;
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (rows * (D / 8) + 255) / 256;
    if (blocks > static_cast<long long>(sms) * 8) blocks = static_cast<long long>(sms) * 8;
    if (blocks < 1) blocks = 1;
    bwd_rowdot_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
        static_cast<const uint4*>(a.out), static_cast<const uint4*>(a.dout), a.dvec, rows);
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
    p.P = a.P;
    p.Ls = a.L / a.P;
    p.causal = a.causal;
    p.n_t = (p.Ls + kRows - 1) / kRows;
    p.scale = 1.0f / sqrtf(static_cast<float>(D));
    p.scale_log2 = kLog2e * p.scale;
    const long long grid = static_cast<long long>(a.B) * a.H * a.P * p.n_t;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    bwd_dkdv_kernel<D><<<static_cast<unsigned>(grid), kThreads, kSmemKV, a.stream>>>(tq, tk, tv, tdo, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dq_kernel<D><<<static_cast<unsigned>(grid), kThreads, kSmemQ, a.stream>>>(tq, tk, tv, tdo, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_bf16(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo)
{
    if (a.D == 64) return launch_bwd_d<64>(a, tq, tk, tv, tdo);
    if (a.D == 128) return launch_bwd_d<128>(a, tq, tk, tv, tdo);
    return cudaErrorInvalidValue;
}

}  // namespace ra
