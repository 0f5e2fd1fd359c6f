// merge.cu -- log-sum-exp merge of two partial attention results, as a
// coalesced 16-byte-vector HBM stream (the juejin ring-attention page, section
// 四, `combine`: lse = logaddexp(lse_a, lse_b), o = o_a e^(lse_a - lse) +
// o_b e^(lse_b - lse)).
//
// A group of G lanes (G = 16-byte vectors per row rounded up to a power of two,
// at most 32) owns one row at a time: every lane of the group reads the two lse
// values, the lanes stream the row's vectors, and after a __syncwarp() the
// group's first lane writes the merged lse.  Reading before the warp barrier
// and writing after it keeps in-place merges (lse_out == lse_a) race-free;
// each output vector is written by the thread that read it, so o_out == o_a
// is race-free as well.  Each lane keeps four rows' loads in flight, and the
// grid is one resident wave (occupancy query).
#include <cuda_bf16.h>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kBlock = 256;

struct Weights {
    float wa, wb, lse;
};

// Partial with lse = -inf covers no key: weight 0.  Both empty: o = 0, lse = -inf.
__device__ __forceinline__ Weights merge_weights(float a, float b)
{
    Weights w;
    if (a == -INFINITY && b == -INFINITY) {
        w.wa = 0.f;
        w.wb = 0.f;
        w.lse = -INFINITY;
        return w;
    }
    const float hi = fmaxf(a, b), lo = fminf(a, b);
    w.lse = hi + log1pf(expf(lo - hi));
    w.wa = expf(a - w.lse);
    w.wb = expf(b - w.lse);
    return w;
}

__device__ __forceinline__ uint4 combine_vec_bf16(uint4 x, uint4 y, float wa, float wb)
{
    const __nv_bfloat162* xa = reinterpret_cast<const __nv_bfloat162*>(&x);
    const __nv_bfloat162* ya = reinterpret_cast<const __nv_bfloat162*>(&y);
    uint4 res;
    __nv_bfloat162* ro = reinterpret_cast<__nv_bfloat162*>(&res);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 fx = __bfloat1622float2(xa[i]);
        const float2 fy = __bfloat1622float2(ya[i]);
        ro[i] = __floats2bfloat162_rn(fmaf(fx.x, wa, fy.x * wb), fmaf(fx.y, wa, fy.y * wb));
    }
    return res;
}

__device__ __forceinline__ uint4 combine_vec_f32(uint4 x, uint4 y, float wa, float wb)
{
    uint4 res;
    res.x = __float_as_uint(fmaf(__uint_as_float(x.x), wa, __uint_as_float(y.x) * wb));
    res.y = __float_as_uint(fmaf(__uint_as_float(x.y), wa, __uint_as_float(y.y) * wb));
    res.z = __float_as_uint(fmaf(__uint_as_float(x.z), wa, __uint_as_float(y.z) * wb));
    res.w = __float_as_uint(fmaf(__uint_as_float(x.w), wa, __uint_as_float(y.w) * wb));
    return res;
}

constexpr int kRowsInFlight = 4;   // row groups per lane group per iteration

template <bool kBf16>
__global__ void __launch_bounds__(kBlock)
    merge_kernel(const uint4* o_a, const float* lse_a, const uint4* o_b, const float* lse_b,
                 uint4* o_out, float* lse_out, long long rows, int vpr, int group_log2,
                 unsigned int* status)
{
    const long long n_vec = rows * vpr;     // extent of the o tensors, 16-byte vectors
    const int lane = threadIdx.x & 31;
    const int G = 1 << group_log2;
    const int rows_per_warp = 32 >> group_log2;
    const int sub = lane & (G - 1);
    const long long warp_global = (static_cast<long long>(blockIdx.x) * kBlock + threadIdx.x) >> 5;
    const long long n_warps = (static_cast<long long>(gridDim.x) * kBlock) >> 5;
    const long long step = n_warps * rows_per_warp;   // rows covered by one sweep of all warps
    for (long long base = warp_global * rows_per_warp; base < rows; base += kRowsInFlight * step) {
        long long row[kRowsInFlight];
        bool valid[kRowsInFlight];
        Weights w[kRowsInFlight];
#pragma unroll
        for (int u = 0; u < kRowsInFlight; ++u) {
            row[u] = base + u * step + (lane >> group_log2);
            valid[u] = row[u] < rows && in_bounds(row[u], 1, rows, status);
            w[u] = Weights{0.f, 0.f, -INFINITY};
        }
        // issue every load of the kRowsInFlight rows before any arithmetic
        float la[kRowsInFlight], lb[kRowsInFlight];
#pragma unroll
        for (int u = 0; u < kRowsInFlight; ++u) {
            la[u] = valid[u] ? lse_a[row[u]] : 0.f;
            lb[u] = valid[u] ? lse_b[row[u]] : 0.f;
        }
        for (int c = sub; c < vpr; c += G) {
            uint4 x[kRowsInFlight], y[kRowsInFlight];
#pragma unroll
            for (int u = 0; u < kRowsInFlight; ++u) {
                if (valid[u] && in_bounds(row[u] * vpr + c, 1, n_vec, status)) {
                    x[u] = __ldcs(o_a + row[u] * vpr + c);
                    y[u] = __ldcs(o_b + row[u] * vpr + c);
                }
            }
#pragma unroll
            for (int u = 0; u < kRowsInFlight; ++u) {
                if (!valid[u]) continue;
                if (c == sub) w[u] = merge_weights(la[u], lb[u]);
                if (!in_bounds(row[u] * vpr + c, 1, n_vec, status)) continue;
                __stcs(o_out + row[u] * vpr + c, kBf16 ? combine_vec_bf16(x[u], y[u], w[u].wa, w[u].wb)
                                                       : combine_vec_f32(x[u], y[u], w[u].wa, w[u].wb));
            }
        }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < kRowsInFlight; ++u)
            if (valid[u] && sub == 0) lse_out[row[u]] = merge_weights(la[u], lb[u]).lse;
        __syncwarp();
    }
}

// Fast path for rows of 1, 2, 4, 8, 16 or 32 vectors: thread v of a sweep owns
// 16-byte vector v, four sweeps in flight per thread.  Consecutive vectors of a
// row land on consecutive lanes of one warp (sweeps start on multiples of 32),
// so reading both lse values before the __syncwarp() and writing lse_out after
// it keeps in-place merges race-free here too.
constexpr int kFlatUnroll = 4;

template <bool kBf16>
__global__ void __launch_bounds__(kBlock)
    merge_flat_kernel(const uint4* o_a, const float* lse_a, const uint4* o_b, const float* lse_b,
                      uint4* o_out, float* lse_out, long long n_vec, int log2_vpr,
                      unsigned int* status)
{
    const long long rows = n_vec >> log2_vpr;
    const long long stride = static_cast<long long>(gridDim.x) * kBlock;
    const long long vpr_mask = (1ll << log2_vpr) - 1;
    for (long long v0 = static_cast<long long>(blockIdx.x) * kBlock + threadIdx.x;
         v0 - threadIdx.x % 32 < n_vec; v0 += kFlatUnroll * stride) {
        long long v[kFlatUnroll];
        bool valid[kFlatUnroll];
        float la[kFlatUnroll], lb[kFlatUnroll];
        uint4 x[kFlatUnroll], y[kFlatUnroll];
#pragma unroll
        for (int u = 0; u < kFlatUnroll; ++u) {
            v[u] = v0 + u * stride;
            valid[u] = v[u] < n_vec && in_bounds(v[u], 1, n_vec, status) &&
                       in_bounds(v[u] >> log2_vpr, 1, rows, status);
            if (valid[u]) {
                const long long row = v[u] >> log2_vpr;
                la[u] = lse_a[row];
                lb[u] = lse_b[row];
                x[u] = __ldcs(o_a + v[u]);
                y[u] = __ldcs(o_b + v[u]);
            }
        }
        float lse_new[kFlatUnroll];
#pragma unroll
        for (int u = 0; u < kFlatUnroll; ++u) {
            if (!valid[u]) continue;
            const Weights w = merge_weights(la[u], lb[u]);
            lse_new[u] = w.lse;
            __stcs(o_out + v[u], kBf16 ? combine_vec_bf16(x[u], y[u], w.wa, w.wb)
                                       : combine_vec_f32(x[u], y[u], w.wa, w.wb));
        }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < kFlatUnroll; ++u)
            if (valid[u] && (v[u] & vpr_mask) == 0) lse_out[v[u] >> log2_vpr] = lse_new[u];
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_merge(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                         void* o_out, float* lse_out, long long rows, int D, int elem_bytes,
                         unsigned int* status, cudaStream_t stream)
{
    const int vpr = D * elem_bytes / 16;
    int group_log2 = 0;
    while ((1 << group_log2) < vpr && group_log2 < 5) ++group_log2;
    const long long rows_per_warp = 32 >> group_log2;
    const long long warps_needed = (rows + rows_per_warp - 1) / rows_per_warp;
    int dev = 0, sms = 148, per_sm = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (elem_bytes == 2)
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, merge_kernel<true>, kBlock, 0);
    else
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, merge_kernel<false>, kBlock, 0);
    long long blocks = (warps_needed * 32 + kBlock - 1) / kBlock;
    const long long cap = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);  // one resident wave
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (vpr <= 32 && (vpr & (vpr - 1)) == 0) {
        int log2_vpr = 0;
        while ((1 << log2_vpr) < vpr) ++log2_vpr;
        const long long n_vec = rows * vpr;
        int fast_per_sm = 1;
        if (elem_bytes == 2)
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fast_per_sm, merge_flat_kernel<true>, kBlock, 0);
        else
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fast_per_sm, merge_flat_kernel<false>, kBlock, 0);
        long long fblocks = (n_vec + kBlock - 1) / kBlock;
        const long long fcap = static_cast<long long>(sms) * (fast_per_sm > 0 ? fast_per_sm : 1);
        if (fblocks > fcap) fblocks = fcap;
        if (fblocks < 1) fblocks = 1;
        if (elem_bytes == 2)
            merge_flat_kernel<true><<<static_cast<unsigned>(fblocks), kBlock, 0, stream>>>(
                static_cast<const uint4*>(o_a), lse_a, static_cast<const uint4*>(o_b), lse_b,
                static_cast<uint4*>(o_out), lse_out, n_vec, log2_vpr, status);
        else
            merge_flat_kernel<false><<<static_cast<unsigned>(fblocks), kBlock, 0, stream>>>(
                static_cast<const uint4*>(o_a), lse_a, static_cast<const uint4*>(o_b), lse_b,
                static_cast<uint4*>(o_out), lse_out, n_vec, log2_vpr, status);
        return cudaGetLastError();
    }
    if (elem_bytes == 2)
        merge_kernel<true><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(
            static_cast<const uint4*>(o_a), lse_a, static_cast<const uint4*>(o_b), lse_b,
            static_cast<uint4*>(o_out), lse_out, rows, vpr, group_log2, status);
    else
        merge_kernel<false><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(
            static_cast<const uint4*>(o_a), lse_a, static_cast<const uint4*>(o_b), lse_b,
            static_cast<uint4*>(o_out), lse_out, rows, vpr, group_log2, status);
    return cudaGetLastError();
}

}  // namespace ra
