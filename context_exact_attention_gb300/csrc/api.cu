// api.cu -- the extern "C" entry points of libringattn.so: host-side argument
// checks (nothing is launched on a bad argument), TMA tensor-map encoding
// through the driver entry point, dispatch to the kernels, and the per-device
// status word that bounded device-side waits report into.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace {

constexpr unsigned long long kWaitLimitNs = 4000000000ull;   // 4 s for any single wait

// Status word of each device: bit RA_STATUS_TIMEOUT is set by a kernel whose
// bounded wait ran out.  Read and cleared by ra_check_status().
__device__ unsigned int g_status_word;

// Device address of the current device's status word.  Looked up on every call (a
// table lookup once the module is loaded): a cached address would go stale if the
// caller reset the device and the module were loaded again elsewhere.
ra_status status_word(unsigned int** out)
{
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return RA_ERR_CUDA;
    *out = static_cast<unsigned int*>(p);
    return RA_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// q/k/v as a 4-D bf16 tensor {D, H, L, B} (innermost first); boxes of 64 head-dim
// elements (128 bytes, the swizzle span) by box_rows sequence rows, 128-byte swizzle.
bool encode_qkv_map(CUtensorMap* map, const void* base, int B, int L, int H, int D,
                    int box_rows = 128)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(H) * D * 2,
                                   static_cast<cuuint64_t>(L) * H * D * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A sequence-sharded Ulysses buffer [P][B][L/P][H][D] as a 5-D bf16 tensor
// {D, H, L/P, B, P} (innermost first), same boxes and swizzle as encode_qkv_map: a box of
// 128 rows stays inside one shard when (L/P) % 128 == 0.
// The sequence-sharded buffer [P][B][L/P][H][D] of the Ulysses transposes as the 5-D
// view {D, H/P, P, L/P, P*B} (innermost first: head dim, head within a group, group,
// position within the shard, source rank and batch), box {D, H/P, 1, R, 1}: one group's
// heads at R consecutive positions.  No swizzle, so a box lands in shared memory as the
// dense run [R][H/P][D] it is on the head-sharded side; elements are moved as 16- or
// 32-bit words.
bool encode_permute_map(CUtensorMap* map, const void* base, int B, int L, int H, int D, int P,
                        int elem_bytes, int R)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t e = static_cast<cuuint64_t>(elem_bytes);
    const cuuint64_t hg = static_cast<cuuint64_t>(H / P), Ls = static_cast<cuuint64_t>(L / P);
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(D), hg, static_cast<cuuint64_t>(P), Ls,
                                static_cast<cuuint64_t>(P) * B};
    const cuuint64_t strides[4] = {D * e, hg * D * e, static_cast<cuuint64_t>(H) * D * e,
                                   Ls * H * D * e};
    const cuuint32_t box[5] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(hg), 1,
                               static_cast<cuuint32_t>(R), 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32, 5,
              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_seq_shard_map(CUtensorMap* map, const void* base, int P, int B, int L, int H, int D,
                          int box_rows = 128)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t Ls = static_cast<cuuint64_t>(L / P);
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), Ls,
                                static_cast<cuuint64_t>(B), static_cast<cuuint64_t>(P)};
    const cuuint64_t row = static_cast<cuuint64_t>(H) * D * 2;
    const cuuint64_t strides[4] = {static_cast<cuuint64_t>(D) * 2, row, Ls * row, Ls * row * B};
    const cuuint32_t box[5] = {64, 1, static_cast<cuuint32_t>(box_rows), 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void* a, unsigned long long na, const void* b, unsigned long long nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

ra_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RA_OK : RA_ERR_CUDA; }

// Shared checks of the attention entry points.  elem: element bytes; Hkv: key/value
// heads (k and v are [B, L, Hkv, D]; H must be a multiple of Hkv).
ra_status check_attn(const void* q, const void* k, const void* v, const void* out,
                     const float* lse, int B, int L, int H, int D, int P, int elem,
                     unsigned long long* elems, int Hkv = -1)
{
    if (Hkv < 0) Hkv = H;
    if (!q || !k || !v || !out) return RA_ERR_INVALID_ARG;
    if (B < 1 || L < 1 || H < 1 || D < 1 || P < 1 || Hkv < 1) return RA_ERR_INVALID_ARG;
    const unsigned long long n = static_cast<unsigned long long>(B) * L * H * D;
    if (n >= (1ull << 40)) return RA_ERR_INVALID_ARG;
    if (L % P != 0 || H % Hkv != 0) return RA_ERR_NOT_DIVISIBLE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return RA_ERR_MISALIGNED;
    if (lse && !aligned(lse, 4)) return RA_ERR_MISALIGNED;
    const unsigned long long bytes = n * elem;
    const unsigned long long kv_bytes = static_cast<unsigned long long>(B) * L * Hkv * D * elem;
    if (overlap(out, bytes, q, bytes) || overlap(out, bytes, k, kv_bytes) ||
        overlap(out, bytes, v, kv_bytes))
        return RA_ERR_INVALID_ARG;
    if (lse) {
        const unsigned long long lb = static_cast<unsigned long long>(B) * L * H * 4;
        if (overlap(lse, lb, q, bytes) || overlap(lse, lb, k, kv_bytes) ||
            overlap(lse, lb, v, kv_bytes) || overlap(lse, lb, out, bytes))
            return RA_ERR_INVALID_ARG;
    }
    *elems = n;
    return RA_OK;
}

ra_status attn_impl(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                    int L, int H, int D, int P, int causal, ra_dtype dtype, int* trace,
                    cudaStream_t stream, int Hkv = -1, int zigzag = 0,
                    const int* cu_seqlens = nullptr, int n_seqs = 0, int ulysses_P = 0,
                    const int* schedule = nullptr)
{
    if (Hkv < 0) Hkv = H;
    if (dtype != RA_BF16 && dtype != RA_F32) return RA_ERR_UNSUPPORTED;
    const int elem = dtype == RA_BF16 ? 2 : 4;
    unsigned long long n = 0;
    ra_status st = check_attn(q, k, v, out, lse, B, L, H, D, P, elem, &n, Hkv);
    if (st != RA_OK) return st;
    if (schedule) {
        const unsigned long long sb = ring_attn_varlen_schedule_bytes(L, P);
        if (overlap(schedule, sb, out, n * elem) ||
            (lse && overlap(schedule, sb, lse, static_cast<unsigned long long>(B) * L * H * 4)))
            return RA_ERR_INVALID_ARG;
    }
    if (dtype == RA_BF16 && D != 64 && D != 128) return RA_ERR_UNSUPPORTED;
    if (dtype == RA_F32 && (D % 4 != 0 || D > 256)) return RA_ERR_UNSUPPORTED;
    if (trace) {
        if (!aligned(trace, 4)) return RA_ERR_MISALIGNED;
        const unsigned long long tb = static_cast<unsigned long long>(P) * P * 4;
        if (overlap(trace, tb, out, n * elem)) return RA_ERR_INVALID_ARG;
    }
    ra::AttnArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.lse = lse;
    a.trace = trace;
    a.B = B;
    a.L = L;
    a.H = H;
    a.D = D;
    a.P = P;
    a.causal = causal ? 1 : 0;
    a.Hkv = Hkv;
    a.zigzag = zigzag;
    a.cu_seqlens = cu_seqlens;
    a.n_seqs = n_seqs;
    a.schedule = schedule;
    a.u_P = 0;
    a.u_B = 0;
    a.u_H = 0;
    a.timeout_ns = kWaitLimitNs;
    a.stream = stream;
    st = status_word(&a.status);
    if (st != RA_OK) return st;
    if (ulysses_P > 0) {
        // the kernel sees ulysses_P * B head-group batches of H / ulysses_P heads (ring P = 1)
        // and addresses the sequence-sharded sources through 5-D tensor maps
        CUtensorMap tq, tk, tv;
        a.u_P = ulysses_P;
        a.u_B = B;
        a.u_H = H;
        a.B = ulysses_P * B;
        a.H = H / ulysses_P;
        a.Hkv = Hkv / ulysses_P;
        const int k_rows = ra::attn_bf16_pair_applies(a) ? 64 : 128;
        if (!encode_seq_shard_map(&tq, q, ulysses_P, B, L, H, D) ||
            !encode_seq_shard_map(&tk, k, ulysses_P, B, L, Hkv, D, k_rows) ||
            !encode_seq_shard_map(&tv, v, ulysses_P, B, L, Hkv, D))
            return RA_ERR_CUDA;
        return from_cuda(ra::launch_attn_bf16(a, tq, tk, tv));
    }
    if (dtype == RA_F32) return from_cuda(ra::launch_attn_f32(a));
    CUtensorMap tq, tk, tv;
    const int k_rows = ra::attn_bf16_pair_applies(a) ? 64 : 128;
    if (!encode_qkv_map(&tq, q, B, L, H, D) || !encode_qkv_map(&tk, k, B, L, Hkv, D, k_rows) ||
        !encode_qkv_map(&tv, v, B, L, Hkv, D))
        return RA_ERR_CUDA;
    return from_cuda(ra::launch_attn_bf16(a, tq, tk, tv));
}

ra_status permute_impl(const void* in, void* out, int B, int L, int H, int D, int P,
                       int elem_bytes, int dir, cudaStream_t stream)
{
    if (!in || !out) return RA_ERR_INVALID_ARG;
    if (B < 1 || L < 1 || H < 1 || D < 1 || P < 1) return RA_ERR_INVALID_ARG;
    if (elem_bytes != 2 && elem_bytes != 4) return RA_ERR_UNSUPPORTED;
    const unsigned long long n = static_cast<unsigned long long>(B) * L * H * D;
    if (n >= (1ull << 40)) return RA_ERR_INVALID_ARG;
    if (L % P != 0 || H % P != 0) return RA_ERR_NOT_DIVISIBLE;
    if ((D * elem_bytes) % 16 != 0) return RA_ERR_UNSUPPORTED;
    if (!aligned(in, 16) || !aligned(out, 16)) return RA_ERR_MISALIGNED;
    const unsigned long long bytes = n * elem_bytes;
    if (overlap(in, bytes, out, bytes)) return RA_ERR_INVALID_ARG;
    unsigned int* status = nullptr;
    const ra_status st = status_word(&status);
    if (st != RA_OK) return st;
    if (ra::ulysses_permute_tma_fits(H, D, P, elem_bytes)) {
        // copy engines: the sequence-sharded side as a 5-D view {D, H/P, P, L/P, P*B}
        const int R = ra::ulysses_permute_tma_rows(L, H, D, P, elem_bytes);
        CUtensorMap map;
        const void* seq_side = dir == 0 ? in : out;
        void* head_side = dir == 0 ? out : const_cast<void*>(in);
        if (encode_permute_map(&map, seq_side, B, L, H, D, P, elem_bytes, R))
            return from_cuda(ra::launch_ulysses_permute_tma(map, head_side, B, L, H, D, P, elem_bytes,
                                                            dir, R, status, kWaitLimitNs, stream));
    }
    return from_cuda(
        ra::launch_ulysses_permute(in, out, B, L, H, D, P, elem_bytes, dir, status, stream));
}

}  // namespace

namespace ra {
namespace {

__global__ void wait_probe_kernel(unsigned int* status, unsigned long long timeout_ns)
{
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        const uint32_t bar = smem_addr(&bar_storage);
        abort_flag = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
        const WaitCtx w{&abort_flag, status, timeout_ns};
        // nobody arrives: the wait can only end by running out of time
        mbar_wait(bar, 0, w);
    }
}

}  // namespace

cudaError_t launch_wait_probe(unsigned int* status, unsigned long long timeout_ns,
                              cudaStream_t stream)
{
    wait_probe_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

ra_status current_status_word(unsigned int** out) { return status_word(out); }

namespace {

__device__ unsigned int g_bounds_probe_sink;

// One checked access that must fail: index 1 of a one-element extent.  The write it
// guards goes to a word of this library, so it is harmless even if the check passed.
__global__ void bounds_probe_kernel(unsigned int* status)
{
    if (in_bounds(1, 1, 1, status)) g_bounds_probe_sink = 1u;
}

}  // namespace

cudaError_t launch_bounds_probe(unsigned int* status, cudaStream_t stream)
{
    bounds_probe_kernel<<<1, 1, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace ra

extern "C" {

ra_status ring_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                        int B, int L, int H, int D, int P, int causal, ra_stream_t stream)
{
    return attn_impl(q, k, v, out, lse, B, L, H, D, P, causal, RA_BF16, nullptr,
                     reinterpret_cast<cudaStream_t>(stream));
}

ra_status ring_attn_fwd_f32(const float* q, const float* k, const float* v, float* out,
                            float* lse, int B, int L, int H, int D, int P, int causal,
                            ra_stream_t stream)
{
    return attn_impl(q, k, v, out, lse, B, L, H, D, P, causal, RA_F32, nullptr,
                     reinterpret_cast<cudaStream_t>(stream));
}

ra_status ring_attn_fwd_trace(const void* q, const void* k, const void* v, void* out, float* lse,
                              int B, int L, int H, int D, int P, int causal, ra_dtype dtype,
                              int* trace, ra_stream_t stream)
{
    if (!trace) return RA_ERR_INVALID_ARG;
    return attn_impl(q, k, v, out, lse, B, L, H, D, P, causal, dtype, trace,
                     reinterpret_cast<cudaStream_t>(stream));
}

ra_status ring_attn_fwd_gqa(const void* q, const void* k, const void* v, void* out, float* lse,
                            int B, int L, int H, int H_kv, int D, int P, int causal,
                            ra_dtype dtype, ra_stream_t stream)
{
    if (H_kv < 1) return RA_ERR_INVALID_ARG;
    return attn_impl(q, k, v, out, lse, B, L, H, D, P, causal, dtype, nullptr,
                     reinterpret_cast<cudaStream_t>(stream), H_kv);
}

ra_status ring_attn_fwd_zigzag(const void* q, const void* k, const void* v, void* out,
                               float* lse, int B, int L, int H, int D, int P, ra_dtype dtype,
                               int* trace, ra_stream_t stream)
{
    if (P < 1 || L < 1) return RA_ERR_INVALID_ARG;
    if (L % (2 * P) != 0) return RA_ERR_NOT_DIVISIBLE;
    // bf16 key/query tiles of 128 must not straddle the two chunks of a shard
    if (dtype == RA_BF16 && (L / (2 * P)) % 128 != 0) return RA_ERR_UNSUPPORTED;
    return attn_impl(q, k, v, out, lse, B, L, H, D, P, 1, dtype, trace,
                     reinterpret_cast<cudaStream_t>(stream), H, 1);
}

ra_status ring_attn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                               float* lse, const int* cu_seqlens, int n_seqs, int L, int H, int D,
                               int P, int causal, ra_dtype dtype, int* trace, ra_stream_t stream)
{
    if (!cu_seqlens || n_seqs < 1) return RA_ERR_INVALID_ARG;
    if (!aligned(cu_seqlens, 4)) return RA_ERR_MISALIGNED;
    return attn_impl(q, k, v, out, lse, 1, L, H, D, P, causal, dtype, trace,
                     reinterpret_cast<cudaStream_t>(stream), H, 0, cu_seqlens, n_seqs);
}

ra_status ulysses_attention_fused(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int B, int L, int H, int H_kv, int D, int P,
                                  int causal, ra_stream_t stream)
{
    if (P < 1 || L < 1 || H < 1 || H_kv < 1) return RA_ERR_INVALID_ARG;
    if (L % P != 0 || H % P != 0 || H_kv % P != 0) return RA_ERR_NOT_DIVISIBLE;
    // a 128-row tile must come from one sequence shard
    if ((L / P) % 128 != 0) return RA_ERR_UNSUPPORTED;
    // q, k, v, out hold as many elements as [B, L, H(_kv), D]: the common checks apply
    // with one ring shard
    return attn_impl(q, k, v, out, lse, B, L, H, D, 1, causal, RA_BF16, nullptr,
                     reinterpret_cast<cudaStream_t>(stream), H_kv, 0, nullptr, 0, P);
}

ra_status attn_merge_partials(const void* o_a, const float* lse_a, const void* o_b,
                              const float* lse_b, void* o_out, float* lse_out, long long rows,
                              int D, ra_dtype dtype, ra_stream_t stream)
{
    if (dtype != RA_BF16 && dtype != RA_F32) return RA_ERR_UNSUPPORTED;
    if (rows < 0 || D < 1) return RA_ERR_INVALID_ARG;
    if (rows == 0) return RA_OK;
    if (!o_a || !lse_a || !o_b || !lse_b || !o_out || !lse_out) return RA_ERR_INVALID_ARG;
    const int elem = dtype == RA_BF16 ? 2 : 4;
    if ((D * elem) % 16 != 0) return RA_ERR_UNSUPPORTED;
    if (static_cast<unsigned long long>(rows) * D >= (1ull << 40)) return RA_ERR_INVALID_ARG;
    if (!aligned(o_a, 16) || !aligned(o_b, 16) || !aligned(o_out, 16) || !aligned(lse_a, 4) ||
        !aligned(lse_b, 4) || !aligned(lse_out, 4))
        return RA_ERR_MISALIGNED;
    const unsigned long long ob = static_cast<unsigned long long>(rows) * D * elem;
    const unsigned long long lb = static_cast<unsigned long long>(rows) * 4;
    // in place is allowed (same base pointer); any partial overlap is not
    if ((o_out != o_a && overlap(o_out, ob, o_a, ob)) || (o_out != o_b && overlap(o_out, ob, o_b, ob)))
        return RA_ERR_INVALID_ARG;
    if ((lse_out != lse_a && overlap(lse_out, lb, lse_a, lb)) ||
        (lse_out != lse_b && overlap(lse_out, lb, lse_b, lb)))
        return RA_ERR_INVALID_ARG;
    if (overlap(o_out, ob, lse_out, lb) || overlap(o_out, ob, lse_a, lb) ||
        overlap(o_out, ob, lse_b, lb))
        return RA_ERR_INVALID_ARG;
    unsigned int* status = nullptr;
    const ra_status st = status_word(&status);
    if (st != RA_OK) return st;
    return from_cuda(ra::launch_merge(o_a, lse_a, o_b, lse_b, o_out, lse_out, rows, D, elem, status,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

ra_status ulysses_seq2head(const void* in, void* out, int B, int L, int H, int D, int P,
                           int elem_bytes, ra_stream_t stream)
{
    return permute_impl(in, out, B, L, H, D, P, elem_bytes, 0,
                        reinterpret_cast<cudaStream_t>(stream));
}

ra_status ulysses_head2seq(const void* in, void* out, int B, int L, int H, int D, int P,
                           int elem_bytes, ra_stream_t stream)
{
    return permute_impl(in, out, B, L, H, D, P, elem_bytes, 1,
                        reinterpret_cast<cudaStream_t>(stream));
}

unsigned long long ring_attn_bwd_workspace_bytes(int B, int L, int H)
{
    if (B < 1 || L < 1 || H < 1) return 0;
    return static_cast<unsigned long long>(B) * L * H * sizeof(float);
}

}  // extern "C"

namespace {

ra_status bwd_impl(const void* q, const void* k, const void* v, const void* out, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, void* workspace,
                   unsigned long long workspace_bytes, int B, int L, int H, int Hkv, int D, int P,
                   int causal, ra_stream_t stream, int zigzag = 0, const int* cu_seqlens = nullptr,
                   int n_seqs = 0, const int* schedule = nullptr)
{
    unsigned long long n = 0;
    ra_status st = check_attn(q, k, v, out, lse, B, L, H, D, P, 2, &n, Hkv);
    if (st != RA_OK) return st;
    if (!lse || !dout || !dq || !dk || !dv || !workspace) return RA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return RA_ERR_UNSUPPORTED;
    if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
        !aligned(workspace, 16))
        return RA_ERR_MISALIGNED;
    const unsigned long long ws = ring_attn_bwd_workspace_bytes(B, L, H);
    if (workspace_bytes < ws) return RA_ERR_INVALID_ARG;
    const unsigned long long bytes = n * 2;                       // q, out, dout, dq
    const unsigned long long kv_bytes = bytes / H * Hkv;          // k, v, dk, dv
    const void* ins[6] = {q, k, v, out, dout, lse};
    const unsigned long long in_bytes[6] = {bytes, kv_bytes, kv_bytes, bytes, bytes, ws};
    void* outs[4] = {dq, dk, dv, workspace};
    const unsigned long long out_bytes[4] = {bytes, kv_bytes, kv_bytes, ws};
    for (int i = 0; i < 4; ++i) {
        for (int j = 0; j < 6; ++j)
            if (overlap(outs[i], out_bytes[i], ins[j], in_bytes[j])) return RA_ERR_INVALID_ARG;
        for (int j = i + 1; j < 4; ++j)
            if (overlap(outs[i], out_bytes[i], outs[j], out_bytes[j])) return RA_ERR_INVALID_ARG;
        if (schedule &&
            overlap(outs[i], out_bytes[i], schedule, ring_attn_varlen_schedule_bytes(L, P)))
            return RA_ERR_INVALID_ARG;
    }
    ra::BwdArgs a;
    a.out = out;
    a.dout = dout;
    a.lse = lse;
    a.dvec = static_cast<float*>(workspace);
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.L = L;
    a.H = H;
    a.Hkv = Hkv;
    a.D = D;
    a.P = P;
    a.causal = causal ? 1 : 0;
    a.zigzag = zigzag;
    a.cu_seqlens = cu_seqlens;
    a.n_seqs = n_seqs;
    a.schedule = schedule;
    a.timeout_ns = kWaitLimitNs;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    st = status_word(&a.status);
    if (st != RA_OK) return st;
    CUtensorMap tq, tk, tv, tdo, tk64, tv64;
    if (!encode_qkv_map(&tq, q, B, L, H, D) || !encode_qkv_map(&tk, k, B, L, Hkv, D) ||
        !encode_qkv_map(&tv, v, B, L, Hkv, D) || !encode_qkv_map(&tdo, dout, B, L, H, D))
        return RA_ERR_CUDA;
    const bool pair = ra::bwd_dq_pair_applies(a);
    if (pair && (!encode_qkv_map(&tk64, k, B, L, Hkv, D, 64) ||
                 !encode_qkv_map(&tv64, v, B, L, Hkv, D, 64)))
        return RA_ERR_CUDA;
    return from_cuda(ra::launch_attn_bwd_bf16(a, tq, tk, tv, tdo, pair ? &tk64 : nullptr,
                                              pair ? &tv64 : nullptr));
}

}  // namespace

extern "C" {

ra_status ring_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        void* workspace, unsigned long long workspace_bytes, int B, int L, int H,
                        int D, int P, int causal, ra_stream_t stream)
{
    return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, L, H, H, D,
                    P, causal, stream);
}

ra_status ring_attn_bwd_gqa(const void* q, const void* k, const void* v, const void* out,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            void* workspace, unsigned long long workspace_bytes, int B, int L,
                            int H, int H_kv, int D, int P, int causal, ra_stream_t stream)
{
    if (H_kv < 1) return RA_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, L, H, H_kv,
                    D, P, causal, stream);
}

ra_status ring_attn_bwd_zigzag(const void* q, const void* k, const void* v, const void* out,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               void* workspace, unsigned long long workspace_bytes, int B, int L,
                               int H, int D, int P, ra_stream_t stream)
{
    if (P < 1 || L < 1) return RA_ERR_INVALID_ARG;
    if (L % (2 * P) != 0) return RA_ERR_NOT_DIVISIBLE;
    // 128-row tiles must not straddle the two chunks of a shard
    if ((L / (2 * P)) % 128 != 0) return RA_ERR_UNSUPPORTED;
    return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, L, H, H, D,
                    P, 1, stream, 1);
}

ra_status ring_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* out,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               void* workspace, unsigned long long workspace_bytes,
                               const int* cu_seqlens, int n_seqs, int L, int H, int D, int P,
                               int causal, ra_stream_t stream)
{
    if (!cu_seqlens || n_seqs < 1) return RA_ERR_INVALID_ARG;
    if (!aligned(cu_seqlens, 4)) return RA_ERR_MISALIGNED;
    return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, 1, L, H, H, D,
                    P, causal, stream, 0, cu_seqlens, n_seqs);
}

// The layout part of a descriptor, checked: zigzag flag, packed boundaries and
// schedule, batch.
static ra_status desc_layout(const ra_attn_desc* d, int bf16, int* zig, const int** cu,
                             int* n_seqs, const int** sched)
{
    if (!d) return RA_ERR_INVALID_ARG;
    if (d->B < 1 || d->L < 1 || d->H < 1 || d->H_kv < 1 || d->D < 1 || d->P < 1)
        return RA_ERR_INVALID_ARG;
    *zig = 0;
    *cu = nullptr;
    *n_seqs = 0;
    *sched = nullptr;
    if (d->layout != RA_LAYOUT_PACKED && d->schedule) return RA_ERR_INVALID_ARG;
    switch (d->layout) {
    case RA_LAYOUT_CONTIGUOUS:
        if (d->cu_seqlens) return RA_ERR_INVALID_ARG;
        return RA_OK;
    case RA_LAYOUT_ZIGZAG:
        if (d->cu_seqlens) return RA_ERR_INVALID_ARG;
        if (!d->causal) return RA_ERR_UNSUPPORTED;            // the layout exists for causal balance
        if (d->L % (2 * d->P) != 0) return RA_ERR_NOT_DIVISIBLE;
        if (bf16 && (d->L / (2 * d->P)) % 128 != 0) return RA_ERR_UNSUPPORTED;
        *zig = 1;
        return RA_OK;
    case RA_LAYOUT_PACKED:
        if (!d->cu_seqlens || d->n_seqs < 1 || d->B != 1) return RA_ERR_INVALID_ARG;
        if (!aligned(d->cu_seqlens, 4)) return RA_ERR_MISALIGNED;
        if (d->schedule && !aligned(d->schedule, 4)) return RA_ERR_MISALIGNED;
        *cu = d->cu_seqlens;
        *n_seqs = d->n_seqs;
        *sched = d->schedule;
        return RA_OK;
    }
    return RA_ERR_INVALID_ARG;
}

ra_status ring_attn_fwd_ex(const ra_attn_desc* desc, const void* q, const void* k, const void* v,
                           void* out, float* lse, int* trace, ra_stream_t stream)
{
    int zig = 0, n_seqs = 0;
    const int* cu = nullptr;
    const int* sched = nullptr;
    const ra_status st =
        desc_layout(desc, desc && desc->dtype == RA_BF16, &zig, &cu, &n_seqs, &sched);
    if (st != RA_OK) return st;
    return attn_impl(q, k, v, out, lse, desc->B, desc->L, desc->H, desc->D, desc->P, desc->causal,
                     desc->dtype, trace, reinterpret_cast<cudaStream_t>(stream), desc->H_kv, zig,
                     cu, n_seqs, 0, sched);
}

ra_status ring_attn_bwd_ex(const ra_attn_desc* desc, const void* q, const void* k, const void* v,
                           const void* out, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* workspace, unsigned long long workspace_bytes,
                           ra_stream_t stream)
{
    int zig = 0, n_seqs = 0;
    const int* cu = nullptr;
    const int* sched = nullptr;
    const ra_status st = desc_layout(desc, 1, &zig, &cu, &n_seqs, &sched);
    if (st != RA_OK) return st;
    if (desc->dtype != RA_BF16) return RA_ERR_UNSUPPORTED;
    return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, desc->B,
                    desc->L, desc->H, desc->H_kv, desc->D, desc->P, desc->causal, stream, zig, cu,
                    n_seqs, sched);
}

unsigned long long ring_attn_varlen_schedule_bytes(int L, int P)
{
    if (L < 1 || P < 1 || P > L || L % P != 0) return 0;
    return static_cast<unsigned long long>(ra::varlen_sched_layout(L, P).total) * sizeof(int);
}

ra_status ring_attn_varlen_schedule(const int* cu_seqlens, int n_seqs, int L, int P, int causal,
                                    int* schedule, unsigned long long schedule_bytes,
                                    ra_stream_t stream)
{
    if (!cu_seqlens || !schedule || n_seqs < 1 || L < 1 || P < 1 || P > L)
        return RA_ERR_INVALID_ARG;
    if (L % P != 0) return RA_ERR_NOT_DIVISIBLE;
    if (!aligned(cu_seqlens, 4) || !aligned(schedule, 4)) return RA_ERR_MISALIGNED;
    const unsigned long long need = ring_attn_varlen_schedule_bytes(L, P);
    if (schedule_bytes < need) return RA_ERR_INVALID_ARG;
    if (overlap(schedule, need, cu_seqlens, (static_cast<unsigned long long>(n_seqs) + 1) * 4))
        return RA_ERR_INVALID_ARG;
    unsigned int* status = nullptr;
    const ra_status st = status_word(&status);
    if (st != RA_OK) return st;
    return from_cuda(ra::launch_varlen_schedule(cu_seqlens, n_seqs, L, P, causal, schedule, status,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

long long ra_padded_length(long long total, int P, int multiple)
{
    if (total < 0 || P < 1 || multiple < 1) return -1;
    const long long step = static_cast<long long>(P) * multiple;   // < 2^62: no overflow
    const long long n = (total + step - 1) / step * step;          // total < 2^63 - step
    if (total > 0x7fffffffLL || n > 0x7fffffffLL) return -1;
    return n;
}

ra_status ra_check_status(ra_stream_t stream)
{
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return RA_ERR_CUDA;
    unsigned int* word = nullptr;
    ra_status st = status_word(&word);
    if (st != RA_OK) return st;
    unsigned int value = 0;
    if (cudaMemcpy(&value, word, sizeof(value), cudaMemcpyDeviceToHost) != cudaSuccess)
        return RA_ERR_CUDA;
    if (value == 0) return RA_OK;
    if (cudaMemset(word, 0, sizeof(value)) != cudaSuccess) return RA_ERR_CUDA;
    if (value & RA_STATUS_TIMEOUT) return RA_ERR_TIMEOUT;
    return (value & RA_STATUS_BOUNDS) ? RA_ERR_BOUNDS : RA_ERR_CUDA;
}

const char* ra_status_string(ra_status status)
{
    switch (status) {
    case RA_OK: return "ok";
    case RA_ERR_INVALID_ARG: return "invalid argument";
    case RA_ERR_UNSUPPORTED: return "unsupported head dim, element size or dtype";
    case RA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case RA_ERR_NOT_DIVISIBLE: return "sequence (or head) count not divisible by P";
    case RA_ERR_CUDA: return "CUDA error";
    case RA_ERR_TIMEOUT: return "a device-side wait ran out of time";
    case RA_ERR_BOUNDS: return "an index check of the debug build failed (access skipped)";
    }
    return "unknown status";
}

ra_status ra_probe_bounds_check(ra_stream_t stream)
{
    if (!ra::kCheckBounds) return RA_ERR_UNSUPPORTED;
    unsigned int* word = nullptr;
    ra_status st = status_word(&word);
    if (st != RA_OK) return st;
    return from_cuda(ra::launch_bounds_probe(word, reinterpret_cast<cudaStream_t>(stream)));
}

ra_status ra_probe_wait_timeout(unsigned long long timeout_ns, ra_stream_t stream)
{
    if (timeout_ns < 1 || timeout_ns > 1000000000ull) return RA_ERR_INVALID_ARG;
    unsigned int* word = nullptr;
    ra_status st = status_word(&word);
    if (st != RA_OK) return st;
    return from_cuda(ra::launch_wait_probe(word, timeout_ns, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
