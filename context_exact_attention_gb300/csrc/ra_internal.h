// ra_internal.h -- host-side interface between the C ABI layer (api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "ring_attn.h"

namespace ra {

constexpr int kMaxDevices = 64;

// Raises a kernel's dynamic shared-memory limit the first time a device launches it.
// `done` is one flag per device (static storage: starts at zero).  Safe to call from
// several host threads at once: the flag is atomic, and the attribute call is
// idempotent, so two threads that both see the flag clear both make it harmlessly.
template <typename Kernel>
cudaError_t smem_limit_once(std::atomic<int>* done, int dev, Kernel kernel, int bytes)
{
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
}

// Everything one attention launch needs; validated by the ABI layer.
struct AttnArgs {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    float* lse;      // may be null
    int* trace;      // may be null
    int B, L, H, D, P, causal;
    int Hkv;                       // key/value heads (H for plain attention)
    int zigzag;                    // zigzag shard layout (causal)
    const int* cu_seqlens;         // packed sequences (device), or null
    int n_seqs;
    const int* schedule;           // packed sequences: unit orders (VarlenSchedLayout), or null
    // Ulysses head groups read from / written to the sequence-sharded buffers
    // [u_P][u_B][L/u_P][u_H][D] (0 = not used): B = u_P * u_B head-group batches of
    // H = u_H / u_P heads, ring P = 1; the tensor maps are then 5-D.
    int u_P, u_B, u_H;
    unsigned int* status;          // device status word
    unsigned long long timeout_ns; // limit of one bounded wait
    cudaStream_t stream;
};

// Packed-sequence schedule (ring_attn_varlen_schedule), in int32 entries: the forward's
// query-tile pairs, the backward's key tiles and query tiles, each a permutation of the
// units of one (batch, head) given by their natural index (shard * per-shard units +
// tile or pair), heaviest first; then scratch for the work counts of all three; then
// kCounters work counters of the persistent kernels (a claim counter and a finished-CTA
// counter per kernel: forward, backward key tiles, backward query tiles), zeroed by the
// schedule kernel and reset to zero by the last CTA of each launch that uses them.
constexpr int kCounters = 8;
struct VarlenSchedLayout {
    long long n_t, n_pair;           // 128-row tiles and tile pairs per shard
    long long fwd, bwd_k, bwd_q;     // offsets of the three orders
    long long scratch;               // offset of the scratch
    long long counters;              // offset of the work counters
    long long total;                 // total entries
};
inline VarlenSchedLayout varlen_sched_layout(int L, int P)
{
    VarlenSchedLayout s;
    const long long Ls = static_cast<long long>(L) / P;
    s.n_t = (Ls + 127) / 128;
    s.n_pair = (s.n_t + 1) / 2;
    s.fwd = 0;
    s.bwd_k = s.fwd + P * s.n_pair;
    s.bwd_q = s.bwd_k + P * s.n_t;
    s.scratch = s.bwd_q + P * s.n_t;
    s.counters = s.scratch + s.scratch;
    s.total = s.counters + kCounters;
    return s;
}
cudaError_t launch_varlen_schedule(const int* cu_seqlens, int n_seqs, int L, int P, int causal,
                                   int* schedule, unsigned int* status, cudaStream_t stream);

// bf16 tcgen05 kernel; tensor maps describe q, k, v as 4-D [B][L][H][D] with
// 64-element, 128-byte-swizzled boxes of 128 rows -- except that k has boxes of 64 rows
// when attn_bf16_pair_applies(a) (the pair-of-SMs kernel loads half a key block per CTA).
bool attn_bf16_pair_applies(const AttnArgs& a);
cudaError_t launch_attn_bf16(const AttnArgs& a, const CUtensorMap& tmap_q,
                             const CUtensorMap& tmap_k, const CUtensorMap& tmap_v);

// fp32 SIMT kernel.
cudaError_t launch_attn_f32(const AttnArgs& a);

// Backward (bf16): Dvec into the workspace, then the dK/dV and dQ kernels.
struct BwdArgs {
    const void* out;     // forward output O
    const void* dout;    // upstream gradient dO
    const float* lse;    // forward lse [B, L, H]
    float* dvec;         // workspace [B, L, H]
    void* dq;
    void* dk;
    void* dv;
    int B, L, H, D, P, causal;
    int Hkv;             // key/value heads (H % Hkv == 0); dk, dv are [B, L, Hkv, D]
    int zigzag;          // zigzag shard layout (causal; Hkv == H)
    const int* cu_seqlens;   // packed sequences (device; B == 1, Hkv == H), or null
    int n_seqs;
    const int* schedule;     // packed sequences: unit orders (VarlenSchedLayout), or null
    unsigned int* status;
    unsigned long long timeout_ns;
    cudaStream_t stream;
};
// tmap_k64, tmap_v64: k and v with 64-row boxes, required when bwd_dq_pair_applies(a) (the
// pair-of-SMs dQ kernel stages half a key block per CTA), else null.
cudaError_t launch_attn_bwd_bf16(const BwdArgs& a, const CUtensorMap& tmap_q,
                                 const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                 const CUtensorMap& tmap_do, const CUtensorMap* tmap_k64,
                                 const CUtensorMap* tmap_v64);
bool bwd_dq_pair_applies(const BwdArgs& a);

cudaError_t launch_merge(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                         void* o_out, float* lse_out, long long rows, int D, int elem_bytes,
                         unsigned int* status, cudaStream_t stream);

// dir = 0: seq2head, dir = 1: head2seq.
// Copy-engine path of the same transposes: seq_map is the 5-D view {D, H/P, P, L/P, P*B}
// of the sequence-sharded buffer with box {D, H/P, 1, R, 1} (encoded by the caller),
// head_side the head-sharded buffer.  Valid when ulysses_permute_tma_fits.
bool ulysses_permute_tma_fits(int H, int D, int P, int elem_bytes);
int ulysses_permute_tma_rows(int L, int H, int D, int P, int elem_bytes);
cudaError_t launch_ulysses_permute_tma(const CUtensorMap& seq_map, void* head_side, int B, int L,
                                       int H, int D, int P, int elem_bytes, int dir, int R,
                                       unsigned int* status, unsigned long long timeout_ns,
                                       cudaStream_t stream);

cudaError_t launch_ulysses_permute(const void* in, void* out, int B, int L, int H, int D, int P,
                                   int elem_bytes, int dir, unsigned int* status, cudaStream_t stream);

cudaError_t launch_wait_probe(unsigned int* status, unsigned long long timeout_ns,
                              cudaStream_t stream);

// Device address of the current device's status word (api.cu).
ra_status current_status_word(unsigned int** out);

// One thread whose index check fails (debug build): exercises RA_STATUS_BOUNDS.
cudaError_t launch_bounds_probe(unsigned int* status, cudaStream_t stream);

}  // namespace ra
