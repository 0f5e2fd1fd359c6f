/*
 * ring_attn.h -- C ABI of libringattn.so: exact context-parallel attention on
 * one GB300 (sm_103a), with P virtual sequence shards living in one HBM.
 *
 * Common conventions
 * ------------------
 * - Every pointer argument named q, k, v, out, lse, o_*, in, trace is a DEVICE
 *   pointer owned by the caller; the library never allocates, frees or keeps
 *   them.  All calls are asynchronous on `stream` (NULL = the legacy default
 *   stream) and never synchronise the host, except ra_check_status().
 * - Sequence tensors are contiguous row-major [B, L, H, D] (batch, sequence,
 *   head, head dim), the layout of the verify script in the juejin.cn article
 *   on debugging a ring-attention library (section 三: batch, sequence, head, head dim).
 *   lse tensors are fp32 [B, L, H], natural logarithm (same article, section 五).
 * - Virtual shard r (0 <= r < P) is the token range [r*L/P, (r+1)*L/P); L must be
 *   divisible by P ("序列并行与 Ring Attention", section 6.4; "Finalize
 *   Guidelines for Ulysses based context parallel attention", section 四).
 * - Argument errors are detected on the host before anything is launched and
 *   reported through the return value; nothing is written in that case.
 *   Launch failures return RA_ERR_CUDA.  Kernels that give up waiting (a
 *   bounded wait ran out) record RA_ERR_TIMEOUT in a per-device status word
 *   that ra_check_status() reads and clears; they never trap.  A kernel that
 *   finds its dynamic shared memory too misaligned to lay out its tiles writes
 *   nothing and records an error that ra_check_status() reports as RA_ERR_CUDA.
 */
#ifndef RING_ATTN_H
#define RING_ATTN_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* ra_stream_t;

typedef enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, overlapping in/out, overflow */
    RA_ERR_UNSUPPORTED = 2,   /* head dim or dtype the kernels do not implement */
    RA_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    RA_ERR_NOT_DIVISIBLE = 4, /* L % P != 0, or H % P != 0 for the Ulysses transposes */
    RA_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
    RA_ERR_TIMEOUT = 6,       /* a kernel's bounded wait ran out (reported by ra_check_status) */
    RA_ERR_BOUNDS = 7         /* debug build only: an index check failed and its access was
                                 skipped (reported by ra_check_status) */
} ra_status;

typedef enum { RA_BF16 = 0, RA_F32 = 1 } ra_dtype;

/*
 * ring_attn_fwd -- bf16 exact attention forward over P virtual ring shards.
 *
 * Computes, for every batch b, head h and query row i,
 *   out[b,i,h,:] = sum_j softmax_j( q[b,i,h,:] . k[b,j,h,:] / sqrt(D) ) v[b,j,h,:]
 *   lse[b,i,h]   = ln sum_j exp( q[b,i,h,:] . k[b,j,h,:] / sqrt(D) )
 * ("序列并行与 Ring Attention", section 3.1), using the blockwise online-softmax
 * recurrence of section 3.2 with the ring schedule of section 3.3: the queries
 * of shard r meet the K/V of shard (r - t) mod P at step t = 0..P-1.  With
 * causal != 0 key j is visible to query i iff j <= i in GLOBAL positions, and
 * shards wholly in the future of shard r are skipped (section 3.4).
 *
 * q, k, v, out: device bf16 [B, L, H, D], 16-byte aligned; out must not overlap
 *               q, k or v.  D must be 64 or 128.
 * lse:          device fp32 [B, L, H] or NULL (not written).
 * Scores and the softmax run in fp32 on tensor-core accumulators; out is
 * rounded to bf16 (round to nearest even).  Repeated calls on the same inputs
 * give bit-identical results (no atomics in the reduction).
 * Limits: B, L, H, P >= 1; L % P == 0; B*L*H*D < 2^40; L < 2^31.
 */
ra_status ring_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                        int B, int L, int H, int D, int P, int causal, ra_stream_t stream);

/*
 * ring_attn_fwd_f32 -- the same operation on fp32 tensors, computed in fp32
 * (SIMT, no tensor cores), for checks at fp32 tolerance.  Any D with
 * 4 <= D <= 256 and D % 4 == 0.  Same layout, limits and errors as above.
 */
ra_status ring_attn_fwd_f32(const float* q, const float* k, const float* v, float* out,
                            float* lse, int B, int L, int H, int D, int P, int causal,
                            ra_stream_t stream);

/*
 * ring_attn_fwd_trace -- ring_attn_fwd (dtype RA_BF16) or ring_attn_fwd_f32
 * (RA_F32) that also records the schedule it ran: trace is a device int32
 * [P, P] array; trace[r*P + t] receives the source shard whose K/V the queries
 * of shard r met at ring step t, or -1 if that step was skipped as wholly
 * future ("序列并行与 Ring Attention", section 6.6: dump the K/V source of every
 * round).  Identical numerics to the untraced call.
 */
ra_status ring_attn_fwd_trace(const void* q, const void* k, const void* v, void* out, float* lse,
                              int B, int L, int H, int D, int P, int causal, ra_dtype dtype,
                              int* trace, ra_stream_t stream);

/*
 * ring_attn_fwd_gqa -- ring_attn_fwd (dtype RA_BF16) or ring_attn_fwd_f32
 * (RA_F32) with grouped key/value heads (GQA; MQA when H_kv == 1): q and out are
 * [B, L, H, D], k and v are [B, L, H_kv, D], and the H / H_kv consecutive query
 * heads h = g*(H/H_kv) .. (g+1)*(H/H_kv) - 1 all attend with key/value head g.
 * "序列并行与 Ring Attention" (sections 3.5 and 6.4) counts key/value heads apart
 * from query heads; the consecutive grouping is this library's reading.
 * H % H_kv != 0 returns RA_ERR_NOT_DIVISIBLE.  Otherwise as ring_attn_fwd.
 */
ra_status ring_attn_fwd_gqa(const void* q, const void* k, const void* v, void* out, float* lse,
                            int B, int L, int H, int H_kv, int D, int P, int causal,
                            ra_dtype dtype, ra_stream_t stream);

/*
 * ring_attn_fwd_zigzag -- causal ring attention (dtype RA_BF16 or RA_F32) over
 * the zigzag shard layout that balances causal work across shards
 * ("序列并行与 Ring Attention", section 3.4).  The sequence is cut into 2P
 * chunks of c = L/(2P) positions and virtual shard r holds chunk r followed by
 * chunk 2P-1-r: row i of q, k, v, out (and lse) sits at global position
 *   r*c + i'            for i' = i - r*L/P < c, and
 *   (2P-1-r)*c + i' - c otherwise,
 * and the causal rule compares those global positions.  The result is causal
 * attention of the sequence in position order, returned in the zigzag row order.
 * Every ring step now meets a shard with visible keys, and every shard does the
 * same amount of work.  trace, if not NULL, is filled as by ring_attn_fwd_trace.
 * Requires L % (2P) == 0 (RA_ERR_NOT_DIVISIBLE), and for bf16 c % 128 == 0
 * (RA_ERR_UNSUPPORTED).  Otherwise as ring_attn_fwd.
 */
ra_status ring_attn_fwd_zigzag(const void* q, const void* k, const void* v, void* out,
                               float* lse, int B, int L, int H, int D, int P, ra_dtype dtype,
                               int* trace, ra_stream_t stream);

/*
 * ring_attn_fwd_varlen -- ring attention (dtype RA_BF16 or RA_F32) over packed
 * variable-length sequences: q, k, v, out are [L, H, D] (one batch), lse [L, H],
 * and sequence g occupies rows [cu_seqlens[g], cu_seqlens[g+1]).  A query sees
 * only keys of its own sequence (causal: not after itself), so no sample attends
 * to another ("序列并行与 Ring Attention", section 6.5, packed sequences must
 * carry their boundaries).  The P virtual shards still split the packed rows
 * evenly (L % P == 0); a sequence may span shards.  Padding to a multiple of P:
 * add the padding rows as one more sequence and ignore its output (the
 * Ulysses guideline page's padded_seq_len rule, section 四/六).
 *
 * cu_seqlens: DEVICE int32 [n_seqs + 1] with cu_seqlens[0] == 0, non-decreasing,
 *             cu_seqlens[n_seqs] == L.  The kernels read it as given; other
 *             contents give undefined results (never out-of-bounds accesses).
 * A query row that sees no key (only with malformed cu_seqlens) gets 0 and -inf.
 */
ra_status ring_attn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                               float* lse, const int* cu_seqlens, int n_seqs, int L, int H, int D,
                               int P, int causal, ra_dtype dtype, int* trace, ra_stream_t stream);

/*
 * ra_padded_length -- the pad rule for packed sequences that do not fill a multiple
 * of P shards ("Finalize Guidelines for Ulysses based context parallel attention",
 * sections 四 and 六, padded_seq_len): the smallest length >= total that P shards of
 * a multiple of `multiple` rows each divide,
 *   ceil(total / (P * multiple)) * P * multiple,
 * e.g. 3000 tokens over P = 4 shards with multiple 8 -> 3008.  The caller appends
 * the padding rows to cu_seqlens as one more sequence and ignores its output.
 * Pure host arithmetic (no device, no stream).  Returns -1 for total < 0, P < 1,
 * multiple < 1, or a result above 2^31 - 1 (the longest L the kernels take).
 */
long long ra_padded_length(long long total, int P, int multiple);

/*
 * ring_attn_fwd_host -- ring_attn_fwd (bf16) on tensors in HOST memory, with the
 * host<->device copies overlapped with the attention (no counterpart on the pages:
 * an addition of this library for callers whose activations live on the host).
 *
 * The operation and the result are exactly those of ring_attn_fwd on the same
 * values (bit-identical: attention is independent per head, and each head goes
 * through the same kernel).  Heads are processed in groups of heads_per_group:
 * group g's q, k, v are copied to the device while group g-1 computes, and its
 * output is copied back while later groups compute.
 *
 * q_host, k_host, v_host, out_host: host bf16 [B, L, H, D]; lse_host: host fp32
 *     [B, L, H] or NULL.  Page-locked memory (cudaHostAlloc, torch pin_memory) is
 *     needed for the copies to overlap anything; pageable memory gives correct
 *     results with copies the runtime stages and serialises.  out_host and
 *     lse_host must not overlap the inputs.
 * workspace: device memory of at least
 *     ring_attn_fwd_host_workspace_bytes(B, L, H, D, heads_per_group) bytes,
 *     256-byte aligned, owned by the caller; no other work may use it until the
 *     call's work on `stream` has completed.  Contents need no initialisation.
 * heads_per_group: 1 <= heads_per_group <= H, H % heads_per_group == 0
 *     (RA_ERR_NOT_DIVISIBLE otherwise).  Smaller groups overlap more of the copies;
 *     each group is one kernel launch over B * heads_per_group heads.
 * Streams: the work starts after the caller's earlier work on `stream`, and later
 * work on `stream` (or cudaStreamSynchronize(stream)) sees out_host and lse_host
 * complete.  The library runs the copies and the groups' kernels on its own
 * streams (two copy streams and two compute streams per device, created on first
 * use and kept until exit); enqueueing holds a per-device lock.
 * Errors: as ring_attn_fwd, plus RA_ERR_INVALID_ARG for a short workspace and
 * RA_ERR_MISALIGNED for a workspace not 256-byte aligned.
 */
unsigned long long ring_attn_fwd_host_workspace_bytes(int B, int L, int H, int D,
                                                      int heads_per_group);
ra_status ring_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                             void* out_host, float* lse_host, void* workspace,
                             unsigned long long workspace_bytes, int B, int L, int H, int D, int P,
                             int causal, int heads_per_group, ra_stream_t stream);

/*
 * attn_merge_partials -- log-sum-exp merge of two partial attention results
 * over disjoint key sets (the `combine` of the juejin.cn ring-attention article, section 四):
 *   lse_out = ln(e^lse_a + e^lse_b)
 *   o_out   = o_a * e^(lse_a - lse_out) + o_b * e^(lse_b - lse_out)
 * A partial with lse = -inf (it saw no key) gets weight 0; if both are -inf,
 * o_out = 0 and lse_out = -inf.
 *
 * o_a, o_b, o_out: device [rows, D] of dtype (RA_BF16 or RA_F32), 16-byte
 *                  aligned; D*sizeof(dtype) must be a multiple of 16.
 * lse_a, lse_b, lse_out: device fp32 [rows].
 * o_out may be the same pointer as o_a or o_b and lse_out the same as lse_a or
 * lse_b (in-place merge); any other overlap is rejected.  Math in fp32; bf16
 * results are rounded to nearest even.
 */
ra_status attn_merge_partials(const void* o_a, const float* lse_a, const void* o_b,
                              const float* lse_b, void* o_out, float* lse_out, long long rows,
                              int D, ra_dtype dtype, ra_stream_t stream);

/*
 * ulysses_seq2head -- the Ulysses all-to-all as a layout transpose on one
 * device ("序列并行与 Ring Attention", section 3.5: [B, L/P, H, D] per rank ->
 * [B, L, H/P, D] per rank).
 *
 * in:  sequence-sharded buffer [P][B][L/P][H][D]: slice r is what rank r holds.
 * out: head-sharded buffer [P][B][L][H/P][D]: slice g is what rank g holds,
 *   out[g][b][r*L/P + l][hh][d] = in[r][b][l][g*H/P + hh][d].
 * elem_bytes: 2 or 4 (bit copy; values are never interpreted).  Requires
 * L % P == 0, H % P == 0, (D*elem_bytes) % 16 == 0, 16-byte aligned pointers,
 * and non-overlapping in/out.  The whole of `out` is a [P*B, L, H/P, D]
 * batch that ring_attn_fwd accepts directly (with P = 1).
 */
ra_status ulysses_seq2head(const void* in, void* out, int B, int L, int H, int D, int P,
                           int elem_bytes, ra_stream_t stream);

/* ulysses_head2seq -- the inverse transpose (head-sharded -> sequence-sharded):
 *   out[r][b][l][g*H/P + hh][d] = in[g][b][r*L/P + l][hh][d].
 * Same requirements as ulysses_seq2head. */
ra_status ulysses_head2seq(const void* in, void* out, int B, int L, int H, int D, int P,
                           int elem_bytes, ra_stream_t stream);

/*
 * ulysses_attention_fused -- the whole Ulysses step of "序列并行与 Ring Attention",
 * section 3.5 (all-to-all to head shards, attention over the full sequence for each
 * head group, all-to-all back) without materialising the head-sharded buffers: the
 * attention kernel's tensor maps address the sequence-sharded inputs directly, so head
 * group g's query tile of positions [l, l+128) is read from shard l / (L/P), rows
 * l % (L/P), heads g*H/P .. (g+1)*H/P - 1, and each output row is written back to its
 * sequence shard.  The result is bit-identical to ulysses_seq2head on q, k, v, then
 * ring_attn_fwd_gqa(B' = P*B, H' = H/P, H_kv' = H_kv/P, P = 1), then ulysses_head2seq.
 *
 * q, out:   device bf16 sequence-sharded [P][B][L/P][H][D];
 * k, v:     device bf16 [P][B][L/P][H_kv][D] (query head h reads key/value head
 *           h / (H / H_kv), as ring_attn_fwd_gqa);
 * lse:      device fp32 [P][B][L/P][H] or NULL;
 * causal:   0 / 1 on the global position r*L/P + l.
 * Requires L % P == 0, H % P == 0, H_kv % P == 0 (RA_ERR_NOT_DIVISIBLE), (L/P) % 128 == 0
 * and D in {64, 128} (RA_ERR_UNSUPPORTED); alignment and overlap as ring_attn_fwd.
 * (On several GPUs the all-to-all moves data between devices; with every shard in one
 * HBM it reduces to the addressing above.)
 */
ra_status ulysses_attention_fused(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int B, int L, int H, int H_kv, int D, int P,
                                  int causal, ra_stream_t stream);

/*
 * ring_attn_bwd_workspace_bytes -- bytes of device workspace ring_attn_bwd needs
 * for a [B, L, H] problem (one fp32 per query row); 0 for invalid sizes.
 */
unsigned long long ring_attn_bwd_workspace_bytes(int B, int L, int H);

/*
 * ring_attn_bwd -- gradients of ring_attn_fwd (bf16).  With S = q k^T / sqrt(D),
 * P = softmax(S) under the same visibility rule as the forward, and the upstream
 * gradient dout:
 *   dv = P^T dout,  dS = P o (dout v^T - rowsum(dout o out)),
 *   dq = dS k / sqrt(D),  dk = dS^T q / sqrt(D).
 * P is recomputed from the forward's lse rather than stored; each K/V block meets
 * the query shards in ring order (r = (s + t) mod P, shards before s skipped under
 * causal masking) and its dk, dv are written once, to the rows of the shard that
 * owns it ("序列并行与 Ring Attention", sections 3.3 and 6.2).
 *
 * q, k, v, out, dout: device bf16 [B, L, H, D] (out and lse as ring_attn_fwd
 *                     produced them for these q, k, v, P, causal);
 * lse:                device fp32 [B, L, H];
 * dq, dk, dv:         device bf16 [B, L, H, D] outputs, overlapping nothing;
 * workspace:          device scratch of at least ring_attn_bwd_workspace_bytes
 *                     (contents need no initialisation; overwritten).
 * D must be 64 or 128; all pointers 16-byte aligned.  Deterministic (no atomics).
 */
ra_status ring_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        void* workspace, unsigned long long workspace_bytes, int B, int L, int H,
                        int D, int P, int causal, ra_stream_t stream);

/*
 * ring_attn_bwd_gqa -- ring_attn_bwd with grouped key/value heads (the backward of
 * ring_attn_fwd_gqa): q, out, dout, dq are [B, L, H, D]; k, v, dk, dv are
 * [B, L, H_kv, D]; query head h reads key/value head h / (H / H_kv).  K/V head g is
 * used by the H / H_kv query heads of its group, so its gradients are the sums over
 * them: dk_g = sum over h in the group of dS_h^T q_h / sqrt(D), dv_g = sum of P_h^T dout_h
 * ("序列并行与 Ring Attention", sections 3.5 and 6.4 count key/value heads apart from query
 * heads; the chain rule through the shared head gives the sums).  H % H_kv != 0 returns
 * RA_ERR_NOT_DIVISIBLE.  The workspace is ring_attn_bwd_workspace_bytes(B, L, H).
 * Otherwise as ring_attn_bwd (deterministic, no atomics: each dk/dv row is written once by
 * the CTA that owns its key tile, after walking every query head of the group).
 */
ra_status ring_attn_bwd_gqa(const void* q, const void* k, const void* v, const void* out,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            void* workspace, unsigned long long workspace_bytes, int B, int L,
                            int H, int H_kv, int D, int P, int causal, ra_stream_t stream);

/*
 * ring_attn_bwd_zigzag -- gradients of ring_attn_fwd_zigzag (bf16, causal): the
 * backward of causal attention over the zigzag shard layout ("序列并行与 Ring
 * Attention", section 3.4: shard r holds chunks r and 2P-1-r of 2P chunks; the causal
 * rule compares global positions), with the exchange of sections 3.3 and 6.2: each
 * K/V tile meets the query tiles of every shard in ring order from its owner's side,
 * (s + t) mod P, and its dk, dv are written once to the owner's rows.
 *
 * q, k, v, out, dout, dq, dk, dv: device bf16 [B, L, H, D] in the zigzag row order
 * (row i of shard r at the global position ring_attn_fwd_zigzag states); lse: the
 * forward's fp32 [B, L, H].  Requires L % (2P) == 0 (RA_ERR_NOT_DIVISIBLE) and
 * L/(2P) % 128 == 0 (RA_ERR_UNSUPPORTED).  Workspace, alignment, D and errors as
 * ring_attn_bwd.  The result equals ring_attn_bwd of the position-ordered causal
 * problem with its rows permuted into the zigzag order.
 */
ra_status ring_attn_bwd_zigzag(const void* q, const void* k, const void* v, const void* out,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               void* workspace, unsigned long long workspace_bytes, int B, int L,
                               int H, int D, int P, ra_stream_t stream);

/*
 * ring_attn_bwd_varlen -- gradients of ring_attn_fwd_varlen (bf16): packed
 * variable-length sequences, where a query sees only keys of its own sequence
 * (causal: not after itself; "序列并行与 Ring Attention", section 6.5), so every
 * gradient row depends only on its own sequence.  q, k, v, out, dout, dq, dk, dv:
 * device bf16 [L, H, D]; lse: the forward's fp32 [L, H]; cu_seqlens: the forward's
 * DEVICE int32 [n_seqs + 1] (0, ..., L; non-decreasing).  The P virtual shards split
 * the packed rows evenly (L % P == 0); tiles are walked in ring order as in
 * ring_attn_bwd.  Workspace: ring_attn_bwd_workspace_bytes(1, L, H).  With malformed
 * cu_seqlens the results are undefined, but every access stays in bounds.  Alignment,
 * D and errors as ring_attn_bwd.
 */
ra_status ring_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* out,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               void* workspace, unsigned long long workspace_bytes,
                               const int* cu_seqlens, int n_seqs, int L, int H, int D, int P,
                               int causal, ra_stream_t stream);

/*
 * ring_attn_bwd_noalloc -- ring_attn_bwd for callers that cannot allocate device
 * memory (no counterpart on the pages: an addition of this library).
 *
 * Same operation, arguments, layout and errors as ring_attn_bwd, minus the
 * workspace: it uses a fixed array compiled into the library instead, so it
 * never calls cudaMalloc, cudaFree or any other allocating routine.  Meant for
 * code that is handed only its tensors (plugins), runs inside a runtime that owns
 * all device memory, or must not allocate after warm-up.
 *
 * Limits and sharing:
 * - B*L*H must not exceed RA_BWD_NOALLOC_MAX_ROWS; larger problems return
 *   RA_ERR_INVALID_ARG without launching anything (use ring_attn_bwd for them).
 * - The array holds 4 MiB on every GPU that loads the library, until exit.  It
 *   comes into being when the CUDA runtime loads the library's module on a
 *   device: at context creation under CUDA_MODULE_LOADING=EAGER, otherwise (lazy
 *   loading, the default) during the first call on that device.  A caller that
 *   must not allocate after some point should make one call on each device
 *   before it.
 * - Every call looks up the array's device address with the device current (a
 *   table lookup once the module is loaded), so a device reset leaves no stale
 *   address behind.
 * - All calls on a device share the array; calls whose GPU work overlaps (for
 *   example on different streams) race and must be ordered by the caller.
 *   Nothing in it needs clearing: each call writes every row before reading it.
 */
#define RA_BWD_NOALLOC_MAX_ROWS 1048576ull
ra_status ring_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                int B, int L, int H, int D, int P, int causal, ra_stream_t stream);

/*
 * Shard layouts of the general entry points below.
 *   RA_LAYOUT_CONTIGUOUS  shard r holds positions [r L/P, (r+1) L/P) (ring_attn_fwd);
 *   RA_LAYOUT_ZIGZAG      shard r holds chunks r and 2P-1-r of 2P chunks
 *                         (ring_attn_fwd_zigzag; causal only);
 *   RA_LAYOUT_PACKED      packed variable-length sequences over contiguous shards,
 *                         boundaries in cu_seqlens (ring_attn_fwd_varlen; B == 1).
 */
typedef enum { RA_LAYOUT_CONTIGUOUS = 0, RA_LAYOUT_ZIGZAG = 1, RA_LAYOUT_PACKED = 2 } ra_layout;

/*
 * Problem description of ring_attn_fwd_ex / ring_attn_bwd_ex: every option of the
 * specialised entry points in one place, so that they combine -- grouped key/value
 * heads with the zigzag or the packed layout in particular (a grouped-head model
 * trained with zigzag ring shards or packed samples needs both at once).
 *   B, L, H, D, P  as ring_attn_fwd; H_kv key/value heads (H % H_kv == 0; H_kv == H
 *                  for plain attention), query head h reading head h / (H / H_kv);
 *   causal         0 / 1 (RA_LAYOUT_ZIGZAG requires 1: RA_ERR_UNSUPPORTED otherwise);
 *   layout         one of ra_layout;
 *   cu_seqlens     RA_LAYOUT_PACKED only (else NULL): device int32 [n_seqs + 1], as
 *                  ring_attn_fwd_varlen takes it;
 *   dtype          RA_BF16 or RA_F32 for the forward, RA_BF16 for the backward;
 *   schedule       RA_LAYOUT_PACKED only (else NULL): NULL, or the device array that
 *                  ring_attn_varlen_schedule wrote for the same cu_seqlens, L and P
 *                  (at least ring_attn_varlen_schedule_bytes(L, P) bytes: the kernels
 *                  read its entries by unit index, and the descriptor carries no size
 *                  to check).  It sets only which work unit runs when (heaviest first
 *                  instead of position order, and with it the forward runs one
 *                  persistent CTA per SM that claims units from a counter): the
 *                  results are the same bits either way.  Other contents of an array
 *                  of that size give undefined results, never out-of-bounds accesses.
 *                  The forward writes that work counter (the array's last entries):
 *                  it zeroes it in stream order before its kernel, so the counter's
 *                  previous contents do not matter, but calls that share one
 *                  schedule array must not overlap on the GPU (order them on one
 *                  stream).
 * The descriptor is read during the call only.
 */
typedef struct {
    int B, L, H, H_kv, D, P;
    int causal;
    ra_layout layout;
    const int* cu_seqlens;
    int n_seqs;
    ra_dtype dtype;
    const int* schedule;
} ra_attn_desc;

/*
 * ring_attn_varlen_schedule_bytes -- device bytes ring_attn_varlen_schedule writes for
 * L packed rows over P shards (0 when L < 1, P < 1 or L % P != 0): with n_t = ceil(L/P
 * / 128) tiles and n_pair = ceil(n_t / 2) tile pairs per shard,
 * 4 * (2 * P * (n_pair + 2 * n_t) + 8).
 */
unsigned long long ring_attn_varlen_schedule_bytes(int L, int P);

/*
 * ring_attn_varlen_schedule -- the order, heaviest first, in which the packed-layout
 * kernels of ring_attn_fwd_ex / ring_attn_bwd_ex take their work units (no counterpart
 * on the pages: an addition of this library).
 *
 * With packed sequences (section 6.5 of "序列并行与 Ring Attention") the work of a unit
 * -- the key tiles a query tile sees, or the query tiles that see a key tile -- grows
 * with the tile's offset inside its sequence, which only cu_seqlens tells.  Without a
 * schedule the kernels take units in position order, which can leave the heaviest ones
 * for the end of the grid while most SMs idle.  This call launches one CTA on `stream`
 * that counts each unit's tiles from cu_seqlens (same visibility rule as the kernels:
 * own sequence, causal or not) and writes three orders, heaviest first and ties in
 * position order: the forward's query-tile pairs, the backward's key tiles and its
 * query tiles.  Pass the array as ra_attn_desc.schedule with the same cu_seqlens, L and
 * P (a schedule made for the other causal flag is valid but less balanced).  It depends
 * only on these arguments, so one schedule serves every head, layer and the backward of
 * a batch.
 *
 * cu_seqlens: DEVICE int32 [n_seqs + 1], as ring_attn_fwd_varlen takes it (malformed
 *             contents give a poor order, never out-of-bounds accesses).
 * schedule:   DEVICE memory of at least ring_attn_varlen_schedule_bytes(L, P) bytes,
 *             4-byte aligned, owned by the caller; written by the launched kernel, so
 *             read it only in work ordered after it on the device.  Layout (int32):
 *             the three orders, a scratch area of the same size, then eight work
 *             counters of the persistent kernels that use the schedule.
 * Errors: RA_ERR_INVALID_ARG (NULL pointer, n_seqs < 1, L < 1, P < 1, P > L, short
 * schedule), RA_ERR_NOT_DIVISIBLE (L % P != 0), RA_ERR_MISALIGNED, RA_ERR_CUDA.
 */
ra_status ring_attn_varlen_schedule(const int* cu_seqlens, int n_seqs, int L, int P, int causal,
                                    int* schedule, unsigned long long schedule_bytes,
                                    ra_stream_t stream);

/*
 * ring_attn_fwd_ex -- the forward for any combination of the options in *desc: the
 * operation of ring_attn_fwd ("序列并行与 Ring Attention", sections 3.1-3.4) with the
 * key/value head grouping of ring_attn_fwd_gqa (sections 3.5, 6.4), the zigzag layout
 * of ring_attn_fwd_zigzag (section 3.4) or the packed sequences of
 * ring_attn_fwd_varlen (section 6.5).  q, out: [B, L, H, D]; k, v: [B, L, H_kv, D];
 * lse [B, L, H] or NULL; trace [P, P] or NULL (as ring_attn_fwd_trace).  Argument
 * checks and errors: those of the specialised entry point of the same options, plus
 * RA_ERR_INVALID_ARG for a NULL descriptor, an unknown layout, cu_seqlens or schedule
 * with a non-packed layout or B != 1 with the packed one, and RA_ERR_MISALIGNED for a
 * schedule not 4-byte aligned.  With the options of a specialised
 * entry point it launches the same kernel on the same arguments (same bits).
 */
ra_status ring_attn_fwd_ex(const ra_attn_desc* desc, const void* q, const void* k, const void* v,
                           void* out, float* lse, int* trace, ra_stream_t stream);

/*
 * ring_attn_bwd_ex -- the backward of ring_attn_fwd_ex (bf16) for the same *desc:
 * the operation of ring_attn_bwd (sections 3.3 and 6.2) under the descriptor's
 * visibility rule and head grouping.  q, out, dout, dq: [B, L, H, D]; k, v, dk, dv:
 * [B, L, H_kv, D], each key/value head's gradients summed over its query heads (as
 * ring_attn_bwd_gqa); lse: the forward's [B, L, H]; workspace of at least
 * ring_attn_bwd_workspace_bytes(B, L, H).  Deterministic (no atomics).  Checks and
 * errors as ring_attn_fwd_ex and ring_attn_bwd; dtype other than RA_BF16 returns
 * RA_ERR_UNSUPPORTED.
 */
ra_status ring_attn_bwd_ex(const ra_attn_desc* desc, const void* q, const void* k, const void* v,
                           const void* out, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* workspace, unsigned long long workspace_bytes,
                           ra_stream_t stream);

/*
 * ra_check_status -- synchronise `stream`, then read and clear the status word
 * of the current device.  Returns RA_ERR_TIMEOUT if a kernel gave up on a
 * bounded wait since the last check, RA_ERR_BOUNDS (debug build) if an index
 * check failed, RA_ERR_CUDA if the stream reports an error or a kernel could not
 * lay out its shared memory, RA_OK otherwise.
 *
 * The debug build.  The library is also built as libringattn_debug.so with the
 * same entry points, in which every global load and store that a kernel
 * addresses by a computed index is first checked against the extent of its
 * tensor (as the arguments of the call define it); a failed check records
 * RA_ERR_BOUNDS and skips the access (a load yields 0) instead of touching
 * memory outside the tensor.  Loads by TMA tensor maps are bounded by the maps
 * in hardware and need no check.  Results are the same bits as the normal
 * build's.  No page has a counterpart: it stands in for a memory checker.
 */
ra_status ra_check_status(ra_stream_t stream);

/*
 * ra_probe_bounds_check -- exercises the debug build's index check without
 * touching memory outside any buffer: launches one thread that checks an index
 * one past the end of a one-element extent and, only if the check passed, writes
 * a word inside the library.  In the debug build the check fails, the write is
 * skipped and ra_check_status then returns RA_ERR_BOUNDS.  The normal build has
 * no checks and returns RA_ERR_UNSUPPORTED without launching anything.
 */
ra_status ra_probe_bounds_check(ra_stream_t stream);

/* Static English text for a status code (never NULL). */
const char* ra_status_string(ra_status status);

/*
 * ra_probe_wait_timeout -- launch one CTA that waits on a shared-memory
 * barrier nothing will ever complete, with a limit of timeout_ns nanoseconds
 * (1 .. 10^9).  The wait runs out, the kernel records RA_ERR_TIMEOUT in the
 * status word and returns normally.  Exercises the give-up path that every
 * kernel's waits share, without faulting or hanging the device.
 */
ra_status ra_probe_wait_timeout(unsigned long long timeout_ns, ra_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RING_ATTN_H */
