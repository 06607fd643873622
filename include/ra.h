/*
 * ra.h - exact blockwise attention, log-sum-exp merge and a one-GPU ring simulation.
 *
 * C ABI of libra.so (CUDA, sm_103a).  Plain pointers and sizes; no C++ or torch types.
 *
 * Tensors
 *   ra_tensor describes a 4-D strided array [B, H, N, D] in device memory:
 *   data (device pointer), dtype, shape[4] = {B, H, N, D} and stride[4] in ELEMENTS.
 *   stride[3] must be 1 (rows of D contiguous).  The caller owns every buffer.
 *   q is [B, Hq, N, D]; k and v are [B, Hkv, N, D] with Hq % Hkv == 0; query head h
 *   reads key/value head h / (Hq / Hkv) (consecutive query heads share a KV head).
 *   o has q's shape and dtype.  lse is a contiguous float32 [B, Hq, N] array.
 *
 * Scale
 *   scale <= 0 selects 1/sqrt(D), the default of the pages' attention definition.
 *
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 * Argument errors are reported synchronously as a status; the message of the last
 * non-OK status of the calling thread is ra_last_error().  Device-side failures
 * (a pipeline wait that exceeded its time limit) are recorded in a device error word
 * that ra_check_device_error() reads.
 *
 * Paths (all on the GPU; there is no CPU path):
 *   bf16, D in {64, 128}, 16-byte aligned base and row strides: tcgen05 tensor-core
 *     kernel (TMA-fed shared-memory pipeline, S and O accumulated in tensor memory).
 *     Its persistent launches take their work items from one of 1024 work-counter pairs
 *     per device, in rotation, and each launch zeroes its pair again when it ends; so at
 *     most 1024 tensor-core launches of the library may be in flight on one device at a
 *     time (launches on one stream run in order; only launches on many streams at once
 *     could reach that).
 *   anything else with D <= 128 (float32 inputs, other head sizes, unaligned strides):
 *     a CUDA-core kernel computing in float32.
 *   D > 128: RA_ERR_UNSUPPORTED.
 */
#ifndef RA_H
#define RA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = 1, /* null pointer, bad shape/stride/dtype/size rule */
    RA_ERR_UNSUPPORTED = 2, /* well-formed but outside what the library implements */
    RA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    RA_ERR_TIMEOUT = 4,     /* a device-side pipeline wait exceeded its limit */
    RA_ERR_BOUNDS = 5       /* debug builds only: a device-side bounds check failed */
} ra_status;

typedef enum { RA_F32 = 0, RA_BF16 = 1 } ra_dtype;

typedef enum { RA_LAYOUT_CONTIG = 0, RA_LAYOUT_ZIGZAG = 1, RA_LAYOUT_STRIPED = 2 } ra_layout;

typedef struct {
    void *data;        /* device pointer */
    int32_t dtype;     /* ra_dtype */
    int32_t reserved;  /* must be 0 */
    int64_t shape[4];  /* B, H, N, D */
    int64_t stride[4]; /* in elements; stride[3] == 1 */
} ra_tensor;

/*
 * ra_attn_fwd - exact attention of one sequence block, O = softmax(scale Q K^T) V,
 * and the per-row natural-log LSE = ln sum_j exp(scale q_i . k_j).
 *
 * Defined by the standard attention formula of "Ring Attention explained"
 * (guijiagi.com), section "朴素 Attention 的显存墙", computed blockwise with the
 * online softmax of its section "在线 Softmax 算法" and the deferred normalisation of
 * "第12章 FlashAttention原理与实现" (FlashAttention-2 paragraph).  With causal != 0,
 * key j is visible to query i iff j <= i ("因果掩码处理": the diagonal block is
 * lower-triangular).  Any N >= 0 (ragged tails are masked); N == 0, B == 0 or
 * H == 0 is a no-op.
 *
 *   q, k, v  inputs as described above (read only)
 *   o        output [B, Hq, N, D], same dtype as q (written)
 *   lse      output float32 [B, Hq, N], contiguous (written)
 *   causal   0 or 1
 *   scale    softmax scale; <= 0 means 1/sqrt(D)
 *   stream   cudaStream_t
 * Errors: RA_ERR_INVALID_ARG (null pointers, shape or dtype mismatch, stride[3] != 1,
 *   NaN scale), RA_ERR_UNSUPPORTED (D > 128), RA_ERR_CUDA (launch failure).
 */
ra_status ra_attn_fwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v, ra_tensor *o,
                      float *lse, int causal, float scale, void *stream);

/*
 * ra_lse_merge - fold a block partial into a running partial, row by row:
 *   L       = ln(e^a + e^b)           with a = lse_acc[row], b = lse_blk[row]
 *   o_acc  <- e^(a-L) o_acc + e^(b-L) o_blk
 *   lse_acc <- L
 * This is `update_out_and_lse` of "序列并行与 Ring Attention：超长上下文训练技术解析"
 * (section "前向传播：ZigZag Ring FlashAttention"), evaluated in the max-shifted form
 * (same value; no overflow).  The identity partial is (o = 0, lse = -inf): a side with
 * lse = -inf contributes nothing, and two identities give the identity.
 *
 *   o_acc    [B, H, N, D] float32 (read and written)
 *   lse_acc  float32 [B, H, N] contiguous (read and written)
 *   o_blk    [B, H, N, D] float32 or bf16 (read)
 *   lse_blk  float32 [B, H, N] contiguous (read)
 * Errors: RA_ERR_INVALID_ARG (null pointers, shape mismatch, o_acc not float32,
 *   stride[3] != 1), RA_ERR_CUDA.
 */
ra_status ra_lse_merge(ra_tensor *o_acc, float *lse_acc, const ra_tensor *o_blk,
                       const float *lse_blk, void *stream);

/*
 * ra_ring_sim_workspace_bytes - an upper bound, valid for every call with this q, of the
 * device workspace ra_ring_sim_fwd needs for its float32 running output: B*Hq*N*D*4 bytes
 * when ring_size > 1, else 0.  Returns 0 on bad arguments.
 * ra_ring_sim_workspace_bytes_for gives the exact need of one call.
 */
size_t ra_ring_sim_workspace_bytes(const ra_tensor *q, int ring_size);

/*
 * ra_ring_sim_workspace_bytes_for - the device workspace ra_ring_sim_fwd needs for exactly
 * these arguments: 0 when ring_size == 1, and 0 when the call runs the fused ring (bf16,
 * D in {64, 128}, 16-byte aligned q, k, v, o; a contiguous or zigzag layout of at most
 * 128 chunks, or the striped layout with at most 128 ranks of whole 128-row tiles), whose
 * running result stays inside the kernel; otherwise B*Hq*N*D*4 bytes for the float32
 * running output of the per-step launches.  ra_ring_sim_fwd accepts a NULL workspace
 * exactly when this is 0.  Returns 0 on bad arguments (the call then reports them; the
 * message is in ra_last_error()).
 */
size_t ra_ring_sim_workspace_bytes_for(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                                       const ra_tensor *o, int ring_size, ra_layout layout, int causal);

/*
 * ra_ring_sim_fwd - ring attention over ring_size simulated ranks on one GPU.
 *
 * The sequence is split among the ranks ("Ring Attention" glossary page,
 * ultralytics.com, section on how ring attention works):
 *   RA_LAYOUT_CONTIG  rank r holds rows [r c, (r+1) c), c = N / ring_size
 *   RA_LAYOUT_ZIGZAG  2*ring_size chunks; rank r holds chunk r and chunk 2R-1-r
 *                     ("序列并行与 Ring Attention", section "2. ZigZag Ring Attention")
 *   RA_LAYOUT_STRIPED rank r holds positions r, r + R, r + 2R, ... (tokens spread evenly
 *                     over the ranks: Striped Attention, named on the glossary page for
 *                     balancing causal work)
 * At step s rank r holds the key/value block of rank (r - s) mod R; the step's
 * partial for each rank's query rows (causality on global positions, so later
 * blocks are skipped and the diagonal block masked) is merged into the rank's running
 * result.  Two executions:
 *   - bf16, D in {64, 128}, contiguous or zigzag layout with up to 128 chunks, or the
 *     striped layout with up to 128 ranks of whole 128-row tiles: one launch walks every
 *     step; each query block's running (max, sum, O) stays in the kernel across the step
 *     boundaries (the LSE merge of consecutive steps' partials is the online-softmax
 *     rescale), and each row is written once.
 *   - otherwise (float32, other D, other striped sizes): one launch per step covering
 *     every simulated rank, merging into a float32 running result in the workspace by the
 *     LSE merge above, inside the attention kernel's epilogue.
 * The result equals ra_attn_fwd on the whole sequence (up to rounding); inputs and
 * outputs are in natural sequence order; ring_size == 1 is ra_attn_fwd.
 *
 *   ring_size  >= 1; contig and striped need N % ring_size == 0, zigzag
 *              N % (2 ring_size) == 0
 *   layout     ra_layout
 *   workspace  device buffer of ra_ring_sim_workspace_bytes_for() bytes, 16-byte
 *              aligned (may be NULL when that is 0: the single pass and the fused ring
 *              need none); contents on entry are ignored; owned by the caller
 * Errors: as ra_attn_fwd, plus RA_ERR_INVALID_ARG for a bad ring size / layout /
 *   divisibility or a missing workspace.
 */
ra_status ra_ring_sim_fwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                          ra_tensor *o, float *lse, int ring_size, ra_layout layout, int causal,
                          float scale, void *workspace, void *stream);

/*
 * ra_attn_varlen_fwd - exact attention over a packed batch of variable-length sequences.
 *
 * Sequence i occupies rows [cu_seqlens[i], cu_seqlens[i+1]) of the packed axis; a row
 * attends only to keys of its own sequence (causal within it when causal != 0), the
 * block-diagonal mask of packed batches ("序列并行与 Ring Attention：超长上下文训练技术解析":
 * varlen FlashAttention over `cu_seqlens`, padding excluded by the attention mask;
 * "第12章 FlashAttention原理与实现": `flash_attn_varlen_func` for samples of different
 * lengths).  Rows outside every sequence (padding) get the identity, O = 0 and
 * LSE = -inf.
 *
 *   q, k, v    [1, Hq, total, D] / [1, Hkv, total, D] (B must be 1)
 *   o, lse     outputs as in ra_attn_fwd
 *   cu_seqlens HOST array of num_seqs + 1 non-decreasing offsets, cu_seqlens[num_seqs]
 *              <= total (read during the call only; empty sequences are allowed)
 * Errors: as ra_attn_fwd, plus RA_ERR_INVALID_ARG for B != 1 or bad cu_seqlens.
 */
ra_status ra_attn_varlen_fwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                             ra_tensor *o, float *lse, const int32_t *cu_seqlens, int num_seqs,
                             int causal, float scale, void *stream);

/*
 * ra_attn_bwd - gradients of ra_attn_fwd for the loss L = sum(dout * O).
 *
 * Recomputes P = exp(scale Q K^T - LSE) from the forward's LSE and follows the backward
 * of the `ring_attention_backward` listing of "Ring Attention 论文解析" over the whole key
 * axis: D = rowsum(dout * O), dV = P^T dout, dS = P * (dout V^T - D),
 * dQ = scale dS K, dK = scale dS^T Q (grouped query heads summed into their KV head).
 *
 *   q, k, v, o, lse  the forward's inputs and outputs (o and lse as ra_attn_fwd wrote them)
 *   dout             [B, Hq, N, D] gradient of O (q's dtype)
 *   dq               [B, Hq, N, D] (written); dk, dv [B, Hkv, N, D] (written)
 *   workspace        device buffer of ra_attn_bwd_workspace_bytes() bytes, 16-byte aligned
 * Errors: as ra_attn_fwd, plus RA_ERR_INVALID_ARG for gradient shape/dtype mismatches or a
 *   missing workspace.
 */
size_t ra_attn_bwd_workspace_bytes(const ra_tensor *q);
ra_status ra_attn_bwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v, const ra_tensor *o,
                      const float *lse, const ra_tensor *dout, ra_tensor *dq, ra_tensor *dk,
                      ra_tensor *dv, int causal, float scale, void *workspace, void *stream);

/*
 * ra_ring_sim_fwd_host - ra_ring_sim_fwd on HOST buffers (no counterpart in the pages:
 * the call a program makes when its tensors live in host memory).
 *
 * q, k, v, o and lse are host pointers (page-locked memory lets the copies run
 * asynchronously; pageable memory works but each copy then waits).  The tensors must be
 * contiguous [B, H, N, D]; lse is [B, Hq, N] float32.  The call stages through the
 * caller's device workspace and pipelines by groups of whole KV heads (up to 8; fewer
 * when the kernels dominate and a group's launch would not fill the GPU; when the copies
 * dominate and there are at least three KV heads per group, group sizes fall along the
 * pipeline), one launch per group over every batch: the next
 * group's q/k/v go in on one internal stream while the current group computes on
 * `stream`, and finished groups' o/lse come out on another, so both directions of the
 * host link overlap the kernels.  The call is ordered on `stream`: the host buffers may
 * be read or reused once `stream` has reached this point (e.g. after
 * cudaStreamSynchronize).  Calls for one device are serialised on the host while they
 * enqueue.
 *
 *   workspace  device buffer of ra_ring_sim_fwd_host_workspace_bytes(q, k, ring_size)
 *              bytes, 256-byte aligned, owned by the caller
 * Errors: as ra_ring_sim_fwd, plus RA_ERR_INVALID_ARG for non-contiguous tensors or a
 *   missing / small / misaligned workspace.
 */
size_t ra_ring_sim_fwd_host_workspace_bytes(const ra_tensor *q, const ra_tensor *k, int ring_size);
ra_status ra_ring_sim_fwd_host(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v, ra_tensor *o,
                               float *lse, int ring_size, ra_layout layout, int causal, float scale,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * ra_ring_sim_bwd - gradients of ra_ring_sim_fwd on the ring schedule of ring_size
 * simulated ranks, on one GPU.
 *
 * The `ring_attention_backward` listing of "Ring Attention 论文解析": at step s rank r
 * holds the key/value block of rank (r - s) mod R (the forward's rotation), recomputes
 * P = exp(scale Q K^T - LSE) of its queries against that block with the forward's LSE and
 * D = rowsum(dout * O), adds dS K to its own dQ, and returns the block's dK = scale dS^T Q
 * and dV = P^T dout to the block's rank, which sums them over the steps.  Each step
 * applies the forward's causal rule (skipped, diagonal or full blocks; the striped
 * interleave's offset).  bf16 with D in {64, 128} and a contiguous or zigzag layout of
 * up to 128 chunks, or the striped layout with up to 128 ranks of whole 128-row tiles:
 * one dQ launch walks each query chunk's partner blocks over all steps and one dK/dV
 * launch walks each key chunk's partner ranks, (j + s) mod R at step s (the reverse
 * ring), with both gradients kept in the kernels across steps.  Otherwise
 * one launch of each kernel per step covers every rank, and gradients that several steps
 * write are carried between steps in fp32 in the workspace.  The sum over steps is the
 * gradient of the whole sequence, so ring_size = 1 (any layout) is ra_attn_bwd.
 *
 *   q, k, v, o, lse  the forward's inputs and outputs (natural sequence order)
 *   dout             [B, Hq, N, D] gradient of O (q's dtype)
 *   dq               [B, Hq, N, D] (written); dk, dv [B, Hkv, N, D] (written)
 *   ring_size, layout  as ra_ring_sim_fwd (N divisible as it requires)
 *   workspace        device buffer of ra_ring_sim_bwd_workspace_bytes(q, k, ring_size)
 *                    bytes, 16-byte aligned, owned by the caller, overwritten
 * Errors: as ra_attn_bwd, plus the ring-size/layout checks of ra_ring_sim_fwd.
 */
size_t ra_ring_sim_bwd_workspace_bytes(const ra_tensor *q, const ra_tensor *k, int ring_size);
ra_status ra_ring_sim_bwd(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v, const ra_tensor *o,
                          const float *lse, const ra_tensor *dout, ra_tensor *dq, ra_tensor *dk, ra_tensor *dv,
                          int ring_size, ra_layout layout, int causal, float scale, void *workspace,
                          void *stream);

/*
 * ra_ulysses_all_to_all - the Ulysses sequence <-> head exchange of sp ranks, restated as a
 * layout transform of one GPU's memory ("序列并行与 Ring Attention：超长上下文训练技术解析",
 * section "1. Ulysses (All-to-All)": scatter the head axis, gather the sequence axis).
 *
 *   to_heads != 0: in  = sequence shards [sp, S/sp, H, D] (rank r holds positions
 *                        [r S/sp, (r+1) S/sp), all heads)
 *                  out = head shards     [sp, S, H/sp, D] (rank r holds heads
 *                        [r H/sp, (r+1) H/sp), whole sequence)
 *   to_heads == 0: the inverse (in = head shards, out = sequence shards).
 * Element strides are free (dim 3 contiguous); H % sp == 0.  The copy is exact.
 * Errors: RA_ERR_INVALID_ARG for mismatched shapes or dtypes, RA_ERR_CUDA.
 */
ra_status ra_ulysses_all_to_all(const ra_tensor *in, ra_tensor *out, int sp, int to_heads,
                                void *stream);

/*
 * ra_ring_sim_plan - host-only description of the ring schedule (no GPU work).
 * For step `step`, writes up to `cap` segments; each segment is 12 int64 values:
 *   q0, q1          query indices [q0, q1) of one chunk of one simulated rank
 *   k0a, k1a        first key index range [k0a, k1a)
 *   k0b, k1b        second key index range (k0b == k1b when absent)
 *   flags           bit 0: first partial of these rows, bit 1: last partial
 *   rank            the simulated rank
 *   q_rank, kv_rank, diag, rs
 *                   index i of the query chunk is sequence position i*rs + q_rank and
 *                   key index j is position j*rs + kv_rank; under causality key j is
 *                   visible to row i iff j + diag <= i (rs = ring_size for the striped
 *                   layout, else 1 with ranks and diag 0)
 * Returns the number of segments of that step (which may exceed cap), or -1 on bad
 * arguments.
 */
int64_t ra_ring_sim_plan(int64_t N, int ring_size, ra_layout layout, int causal, int step,
                         int64_t *segments, int64_t cap);

/*
 * ra_ring_sim_bwd_plan - host-only description of one step of ra_ring_sim_bwd (no GPU
 * work).  kind 0: the segments of the dQ kernel (fixed range = a query chunk, streamed
 * ranges = the key chunks of the block it holds); kind 1: the segments of the dK/dV
 * kernel (fixed range = a key chunk, streamed ranges = the query chunks of the rank that
 * holds it at this step).  Each segment is 10 int64 values:
 *   f0, f1          fixed index range
 *   s0a, s1a        first streamed index range
 *   s0b, s1b        second streamed index range (s0b == s1b when absent)
 *   f_rank, s_rank  striped layout: ranks of the fixed and streamed ranges (0 otherwise;
 *                   index i of rank r is sequence position i * ring_size + r)
 *   diag            under causality key c is visible to row i iff c + diag <= i
 *   flags           bit 0: no earlier step writes the fixed range's gradient,
 *                   bit 1: no later step does
 * Returns the number of segments (which may exceed cap), or -1 on bad arguments.
 */
int64_t ra_ring_sim_bwd_plan(int64_t N, int ring_size, ra_layout layout, int causal, int step, int kind,
                             int64_t *out, int64_t cap);

/*
 * ra_ring_sim_fwd_noalloc - ra_ring_sim_fwd for callers that cannot have device memory
 * allocated on their behalf: a framework whose memory pool owns the device, a
 * latency-critical loop where cudaMalloc/cudaFree would synchronise the device, or a
 * host application that gives a plugin only its input and output buffers.  The pages
 * have no counterpart; this is a property of the library, not of the method.
 *
 * Same arguments, result and errors as ra_ring_sim_fwd, without the workspace, and the
 * same schedule.  A call that runs the fused ring (ra_ring_sim_workspace_bytes_for() == 0:
 * bf16, D in {64, 128}, aligned, a layout the fused kernel walks) needs no scratch at all.
 * Otherwise the float32 running output lives in a fixed device array inside the library,
 * 8 Mi floats (32 MiB), which every GPU that loads the library holds until the process
 * exits.
 *   - Calls that need the array: B*Hq*N*D must be <= 8388608 and ring_size <= 64;
 *     larger ones get RA_ERR_UNSUPPORTED (use ra_ring_sim_fwd with a workspace).
 *   - The call allocates nothing: no cudaMalloc/cudaFree, no host heap on success.
 *   - The first call on a device that needs the array looks up its device address (once
 *     per device, with that device current).
 *   - Every such call shares the array and it keeps the last call's contents.  Nothing in
 *     it needs clearing: each row's first partial is written, never merged.  Calls that
 *     overlap on the GPU (different streams, or different host threads) race on it:
 *     serialise them.
 */
ra_status ra_ring_sim_fwd_noalloc(const ra_tensor *q, const ra_tensor *k, const ra_tensor *v,
                                  ra_tensor *o, float *lse, int ring_size, ra_layout layout,
                                  int causal, float scale, void *stream);

/*
 * ra_check_device_error - synchronise `stream`, then read and clear the device error
 * word of the current device.  RA_ERR_TIMEOUT if a kernel recorded a wait timeout,
 * RA_ERR_CUDA if the synchronisation failed, else RA_OK.
 */
ra_status ra_check_device_error(void *stream);

/*
 * ra_debug_set_wait_limit_ns - time limit of the kernels' pipeline waits (default 2e9 ns).
 * A wait that exceeds it records RA_ERR_TIMEOUT and the kernel winds down cleanly (its
 * copies and MMAs in flight complete, tensor memory is released) and returns.  The limit
 * is read after a few dozen blocking probes of the barrier, each of which the hardware
 * may suspend for a while, so it bounds long waits, not short ones.  Values < 0 restore
 * the default.  Diagnostic hook.
 *
 * ra_debug_set_producer_delay_ns - the tensor-core kernels' TMA producers pause this long
 * (at most 0.1 s; default 0) before their first copy.  With a short wait limit the
 * consumers' waits then run out for real: the timeout path can be tested on any input
 * without a fault or a hang.  Diagnostic hook.
 * Both settings are process-wide and apply to the calls made after them.
 */
void ra_debug_set_wait_limit_ns(int64_t ns);
void ra_debug_set_producer_delay_ns(int64_t ns);

/*
 * ra_debug_fail_next_launches - make the calling thread's next n kernel launches fail on
 * the host, before they reach the GPU: each reports RA_ERR_CUDA with a message that names
 * this hook, as a real launch failure would.  n <= 0 clears it.  Diagnostic hook, for
 * testing the callers' error paths without a GPU fault.
 */
void ra_debug_fail_next_launches(int n);

/*
 * ra_debug_time_launches - while enable != 0, each kernel launch of the calling thread is
 * bracketed by two CUDA events recorded on its stream, so that every kernel of a call is
 * timed on its own (the events also keep launches that would overlap - a ring step's tail
 * and the next launch - apart).  For profiling; costs two event records per launch.
 * ra_debug_launch_times - waits for the timed launches since the previous read, writes
 * up to `cap` durations in milliseconds (-1 where an event failed) and kernel names (each
 * NUL-terminated in a slot of name_len bytes; names may be NULL) in launch order, forgets
 * them, and returns how many there were (which may exceed cap).
 */
void ra_debug_time_launches(int enable);
int ra_debug_launch_times(float *ms, int cap, char *names, int name_len);

/*
 * ra_debug_work_counters_in_use - synchronise `stream`, then count the work-counter pairs
 * of the current device that are not zero.  Each tensor-core forward launch takes its work
 * items from one of 1024 counter pairs (in rotation) and its last block to finish zeroes
 * the pair again, also when the launch ends early on a wait timeout; so with no launch in
 * flight on the device this is 0.  -1 if the device or the copy fails.  Diagnostic hook.
 */
int ra_debug_work_counters_in_use(void *stream);

/*
 * ra_debug_host_group_bounds - the head groups ra_ring_sim_fwd_host would use for `hkv` KV
 * heads in `ng` groups (1 <= ng <= min(8, hkv)): writes ng + 1 boundaries (in KV heads,
 * 0 = out[0] < out[1] < ... < out[ng] = hkv) to `out` and returns ng, or -1 for arguments
 * out of range.  copy_bound != 0: the schedule used when the copies dominate (once
 * hkv >= 3 ng and ng >= 4, sizes in proportion to ng, ng - 1, ..., 1).  Host only;
 * diagnostic hook.
 */
int ra_debug_host_group_bounds(int64_t hkv, int ng, int copy_bound, int64_t *out);

/*
 * Debug builds.  Built with RA_DEBUG_BOUNDS defined (libra_debug.so, build.py
 * debug_bounds=True), the kernels check every tile coordinate and row index against its
 * tensor before a global-memory access; a failed check records RA_ERR_BOUNDS in the device
 * error word (read by ra_check_device_error) and skips the access instead of trapping (a
 * skipped tile load then ends in a bounded wait that times out).  Release builds compile
 * the checks away.
 *
 * ra_debug_bounds_checked - 1 in a debug build, else 0.
 * ra_debug_bounds_selftest - launch one block whose bounds check fails on purpose (no
 *   memory is accessed), so that ra_check_device_error returns RA_ERR_BOUNDS.
 *   RA_ERR_UNSUPPORTED in release builds.
 */
int ra_debug_bounds_checked(void);
ra_status ra_debug_bounds_selftest(void *stream);

/*
 * ra_debug_wait_selftest - launch one block that waits, bounded by `limit_ns`, on a
 * shared-memory barrier that nothing completes, then records RA_ERR_TIMEOUT in the
 * device error word.  Exercises the timeout path without touching any pipeline.
 */
ra_status ra_debug_wait_selftest(int64_t limit_ns, void *stream);

/* Message of the calling thread's last non-OK status ("" if none). */
const char *ra_last_error(void);

/* Number of kernel launches issued by the calling thread since the last reset. */
int64_t ra_launch_count(int reset);

/* Library version, 100 * major + minor. */
int ra_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RA_H */
