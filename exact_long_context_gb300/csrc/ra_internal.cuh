// ra_internal.cuh - launch parameters and device helpers shared by the attention kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ra.h"

namespace ra {

// One query chunk of one simulated rank against the key/value block it holds in a
// ring step.  Rows and keys are indices along the sequence axis as seen through a rank
// interleave of stride StepParams::rs: index i of the query chunk is sequence position
// i * rs + q_rank, index j of a key range is position j * rs + kv_rank (rs = 1 and
// ranks 0 for contiguous and zigzag layouts, rs = R for the striped layout).  Key ranges
// are disjoint and increasing; the second may be empty (k0[1] == k1[1]).  Under
// causality key index j is visible to row index i iff j + diag <= i (diag = 1 when the
// key rank follows the query rank in the interleave, else 0).
struct Seg {
    int32_t q0, q1;
    int32_t k0[2], k1[2];
    int32_t flags;
    int32_t rank;
    int32_t blk0;  // first work block of this segment (variable-length launches)
    int32_t q_rank, kv_rank;
    int32_t diag;
};

enum : int32_t { SEG_FIRST = 1, SEG_FINAL = 2 };

constexpr int kMaxSeg = 128;

// Everything one step launch needs.  Every segment of a launch has the same number
// of query rows, so a work block decodes to (segment, local block) arithmetically.
struct StepParams {
    const void *q, *k, *v;
    int64_t sq[3], sk[3], sv[3];  // strides (elements) of dims B, H, N
    void *o;
    int64_t so[3];
    float *lse;   // [B, Hq, N] contiguous; also the running LSE across steps
    float *oacc;  // [B, Hq, N, D] contiguous float32 running output (steps > 1)
    int32_t B, Hq, Hkv, N, D;
    int32_t in_bf16;   // q, k, v, o are bf16 (else float32)
    int32_t causal;
    float scale_log2;  // softmax scale * log2(e)
    int32_t nseg;
    int32_t blocks_per_seg;  // work blocks per segment
    int32_t rows_per_block;  // query rows per work block
    int32_t total_items;     // persistent kernels: work items in this launch
    int32_t chained;         // launched as a dependent of the previous ring step's kernel
    int32_t var_blocks;      // segments have different lengths: decode through Seg::blk0
    int32_t pair_items;      // tensor-core kernel: items are pairs of blocks (set at launch)
    int32_t prefer_pairs;    // host: a ring step (tails overlap the next step's launch)
    int32_t ring_fused;      // one launch walks every ring step: Seg = a query chunk of rank Seg::rank
    int32_t ring_R, ring_layout;  // fused ring: ring size, RA_LAYOUT_CONTIG (0), ZIGZAG (1) or STRIPED (2)
    int32_t rs;              // rank interleave stride of the sequence axis (1 unless striped)
    int32_t o_tma;           // tensor-core kernel: final O rows leave through bulk tensor stores
    int64_t wait_limit_ns;
    int64_t producer_delay_ns;  // diagnostic: the TMA producer pauses this long before its first copy
    int *err;  // device error word
    // tensor-core kernel: this launch's work counter pair (next item, CTAs finished), zero on
    // entry and reset to zero by the last CTA (required)
    int *sched;
    int32_t blocks_y;    // work blocks per head (set at launch)
    int32_t head_group;  // single-block items: query heads per group of consecutive items (0: all)
    Seg seg[kMaxSeg];
};

// Standalone LSE merge of a block partial into a running partial (see lse_merge.cu).
struct MergeParams {
    float *oacc;
    int64_t sa[3];
    float *lse_acc;
    const void *oblk;
    int64_t sb[3];
    const float *lse_blk;
    int32_t blk_bf16;
    int32_t H, N, D;
    int32_t vec;  // rows are 16-byte aligned (8 for bf16) and D % 4 == 0
    int32_t half_warp;  // vec, D <= 128 and bf16 rows 16-byte aligned: half a warp per row
    int64_t rows;
};

// Gradients of attention (see attn_bwd_simt.cu).
// One unit of backward work in a ring step: a fixed range (query rows for the dQ kernels,
// keys for the dK/dV kernels) of one rank against up to two streamed ranges of the
// partner rank, in the layout's index space (absolute positions for the contiguous and
// zigzag layouts; indices within a rank's interleave for the striped layout, where the
// position of index i of rank r is i * rs + r).  Under causality key c is visible to
// row i iff c + diag <= i.
struct BSeg {
    int32_t f0, f1;
    int32_t s0[2], s1[2];  // s0[1] == s1[1] when the second range is unused
    int32_t f_rank, s_rank;
    int32_t diag;
    int32_t flags;  // SEG_FIRST: no earlier step wrote the fixed range; SEG_FINAL: no later step will
    int32_t rank;   // fused ring: the rank owning the fixed range (its partners follow from it)
};
constexpr int kMaxBSeg = 128;

struct BwdParams {
    const void *q, *k, *v, *o, *dout;
    void *dq, *dk, *dv;
    int64_t sq[3], sk[3], sv[3], so[3], sdo[3], sdq[3], sdk[3], sdv[3];
    const float *lse;  // [B, Hq, N]
    float *dvec;       // [B, Hq, N] rowsum(dO * O)
    float *acc_q;      // [B, Hq, N, D] fp32 running dQ between ring steps (final units)
    float *acc_k, *acc_v;  // [B, Hkv, N, D] fp32 running dK, dV
    int32_t B, Hq, Hkv, N, D;
    int32_t bf16;
    int32_t causal;
    float scale, scale_log2;
    int32_t rs;    // rank interleave of the striped layout (1 otherwise)
    int32_t flen;  // length of every segment's fixed range
    int32_t nseg;
    int32_t ring_fused;           // one launch walks every ring step (striped: ranks of whole tiles)
    int32_t ring_R, ring_layout;  // fused ring: ring size, RA_LAYOUT_CONTIG (0), ZIGZAG (1) or STRIPED (2)
    int64_t producer_delay_ns;    // diagnostic: the TMA producer pauses this long before its first copy
    int *sched;                   // tensor-core kernels: work counter pair of this launch (required)
    int32_t single;               // one-segment launch: single-tile items, longest first
    int32_t head_group;           // single-tile items: units (heads) per group of consecutive items (0: one group)
    int32_t dkv_tma;              // dK/dV kernel: final rows leave through bulk tensor stores
    BSeg seg[kMaxBSeg];
};

// Ulysses all-to-all as a layout transform (see ulysses.cu).
struct UlyssesParams {
    const void *in;
    void *out;
    int64_t si[4], so[4];  // element strides of in / out (dims 0..3)
    int32_t sp, S, H, D;   // full sequence S, all heads H
    int32_t esize;         // 2 or 4 bytes
    int32_t to_heads;      // 1: seq shards -> head shards, 0: inverse
    int32_t vec;           // rows are 16-byte aligned and D * esize % 16 == 0
};

// Device error codes (first one wins).
enum : int { DERR_TIMEOUT = 1, DERR_BOUNDS = 2 };

__device__ __forceinline__ void record_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Bounds check of a tile coordinate or row index before a global-memory access:
// in_bounds(cond, err).  Debug builds (RA_DEBUG_BOUNDS defined, see build.py) record
// DERR_BOUNDS in the device error word when cond is false and yield false, and the caller
// skips the access (a skipped tile load then ends in a bounded wait that times out:
// nothing traps or hangs).  Release builds yield true without evaluating cond.
__device__ __forceinline__ bool bounds_check(bool ok, int *err) {
    if (!ok) record_error(err, DERR_BOUNDS);
    return ok;
}
#ifdef RA_DEBUG_BOUNDS
#define in_bounds(cond, err) ::ra::bounds_check((cond), (err))
constexpr bool kDebugBounds = true;
#else
#define in_bounds(cond, err) true
constexpr bool kDebugBounds = false;
#endif

// End of a CTA of a launch with a work counter pair: the last CTA to finish zeroes the pair
// for the launch that next uses it (every CTA has taken its last item number by then).
__device__ __forceinline__ void sched_finish(int *sched) {
    __threadfence();
    if (atomicAdd(&sched[1], 1) == (int)(gridDim.x * gridDim.y * gridDim.z) - 1) {
        atomicExch(&sched[0], 0);
        atomicExch(&sched[1], 0);
        __threadfence();
    }
}

// Diagnostic pause of a pipeline's producer before its first copy (0: none), so that the
// consumers' bounded waits run past a short limit and take the timeout path for real.
__device__ __forceinline__ void producer_delay(int64_t ns) {
    if (ns <= 0) return;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if ((int64_t)(t - t0) >= ns) return;
        __nanosleep(1000);
    }
}

// Decode a work-block index into (segment, local block).
// Equal-length segments: blocks are numbered round-robin over segments.
// Variable-length segments (sorted longest first by the host): segment si owns blocks
// [blk0, blk0 + its block count).
// Either way the local block counts down, so the last (under causality the heaviest)
// blocks of a segment are dispatched first.
__device__ __forceinline__ void decode_work(const StepParams &P, int w, int &si, int &lb) {
    if (!P.var_blocks) {
        const int round = w / P.nseg;
        si = w - round * P.nseg;
        lb = P.blocks_per_seg - 1 - round;
        return;
    }
    int lo = 0, hi = P.nseg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.seg[mid].blk0 <= w)
            lo = mid;
        else
            hi = mid - 1;
    }
    si = lo;
    const int nb = (P.seg[si].q1 - P.seg[si].q0 + P.rows_per_block - 1) / P.rows_per_block;
    lb = nb - 1 - (w - P.seg[si].blk0);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Per-row epilogue weights for folding a block partial with LSE `b` into the running
// partial with LSE `a` (natural logs): L = ln(e^a + e^b), w_a = e^(a-L), w_b = e^(b-L).
struct MergeW {
    float wa, wb, L;
};

__device__ __forceinline__ MergeW merge_weights(float a, float b) {
    MergeW m;
    if (a == -INFINITY) {
        m.wa = 0.f;
        m.wb = (b == -INFINITY) ? 0.f : 1.f;
        m.L = b;
        return m;
    }
    if (b == -INFINITY) {
        m.wa = 1.f;
        m.wb = 0.f;
        m.L = a;
        return m;
    }
    const float mx = fmaxf(a, b);
    const float L = mx + log1pf(expf(-fabsf(a - b)));
    m.wa = expf(a - L);
    m.wb = expf(b - L);
    m.L = L;
    return m;
}

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

}  // namespace ra
