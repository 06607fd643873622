// attn_tc.cu - exact attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA owns a block of 256 query rows of one (batch, head) - two 128-row halves -
// and streams the key/value tiles of its ring-step segment through shared memory.
//
//   warp 0        TMA producer: decodes each work item once and hands it to the other
//                 roles through a ring in shared memory; Q halves once per item, then
//                 (V_t, K_t+1) stages into a ring of buffer pairs
//   warp 1        MMA issuer (one lane) and tensor-memory owner:
//                   S_h = Q_h K_t^T      (tcgen05.mma, A and B from shared memory)
//                   O_h += P_h V_t       (tcgen05.mma, A = P from tensor memory)
//   warps 4-7     softmax of half 0, one thread per query row, and its epilogue
//   warps 8-11    softmax of half 1
//
// Outside the fused ring a causal item walks its key tiles last first: half 0 sits out
// the first tile, the halves start staggered and end on the same tile.
//
// Tensor memory (512 columns x 128 lanes x 32 bit): S_0 | S_1 | O_0 | O_1.  The bf16
// P_h overwrites the first 64 columns of S_h once the softmax threads hold S_h in
// registers; the next S_h is issued after the P_h V MMA, and tcgen05 MMAs of one
// thread run in issue order.
//
// The arithmetic per query row is the online softmax of "Ring Attention explained"
// (guijiagi.com), section "在线 Softmax 算法" - running max, running sum, rescaled
// unnormalised output - in log2 units (scale * log2 e folded into one FFMA before
// exp2), with the normalisation deferred to the end ("第12章 FlashAttention原理与实现",
// FlashAttention-2 paragraph).  The running max is only moved when a tile's max
// exceeds it by more than 2^8; the final O / l and LSE are the same quantities for
// any reference value, and this skips most rescales of O.
//
// Causality is decided per 128x128 tile on global positions: tiles entirely after
// the half's last row are never issued, tiles that straddle the diagonal or a key
// range end are masked element-wise (key j visible to row i iff j <= i: the block
// classes of the `ring_attention_causal_step` listing of "Ring Attention 论文解析").
//
// Epilogue (per row): O / l and LSE = ln sum exp, then, by segment flags, a direct
// write, or the log-sum-exp merge of the Twinkle page's `update_out_and_lse` into the
// float32 running output - so a ring step's partial never goes to HBM unnormalised.
// Final bf16 rows go out through per-warp shared-memory buffers and bulk tensor stores.
//
// Every mbarrier wait is bounded (globaltimer).  On a timeout the CTA records
// DERR_TIMEOUT in the device error word, every role stops, waits (bounded) for its
// own copies and MMAs in flight, and the tensor memory is released before exit.
#include <cuda.h>
#include <stddef.h>
#include <string.h>

#include <algorithm>

#include "tc_common.cuh"

namespace ra {
namespace tc {

constexpr int BM = 128;  // query rows per half (MMA M)
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;      // log2 units


template <int HD>
struct Cfg {
    static constexpr int SLABS = HD / 64;          // 128-byte column slabs per tile row
    static constexpr int TILE_BYTES = 128 * HD * 2;  // one Q half or one K/V tile (bf16)
    static constexpr int SLAB_BYTES = 128 * 128;     // 128 rows x 128 bytes
    static constexpr int NSLOT = (HD == 128) ? 4 : 8;  // tile buffers
    static constexpr int NSTAGE = NSLOT / 2;            // a stage = (V_t, K_t+1) buffer pair
    static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 256 + HD;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int STAGE_BYTES = 8 * 4096;  // O staging: 2 x (32 rows x 32 columns) per softmax warp
    static constexpr int BAR_BYTES = 1024;
    static constexpr int SMEM_BYTES = 1024 + (2 + NSLOT) * TILE_BYTES + STAGE_BYTES + BAR_BYTES;
};

struct Bars {
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t s_full[2];
    uint64_t it_full[4], it_empty[4];  // decoded-item ring: producer -> MMA issuer, softmax warps
    int32_t it_info[4][24];            // a decoded Item (nmax < 0: no more items)
    uint64_t o_full[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
    uint32_t p_count[2];  // P_h tiles published by the softmax warps (4 per tile)
};
static_assert(sizeof(Bars) <= 1024, "barrier block");

// Register split between warpgroups (launch: 168 per thread x 384 threads = 64512).
// Warpgroup 0 (TMA + MMA warps) gives back to 88, the two softmax warpgroups take 208:
// 88 * 128 + 208 * 256 = 64512.  (setmaxnreg needs the waits inlined: no calls.)
constexpr uint32_t kRegsControl = 88;
constexpr uint32_t kRegsSoftmax = 208;
static_assert(kRegsControl * 128 + kRegsSoftmax * 256 <= 168 * 384, "register split");

template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- tile bookkeeping

struct KTiles {
    int k0[2], k1[2];
    int nt0, ntot;
    __device__ __forceinline__ int start(int t) const {
        return t < nt0 ? k0[0] + BN * t : k0[1] + BN * (t - nt0);
    }
    __device__ __forceinline__ int range_end(int t) const { return t < nt0 ? k1[0] : k1[1]; }
    // Number of leading tiles whose first key is <= last_row (the tiles some row
    // <= last_row can see under causality).
    __device__ __forceinline__ int visible_prefix(int last_row) const {
        int c = 0;
        if (last_row >= k0[0]) c += min(nt0, (last_row - k0[0]) / BN + 1);
        if (ntot > nt0 && last_row >= k0[1]) c += min(ntot - nt0, (last_row - k0[1]) / BN + 1);
        return c;
    }
};

// ---------------------------------------------------------------- work items

// One work item: 256 query rows (two 128-row halves) of one (batch, head) against the
// key tiles of one segment.  Every role decodes the same items in the same order.
struct __align__(16) Item {
    int b, h, hk;
    int q_rank, kv_rank, diag;
    int qrow0, q1;
    int flags;
    int rank;   // the query chunk's rank (fused ring: the key ranges of every step follow from it)
    int nh[2];  // key tiles each half takes part in
    int nmax;   // key tiles of the item (T)
    int T0;     // tiles of the first step (the only one with a diagonal range)
    int skip0;  // the one tile half 0 sits out, or -1 (-2: the first tile of every step)
    int tps;    // fused striped ring: tiles per step (every step the same), else 0
    int rev;    // the first `rev` tiles are walked last key tile first (0: in key order)
    KTiles kt;  // the first step's key ranges
    // key tile of the item's t-th tile
    __device__ __forceinline__ int tile(int t) const { return t < rev ? rev - 1 - t : t; }
    // Half 1 (the later rows) takes part in every tile; half 0 in every tile but the last
    // of the first step when that tile starts past its last row.
    __device__ __forceinline__ bool part(int hh, int t) const {
        return hh ? nh[1] > 0 : (nh[0] > 0 && t != skip0);
    }
    __device__ __forceinline__ int last(int hh) const { return (!hh && skip0 == nmax - 1) ? nmax - 2 : nmax - 1; }
};

// What the MMA issuer needs of an item (handed over by the producer through shared memory).
struct MItem {
    int nh[2], nmax, skip0, tps;
    __device__ __forceinline__ bool part(int hh, int t) const {
        return hh ? nh[1] > 0 : (nh[0] > 0 && t != skip0);
    }
    __device__ __forceinline__ int last(int hh) const { return (!hh && skip0 == nmax - 1) ? nmax - 2 : nmax - 1; }
};
constexpr int kItemRing = 4;  // decoded items in flight from the producer to the other roles
constexpr uint32_t kItemReaders = 9;  // the MMA thread and one lane per softmax warp
static_assert(sizeof(Bars::it_info) / sizeof(Bars::it_info[0]) == kItemRing, "item ring");
static_assert(sizeof(Item) <= sizeof(Bars::it_info[0]) && sizeof(Item) % 16 == 0, "item record");
static_assert(offsetof(Bars, it_info) % 16 == 0, "16-byte item records");

__device__ __forceinline__ void item_store(int32_t *dst, const Item &it) {
    const int4 *src = reinterpret_cast<const int4 *>(&it);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(Item) / 16); ++i) reinterpret_cast<int4 *>(dst)[i] = src[i];
}
__device__ __forceinline__ void item_load(const int32_t *src, Item &it) {
    int4 *dst = reinterpret_cast<int4 *>(&it);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(Item) / 16); ++i) dst[i] = reinterpret_cast<const int4 *>(src)[i];
}

// Fused ring (contiguous or zigzag layout): the key ranges rank r's query chunk ending at
// q1 sees at step s, those of rank (r - s) mod R, with the forward's causal rule (a range
// starting after the chunk's last row is skipped).  Only step 0, the rank's own block, can
// hold a diagonal range, and it is that step's last.
__device__ __forceinline__ int ring_ranges(const StepParams &P, int r, int q1, int s, int &a0, int &b0,
                                           int &a1, int &b1) {
    const int R = P.ring_R;
    const int j = ((r - s) % R + R) % R;
    int ca0, cb0, ca1 = 0, cb1 = 0, nc;
    if (P.ring_layout == 0) {
        const int c = P.N / R;
        ca0 = j * c;
        cb0 = ca0 + c;
        nc = 1;
    } else {
        const int h = P.N / (2 * R);
        ca0 = j * h;
        cb0 = ca0 + h;
        ca1 = (2 * R - 1 - j) * h;
        cb1 = ca1 + h;
        nc = 2;
    }
    int n = 0;
    a0 = b0 = a1 = b1 = 0;
    for (int i = 0; i < nc; ++i) {
        const int ca = i ? ca1 : ca0, cb = i ? cb1 : cb0;
        if (cb <= ca || (P.causal && ca > q1 - 1)) continue;
        if (n == 0) {
            a0 = ca;
            b0 = cb;
        } else {
            a1 = ca;
            b1 = cb;
        }
        ++n;
    }
    return n;
}

// Fused ring, striped layout: the keys of step s in the rank-local index space.  At step
// s rank r holds rank j = (r - s) mod R's keys; under causality row i of rank r sees key
// index k of rank j iff k + [j > r] <= i (the interleave puts rank j's k-th position
// after rank r's k-th exactly when j > r), so rows ending before qend see [0, min(c,
// qend - [j > r])).  Every step is a causal prefix with its own diagonal offset d.
__device__ __forceinline__ void striped_range(const StepParams &P, int r, int qend, int s, int &end, int &j, int &d) {
    const int R = P.ring_R, c = P.N / R;
    j = ((r - s) % R + R) % R;
    d = (P.causal && j > r) ? 1 : 0;
    end = P.causal ? min(c, qend - d) : c;
}

// Walk of a fused striped item: step s, tile u of the step's tps tiles, each step's
// tiles last key tile first (half 0 then sits out the first tile of each step, as an
// item outside the fused ring sits out its first).
struct StripeWalk {
    int s, u, j, d, end;
    __device__ __forceinline__ int start(int tps) const { return (tps - 1 - u) * BN; }
};
__device__ __forceinline__ void stripe_begin(const StepParams &P, const Item &it, StripeWalk &w) {
    w.s = 0;
    w.u = 0;
    striped_range(P, it.rank, min(it.qrow0 + 2 * BM, it.q1), 0, w.end, w.j, w.d);
}
__device__ __forceinline__ void stripe_next(const StepParams &P, const Item &it, StripeWalk &w) {
    if (++w.u < it.tps) return;
    w.u = 0;
    ++w.s;
    striped_range(P, it.rank, min(it.qrow0 + 2 * BM, it.q1), w.s, w.end, w.j, w.d);
}

// Whether half hh takes part in tile t, given the tile's position in its step (MODE 2, the
// fused striped ring: half 0 sits out each step's first tile; the callers count the
// position, since a division per test would sit between the MMA thread's products), and
// its last tile.
template <int MODE, class I>
__device__ __forceinline__ bool part_pos(const I &it, int hh, int t, int pos) {
    if constexpr (MODE == 2)
        return hh ? it.nh[1] > 0 : (it.nh[0] > 0 && !(it.skip0 == -2 && pos == 0));
    else
        return it.part(hh, t);
}
template <int MODE, class I>
__device__ __forceinline__ int last_t(const I &it, int hh) {
    if constexpr (MODE == 2)
        return it.nmax - 1;
    else
        return it.last(hh);
}

// Walks an item's key tiles in order: the first T0 tiles of step 0's ranges (the tiles
// some row of the item sees: the diagonal range is cut at the causal prefix), then every
// tile of step 1's ranges, of step 2's, ...
struct TileCursor {
    int s, ri, nr, ti, nti;
    int left0;  // tiles of step 0 still to come
    int a0, b0, a1, b1;
    __device__ __forceinline__ int start() const { return (ri ? a1 : a0) + ti * BN; }
    __device__ __forceinline__ int end() const { return ri ? b1 : b0; }
};
__device__ __forceinline__ int ntiles(int a, int b) { return b > a ? (b - a + BN - 1) / BN : 0; }
__device__ __forceinline__ void cursor_seek(const StepParams &P, const Item &it, TileCursor &c) {
    const int steps = P.ring_fused ? P.ring_R : 1;
    for (; c.s < steps; ++c.s) {
        if (c.s == 0) {
            c.a0 = it.kt.k0[0];
            c.b0 = it.kt.k1[0];
            c.a1 = it.kt.k0[1];
            c.b1 = it.kt.k1[1];
            c.nr = (c.b0 > c.a0) + (c.b1 > c.a1);
            if (c.b0 <= c.a0) {
                c.a0 = c.a1;
                c.b0 = c.b1;
            }
        } else {
            c.nr = ring_ranges(P, it.rank, it.q1, c.s, c.a0, c.b0, c.a1, c.b1);
        }
        if (c.nr > 0) {
            c.ri = 0;
            c.ti = 0;
            c.nti = ntiles(c.a0, c.b0);
            return;
        }
    }
}
__device__ __forceinline__ void cursor_begin(const StepParams &P, const Item &it, TileCursor &c) {
    c.s = 0;
    c.left0 = it.T0;
    cursor_seek(P, it, c);
}
__device__ __forceinline__ void cursor_next(const StepParams &P, const Item &it, TileCursor &c) {
    if (c.s == 0 && --c.left0 <= 0) {  // past step 0's visible prefix
        c.s = 1;
        cursor_seek(P, it, c);
        return;
    }
    if (++c.ti < c.nti) return;
    if (c.ri + 1 < c.nr) {
        c.ri = 1;
        c.ti = 0;
        c.nti = ntiles(c.a1, c.b1);
        return;
    }
    ++c.s;
    cursor_seek(P, it, c);
}

// Items of a launch are numbered heaviest first (decode_item); each CTA's producer takes
// the next item number from the launch's work counter (P.sched) when it needs one, so the
// persistent grid balances whatever the items' costs.

// Work item L, part `sub`.  With P.pair_items (segments of equal length): an item is a
// pair of 256-row blocks of one segment and one head, block p and block nb-1-p, so under
// causality every item of a segment costs the same; items are numbered segment
// (heaviest first, as the host orders them), then head, then pair, so the CTAs that run
// at the same time share the K/V tiles of a few heads in L2.  `sub` 0 is the later
// block, 1 the earlier one (false when the pair has a single middle block).  Otherwise
// an item is one block, as decode_work numbers them (heaviest first) with the heads
// innermost, which balances best when there are few items per CTA (in the fused ring,
// chunk by chunk); `sub` 1 is empty.
__device__ __forceinline__ bool decode_item(const StepParams &P, int L, int sub, Item &it) {
    const int BH = P.B * P.Hq;
    int si, lb, bh;
    if (!P.pair_items) {
        if (sub) return false;
        // single blocks: block rank w (heaviest first) outside, heads inside; with head groups,
        // the heads of one group of P.head_group consecutive (batch, head) units go first, so
        // the CTAs that run together read the K/V of those heads only (they stay in L2)
        int w;
        if (P.head_group > 0 && P.head_group < BH) {
            const int per_group = P.head_group * P.blocks_y;
            const int g = L / per_group;
            const int r = L - g * per_group;
            const int gsize = min(P.head_group, BH - g * P.head_group);
            w = r / gsize;
            bh = g * P.head_group + (r - w * gsize);
        } else {
            w = L / BH;
            bh = L - w * BH;
        }
        if (P.ring_fused && P.ring_layout == 2) {
            // fused striped ring: every rank's chunk costs the same block by block (block lb
            // walks R steps of 2 lb + 2 tiles), so items go block by block across the ranks,
            // the last (heaviest) block first: longest first over the whole launch
            const int wb = w / P.nseg;
            si = w - wb * P.nseg;
            lb = P.blocks_per_seg - 1 - wb;
        } else if (P.ring_fused) {
            // fused ring: a block's cost is mostly its chunk's later steps, so items go
            // chunk by chunk (heaviest first, as the host orders them), last block first
            si = w / P.blocks_per_seg;
            lb = P.blocks_per_seg - 1 - (w - si * P.blocks_per_seg);
        } else {
            decode_work(P, w, si, lb);
        }
    } else {
        const int np = (P.blocks_per_seg + 1) >> 1;
        const int per_seg = BH * np;
        si = L / per_seg;
        const int rem = L - si * per_seg;
        bh = rem / np;
        const int pp = rem - bh * np;
        lb = sub ? pp : P.blocks_per_seg - 1 - pp;
        if (sub && lb == P.blocks_per_seg - 1 - pp) return false;
    }
    it.b = bh / P.Hq;
    it.h = bh - it.b * P.Hq;
    it.hk = it.h / (P.Hq / P.Hkv);
    it.nmax = 0;
    it.nh[0] = it.nh[1] = 0;
    it.T0 = 0;
    it.skip0 = -1;
    it.tps = 0;
    it.rev = 0;
    if (lb < 0) return true;
    const Seg &S = P.seg[si];
    it.rank = S.rank;
    it.qrow0 = S.q0 + lb * 2 * BM;
    it.q1 = S.q1;
    it.q_rank = S.q_rank;
    it.kv_rank = S.kv_rank;
    it.diag = S.diag;
    it.flags = S.flags;
    if (P.ring_fused && P.ring_layout == 2) {
        // striped: every step is a causal prefix of the same tile count T (the chunk and
        // the items' rows are whole 128-row tiles); half 0 sits out one tile per step when
        // half 1 has rows
        int end, j, d;
        striped_range(P, S.rank, min(it.qrow0 + 2 * BM, S.q1), 0, end, j, d);
        const int T = ntiles(0, end);
        const bool two = it.qrow0 + BM < S.q1;
        it.tps = T;
        it.nmax = P.ring_R * T;
        it.nh[1] = two ? it.nmax : 0;
        it.nh[0] = (two && P.causal) ? P.ring_R * (T - 1) : it.nmax;
        it.skip0 = (two && P.causal) ? -2 : -1;
        it.T0 = T;
        it.kt.k0[0] = it.kt.k1[0] = it.kt.k0[1] = it.kt.k1[1] = 0;
        it.kt.nt0 = it.kt.ntot = 0;
        return true;
    }
    if (P.ring_fused) {  // step 0's ranges: the rank's own block
        int a0, b0, a1, b1;
        const int nr = ring_ranges(P, S.rank, S.q1, 0, a0, b0, a1, b1);
        it.kt.k0[0] = a0;
        it.kt.k1[0] = b0;
        it.kt.k0[1] = nr > 1 ? a1 : b0;
        it.kt.k1[1] = nr > 1 ? b1 : b0;
    } else {
        it.kt.k0[0] = S.k0[0];
        it.kt.k1[0] = S.k1[0];
        it.kt.k0[1] = S.k0[1];
        it.kt.k1[1] = S.k1[1];
    }
    it.kt.nt0 = ntiles(it.kt.k0[0], it.kt.k1[0]);
    it.kt.ntot = it.kt.nt0 + ntiles(it.kt.k0[1], it.kt.k1[1]);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int r0 = it.qrow0 + hh * BM;
        if (r0 >= S.q1)
            it.nh[hh] = 0;
        else if (!P.causal)
            it.nh[hh] = it.kt.ntot;
        else
            it.nh[hh] = it.kt.visible_prefix(min(r0 + BM, S.q1) - 1 - S.diag);
    }
    // the first step: each half a prefix of its tiles; the later steps (fused ring): every
    // tile for both halves (their ranges lie wholly before or wholly after the chunk)
    it.T0 = max(it.nh[0], it.nh[1]);
    // half 1 sees every first-step tile (its rows come later); half 0 at most one fewer:
    // the last one.  Outside the fused ring the item walks its tiles last first, so that
    // half 0 sits out the first tile: the halves start staggered (half 0's first S is
    // computed before half 1's first P is in) and end together, and neither half's
    // epilogue delays the other's start on the next item.
    if (it.nh[0] > 0 && it.nh[0] < it.T0) {
        if (P.ring_fused) {
            it.skip0 = it.T0 - 1;
        } else {
            it.skip0 = 0;
            it.rev = it.T0;
        }
    }
    int later = 0;
    if (P.ring_fused && it.T0 > 0)
        for (int s = 1; s < P.ring_R; ++s) {
            int a0, b0, a1, b1;
            const int nr = ring_ranges(P, S.rank, S.q1, s, a0, b0, a1, b1);
            later += (nr > 0 ? ntiles(a0, b0) : 0) + (nr > 1 ? ntiles(a1, b1) : 0);
        }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
        if (it.nh[hh] > 0) it.nh[hh] += later;
    it.nmax = it.T0 + later;
    return true;
}

// ---------------------------------------------------------------- the kernel
//
// Persistent: one CTA per SM walks its work items.  Barrier phases run on across items
// (every wait uses a running count), so the next item's Q/K/V loads and first Q K^T
// overlap the current item's last P V products and epilogue.  Q_h is reloaded once
// the MMA thread has issued the item's last Q_h K^T (q_empty[h]); the softmax
// warpgroup of half h finishes its epilogue (reads O_h) before it signals the next
// item's first P_h, and only then is O_h overwritten.

// MODE 0: one ring step (or the single pass): key tiles come from the item's segment
// ranges.  MODE 1: a fused contiguous or zigzag ring (P.ring_fused): the launch walks
// every step, key tiles from a cursor over the steps' ranges.  MODE 2: a fused striped
// ring: every step a causal prefix, walked last tile first (StripeWalk).
template <int HD, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const __grid_constant__ StepParams P) {
    using C = Cfg<HD>;
    constexpr bool FUSED = MODE != 0;
    constexpr bool STRIPED = MODE == 2;
    // Outside the fused ring, half 0 (the half the MMA thread serves last in each tile)
    // learns that its next S is ready from the stage's release (a commit after that S's
    // product, which is the stage's last), not from a commit of its own: two commits back
    // to back hold the MMA thread until the products before them complete.  (Measured:
    // +1.2 % on the dense pass; in the fused ring, with half 1 last, it cost 3-4 %.)
    constexpr int kLastHalf = MODE == 1 ? -1 : 0;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sQ = base;
    const uint32_t sKV = base + 2 * C::TILE_BYTES;
    const uint32_t sStage = base + (2 + C::NSLOT) * C::TILE_BYTES;  // 1024-byte aligned
    Bars *bars = reinterpret_cast<Bars *>(base_ptr + (2 + C::NSLOT) * C::TILE_BYTES + C::STAGE_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = P.total_items;
    if ((int)blockIdx.x >= total) {
        if (threadIdx.x == 0) sched_finish(P.sched);
        return;
    }

    const uint32_t b_drain = smem_u32(&bars->drain);
    volatile int32_t *abort_flag = &bars->abort;

    // ---- set-up (once per CTA)
    if (threadIdx.x == 0) {
        bars->abort = 0;
#pragma unroll
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            mbar_init(smem_u32(&bars->q_full[hh]), 1);
            mbar_init(smem_u32(&bars->q_empty[hh]), 1);
            mbar_init(smem_u32(&bars->s_full[hh]), 1);
            mbar_init(smem_u32(&bars->o_full[hh]), 1);
        }
        mbar_init(b_drain, 1);
#pragma unroll
        for (int i = 0; i < kItemRing; ++i) {
            mbar_init(smem_u32(&bars->it_full[i]), 1);
            mbar_init(smem_u32(&bars->it_empty[i]), kItemReaders);
        }
        bars->p_count[0] = bars->p_count[1] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_u32(&bars->tmem_base), C::TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // The next ring step's kernel may start on SMs this grid frees; it only waits for
    // this grid before its epilogue touches the running result (griddepcontrol.wait).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < 4) {
      regs_dec<kRegsControl>();
      if (warp == 0) {
        // ================= TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            producer_delay(P.producer_delay_ns);
            int slot = 0;
            uint32_t ph = 0;
            uint32_t issued = 0, last_ph = 0;  // per-slot bit sets
            uint32_t qcnt[2] = {0u, 0u};       // Q_h loads issued
            uint32_t icnt = 0;                 // items handed to the MMA issuer
            // hand a decoded item to the MMA issuer and the softmax warps once its ring slot
            // is free
            auto hand_over = [&](const Item &x) -> bool {
                const int islot = icnt & (kItemRing - 1);
                if (icnt >= (uint32_t)kItemRing &&
                    !wait_phase(smem_u32(&bars->it_empty[islot]), (icnt / kItemRing - 1u) & 1u, abort_flag,
                                P.wait_limit_ns, P.err))
                    return false;
                item_store(&bars->it_info[islot][0], x);
                mbar_arrive(smem_u32(&bars->it_full[islot]));  // release: the fields are visible
                ++icnt;
                return true;
            };
            bool ok = true;
            int L = 0;
            for (int k2 = 0; ok; ++k2) {  // (item, part)
                if (!(k2 & 1)) L = atomicAdd(&P.sched[0], 1);  // the next item number
                if (L >= total) break;
                Item it;
                if (!decode_item(P, L, k2 & 1, it)) continue;
                if (it.nmax == 0) continue;
                if (!hand_over(it)) {
                    ok = false;
                    break;
                }
                // Stages of an item: (K_0), then (V_t, K_t+1) for t = 0..n-1 (the last one
                // V only).  Stage (K_0) first - it only needs a free buffer pair - then Q,
                // which waits until the previous item has issued its last Q K^T.
                TileCursor cur;
                StripeWalk sw;
                if constexpr (STRIPED)
                    stripe_begin(P, it, sw);
                else if constexpr (FUSED)
                    cursor_begin(P, it, cur);
                int vstart = 0, vrank = it.kv_rank;  // V_t is the tile K_t came from
                for (int st = -1; st < it.nmax && ok; ++st) {
                    const uint32_t b_empty = smem_u32(&bars->empty[slot]);
                    const uint32_t b_full = smem_u32(&bars->full[slot]);
                    if (!wait_phase(b_empty, ph ^ 1u, abort_flag, P.wait_limit_ns, P.err)) {
                        ok = false;
                        break;
                    }
                    const bool has_v = st >= 0;
                    const bool has_k = st + 1 < it.nmax;
                    mbar_expect_tx(b_full, (has_v + has_k) * C::TILE_BYTES);
                    const uint32_t vbuf = sKV + (2 * slot) * C::TILE_BYTES;
                    const uint32_t kbuf = sKV + (2 * slot + 1) * C::TILE_BYTES;
                    if (has_v) {
                        const int vs = FUSED ? vstart : it.kt.start(it.tile(st));
                        if (in_bounds(vrank >= 0 && vrank < P.rs && vs >= 0 && vs < P.N / P.rs && it.hk >= 0 &&
                                          it.hk < P.Hkv && it.b >= 0 && it.b < P.B,
                                      P.err))
#pragma unroll
                            for (int c = 0; c < C::SLABS; ++c)
                                tma_load_5d(vbuf + c * C::SLAB_BYTES, &tm_v, b_full, c * 64, vrank, vs, it.hk, it.b);
                    }
                    if (has_k) {
                        int ks, kr = it.kv_rank;
                        if constexpr (STRIPED) {
                            ks = sw.start(it.tps);
                            kr = sw.j;
                            vstart = ks;
                            vrank = kr;
                            stripe_next(P, it, sw);
                        } else if constexpr (FUSED) {
                            ks = cur.start();
                            vstart = ks;
                            cursor_next(P, it, cur);
                        } else {
                            ks = it.kt.start(it.tile(st + 1));
                        }
                        if (in_bounds(kr >= 0 && kr < P.rs && ks >= 0 && ks < P.N / P.rs && it.hk >= 0 &&
                                          it.hk < P.Hkv && it.b >= 0 && it.b < P.B,
                                      P.err))
#pragma unroll
                            for (int c = 0; c < C::SLABS; ++c)
                                tma_load_5d(kbuf + c * C::SLAB_BYTES, &tm_k, b_full, c * 64, kr, ks, it.hk, it.b);
                    }
                    issued |= 1u << slot;
                    last_ph = (last_ph & ~(1u << slot)) | (ph << slot);
                    if (++slot == C::NSTAGE) {
                        slot = 0;
                        ph ^= 1u;
                    }
                    if (st == -1) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            if (it.nh[hh] == 0 || !ok) continue;
                            const uint32_t qf = smem_u32(&bars->q_full[hh]);
                            if (!wait_phase(smem_u32(&bars->q_empty[hh]), (qcnt[hh] & 1u) ^ 1u,
                                            abort_flag, P.wait_limit_ns, P.err)) {
                                ok = false;
                                break;
                            }
                            mbar_expect_tx(qf, C::TILE_BYTES);
                            if (in_bounds(it.q_rank >= 0 && it.q_rank < P.rs && it.qrow0 + hh * BM >= 0 &&
                                              it.qrow0 + hh * BM < P.N / P.rs && it.h >= 0 && it.h < P.Hq &&
                                              it.b >= 0 && it.b < P.B,
                                          P.err))
#pragma unroll
                            for (int c = 0; c < C::SLABS; ++c)
                                tma_load_5d(sQ + hh * C::TILE_BYTES + c * C::SLAB_BYTES, &tm_q, qf,
                                            c * 64, it.q_rank, it.qrow0 + hh * BM, it.h, it.b);
                            ++qcnt[hh];
                        }
                    }
                }
            }
            if (ok) {  // no more items
                Item end;
                memset(&end, 0, sizeof end);
                end.nmax = -1;
                ok = hand_over(end);
            }
            if (!ok) {  // wind down: let every copy this thread issued land
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    if (qcnt[hh]) wait_phase_drain(smem_u32(&bars->q_full[hh]), (qcnt[hh] - 1u) & 1u);
                for (int s2 = 0; s2 < C::NSTAGE; ++s2)
                    if (issued & (1u << s2))
                        wait_phase_drain(smem_u32(&bars->full[s2]), (last_ph >> s2) & 1u);
            }
        }
      } else if (warp == 1) {
        // ================= MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(BM, HD, true);
            // descriptors of the two Q halves, built once; K and V ones once per stage
            const SDesc qd0 = sdesc_split(sQ, 16, 1024), qd1 = sdesc_split(sQ + C::TILE_BYTES, 16, 1024);
            auto issue_qk = [=](int hh, uint32_t kb) {
                const uint32_t d = tmem + (hh ? C::TM_S1 : C::TM_S0);
                const SDesc qd = hh ? qd1 : qd0;
                const SDesc kd = sdesc_split(kb, 16, 1024);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    const uint32_t off = (k >> 2) * C::SLAB_BYTES + (k & 3) * 32;
                    mma_ss(d, qd.at(off), kd.at(off), IDESC_QK, k > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [=](int hh, uint32_t vb, bool acc_in) {
                const uint32_t d = tmem + (hh ? C::TM_O1 : C::TM_O0);
                const uint32_t p = tmem + (hh ? C::TM_S1 : C::TM_S0);
                const SDesc vd = sdesc_split(vb, C::SLAB_BYTES, 1024);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    mma_ts(d, p + k * 8, vd.at(k * 16 * 128), IDESC_PV, (acc_in || k > 0) ? 1u : 0u);
            };
            int slot = 0;
            uint32_t ph = 0;
            uint32_t qcnt[2] = {0u, 0u};  // Q_h loads consumed
            uint32_t pcnt[2] = {0u, 0u};  // P_h tiles consumed
            bool ok = true;
            // items come decoded from the producer (which runs ahead): the MMA thread's
            // own decode would sit between an item's last P V and the next one's Q K^T
            uint32_t icnt = 0;
            for (;;) {
                MItem it;
                {
                    const int islot = icnt & (kItemRing - 1);
                    ok = wait_phase(smem_u32(&bars->it_full[islot]), (icnt / kItemRing) & 1u, abort_flag,
                                    P.wait_limit_ns, P.err);
                    if (!ok) break;
                    const Item &v = *reinterpret_cast<const Item *>(&bars->it_info[islot][0]);
                    it.nh[0] = v.nh[0];
                    it.nh[1] = v.nh[1];
                    it.nmax = v.nmax;
                    it.skip0 = v.skip0;
                    it.tps = v.tps;
                    mbar_arrive(smem_u32(&bars->it_empty[islot]));
                    ++icnt;
                }
                if (it.nmax < 0) break;  // no more items
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (it.nh[hh] == 0 || !ok) continue;
                    ok = wait_phase(smem_u32(&bars->q_full[hh]), qcnt[hh] & 1u, abort_flag,
                                    P.wait_limit_ns, P.err);
                    ++qcnt[hh];
                }
                if (!ok) break;
                // stage (K_0): the first Q K^T of both halves
                ok = wait_phase(smem_u32(&bars->full[slot]), ph, abort_flag, P.wait_limit_ns, P.err);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (part_pos<MODE>(it, hh, 0, 0)) {
                        issue_qk(hh, sKV + (2 * slot + 1) * C::TILE_BYTES);
                        if (hh != kLastHalf) mma_commit(smem_u32(&bars->s_full[hh]));
                        if (last_t<MODE>(it, hh) == 0) mma_commit(smem_u32(&bars->q_empty[hh]));
                    }
                }
                mma_commit(smem_u32(&bars->empty[slot]));
                if (++slot == C::NSTAGE) {
                    slot = 0;
                    ph ^= 1u;
                }
                // stage (V_t, K_t+1): P_h V_t and the next Q_h K^T of each half (a half
                // issues the next Q K^T of a tile it takes part in even when it sat this
                // tile out: its last P was read by the P V issued before)
                bool started[2] = {false, false};
                int upos = 0;  // MODE 2: tile t's position in its step
                for (int t = 0; ok && t < it.nmax; ++t) {
                    const int unext = (upos + 1 == it.tps) ? 0 : upos + 1;
                    bool o_due = false;  // the half signalled by stage releases finished its O
                    ok = wait_phase(smem_u32(&bars->full[slot]), ph, abort_flag, P.wait_limit_ns,
                                    P.err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t vb = sKV + (2 * slot) * C::TILE_BYTES;
                    const uint32_t kb = sKV + (2 * slot + 1) * C::TILE_BYTES;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        // outside the fused ring half 1 starts first (half 0 sits out the
                        // item's first tile), and it is served first in every tile
                        const int hh = MODE == 1 ? h2 : 1 - h2;
                        if (part_pos<MODE>(it, hh, t, upos)) {
                            ++pcnt[hh];
                            ok = wait_count(&bars->p_count[hh], 4u * pcnt[hh], abort_flag,
                                            P.wait_limit_ns, P.err);
                            if (!ok) break;
                            tc_fence_after();
                            issue_pv(hh, vb, started[hh]);
                            started[hh] = true;
                            if (t == last_t<MODE>(it, hh)) {
                                if (hh == kLastHalf)
                                    o_due = true;
                                else
                                    mma_commit(smem_u32(&bars->o_full[hh]));
                            }
                        }
                        if (t + 1 < it.nmax && part_pos<MODE>(it, hh, t + 1, unext)) {
                            issue_qk(hh, kb);
                            if (hh != kLastHalf) mma_commit(smem_u32(&bars->s_full[hh]));
                            if (t + 1 == last_t<MODE>(it, hh)) mma_commit(smem_u32(&bars->q_empty[hh]));
                        }
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&bars->empty[slot]));
                    // The O-ready commit of the half signalled by stage releases comes after
                    // the release of the item's last stage.  That half's softmax warps wait
                    // for each S on the release of the stage that computed it, by parity, and
                    // their first such wait in the next item can fall on this stage's buffer:
                    // once they have seen O ready, this release has arrived too, so that wait
                    // cannot pass a phase early.
                    if constexpr (kLastHalf >= 0)
                        if (o_due) mma_commit(smem_u32(&bars->o_full[kLastHalf]));
                    if (++slot == C::NSTAGE) {
                        slot = 0;
                        ph ^= 1u;
                    }
                    upos = unext;
                }
                if (!ok) break;
            }
            // every MMA this thread issued completes before tensor memory is released
            mma_commit(b_drain);
            wait_phase_drain(b_drain, 0);
        }
      }
    } else {
        regs_inc<kRegsSoftmax>();
        // ================= softmax (+ O rescale and epilogue) of one half
        const int hh = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + (hh ? C::TM_S1 : C::TM_S0) + lane_off;
        const uint32_t tO = tmem + (hh ? C::TM_O1 : C::TM_O0) + lane_off;
        const uint32_t b_s = smem_u32(&bars->s_full[hh]);
        const uint32_t b_o = smem_u32(&bars->o_full[hh]);
        const float sl2 = P.scale_log2;
        uint32_t scnt = 0, ocnt = 0;  // S_h tiles and O_h results seen
        uint32_t gstage = 0;          // stages of the items so far: (K_0) and one per tile
        bool ok = true;
        uint32_t icnt = 0;
        for (;;) {  // items, decoded by the producer
            Item it;
            {
                const int islot = icnt & (kItemRing - 1);
                ok = wait_phase(smem_u32(&bars->it_full[islot]), (icnt / kItemRing) & 1u, abort_flag,
                                P.wait_limit_ns, P.err);
                if (!ok) break;
                item_load(&bars->it_info[islot][0], it);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->it_empty[islot]));
                ++icnt;
            }
            if (it.nmax < 0) break;  // no more items
            const int n = hh ? it.nh[1] : it.nh[0];
            const uint32_t sbase = gstage;  // tile t's S is computed in stage sbase + t
            gstage += 1u + (uint32_t)it.nmax;
            if (n == 0) continue;
            const int first_row = it.qrow0 + hh * BM;
            const int row_g = first_row + quarter * 32 + lane;     // index in the segment
            const int pos = row_g * P.rs + it.q_rank;               // position in the sequence
            if (P.oacc && !(it.flags & SEG_FIRST) && row_g < it.q1) {
                // the running row is read by this item's epilogue: stage it in L2 now
                const float *pre = P.oacc + (((int64_t)it.b * P.Hq + it.h) * P.N + pos) * HD;
#pragma unroll
                for (int i = 0; i < HD * 4 / 128; ++i)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(pre + i * 32));
            }
            float m_ref = -INFINITY, l = 0.f;
            TileCursor cur;
            StripeWalk sw;
            if constexpr (STRIPED)
                stripe_begin(P, it, sw);
            else if constexpr (FUSED)
                cursor_begin(P, it, cur);
            bool first_tile = true;
            for (int t = 0; t < it.nmax; ++t) {
                int ks, ke, dg = it.diag;  // the tile's keys and diagonal offset
                int upos = 0;              // (striped) the tile's position in its step
                if constexpr (STRIPED) {
                    upos = sw.u;
                    ks = sw.start(it.tps);
                    ke = sw.end;
                    dg = sw.d;
                    stripe_next(P, it, sw);
                } else if constexpr (FUSED) {
                    ks = cur.start();
                    ke = cur.end();
                    cursor_next(P, it, cur);
                } else {
                    ks = it.kt.start(it.tile(t));
                    ke = it.kt.range_end(it.tile(t));
                }
                if (!part_pos<MODE>(it, hh, t, upos)) continue;
                if (hh == kLastHalf) {
                    const uint32_t gs = sbase + (uint32_t)t;
                    ok = wait_phase(smem_u32(&bars->empty[gs % C::NSTAGE]), (gs / C::NSTAGE) & 1u, abort_flag,
                                    P.wait_limit_ns, P.err);
                } else {
                    ok = wait_phase(b_s, scnt & 1u, abort_flag, P.wait_limit_ns, P.err);
                    ++scnt;
                }
                if (!ok) break;
                tc_fence_after();
                uint32_t r[4][32];
                tmem_ld32(tS + 0, r[0]);
                tmem_ld32(tS + 32, r[1]);
                tmem_ld32(tS + 64, r[2]);
                tmem_ld32(tS + 96, r[3]);
                tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[128]>(&r[0][0]));
                const bool need_mask =
                    (ks + BN > ke) || (P.causal && (min(ks + BN, ke) - 1 + dg > first_row));
                if (need_mask) {
                    const int lim = (P.causal ? min(ke, row_g + 1 - dg) : ke) - ks;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim) r[c >> 5][c & 31] = __float_as_uint(-INFINITY);
                }
                // row max: eight independent chains of 3-input max
                float mc[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c0 = j * 16;
                    float m = fmax3(__uint_as_float(r[c0 >> 5][c0 & 31]),
                                    __uint_as_float(r[c0 >> 5][(c0 & 31) + 1]),
                                    __uint_as_float(r[c0 >> 5][(c0 & 31) + 2]));
#pragma unroll
                    for (int i = 3; i < 15; i += 2)
                        m = fmax3(m, __uint_as_float(r[c0 >> 5][(c0 & 31) + i]),
                                  __uint_as_float(r[c0 >> 5][(c0 & 31) + i + 1]));
                    mc[j] = fmaxf(m, __uint_as_float(r[c0 >> 5][(c0 & 31) + 15]));
                }
                const float mx = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]),
                                       fmaxf(mc[6], mc[7]));
                const float m_tile = mx * sl2;
                float alpha = 1.f;
                bool resc = false;
                if (first_tile) {
                    m_ref = m_tile;
                } else if (m_tile > m_ref + kRescaleThreshold) {
                    alpha = ex2(m_ref - m_tile);
                    m_ref = m_tile;
                    resc = true;
                }
                const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
                // p = 2^(s * scale * log2e - m): paired FFMA, one ex2 per element, bf16
                // pack, four paired partial sums; the first 64 keys go to tensor memory
                // while the rest are computed
                const uint64_t sl2x2 = pack_f32x2(sl2, sl2);
                const uint64_t negm2 = pack_f32x2(neg_m, neg_m);
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int c = j * 64 + 2 * i;
                        const uint64_t x =
                            ffma2(pack_f32x2(__uint_as_float(r[c >> 5][c & 31]),
                                             __uint_as_float(r[c >> 5][(c & 31) + 1])),
                                  sl2x2, negm2);
                        float x0, x1;
                        unpack_f32x2(x, x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        acc2[i & 3] = fadd2(acc2[i & 3], pack_f32x2(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(tS + j * 32, pk);
                }
                float rs;
                {
                    const uint64_t a = fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3]));
                    float a0, a1;
                    unpack_f32x2(a, a0, a1);
                    rs = a0 + a1;
                }
                l = l * alpha + rs;
                if (!first_tile && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_ld_wait_regs(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + c * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) count_release_add(&bars->p_count[hh]);
                first_tile = false;
            }
            if (!ok) break;
            // ---- epilogue: O / l, LSE, then write or LSE-merge into the running result.
            // (The running row was staged in L2 at the start of the item.)
            // the previous ring step wrote the running result (o_acc, lse) and, for its
            // last rows, O: wait for that grid before reading or writing them
            if (P.chained) asm volatile("griddepcontrol.wait;" ::: "memory");
            const bool first = (it.flags & SEG_FIRST) != 0;
            const bool final_ = (it.flags & SEG_FINAL) != 0;
            const int64_t lrow = ((int64_t)it.b * P.Hq + it.h) * P.N + pos;
            const bool valid = row_g < it.q1 && in_bounds(pos >= 0 && pos < P.N && lrow < (int64_t)P.B * P.Hq * P.N, P.err);
            const bool merge = valid && !first;
            float *arow = P.oacc ? P.oacc + lrow * HD : nullptr;
            const float lse_a = merge ? P.lse[lrow] : -INFINITY;
            ok = wait_phase(b_o, ocnt & 1u, abort_flag, P.wait_limit_ns, P.err);
            ++ocnt;
            if (!ok) break;
            tc_fence_after();
            const bool have = l > 0.f;
            const float lse_b = have ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
            const float inv = have ? 1.f / l : 0.f;
            MergeW w;
            w.wa = 0.f;
            w.wb = 1.f;
            w.L = lse_b;
            if (merge) w = merge_weights(lse_a, lse_b);
            const bool use_prev = merge && w.wa != 0.f;
            const float wb = w.wb * inv;
            // Final rows of a half that lies wholly inside its segment (or is clipped by the
            // end of the tensor) leave through shared memory and bulk tensor stores: each warp
            // stores its 32 rows 32 columns at a time from two 2 KiB buffers of its own, so no
            // warp waits for another.  Row-per-thread global stores would issue 32 scattered
            // 16-byte pieces per instruction and clog the SM's memory pipeline.
            const bool tma_o = final_ && P.o_tma && (first_row + BM <= it.q1 || it.q1 == P.N / P.rs);
            if (tma_o) {
                const uint32_t wbuf = sStage + (uint32_t)(hh * 4 + quarter) * 4096u;
#pragma unroll 1
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    float x[32];
                    if (use_prev) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 a = __ldcs(reinterpret_cast<const float4 *>(arow + c * 32 + i));
                            x[i] = w.wa * a.x;
                            x[i + 1] = w.wa * a.y;
                            x[i + 2] = w.wa * a.z;
                            x[i + 3] = w.wa * a.w;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[i] = 0.f;
                    }
                    tmem_ld_wait_regs(o);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(fmaf(wb, __uint_as_float(o[2 * i]), x[2 * i]),
                                            fmaf(wb, __uint_as_float(o[2 * i + 1]), x[2 * i + 1]));
                    // this buffer's previous store (two stores ago) has read it
                    const uint32_t buf = wbuf + (uint32_t)(c & 1) * 2048u;
                    if (lane == 0) bulk_wait_read1();
                    __syncwarp();
                    // 64-byte swizzle, as the tensor map expects: 16-byte piece j of row r
                    // sits at piece j ^ ((r / 2) mod 4)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t a = buf + lane * 64 + ((uint32_t)(j ^ ((lane >> 1) & 3)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pk[4 * j]),
                                     "r"(pk[4 * j + 1]), "r"(pk[4 * j + 2]), "r"(pk[4 * j + 3])
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    // (debug builds: a box wholly past the end of the rows, of a half clipped
                    // by the tensor's end, writes nothing and is skipped unchecked)
                    if (lane == 0 && (!kDebugBounds || (first_row + quarter * 32 < P.N / P.rs &&
                                                        in_bounds(first_row >= 0 && it.q_rank >= 0 &&
                                                                      it.q_rank < P.rs && it.h >= 0 &&
                                                                      it.h < P.Hq && it.b >= 0 && it.b < P.B,
                                                                  P.err)))) {
                        tma_store_5d(&tm_o, buf, c * 32, it.q_rank, first_row + quarter * 32, it.h, it.b);
                        bulk_commit();
                    }
                    __syncwarp();
                }
                if (valid) P.lse[lrow] = first ? lse_b : w.L;
                continue;
            }
            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(P.o) + (int64_t)it.b * P.so[0] +
                                  (int64_t)it.h * P.so[1] + (int64_t)pos * P.so[2];
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                float x[32];
                if (use_prev) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 a = __ldcs(reinterpret_cast<const float4 *>(arow + c * 32 + i));
                        x[i] = w.wa * a.x;
                        x[i + 1] = w.wa * a.y;
                        x[i + 2] = w.wa * a.z;
                        x[i + 3] = w.wa * a.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = 0.f;
                }
                tmem_ld_wait_regs(o);
                if (!valid) continue;
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = fmaf(wb, __uint_as_float(o[i]), x[i]);
                if (final_) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 u;
                        u.x = pack_bf16x2(x[i], x[i + 1]);
                        u.y = pack_bf16x2(x[i + 2], x[i + 3]);
                        u.z = pack_bf16x2(x[i + 4], x[i + 5]);
                        u.w = pack_bf16x2(x[i + 6], x[i + 7]);
                        *reinterpret_cast<uint4 *>(orow + c * 32 + i) = u;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        __stcg(reinterpret_cast<float4 *>(arow + c * 32 + i),
                               make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]));
                }
            }
            if (valid) P.lse[lrow] = first ? lse_b : w.L;
        }
    }

    // the bulk stores of O issued by each softmax warp are complete before exit
    if (warp >= 4 && lane == 0) bulk_wait0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
    if (threadIdx.x == 0) sched_finish(P.sched);
}

// One block, one thread: a bounded wait on a barrier nothing completes.
__global__ void wait_selftest_kernel(int64_t limit_ns, int *err) {
    __shared__ uint64_t bar;
    __shared__ int32_t abort;
    if (threadIdx.x != 0) return;
    abort = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    wait_phase(smem_u32(&bar), 0, &abort, limit_ns, err);
}

// One block, one thread: the device bounds check on an index outside its range (debug
// builds record DERR_BOUNDS; nothing is accessed).
__global__ void bounds_selftest_kernel(int n, int *err) {
    if (threadIdx.x == 0) (void)bounds_check(n < 0, err);
}

}  // namespace tc

// ---------------------------------------------------------------- host side

template <int HD>
static cudaError_t launch_tc_hd(const StepParams &P, int blocks_y, int num_sms,
                                cudaStream_t stream) {
    using C = tc::Cfg<HD>;
    if (!P.sched) return cudaErrorInvalidValue;  // items come from a work counter pair
    static int configured_mask = 0;  // per device ordinal bit (devices < 32)
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(configured_mask & (1 << (dev & 31)))) {
        cudaError_t e = cudaFuncSetAttribute(tc::attn_tc_kernel<HD, 0>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tc::attn_tc_kernel<HD, 1>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tc::attn_tc_kernel<HD, 2>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured_mask |= 1 << (dev & 31);
    }
    CUtensorMap mq, mk, mv, mo;
    if (!encode_map(&mq, P.q, P.B, P.Hq, P.N, P.D, P.sq, P.rs) ||
        !encode_map(&mk, P.k, P.B, P.Hkv, P.N, P.D, P.sk, P.rs) ||
        !encode_map(&mv, P.v, P.B, P.Hkv, P.N, P.D, P.sv, P.rs))
        return cudaErrorInvalidValue;
    // O through bulk tensor stores (32 x 32 boxes, 64-byte swizzle) when its layout allows
    // a map (else row stores)
    const bool o_map = encode_map(&mo, P.o, P.B, P.Hq, P.N, P.D, P.so, P.rs, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!o_map) memset(&mo, 0, sizeof mo);
    // Items: pairs of blocks for a ring step launched per step (its tail overlaps the
    // next step's launch) or when the pairs fill their rounds over the persistent grid to
    // 93 %; single blocks (heaviest first) otherwise, for the fused ring and for packed
    // batches.
    const int64_t singles = (int64_t)P.B * P.Hq * blocks_y;
    const int64_t pairs = (int64_t)P.B * P.Hq * P.nseg * ((P.blocks_per_seg + 1) / 2);
    bool use_pairs = false;
    if (!P.var_blocks && pairs > 0) {
        const int64_t g = std::min<int64_t>(pairs, num_sms);
        const int64_t rounds = (pairs + g - 1) / g;
        // (a fused ring takes single blocks: its pairs differ in cost from chunk to chunk,
        // and with a few rounds of them per CTA the grid ran unbalanced - ring8 zigzag
        // 1245 TFLOP/s with pairs, 1563 with single blocks)
        use_pairs = (P.prefer_pairs && !P.ring_fused) || (double)pairs >= 0.93 * (double)(rounds * g);
    }
    const int64_t total = use_pairs ? pairs : singles;
    if (total > 0x7fffffff) return cudaErrorInvalidValue;
    StepParams Q = P;
    Q.total_items = (int32_t)total;
    Q.pair_items = use_pairs ? 1 : 0;
    Q.blocks_y = blocks_y;
    Q.o_tma = o_map ? 1 : 0;
    const int grid = (int)std::min<int64_t>(total, (int64_t)num_sms);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(tc::kThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (P.chained) {  // only ever chained to the previous step of the same ring run
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (P.ring_fused && P.ring_layout == 2) return cudaLaunchKernelEx(&cfg, tc::attn_tc_kernel<HD, 2>, mq, mk, mv, mo, Q);
    if (P.ring_fused) return cudaLaunchKernelEx(&cfg, tc::attn_tc_kernel<HD, 1>, mq, mk, mv, mo, Q);
    return cudaLaunchKernelEx(&cfg, tc::attn_tc_kernel<HD, 0>, mq, mk, mv, mo, Q);
}

cudaError_t launch_attn_tc(const StepParams &P, int blocks_y, int num_sms, cudaStream_t stream) {
    if (blocks_y <= 0 || P.B * P.Hq <= 0) return cudaSuccess;
    if (P.D == 128) return launch_tc_hd<128>(P, blocks_y, num_sms, stream);
    if (P.D == 64) return launch_tc_hd<64>(P, blocks_y, num_sms, stream);
    return cudaErrorInvalidValue;
}

int attn_tc_rows_per_block() { return 2 * tc::BM; }

cudaError_t launch_bounds_selftest(int *err, cudaStream_t stream) {
#ifdef RA_DEBUG_BOUNDS
    tc::bounds_selftest_kernel<<<1, 32, 0, stream>>>(1, err);
    return cudaGetLastError();
#else
    (void)err;
    (void)stream;
    return cudaErrorNotSupported;
#endif
}

cudaError_t launch_wait_selftest(int64_t limit_ns, int *err, cudaStream_t stream) {
    tc::wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace ra
