// attn_bwd_tc.cu - gradients of exact attention on the sm_103a tensor cores.
//
// The same quantities as attn_bwd_simt.cu (the recompute-from-LSE backward of the
// `ring_attention_backward` listing of "Ring Attention 论文解析"), as two persistent
// kernels with one writer per output element (no atomics):
//
//   dQ kernel   one CTA item = 128 query rows of one segment and one (b, h); for each
//               visible key tile of the segment's streamed ranges:
//                 S  = Q K^T,  dP = dO V^T          (tcgen05, A and B from shared memory)
//                 dS = P * (dP - D),  P = exp(S * scale - LSE)   (one thread per row)
//                 dQ += dS K                        (tcgen05, A = dS from tensor memory)
//   dK/dV kernel one CTA item = 128 keys of one segment and one (b, KV head); for each
//                visible query tile of the streamed ranges, for every query head that
//                reads the KV head:
//                 S^T = K Q^T,  dP^T = V dO^T
//                 P^T, dS^T                         (one thread per key)
//                 dV += P^T dO,  dK += dS^T Q       (A from tensor memory)
//
// Warp roles: warp 0 TMA producer, warp 1 MMA issuer and tensor-memory owner (the dQ
// kernel: S and dP; warp 2 issues its dQ products), warps 4-11 the element-wise work and
// the epilogue: two warps per tensor-memory lane quarter, each owning 64 of a tile's 128
// columns (one warp per scheduler left the exponentials and the tensor-memory round trips
// exposed).  Every S / dP product is a full 128 x 128 tile (narrower products run the
// tensor core below its rate).  The dQ kernel rotates the S and dP of consecutive tiles
// through three tensor-memory slots, so the next tile's S is computed while the
// element-wise warps work on this one; the dK/dV kernel orders its products so that the
// next tile's S^T and dP^T overlap the element-wise work.  The bf16 P / dS overwrite the
// columns of the fp32 S / dP they came from once those are in registers; an issuer puts a
// product that overwrites a slot after the products that read it (tcgen05 MMAs of a
// thread run in order), or, across the dQ kernel's two issuers, waits for their
// completion.  Every wait is bounded like the forward kernel's.
//
// A launch covers the segments of one ring step (struct BSeg): the whole-sequence
// backward is one segment.  On a ring, the gradient of a range that earlier or later
// steps also write is carried between steps in fp32 running buffers (store_grad_chunk).
#include <climits>
#include <cstring>
#include <stddef.h>

#include "tc_common.cuh"

namespace ra {
namespace tcb {

using namespace ra::tc;

constexpr int kT = 128;  // rows per tile (queries or keys); S / dP products are 128 x 128
constexpr int kThreads = 384;
constexpr int kEwWarps = 8;  // warps 4-11: two groups of four, each owning 64 of a tile's 128 columns
constexpr uint32_t kNegInfBits = 0xff800000u;  // -inf as fp32 bits

// Tensor memory (512 columns).  dQ kernel: three 128-column slots that hold the S and dP
// of consecutive tiles in rotation (tile g: S in slot s_slot(g), dP in slot d_slot(g);
// the next tile's S goes to the free slot and its dP to the slot of this tile's S once
// that has been read), dQ accumulator at 384.  dK/dV kernel: S^T at 0, dP^T at 128, dV
// at 256, dK at 256 + HD.  The bf16 P / dS a tile produces (64 packed columns) overwrite
// columns 32..95 of the fp32 S / dP they came from: element-wise group g reads columns
// [64g, 64g + 64) and writes its 32 packed columns at 32 + 32g, inside what it has read
// and clear of the other group's columns (the order of its two 32-column chunks keeps a
// chunk from being overwritten before it is read).
constexpr int kBarBytes = 1024;  // barrier block and the decoded-item ring

template <int HD>
struct BCfg {
    static constexpr int SLABS = HD / 64;
    static constexpr int TILE_BYTES = kT * HD * 2;
    static constexpr int SLAB_BYTES = 128 * 128;
    static constexpr int NST = (HD == 128) ? 2 : 4;  // dK/dV kernel: stages of two tiles (Q, dO)
    // dQ kernel: separate rings of K tiles and V tiles (V is free after the dP product,
    // K only after the dQ product, so K gets the deeper ring)
    static constexpr int KST = (HD == 128) ? 3 : 4;
    static constexpr int VST = (HD == 128) ? 2 : 4;
    static constexpr uint32_t TM_A0 = 256, TM_A1 = 256 + HD;  // dK/dV kernel: dV, dK
    static constexpr uint32_t TM_DQ = 384;                    // dQ kernel: dQ
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int BAR_OFF = (2 + 2 * NST) * TILE_BYTES;
    // dK/dV kernel: per element-wise warp, its LSE/D values, then (outside the fused ring) a
    // 2 KiB staging buffer for the bulk tensor stores of final dK/dV rows (32 rows x 32
    // columns).  The fused ring writes its rows once per long item: there the buffer's
    // shared memory (taken from L1) cost more than the stores gained (ring8 -0.4 % zigzag,
    // -1.6 % striped), so it keeps row stores.
    static constexpr int STG_OFF = BAR_OFF + kBarBytes + kEwWarps * 2 * 64 * 4;
    static constexpr int SMEM_BYTES_FUSED = 1024 + STG_OFF;
    static constexpr int SMEM_BYTES = SMEM_BYTES_FUSED + kEwWarps * 2048;
    static constexpr int BAR_OFF_DQ = (2 + KST + VST) * TILE_BYTES;
    static constexpr int SMEM_BYTES_DQ = 1024 + BAR_OFF_DQ + kBarBytes;
};

struct BBars {
    uint64_t fix_full, fix_empty;  // the item's fixed pair (Q, dO) or (K, V)
    uint64_t full[4], empty[4];    // streamed pairs (dK/dV kernel) or K tiles (dQ kernel)
    uint64_t fullv[4], emptyv[4];  // V tiles (dQ kernel)
    uint64_t s_full[2], o_full, drain;
    uint64_t dq_done[2], drain2;  // dQ kernel: the dQ issuer's products (alternating), its drain
    uint32_t ds_count[2];         // dQ kernel: dS tiles stored, counted apart by tile parity
    uint32_t tmem_base;
    int32_t abort;
    uint32_t p_count[2];
    uint64_t it_full[4], it_empty[4];  // decoded-item ring: producer -> MMA thread, element-wise warps
    int32_t it_rec[4][32];             // a QRec or KRec
};
static_assert(sizeof(BBars) <= kBarBytes, "barrier block");
static_assert(offsetof(BBars, it_rec) % 16 == 0, "16-byte item records");
constexpr int kItemRing = 4;
constexpr uint32_t kItemReaders = 1 + kEwWarps;  // the MMA thread and one lane per element-wise warp
constexpr uint32_t kItemReadersDq = 2 + kEwWarps;  // dQ kernel: its two MMA issuers and the element-wise warps

// Work items are pairs of tiles of one segment and one head: tile p and tile tps-1-p of
// the segment's fixed range.  Under causality the two costs add up to the same total,
// so every item of a segment costs the same; items are numbered segment (heaviest
// first, as the host orders them), then head, then pair, so the CTAs that run at the
// same time share the streamed tiles of a few heads in L2.  `sub` selects the pair's
// first (0) or second (1) tile; false when the pair has a single (middle) tile.
__device__ __forceinline__ int tile_pairs(int tps) { return (tps + 1) >> 1; }

// A launch over one segment whose CTAs take items from a work counter (P.single) uses
// single tiles instead, longest first: equal-cost pairs leave the last round of the
// persistent grid part empty (1024 pairs on 152 SMs is 6.7 rounds), single tiles taken
// heaviest first fill it.  Item L is tile rank w of unit u (a head, or a (batch, KV head)),
// the units innermost within groups of hg consecutive units (hg 0: one group), so the CTAs
// that run together stream the tiles of a few heads only (they stay in L2).
__device__ __forceinline__ void group_decode(int L, int hg, int units, int tiles, int &w, int &u) {
    if (hg > 0 && hg < units) {
        const int per = hg * tiles;
        const int g = L / per;
        const int r = L - g * per;
        const int gs = min(hg, units - g * hg);
        w = r / gs;
        u = g * hg + (r - w * gs);
    } else {
        w = L / units;
        u = L - w * units;
    }
}

// Fused ring (contiguous or zigzag layout): the streamed ranges of step s for a fixed
// range [f0, f1) of rank `rank`.  dQ (kind 0): the key chunks of rank (rank - s) mod R
// that some row of the range sees; dK/dV (kind 1): the query chunks of rank
// (rank + s) mod R that see some key of the range (the rank holding this block at step s).
// Ranges are in increasing position; returns their number (0..2).
// Striped layout (P.ring_layout 2): ranges are in the partner rank's own index space, and
// the fixed range of a dQ item is its query tile [f0, f1): at step s the keys of rank
// j = (rank - s) mod R that a row of the tile can see are [0, min(c, f1)) (the diagonal
// offset of striped_step masks key f1 - 1 when j > rank); the queries of rank
// (rank + s) mod R are [0, c), of which a dK/dV item walks those from its first key on.
__device__ __forceinline__ int ring_ranges_bwd(const BwdParams &P, int kind, int rank, int f0, int f1, int s,
                                               int &a0, int &b0, int &a1, int &b1) {
    const int R = P.ring_R;
    if (P.ring_layout == 2) {
        const int c = P.N / R;
        a0 = a1 = b1 = 0;
        b0 = (kind || !P.causal) ? c : min(c, f1);
        (void)f0;
        (void)s;
        return b0 > 0 ? 1 : 0;
    }
    const int j = kind ? (rank + s) % R : ((rank - s) % R + R) % R;
    int ca0, cb0, ca1 = 0, cb1 = 0, nc;
    if (P.ring_layout == 0) {
        const int c = P.N / R;
        ca0 = j * c;
        cb0 = ca0 + c;
        nc = 1;
    } else {
        const int hc = P.N / (2 * R);
        ca0 = j * hc;
        cb0 = ca0 + hc;
        ca1 = (2 * R - 1 - j) * hc;
        cb1 = ca1 + hc;
        nc = 2;
    }
    int n = 0;
    a0 = b0 = a1 = b1 = 0;
    for (int i = 0; i < nc; ++i) {
        const int ca = i ? ca1 : ca0, cb = i ? cb1 : cb0;
        if (cb <= ca) continue;
        if (P.causal && (kind ? f0 > cb - 1 : ca > f1 - 1)) continue;
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

// Striped layout: the rank holding the streamed tiles of step s and their diagonal offset.
// Rank j's k-th position follows rank r's k-th exactly when j > r, so key k of rank j is
// visible to row i of rank r iff k + [j > r] <= i (dQ: j = (r - s) mod R; dK/dV: the
// queries of rank j = (r + s) mod R see key k of rank r iff k + [r > j] <= i).
__device__ __forceinline__ void striped_step(const BwdParams &P, int kind, int rank, int s, int &srank, int &dg) {
    const int R = P.ring_R;
    const int j = kind ? (rank + s) % R : ((rank - s) % R + R) % R;
    srank = j;
    dg = P.causal ? (kind ? (rank > j ? 1 : 0) : (j > rank ? 1 : 0)) : 0;
}

// Walks the streamed tiles of the later steps (s = 1 .. R-1) of a fused ring item: every
// tile of each range from its first visible one (`vis0` is the first streamed index some
// fixed row pairs with: for dK/dV the query tiles before the range's first visible row
// are skipped; dQ ranges of later steps are wholly visible).
struct BCursor {
    int s, ri, nr, ti, nti;
    int a0, b0, a1, b1, sk0, sk1;
    __device__ __forceinline__ int start() const { return ri ? a1 + (sk1 + ti) * kT : a0 + (sk0 + ti) * kT; }
    __device__ __forceinline__ int end() const { return ri ? b1 : b0; }
};
__device__ __forceinline__ int skip_tiles(int a, int b, int vis0) {
    return vis0 > a ? (min(vis0, b) - a) / kT : 0;
}
__device__ __forceinline__ int vis_tiles(int a, int b, int vis0) {
    const int lo = max(a, vis0);
    return lo < b ? (b - a + kT - 1) / kT - skip_tiles(a, b, vis0) : 0;
}
__device__ __forceinline__ void bcur_seek(const BwdParams &P, int kind, int rank, int f0, int f1, int vis0,
                                          BCursor &c) {
    for (; c.s < P.ring_R; ++c.s) {
        c.nr = ring_ranges_bwd(P, kind, rank, f0, f1, c.s, c.a0, c.b0, c.a1, c.b1);
        c.sk0 = skip_tiles(c.a0, c.b0, vis0);
        c.sk1 = skip_tiles(c.a1, c.b1, vis0);
        const int n0 = c.nr > 0 ? vis_tiles(c.a0, c.b0, vis0) : 0;
        const int n1 = c.nr > 1 ? vis_tiles(c.a1, c.b1, vis0) : 0;
        if (n0 > 0) {
            c.ri = 0;
            c.ti = 0;
            c.nti = n0;
            return;
        }
        if (n1 > 0) {
            c.ri = 1;
            c.ti = 0;
            c.nti = n1;
            return;
        }
    }
}
__device__ __forceinline__ void bcur_begin(const BwdParams &P, int kind, int rank, int f0, int f1, int vis0,
                                           BCursor &c) {
    c.s = 1;
    bcur_seek(P, kind, rank, f0, f1, vis0, c);
}
__device__ __forceinline__ void bcur_next(const BwdParams &P, int kind, int rank, int f0, int f1, int vis0,
                                          BCursor &c) {
    if (++c.ti < c.nti) return;
    if (c.ri == 0 && c.nr > 1) {
        const int n1 = vis_tiles(c.a1, c.b1, vis0);
        if (n1 > 0) {
            c.ri = 1;
            c.ti = 0;
            c.nti = n1;
            return;
        }
    }
    ++c.s;
    bcur_seek(P, kind, rank, f0, f1, vis0, c);
}
// Streamed tiles of the later steps of a fused item.
__device__ __forceinline__ int later_tiles(const BwdParams &P, int kind, int rank, int f0, int f1, int vis0) {
    int n = 0;
    for (int s = 1; s < P.ring_R; ++s) {
        int a0, b0, a1, b1;
        const int nr = ring_ranges_bwd(P, kind, rank, f0, f1, s, a0, b0, a1, b1);
        if (nr > 0) n += vis_tiles(a0, b0, vis0);
        if (nr > 1) n += vis_tiles(a1, b1, vis0);
    }
    return n;
}

// dQ sub-item: query tile of one segment and one (b, h).  Rows [r_lo, r_hi) of the
// segment's fixed range; streamed key tiles: n0 from the first range, then n1 - n0 from
// the second (the first step's ranges sa/sb; for a fused ring, the later steps' tiles
// follow, n in all).
struct QItem {
    int b, h, hk, si, r_lo, r_hi, n0, n1, n;
    int sa0, sb0, sa1, sb1;
};
// The fixed range whose streamed ranges a dQ item walks: its segment's, or under the
// striped layout its own query tile (every step is then a causal prefix of the tile).
__device__ __forceinline__ int q_fix0(const BwdParams &P, const BSeg &S, const QItem &it) {
    return P.ring_layout == 2 ? it.r_lo : S.f0;
}
__device__ __forceinline__ int q_fix1(const BwdParams &P, const BSeg &S, const QItem &it) {
    return P.ring_layout == 2 ? it.r_hi : S.f1;
}
__device__ __forceinline__ bool decode_q(const BwdParams &P, int tps, int L, int sub, QItem &it) {
    const int BH = P.B * P.Hq;
    int bh, qi;
    if (P.single) {  // one segment, single tiles: under causality the last query tile is the heaviest
        if (sub) return false;
        int w;
        group_decode(L, P.head_group, BH, tps, w, bh);
        it.si = 0;
        qi = P.causal ? tps - 1 - w : w;
    } else {
        const int np = tile_pairs(tps);
        const int per_seg = BH * np;
        it.si = L / per_seg;
        const int rem = L - it.si * per_seg;
        bh = rem / np;
        const int pp = rem - bh * np;
        qi = sub ? pp : tps - 1 - pp;  // the later (heavier) query tile first
        if (sub && qi == tps - 1 - pp) return false;
    }
    it.b = bh / P.Hq;
    it.h = bh - it.b * P.Hq;
    it.hk = it.h / (P.Hq / P.Hkv);
    const BSeg &S = P.seg[it.si];
    it.r_lo = S.f0 + qi * kT;
    it.r_hi = min(it.r_lo + kT, S.f1);
    if (P.ring_fused) {
        const int nr = ring_ranges_bwd(P, 0, S.rank, q_fix0(P, S, it), q_fix1(P, S, it), 0, it.sa0, it.sb0, it.sa1,
                                       it.sb1);
        if (nr < 2) it.sa1 = it.sb1 = it.sb0;
    } else {
        it.sa0 = S.s0[0];
        it.sb0 = S.s1[0];
        it.sa1 = S.s0[1];
        it.sb1 = S.s1[1];
    }
    it.n1 = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int a = p ? it.sa1 : it.sa0;
        const int b = p ? it.sb1 : it.sb0;
        const int e = P.causal ? min(b, it.r_hi - S.diag) : b;
        const int np_ = e > a ? (e - a + kT - 1) / kT : 0;
        if (p == 0) it.n0 = np_;
        it.n1 += np_;
    }
    it.n = it.n1;
    if (P.ring_fused && it.n1 > 0) it.n += later_tiles(P, 0, S.rank, q_fix0(P, S, it), q_fix1(P, S, it), 0);
    return true;
}

// Streamed key tile t (t < n1: the first step) of a dQ item: first key index and the end
// of its range.
__device__ __forceinline__ void q_tile(const BSeg &S, const QItem &it, int t, int &k0, int &klim) {
    const int p = t < it.n0 ? 0 : 1;
    k0 = p ? it.sa1 + (t - it.n0) * kT : it.sa0 + t * kT;
    klim = p ? it.sb1 : it.sb0;
    (void)S;
}

// dK/dV sub-item: key tile of one segment and one (b, KV head), the earlier (heavier)
// tile of the pair first; it visits the visible query tiles of both streamed ranges for
// each of the G query heads: n = G * per.
struct KItem {
    int b, hk, si, c_lo, c_hi, t0[2], n0, per0, per, n;
    int sa0, sb0, sa1, sb1;  // the first step's query ranges
};
__device__ __forceinline__ bool decode_kv(const BwdParams &P, int tps, int L, int sub, KItem &it) {
    const int BHk = P.B * P.Hkv;
    int bhk, kj;
    if (P.single) {  // one segment, single tiles: under causality the first key tile is the heaviest
        if (sub) return false;
        group_decode(L, P.head_group, BHk, tps, kj, bhk);
        it.si = 0;
    } else {
        const int np = tile_pairs(tps);
        const int per_seg = BHk * np;
        it.si = L / per_seg;
        const int rem = L - it.si * per_seg;
        bhk = rem / np;
        const int pp = rem - bhk * np;
        kj = sub ? tps - 1 - pp : pp;
        if (sub && kj == pp) return false;
    }
    it.b = bhk / P.Hkv;
    it.hk = bhk - it.b * P.Hkv;
    const BSeg &S = P.seg[it.si];
    it.c_lo = S.f0 + kj * kT;
    it.c_hi = min(it.c_lo + kT, S.f1);
    if (P.ring_fused) {
        const int nr = ring_ranges_bwd(P, 1, S.rank, S.f0, S.f1, 0, it.sa0, it.sb0, it.sa1, it.sb1);
        if (nr < 2) it.sa1 = it.sb1 = it.sb0;
    } else {
        it.sa0 = S.s0[0];
        it.sb0 = S.s1[0];
        it.sa1 = S.s0[1];
        it.sb1 = S.s1[1];
    }
    it.per0 = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int sa = p ? it.sa1 : it.sa0, sb = p ? it.sb1 : it.sb0;
        const int a = P.causal ? max(sa, it.c_lo + S.diag) : sa;
        int np_ = 0, t0 = 0;
        if (a < sb) {
            t0 = (a - sa) / kT;
            np_ = (sb - sa + kT - 1) / kT - t0;
        }
        if (p == 0) {
            it.t0[0] = t0;
            it.n0 = np_;
        } else {
            it.t0[1] = t0;
        }
        it.per0 += np_;
    }
    it.per = it.per0;
    if (P.ring_fused && it.per0 > 0)
        it.per += later_tiles(P, 1, S.rank, S.f0, S.f1, P.causal ? it.c_lo : INT_MIN);
    it.n = (P.Hq / P.Hkv) * it.per;
    return true;
}

// Streamed query tile tt (tt < per0: the first step) of a dK/dV item: first query index
// and the end of its range.
__device__ __forceinline__ void kv_tile0(const KItem &it, int tt, int &q0, int &qlim) {
    const int p = tt < it.n0 ? 0 : 1;
    q0 = p ? it.sa1 + (it.t0[1] + tt - it.n0) * kT : it.sa0 + (it.t0[0] + tt) * kT;
    qlim = p ? it.sb1 : it.sb0;
}

// Sequential walks over an item's streamed tiles (the producer and the element-wise warps
// take them in order): the first step's from the item's ranges, a fused ring's later
// steps from a cursor.
// (The walks avoid runtime divisions per tile where they can: the element-wise warps take a
// tile's walk on their path between tiles, and a division there costs more than the rest of
// the step.)
struct QWalk {
    BCursor c;
    int t = 0;
    int cs = -1, csr = 0, cdg = 0;  // striped: the step whose rank and offset are cached
    // k0, klim: the key tile's first index and its range's end; srank, dg: the rank holding
    // those keys and the tile's diagonal offset (key k visible to row i iff k + dg <= i)
    template <bool FUSED>
    __device__ __forceinline__ void next(const BwdParams &P, const BSeg &S, const QItem &it, int &k0, int &klim,
                                         int &srank, int &dg) {
        srank = S.s_rank;
        dg = S.diag;
        if (!FUSED || t < it.n1) {
            q_tile(S, it, t, k0, klim);
        } else {
            const int f0 = q_fix0(P, S, it), f1 = q_fix1(P, S, it);
            if (t == it.n1) bcur_begin(P, 0, S.rank, f0, f1, 0, c);
            k0 = c.start();
            klim = c.end();
            if (P.ring_layout == 2) {
                if (c.s != cs) {
                    striped_step(P, 0, S.rank, c.s, csr, cdg);
                    cs = c.s;
                }
                srank = csr;
                dg = cdg;
            }
            bcur_next(P, 0, S.rank, f0, f1, 0, c);
        }
        ++t;
    }
};
struct KWalk {
    BCursor c;
    int t = 0;
    // q0, qlim: the query tile's first index and its range's end; g: its query head in the
    // KV head's group; srank, dg: the rank holding those queries and the diagonal offset
    template <bool FUSED>
    __device__ __forceinline__ void next(const BwdParams &P, const BSeg &S, const KItem &it, int &q0, int &qlim,
                                         int &g, int &srank, int &dg) {
        // tile t's query head in the group and its index in that head's walk (one head per
        // KV head: no division)
        g = P.Hq == P.Hkv ? 0 : t / it.per;
        const int tt = t - g * it.per;
        srank = S.s_rank;
        dg = S.diag;
        if (!FUSED || tt < it.per0) {
            kv_tile0(it, tt, q0, qlim);
        } else {
            const int vis0 = P.causal ? it.c_lo : INT_MIN;
            if (tt == it.per0) bcur_begin(P, 1, S.rank, S.f0, S.f1, vis0, c);
            q0 = c.start();
            qlim = c.end();
            if (P.ring_layout == 2) striped_step(P, 1, S.rank, c.s, srank, dg);
            bcur_next(P, 1, S.rank, S.f0, S.f1, vis0, c);
        }
        ++t;
    }
};

// ---------------------------------------------------------------- shared pieces

__device__ __forceinline__ void bwd_init(BBars *bars, int nst, uint32_t readers) {
    bars->abort = 0;
    bars->p_count[0] = bars->p_count[1] = 0;
    bars->ds_count[0] = bars->ds_count[1] = 0;
    mbar_init(smem_u32(&bars->fix_full), 1);
    mbar_init(smem_u32(&bars->fix_empty), 1);
    for (int s = 0; s < nst; ++s) {
        mbar_init(smem_u32(&bars->full[s]), 1);
        mbar_init(smem_u32(&bars->empty[s]), 1);
        mbar_init(smem_u32(&bars->fullv[s]), 1);
        mbar_init(smem_u32(&bars->emptyv[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full[0]), 1);
    mbar_init(smem_u32(&bars->s_full[1]), 1);
    mbar_init(smem_u32(&bars->o_full), 1);
    mbar_init(smem_u32(&bars->drain), 1);
    mbar_init(smem_u32(&bars->dq_done[0]), 1);
    mbar_init(smem_u32(&bars->dq_done[1]), 1);
    mbar_init(smem_u32(&bars->drain2), 1);
    for (int i = 0; i < kItemRing; ++i) {
        mbar_init(smem_u32(&bars->it_full[i]), 1);
        mbar_init(smem_u32(&bars->it_empty[i]), readers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// The producer decodes each work item (item number, segment table) once and hands it,
// with its segment, to the MMA thread and the element-wise warps through a ring in
// shared memory; their own decode would sit between one item's last products and the
// next item's first.  `end` marks the end of the launch's items.
template <class ItemT>
struct __align__(16) Rec {
    ItemT it;
    BSeg seg;
    int end;
};
template <class R>
__device__ __forceinline__ bool ring_put(BBars *bars, uint32_t &cnt, const R &r, volatile int32_t *abort_flag,
                                         int64_t limit, int *err) {
    static_assert(sizeof(R) <= sizeof(bars->it_rec[0]) && sizeof(R) % 16 == 0, "item record");
    const int slot = cnt & (kItemRing - 1);
    if (cnt >= (uint32_t)kItemRing &&
        !wait_phase(smem_u32(&bars->it_empty[slot]), (cnt / kItemRing - 1u) & 1u, abort_flag, limit, err))
        return false;
#pragma unroll
    for (int i = 0; i < (int)(sizeof(R) / 16); ++i)
        reinterpret_cast<int4 *>(&bars->it_rec[slot][0])[i] = reinterpret_cast<const int4 *>(&r)[i];
    mbar_arrive(smem_u32(&bars->it_full[slot]));  // release: the record is visible
    ++cnt;
    return true;
}
// every lane of the calling warp reads the record; `arrive`: this lane frees the slot
template <class R>
__device__ __forceinline__ bool ring_get(BBars *bars, uint32_t &cnt, R &r, bool warp_wide, volatile int32_t *abort_flag,
                                         int64_t limit, int *err) {
    const int slot = cnt & (kItemRing - 1);
    if (!wait_phase(smem_u32(&bars->it_full[slot]), (cnt / kItemRing) & 1u, abort_flag, limit, err)) return false;
#pragma unroll
    for (int i = 0; i < (int)(sizeof(R) / 16); ++i)
        reinterpret_cast<int4 *>(&r)[i] = reinterpret_cast<const int4 *>(&bars->it_rec[slot][0])[i];
    if (warp_wide) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&bars->it_empty[slot]));
    } else {
        mbar_arrive(smem_u32(&bars->it_empty[slot]));
    }
    ++cnt;
    return true;
}


// The fixed pair of an item is read once, from DRAM, and its loads wait until the previous
// item's last product on the pair is done: start it towards L2 as soon as the item is known.
template <int HD>
__device__ __forceinline__ void prefetch_fixed(const CUtensorMap *fa, const CUtensorMap *fb, int f_row, int f_rank,
                                               int fh, int b, bool fix_in) {
    for (int c = 0; c < BCfg<HD>::SLABS && fix_in; ++c) {
        tma_prefetch_5d(fa, c * 64, f_rank, f_row, fh, b);
        tma_prefetch_5d(fb, c * 64, f_rank, f_row, fh, b);
    }
}

// Producer: per item the fixed pair (fa, fb) at index f_row of rank f_rank of (fh, b), then
// `n` streamed pairs (sa, sb) at the index and head coords(t) gives, of rank s_rank.
// fix_in and coords' result: the coordinates lie inside their tensors (always true in
// release builds; a debug build skips the loads of a tile outside, see in_bounds).
// Shared by both kernels.
template <int HD, typename StreamCoords>
__device__ __forceinline__ bool produce_item(BBars *bars, uint32_t fix0, uint32_t st0, int &slot, uint32_t &ph,
                                             uint32_t &fcnt, uint32_t &issued, uint32_t &last_ph,
                                             const CUtensorMap *fa, const CUtensorMap *fb, int f_row, int f_rank,
                                             int fh, const CUtensorMap *sa, const CUtensorMap *sb,
                                             int n, int b, bool fix_in,
                                             StreamCoords coords, volatile int32_t *abort_flag,
                                             int64_t limit, int *err) {
    using C = BCfg<HD>;
    prefetch_fixed<HD>(fa, fb, f_row, f_rank, fh, b, fix_in);
    if (!wait_phase(smem_u32(&bars->fix_empty), (fcnt & 1u) ^ 1u, abort_flag, limit, err)) return false;
    {
        const uint32_t bf = smem_u32(&bars->fix_full);
        mbar_expect_tx(bf, 2 * C::TILE_BYTES);
        for (int c = 0; c < C::SLABS && fix_in; ++c) {
            tma_load_5d(fix0 + c * C::SLAB_BYTES, fa, bf, c * 64, f_rank, f_row, fh, b);
            tma_load_5d(fix0 + C::TILE_BYTES + c * C::SLAB_BYTES, fb, bf, c * 64, f_rank, f_row, fh, b);
        }
        ++fcnt;
    }
    for (int t = 0; t < n; ++t) {
        if (!wait_phase(smem_u32(&bars->empty[slot]), ph ^ 1u, abort_flag, limit, err)) return false;
        int row, head, s_rank;
        const bool in = coords(t, row, head, s_rank);
        const uint32_t bf = smem_u32(&bars->full[slot]);
        mbar_expect_tx(bf, 2 * C::TILE_BYTES);
        const uint32_t a0 = st0 + (2 * slot) * C::TILE_BYTES;
        for (int c = 0; c < C::SLABS && in; ++c) {
            tma_load_5d(a0 + c * C::SLAB_BYTES, sa, bf, c * 64, s_rank, row, head, b);
            tma_load_5d(a0 + C::TILE_BYTES + c * C::SLAB_BYTES, sb, bf, c * 64, s_rank, row, head, b);
        }
        issued |= 1u << slot;
        last_ph = (last_ph & ~(1u << slot)) | (ph << slot);
        if (++slot == C::NST) {
            slot = 0;
            ph ^= 1u;
        }
    }
    return true;
}

// A ring of single-tile buffers: slot, phase, and for a bounded drain on abort the slots
// with loads in flight and their phases.
struct Ring {
    int slot;
    uint32_t ph, issued, last_ph;
    template <int DEPTH>
    __device__ __forceinline__ void advance() {
        if (++slot == DEPTH) {
            slot = 0;
            ph ^= 1u;
        }
    }
};

// Producer of the dQ kernel: per item the fixed pair (Q, dO), then for each streamed tile
// its K into the K ring and its V into the V ring.
template <int HD, typename StreamCoords>
__device__ __forceinline__ bool produce_item_kv(BBars *bars, uint32_t fix0, uint32_t k0, uint32_t v0, Ring &kr,
                                                Ring &vr, uint32_t &fcnt, const CUtensorMap *fa,
                                                const CUtensorMap *fb, int f_row, int f_rank, int fh,
                                                const CUtensorMap *tk, const CUtensorMap *tv, int n,
                                                int b, bool fix_in, StreamCoords coords, volatile int32_t *abort_flag,
                                                int64_t limit, int *err) {
    using C = BCfg<HD>;
    prefetch_fixed<HD>(fa, fb, f_row, f_rank, fh, b, fix_in);
    if (!wait_phase(smem_u32(&bars->fix_empty), (fcnt & 1u) ^ 1u, abort_flag, limit, err)) return false;
    {
        const uint32_t bf = smem_u32(&bars->fix_full);
        mbar_expect_tx(bf, 2 * C::TILE_BYTES);
        for (int c = 0; c < C::SLABS && fix_in; ++c) {
            tma_load_5d(fix0 + c * C::SLAB_BYTES, fa, bf, c * 64, f_rank, f_row, fh, b);
            tma_load_5d(fix0 + C::TILE_BYTES + c * C::SLAB_BYTES, fb, bf, c * 64, f_rank, f_row, fh, b);
        }
        ++fcnt;
    }
    for (int t = 0; t < n; ++t) {
        int row, head, s_rank;
        const bool in = coords(t, row, head, s_rank);
        for (int which = 0; which < 2; ++which) {
            Ring &r = which ? vr : kr;
            uint64_t *emp = which ? bars->emptyv : bars->empty;
            uint64_t *ful = which ? bars->fullv : bars->full;
            if (!wait_phase(smem_u32(&emp[r.slot]), r.ph ^ 1u, abort_flag, limit, err)) return false;
            const uint32_t bf = smem_u32(&ful[r.slot]);
            mbar_expect_tx(bf, C::TILE_BYTES);
            const uint32_t dst = (which ? v0 : k0) + r.slot * C::TILE_BYTES;
            for (int c = 0; c < C::SLABS && in; ++c)
                tma_load_5d(dst + c * C::SLAB_BYTES, which ? tv : tk, bf, c * 64, s_rank, row, head, b);
            r.issued |= 1u << r.slot;
            r.last_ph = (r.last_ph & ~(1u << r.slot)) | (r.ph << r.slot);
            if (which)
                r.advance<C::VST>();
            else
                r.advance<C::KST>();
        }
    }
    return true;
}

// D = A B^T over K = HD into the 128 x 128 fp32 tile at tensor-memory column tcol: A and
// B are 128-row tiles in shared memory, K-major (SWIZZLE_128B slabs of 64 columns).
template <int HD>
__device__ __forceinline__ void issue_nt(uint32_t tcol, uint32_t a, uint32_t b) {
    using C = BCfg<HD>;
    constexpr uint32_t ID = idesc_bf16(kT, kT, false);
    const SDesc ad = sdesc_split(a, 16, 1024), bd = sdesc_split(b, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::SLAB_BYTES + (kk & 3) * 32;
        mma_ss(tcol, ad.at(off), bd.at(off), ID, kk > 0);
    }
}

// acc += X B over K = 128: X (bf16, 128 x 128) in tensor memory at column xcol (64 packed
// columns), B a 128-row tile in shared memory read as an MN-major operand (N = HD).
template <int HD>
__device__ __forceinline__ void issue_tn(uint32_t acc, uint32_t xcol, uint32_t bsrc, bool accumulate) {
    using C = BCfg<HD>;
    constexpr uint32_t ID = idesc_bf16(kT, HD, true);
    const SDesc bd = sdesc_split(bsrc, C::SLAB_BYTES, 1024);
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk)
        mma_ts(acc, xcol + kk * 8, bd.at(kk * 16 * 128), ID, (accumulate || kk > 0) ? 1u : 0u);
}

// Tensor-memory slots of tile g in the dQ kernel's rotation.
__device__ __forceinline__ uint32_t s_slot(uint32_t g) {
    const uint32_t r = g % 3u;
    return r == 0 ? 0u : (r == 1 ? 256u : 128u);
}
__device__ __forceinline__ uint32_t d_slot(uint32_t g) {
    const uint32_t r = g % 3u;
    return r == 0 ? 128u : (r == 1 ? 0u : 256u);
}

// Invisible entries of 32 scores become -inf (P = 0, dS = 0): e < lo or e >= hi.
__device__ __forceinline__ void mask32(uint32_t (&v)[32], int lo, int hi) {
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = (e >= lo && e < hi) ? v[e] : kNegInfBits;
}

// 32 columns of one gradient row: mul * the step's value, plus the running value of earlier
// steps unless the range is new this step; bf16 to the gradient on the range's last step,
// else fp32 to the running buffer.
__device__ __forceinline__ void store_grad_chunk(__nv_bfloat16 *dst, float *acc, const uint32_t (&o)[32],
                                                 float mul, int flags) {
    float x[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) x[e] = mul * __uint_as_float(o[e]);
    if (!(flags & SEG_FIRST)) {
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 a = __ldcs(reinterpret_cast<const float4 *>(acc + e));
            x[e] += a.x;
            x[e + 1] += a.y;
            x[e + 2] += a.z;
            x[e + 3] += a.w;
        }
    }
    if (flags & SEG_FINAL) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
            uint4 v4;
            v4.x = pack_bf16x2(x[e], x[e + 1]);
            v4.y = pack_bf16x2(x[e + 2], x[e + 3]);
            v4.z = pack_bf16x2(x[e + 4], x[e + 5]);
            v4.w = pack_bf16x2(x[e + 6], x[e + 7]);
            *reinterpret_cast<uint4 *>(dst + e) = v4;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
            __stcs(reinterpret_cast<float4 *>(acc + e), make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]));
    }
}

// ---------------------------------------------------------------- dQ kernel

// Element-wise work of one tile in the dQ kernel for this warp's 64 columns: P from the
// S registers (already masked), then dS = P (dP - D) chunk by chunk into the dP slot.
// FIRST is the chunk (0: columns 0-31 of the group, 1: 32-63) processed first.
template <int FIRST>
__device__ __forceinline__ void dq_tile_ew(uint32_t (&sv)[64], uint32_t tD, int grp, float d_r) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = cc == 0 ? FIRST : 1 - FIRST;
        uint32_t dp[32];
        tmem_ld32_wait(tD + grp * 64 + c * 32, dp);
        uint32_t pk[16];
        const uint64_t d2 = pack_f32x2(d_r, d_r);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {  // dS = P (dP - D), two columns per paired op
            const uint64_t ds = fmul2(pack_f32x2(__uint_as_float(sv[c * 32 + e]), __uint_as_float(sv[c * 32 + e + 1])),
                                      fsub2(pack_f32x2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), d2));
            float d0, d1;
            unpack_f32x2(ds, d0, d1);
            pk[e / 2] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tD + 32 + 32 * grp + 16 * c, pk);
    }
}

template <int HD, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ BwdParams P, int total, int64_t limit, int *err) {
    using C = BCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sQ = base, sDo = base + C::TILE_BYTES;
    const uint32_t sK = base + 2 * C::TILE_BYTES;               // ring of K tiles
    const uint32_t sV = base + (2 + C::KST) * C::TILE_BYTES;    // ring of V tiles
    BBars *bars = reinterpret_cast<BBars *>(base_ptr + C::BAR_OFF_DQ);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((int)blockIdx.x >= total) {
        if (threadIdx.x == 0) sched_finish(P.sched);
        return;
    }
    volatile int32_t *abort_flag = &bars->abort;
    const int tps = (P.flen + kT - 1) / kT;
    const float sl2 = P.scale_log2;

    if (threadIdx.x == 0) bwd_init(bars, 4, kItemReadersDq);
    if (warp == 1) tmem_alloc(smem_u32(&bars->tmem_base), C::TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // the dK/dV kernel reads only inputs ready before this launch: it may start on the
    // SMs this grid frees
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            producer_delay(P.producer_delay_ns);
            Ring kr = {0, 0u, 0u, 0u}, vr = {0, 0u, 0u, 0u};
            uint32_t fcnt = 0, rcnt = 0;
            bool ok = true;
            int L = 0;
            for (int k2 = 0; ok; ++k2) {  // (item, tile of the pair)
                if (!(k2 & 1)) L = atomicAdd(&P.sched[0], 1);  // the next item number
                if (L >= total) break;
                Rec<QItem> rec;
                if (!decode_q(P, tps, L, k2 & 1, rec.it)) continue;
                rec.seg = P.seg[rec.it.si];
                rec.end = 0;
                if (!(ok = ring_put(bars, rcnt, rec, abort_flag, limit, err))) break;
                const QItem &it = rec.it;
                if (it.n == 0) continue;
                const BSeg &S = rec.seg;
                const int hk = it.hk;
                QWalk walk;
                auto coords = [&](int t, int &row, int &head, int &srank) -> bool {
                    int klim, dg;
                    walk.next<FUSED>(P, S, it, row, klim, srank, dg);
                    head = hk;
                    (void)t;
                    return in_bounds(row >= 0 && row < P.N / P.rs && hk < P.Hkv && srank >= 0 && srank < P.rs, err);
                };
                const bool fix_in = in_bounds(it.r_lo >= 0 && it.r_lo < P.N / P.rs && it.h < P.Hq &&
                                                  S.f_rank < P.rs && it.b < P.B,
                                              err);
                ok = produce_item_kv<HD>(bars, sQ, sK, sV, kr, vr, fcnt, &tm_q, &tm_do, it.r_lo, S.f_rank, it.h,
                                         &tm_k, &tm_v, it.n, it.b, fix_in, coords, abort_flag, limit, err);
            }
            if (ok) {  // no more items
                Rec<QItem> rec;
                memset(&rec, 0, sizeof rec);
                rec.end = 1;
                ok = ring_put(bars, rcnt, rec, abort_flag, limit, err);
            }
            if (!ok) {
                if (fcnt) wait_phase_drain(smem_u32(&bars->fix_full), (fcnt - 1u) & 1u);
                for (int s2 = 0; s2 < C::KST; ++s2)
                    if (kr.issued & (1u << s2)) wait_phase_drain(smem_u32(&bars->full[s2]), (kr.last_ph >> s2) & 1u);
                for (int s2 = 0; s2 < C::VST; ++s2)
                    if (vr.issued & (1u << s2))
                        wait_phase_drain(smem_u32(&bars->fullv[s2]), (vr.last_ph >> s2) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // S / dP issuer.  Tile g's S goes to the slot that held dS of tile g - 2, so it
            // waits for that tile's dQ product (the other issuer's) to complete; its dP goes
            // to the slot of tile g - 1's S once the element-wise warps have read that.
            Ring kr = {0, 0u, 0u, 0u}, vr = {0, 0u, 0u, 0u};
            uint32_t fcnt = 0, g = 0;
            bool ok = true;
            uint32_t rcnt = 0;
            while (ok) {
                Rec<QItem> rec;
                if (!(ok = ring_get(bars, rcnt, rec, false, abort_flag, limit, err))) break;
                if (rec.end) break;
                const QItem &it = rec.it;
                const int n = it.n;
                if (n == 0) continue;
                ok = wait_phase(smem_u32(&bars->fix_full), fcnt & 1u, abort_flag, limit, err);
                ++fcnt;
                for (int t = 0; ok && t < n; ++t, ++g) {
                    // dq_done[g & 1] completes once per tile of that parity: tile g - 2's is
                    // its completion number (g - 2) / 2
                    if (g >= 2) {
                        ok = wait_phase(smem_u32(&bars->dq_done[g & 1u]), ((g - 2u) >> 1) & 1u, abort_flag, limit, err);
                        if (!ok) break;
                    }
                    ok = wait_phase(smem_u32(&bars->full[kr.slot]), kr.ph, abort_flag, limit, err);
                    if (!ok) break;
                    tc_fence_after();
                    issue_nt<HD>(tmem + s_slot(g), sQ, sK + kr.slot * C::TILE_BYTES);  // S = Q K^T
                    if (g > 0) {  // this tile's dP goes where the previous tile's S was read from
                        ok = wait_count(&bars->p_count[0], (uint32_t)kEwWarps * g, abort_flag, limit, err);
                        if (!ok) break;
                    }
                    ok = wait_phase(smem_u32(&bars->fullv[vr.slot]), vr.ph, abort_flag, limit, err);
                    if (!ok) break;
                    tc_fence_after();
                    issue_nt<HD>(tmem + d_slot(g), sDo, sV + vr.slot * C::TILE_BYTES);  // dP = dO V^T
                    mma_commit(smem_u32(&bars->s_full[0]));
                    mma_commit(smem_u32(&bars->emptyv[vr.slot]));  // the V tile is free
                    vr.advance<C::VST>();
                    if (t == n - 1) mma_commit(smem_u32(&bars->fix_empty));
                    kr.advance<C::KST>();  // (the dQ issuer frees the K tile)
                }
            }
            mma_commit(smem_u32(&bars->drain));
            wait_phase_drain(smem_u32(&bars->drain), 0);
        }
    } else if (warp == 2) {
        if (lane == 0) {
            // dQ issuer: dQ += dS K for each tile once the element-wise warps have stored its
            // dS.  A thread that issues tcgen05 MMAs stalls on each until the tensor pipe
            // takes it, and the pipe runs dry while that thread waits on anything; with the
            // dQ products on their own thread, the waits of each issuer are covered by the
            // other's products.  Tile g's K tile sits in slot g mod KST of the K ring.
            uint32_t g = 0, rcnt = 0;
            bool ok = true;
            while (ok) {
                Rec<QItem> rec;
                if (!(ok = ring_get(bars, rcnt, rec, false, abort_flag, limit, err))) break;
                if (rec.end) break;
                const int n = rec.it.n;
                for (int t = 0; ok && t < n; ++t, ++g) {
                    // every element-wise warp has stored tile g's dS.  A count summed over the
                    // warps can reach 8 (g + 1) early: the warps that are done may already
                    // store tile g + 1's dS (its dP does not wait for this product) while one
                    // still works on tile g.  No warp gets two tiles ahead of another (tile
                    // g + 2's S needs every warp to have read tile g + 1's), so counting the
                    // tiles of each parity apart makes the count exact.
                    ok = wait_count(&bars->ds_count[g & 1u], (uint32_t)kEwWarps * ((g >> 1) + 1u), abort_flag, limit,
                                    err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t ks = g % (uint32_t)C::KST;
                    issue_tn<HD>(tmem + C::TM_DQ, tmem + d_slot(g) + 32, sK + ks * C::TILE_BYTES,
                                 t > 0);  // dQ += dS K
                    mma_commit(smem_u32(&bars->dq_done[g & 1u]));
                    mma_commit(smem_u32(&bars->empty[ks]));  // the K tile is free
                    if (t == n - 1) mma_commit(smem_u32(&bars->o_full));
                }
            }
            mma_commit(smem_u32(&bars->drain2));
            wait_phase_drain(smem_u32(&bars->drain2), 0);
        }
    } else if (warp >= 4) {
        const int quarter = warp & 3;
        const int grp = (warp - 4) >> 2;  // which 64 columns of a tile this warp owns
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t g = 0, icnt = 0, rcnt = 0;
        bool ok = true;
        while (ok) {  // items, decoded by the producer
            Rec<QItem> rec;
            if (!(ok = ring_get(bars, rcnt, rec, true, abort_flag, limit, err))) break;
            if (rec.end) break;
            const QItem &it = rec.it;
            const BSeg &S = rec.seg;
            const int n = it.n;
            const int row = it.r_lo + quarter * 32 + lane;  // index in the fixed range
            const int64_t pos = (int64_t)row * P.rs + S.f_rank;
            const int64_t lrow = ((int64_t)it.b * P.Hq + it.h) * P.N + pos;
            const bool valid = row < it.r_hi && in_bounds(pos < P.N && lrow < (int64_t)P.B * P.Hq * P.N, err);
            // the row's LSE and D, kept as loaded until the first tile's S is in: arithmetic
            // on them here would stall the warp until the loads return
            float lse_raw = 0.f, d_r = 0.f;
            if (valid) {
                lse_raw = P.lse[lrow];
                d_r = P.dvec[lrow];
            }
            float *accp = P.acc_q + lrow * HD;
            if (valid && grp == 0 && !(S.flags & SEG_FIRST))
                for (int i = 0; i < HD * 4; i += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(
                                                          reinterpret_cast<const char *>(accp) + i));
            QWalk walk;
            for (int t = 0; t < n && ok; ++t, ++g) {
                int kt0, klim;
                int srank_t, diag;  // (the keys' rank: the producer's concern here)
                walk.next<FUSED>(P, S, it, kt0, klim, srank_t, diag);
                (void)srank_t;
                ok = wait_phase(smem_u32(&bars->s_full[0]), g & 1u, abort_flag, limit, err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tS = tmem + s_slot(g) + lane_off, tD = tmem + d_slot(g) + lane_off;
                uint32_t sv[64];
                tmem_ld64_wait(tS + grp * 64, sv);
                // S is in registers: its slot may take the next tile's dP
                tc_fence_before();
                __syncwarp();
                if (lane == 0) count_release_add(&bars->p_count[0]);
                // (opaque per tile, so the scaling below stays here and is not hoisted to the load)
                asm volatile("" : "+f"(lse_raw), "+f"(d_r));
                const float nl2 = lse_raw * -kLog2e;  // -LSE in log2 units
                const int k0 = kt0 + grp * 64;  // first key of this warp's columns
                if ((k0 + 64 > klim) || (P.causal && k0 + 63 + diag > row) || !valid) {
                    const int hi = !valid ? 0 : (P.causal ? min(klim, row + 1 - diag) : klim) - k0;
                    mask32(*reinterpret_cast<uint32_t(*)[32]>(&sv[0]), 0, hi);
                    mask32(*reinterpret_cast<uint32_t(*)[32]>(&sv[32]), 0, hi - 32);
                }
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const uint64_t x = ffma2(pack_f32x2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                             pack_f32x2(sl2, sl2), pack_f32x2(nl2, nl2));
                    float x0, x1;
                    unpack_f32x2(x, x0, x1);
                    sv[e] = __float_as_uint(ex2(x0));
                    sv[e + 1] = __float_as_uint(ex2(x1));
                }
                if (grp == 0)
                    dq_tile_ew<1>(sv, tD, 0, d_r);
                else
                    dq_tile_ew<0>(sv, tD, 1, d_r);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) count_release_add(&bars->ds_count[g & 1u]);
            }
            if (!ok) break;
            if (n > 0) {
                ok = wait_phase(smem_u32(&bars->o_full), icnt & 1u, abort_flag, limit, err);
                ++icnt;
                if (!ok) break;
                tc_fence_after();
            }
            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(P.dq) + (int64_t)it.b * P.sdq[0] +
                                  (int64_t)it.h * P.sdq[1] + pos * P.sdq[2];
            for (int c = grp * (HD / 64); c < (grp + 1) * (HD / 64); ++c) {  // this group's columns
                uint32_t o[32];
                if (n > 0) {
                    tmem_ld32_wait(tmem + C::TM_DQ + lane_off + c * 32, o);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (!valid) continue;
                store_grad_chunk(orow + c * 32, accp + c * 32, o, P.scale, S.flags);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
    if (threadIdx.x == 0) sched_finish(P.sched);
}

// ---------------------------------------------------------------- dK / dV kernel

// Pack 64 fp32 values (this warp's columns) to bf16 into the 32 packed columns at
// 32 + 32 * grp of the slot at t, the chunk FIRST first (see the tensor-memory layout).
template <int FIRST>
__device__ __forceinline__ void pack_store64(const uint32_t (&v)[64], uint32_t t, int grp) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = cc == 0 ? FIRST : 1 - FIRST;
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
            pk[e / 2] = pack_bf16x2(__uint_as_float(v[c * 32 + e]), __uint_as_float(v[c * 32 + e + 1]));
        tmem_st16(t + 32 + 32 * grp + 16 * c, pk);
    }
}

// dS = P (dP - D) for this warp's 64 columns, chunk by chunk from the dP slot at tD, into
// the packed columns of that slot, the chunk FIRST first.
template <int FIRST>
__device__ __forceinline__ void ds_tile_ew(const uint32_t (&pv)[64], uint32_t tD, int grp, const float *du) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = cc == 0 ? FIRST : 1 - FIRST;
        uint32_t dp[32];
        tmem_ld32_wait(tD + grp * 64 + c * 32, dp);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {  // two columns per paired op
            const uint64_t ds = fmul2(pack_f32x2(__uint_as_float(pv[c * 32 + e]), __uint_as_float(pv[c * 32 + e + 1])),
                                      fsub2(pack_f32x2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                            pack_f32x2(du[c * 32 + e], du[c * 32 + e + 1])));
            float d0, d1;
            unpack_f32x2(ds, d0, d1);
            pk[e / 2] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tD + 32 + 32 * grp + 16 * c, pk);
    }
}

template <int HD, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                       const __grid_constant__ BwdParams P, int total, int64_t limit, int *err) {
    using C = BCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sK = base, sV = base + C::TILE_BYTES;
    const uint32_t sSt = base + 2 * C::TILE_BYTES;  // stages of (Q, dO)
    BBars *bars = reinterpret_cast<BBars *>(base_ptr + C::BAR_OFF);
    // per element-wise warp: the current query tile's LSE (log2 units) and D values of its columns
    float *s_stage = reinterpret_cast<float *>(base_ptr + C::BAR_OFF + kBarBytes);  // [8 warps][2][64]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((int)blockIdx.x >= total) {
        if (threadIdx.x == 0) sched_finish(P.sched);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    volatile int32_t *abort_flag = &bars->abort;
    const int G = P.Hq / P.Hkv;
    const int tps = (P.flen + kT - 1) / kT;
    const float sl2 = P.scale_log2;

    if (threadIdx.x == 0) bwd_init(bars, C::NST, kItemReaders);
    if (warp == 1) tmem_alloc(smem_u32(&bars->tmem_base), C::TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            producer_delay(P.producer_delay_ns);
            int slot = 0;
            uint32_t ph = 0, fcnt = 0, issued = 0, last_ph = 0, rcnt = 0;
            bool ok = true;
            int L = 0;
            for (int k2 = 0; ok; ++k2) {  // (item, tile of the pair)
                if (!(k2 & 1)) L = atomicAdd(&P.sched[0], 1);  // the next item number
                if (L >= total) break;
                Rec<KItem> rec;
                if (!decode_kv(P, tps, L, k2 & 1, rec.it)) continue;
                rec.seg = P.seg[rec.it.si];
                rec.end = 0;
                if (!(ok = ring_put(bars, rcnt, rec, abort_flag, limit, err))) break;
                const KItem &it = rec.it;
                if (it.n == 0) continue;
                const BSeg &S = rec.seg;
                const int hk = it.hk;
                KWalk walk;
                auto coords = [&](int t, int &row, int &head, int &srank) -> bool {
                    int qlim, g, dg;
                    walk.next<FUSED>(P, S, it, row, qlim, g, srank, dg);
                    head = hk * G + g;
                    (void)t;
                    return in_bounds(row >= 0 && row < P.N / P.rs && head < P.Hq && srank >= 0 && srank < P.rs, err);
                };
                const bool fix_in = in_bounds(it.c_lo >= 0 && it.c_lo < P.N / P.rs && hk < P.Hkv &&
                                                  S.f_rank < P.rs && it.b < P.B,
                                              err);
                ok = produce_item<HD>(bars, sK, sSt, slot, ph, fcnt, issued, last_ph, &tm_k, &tm_v, it.c_lo,
                                      S.f_rank, hk, &tm_q, &tm_do, it.n, it.b, fix_in, coords, abort_flag,
                                      limit, err);
            }
            if (ok) {  // no more items
                Rec<KItem> rec;
                memset(&rec, 0, sizeof rec);
                rec.end = 1;
                ok = ring_put(bars, rcnt, rec, abort_flag, limit, err);
            }
            if (!ok) {
                if (fcnt) wait_phase_drain(smem_u32(&bars->fix_full), (fcnt - 1u) & 1u);
                for (int s2 = 0; s2 < C::NST; ++s2)
                    if (issued & (1u << s2)) wait_phase_drain(smem_u32(&bars->full[s2]), (last_ph >> s2) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int slot = 0;
            uint32_t ph = 0, fcnt = 0, g = 0;
            bool ok = true;
            uint32_t rcnt = 0;
            while (ok) {
                Rec<KItem> rec;
                if (!(ok = ring_get(bars, rcnt, rec, false, abort_flag, limit, err))) break;
                if (rec.end) break;
                const KItem &it = rec.it;
                const int n = it.n;
                if (n == 0) continue;
                ok = wait_phase(smem_u32(&bars->fix_full), fcnt & 1u, abort_flag, limit, err);
                ++fcnt;
                if (!ok) break;
                // Order of the products, tile t: ... dV(t), S^T(t+1), dK(t), dP^T(t+1), dV(t+1) ...
                // S^T(t+1) overwrites P^T(t), read by dV(t) before it; dP^T(t+1) overwrites
                // dS^T(t), read by dK(t) before it (tcgen05 MMAs of a thread run in order).
                // So the next tile's S^T is computed while the element-wise warps work on
                // this tile's dS^T, and its dP^T while they work on its P^T.
                auto load_wait = [&]() -> bool {
                    if (!wait_phase(smem_u32(&bars->full[slot]), ph, abort_flag, limit, err)) return false;
                    tc_fence_after();
                    return true;
                };
                int nslot = slot;
                uint32_t nph = ph;
                auto next_stage = [&]() {
                    if (++nslot == C::NST) {
                        nslot = 0;
                        nph ^= 1u;
                    }
                };
                if (!(ok = load_wait())) break;
                issue_nt<HD>(tmem + 0, sK, sSt + (2 * slot) * C::TILE_BYTES);  // S^T(0) = K Q^T
                mma_commit(smem_u32(&bars->s_full[0]));
                issue_nt<HD>(tmem + 128, sV, sSt + (2 * slot) * C::TILE_BYTES + C::TILE_BYTES);  // dP^T(0)
                mma_commit(smem_u32(&bars->s_full[1]));
                if (n == 1) mma_commit(smem_u32(&bars->fix_empty));
                for (int t = 0; ok && t < n; ++t, ++g) {
                    const uint32_t qb = sSt + (2 * slot) * C::TILE_BYTES;
                    ok = wait_count(&bars->p_count[0], (uint32_t)kEwWarps * (g + 1u), abort_flag, limit, err);
                    if (!ok) break;
                    tc_fence_after();
                    issue_tn<HD>(tmem + C::TM_A0, tmem + 0 + 32, qb + C::TILE_BYTES, t > 0);  // dV += P^T dO
                    nslot = slot;
                    nph = ph;
                    next_stage();
                    const uint32_t nb = sSt + (2 * nslot) * C::TILE_BYTES;
                    if (t + 1 < n) {
                        if (!wait_phase(smem_u32(&bars->full[nslot]), nph, abort_flag, limit, err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_nt<HD>(tmem + 0, sK, nb);  // S^T(t+1)
                        mma_commit(smem_u32(&bars->s_full[0]));
                    }
                    ok = wait_count(&bars->p_count[1], (uint32_t)kEwWarps * (g + 1u), abort_flag, limit, err);
                    if (!ok) break;
                    tc_fence_after();
                    issue_tn<HD>(tmem + C::TM_A1, tmem + 128 + 32, qb, t > 0);  // dK += dS^T Q
                    mma_commit(smem_u32(&bars->empty[slot]));
                    if (t == n - 1) mma_commit(smem_u32(&bars->o_full));
                    if (t + 1 < n) {
                        issue_nt<HD>(tmem + 128, sV, nb + C::TILE_BYTES);  // dP^T(t+1)
                        mma_commit(smem_u32(&bars->s_full[1]));
                        if (t + 2 == n) mma_commit(smem_u32(&bars->fix_empty));
                    }
                    slot = nslot;
                    ph = nph;
                }
            }
            mma_commit(smem_u32(&bars->drain));
            wait_phase_drain(smem_u32(&bars->drain), 0);
        }
    } else if (warp >= 4) {
        const int quarter = warp & 3;
        const int grp = (warp - 4) >> 2;  // which 64 columns of a tile this warp owns
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float *lb = s_stage + (warp - 4) * 2 * 64;  // this warp's columns only: no cross-warp barrier
        float *db = lb + 64;
        uint32_t g = 0, icnt = 0, rcnt = 0;
        bool ok = true;
        while (ok) {  // items, decoded by the producer
            Rec<KItem> rec;
            if (!(ok = ring_get(bars, rcnt, rec, true, abort_flag, limit, err))) break;
            if (rec.end) break;
            const KItem &it = rec.it;
            const BSeg &S = P.seg[it.si];  // (read in place: a register copy would spill)
            const int n = it.n;
            const int key = it.c_lo + quarter * 32 + lane;  // index in the fixed range
            const int64_t kpos = (int64_t)key * P.rs + S.f_rank;
            const int64_t arow = (((int64_t)it.b * P.Hkv + it.hk) * P.N + kpos) * HD;
            const bool kvalid = key < it.c_hi && in_bounds(kpos < P.N && it.hk < P.Hkv && it.b < P.B, err);
            if (kvalid && grp == 0 && !(S.flags & SEG_FIRST))
                for (int i = 0; i < HD * 4; i += 128) {
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(P.acc_k + arow) + i));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(P.acc_v + arow) + i));
                }
            // LSE and D of this lane's two queries of tile t; the next tile's are loaded while
            // this one is processed.  fetch() keeps them as loaded: any arithmetic on them
            // here would stall the warp until the load returns (it did: ~750 cycles a tile).
            // They are scaled to log2 units when staged, a tile later.
            // the walk runs one tile ahead: fetch() takes tile t+1's coordinates and values
            // while tile t is processed, and hands the coordinates on
            KWalk walk;
            int nq0 = 0, nqlim = 0, ngh = 0, ndiag = 0;
            auto fetch = [&](int t, float (&l)[2], float (&d)[2]) {
                int q0, qlim, gh, srank, dg;
                walk.next<FUSED>(P, S, it, q0, qlim, gh, srank, dg);
                nq0 = q0;
                nqlim = qlim;
                ngh = gh;
                ndiag = dg;
                (void)t;
                const int h = it.hk * G + gh;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int qme = q0 + grp * 64 + r * 32 + lane;
                    const int64_t li = ((int64_t)it.b * P.Hq + h) * P.N + (int64_t)qme * P.rs + srank;
                    const bool in = qme < qlim && in_bounds(li < (int64_t)P.B * P.Hq * P.N, err);
                    float lv = 0.f, dv = 0.f;
                    if (in) {
                        lv = P.lse[li];
                        dv = P.dvec[li];
                    }
                    l[r] = lv;
                    d[r] = dv;
                }
            };
            float nl[2] = {0.f, 0.f}, nd[2] = {0.f, 0.f};
            if (n > 0) fetch(0, nl, nd);
            for (int t = 0; t < n && ok; ++t, ++g) {
                const int q0 = nq0, qlim = nqlim, diag = ndiag;
                (void)ngh;
                const int qa = q0 + grp * 64;  // first query of this warp's columns
                __syncwarp();  // every lane is done with the previous tile's values
                lb[lane] = nl[0] * -kLog2e;  // -LSE in log2 units: the exponent's FFMA adds it
                lb[32 + lane] = nl[1] * -kLog2e;
                db[lane] = nd[0];
                db[32 + lane] = nd[1];
                __syncwarp();
                if (t + 1 < n) fetch(t + 1, nl, nd);
                ok = wait_phase(smem_u32(&bars->s_full[0]), g & 1u, abort_flag, limit, err);
                if (!ok) break;
                tc_fence_after();
                uint32_t pv[64];
                tmem_ld64_wait(tmem + lane_off + grp * 64, pv);
                if ((qa + 64 > qlim) || (P.causal && it.c_hi - 1 + diag > qa)) {
                    const int lo = P.causal ? key + diag - qa : 0;  // first visible column
                    const int hi = qlim - qa;
                    mask32(*reinterpret_cast<uint32_t(*)[32]>(&pv[0]), lo, hi);
                    mask32(*reinterpret_cast<uint32_t(*)[32]>(&pv[32]), lo - 32, hi - 32);
                }
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const uint64_t x = ffma2(pack_f32x2(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])),
                                             pack_f32x2(sl2, sl2), pack_f32x2(lb[e], lb[e + 1]));
                    float x0, x1;
                    unpack_f32x2(x, x0, x1);
                    pv[e] = __float_as_uint(ex2(x0));
                    pv[e + 1] = __float_as_uint(ex2(x1));
                }
                const uint32_t tSl = tmem + lane_off, tDl = tmem + 128 + lane_off;
                if (grp == 0)
                    pack_store64<1>(pv, tSl, 0);
                else
                    pack_store64<0>(pv, tSl, 1);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) count_release_add(&bars->p_count[0]);  // P^T is in tensor memory
                ok = wait_phase(smem_u32(&bars->s_full[1]), g & 1u, abort_flag, limit, err);
                if (!ok) break;
                tc_fence_after();
                if (grp == 0)
                    ds_tile_ew<1>(pv, tDl, 0, db);
                else
                    ds_tile_ew<0>(pv, tDl, 1, db);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) count_release_add(&bars->p_count[1]);  // dS^T is in tensor memory
            }
            if (!ok) break;
            if (n > 0) {
                ok = wait_phase(smem_u32(&bars->o_full), icnt & 1u, abort_flag, limit, err);
                ++icnt;
                if (!ok) break;
                tc_fence_after();
            }
            __nv_bfloat16 *vrow = static_cast<__nv_bfloat16 *>(P.dv) + (int64_t)it.b * P.sdv[0] +
                                  (int64_t)it.hk * P.sdv[1] + kpos * P.sdv[2];
            __nv_bfloat16 *krow = static_cast<__nv_bfloat16 *>(P.dk) + (int64_t)it.b * P.sdk[0] +
                                  (int64_t)it.hk * P.sdk[1] + kpos * P.sdk[2];
            // Final rows of a key tile that lies wholly inside its range (or is clipped by the
            // end of the tensor) leave through shared memory and bulk tensor stores, 32 rows x
            // 32 columns per warp at a time: row-per-thread stores would issue 32 scattered
            // 16-byte pieces per instruction (measured: the stores cost 6 % of the dense
            // backward).  The rest are written row by row (store_grad_chunk).
            const int row0 = it.c_lo + quarter * 32;
            // (only rows that no other step adds to: first and final, with no running value)
            const bool tma = !FUSED && n > 0 && (S.flags & SEG_FIRST) && (S.flags & SEG_FINAL) && P.dkv_tma &&
                             (it.c_hi - it.c_lo == kT || it.c_hi == P.N / P.rs);
            const uint32_t stg = smem_u32(base_ptr + C::STG_OFF) + (uint32_t)(warp - 4) * 2048u;
            for (int which = 0; which < 2; ++which) {
                const float mul = which ? P.scale : 1.f;
                __nv_bfloat16 *dst = which ? krow : vrow;
                float *acc = (which ? P.acc_k : P.acc_v) + arow;
                const uint32_t col = which ? C::TM_A1 : C::TM_A0;
                for (int c = grp * (HD / 64); c < (grp + 1) * (HD / 64); ++c) {  // this group's columns
                    uint32_t o[32];
                    if (n > 0) {
                        tmem_ld32_wait(tmem + col + lane_off + c * 32, o);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = 0u;
                    }
                    if (tma) {
                        if (row0 >= P.N / P.rs) continue;  // a box wholly past the rows writes nothing
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(mul * __uint_as_float(o[2 * i]), mul * __uint_as_float(o[2 * i + 1]));
                        if (lane == 0) bulk_wait_read0();  // this warp's previous store has read the buffer
                        __syncwarp();
                        // 64-byte swizzle, as the tensor map expects: 16-byte piece j of row r
                        // sits at piece j ^ ((r / 2) mod 4)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t a = stg + lane * 64 + ((uint32_t)(j ^ ((lane >> 1) & 3)) << 4);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pk[4 * j]),
                                         "r"(pk[4 * j + 1]), "r"(pk[4 * j + 2]), "r"(pk[4 * j + 3])
                                         : "memory");
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && in_bounds(row0 >= 0 && S.f_rank < P.rs && it.hk < P.Hkv && it.b < P.B, err)) {
                            tma_store_5d(which ? &tm_dk : &tm_dv, stg, c * 32, S.f_rank, row0, it.hk, it.b);
                            bulk_commit();
                        }
                        __syncwarp();
                        continue;
                    }
                    if (!kvalid) continue;
                    store_grad_chunk(dst + c * 32, acc + c * 32, o, mul, S.flags);
                }
            }
        }
    }
    // the bulk stores of dK/dV issued by each element-wise warp are complete before exit
    if (warp >= 4 && lane == 0) bulk_wait0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
    if (threadIdx.x == 0) sched_finish(P.sched);
    // when launched to overlap the dQ kernel's tail, finish only after it has: work later
    // in the stream then sees both kernels' writes (a no-op for a plain launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace tcb

// Units per head group of single-tile backward items: whole KV heads whose streamed
// tiles (dQ kernel: K and V, 4 N D bytes per KV head; dK/dV kernel: Q and dO of its G query
// heads) fit in 48 MiB, so they stay in the 129 MB L2 while the group runs; counted in
// query heads for the dQ kernel, in (batch, KV head) units for the dK/dV kernel.  0: one
// group (everything fits).
static int32_t bwd_head_group(const BwdParams &P, int kind) {
    const int64_t G = P.Hkv > 0 ? P.Hq / P.Hkv : 1;
    const double per_kv = 4.0 * (double)P.N * (double)P.D * (kind ? (double)G : 1.0);
    const int64_t units = (int64_t)P.B * P.Hkv;
    const int64_t kv = std::max<int64_t>((int64_t)(48.0 * (1 << 20) / std::max(per_kv, 1.0)), 1);
    if (kv >= units) return 0;
    return (int32_t)std::min<int64_t>(kind ? kv : kv * G, 1 << 30);
}

template <int HD>
static cudaError_t launch_bwd_tc_hd(const BwdParams &P, int parts, int num_sms, int64_t wait_ns, int *err,
                                    cudaStream_t stream, bool after_dq) {
    using C = tcb::BCfg<HD>;
    static int configured_mask = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(configured_mask & (1 << (dev & 31)))) {
        cudaError_t e = cudaFuncSetAttribute(tcb::bwd_dq_tc_kernel<HD, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES_DQ);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tcb::bwd_dq_tc_kernel<HD, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES_DQ);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tcb::bwd_dkdv_tc_kernel<HD, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tcb::bwd_dkdv_tc_kernel<HD, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES_FUSED);
        if (e != cudaSuccess) return e;
        configured_mask |= 1 << (dev & 31);
    }
    CUtensorMap mq, mk, mv, mdo;
    if (!encode_map(&mq, P.q, P.B, P.Hq, P.N, P.D, P.sq, P.rs) ||
        !encode_map(&mk, P.k, P.B, P.Hkv, P.N, P.D, P.sk, P.rs) ||
        !encode_map(&mv, P.v, P.B, P.Hkv, P.N, P.D, P.sv, P.rs) ||
        !encode_map(&mdo, P.dout, P.B, P.Hq, P.N, P.D, P.sdo, P.rs))
        return cudaErrorInvalidValue;
    const int tps = (P.flen + tcb::kT - 1) / tcb::kT;
    const int np = (tps + 1) / 2;  // tile pairs per segment and head
    // a one-segment launch takes single tiles, longest first, in head groups; otherwise
    // equal-cost tile pairs, segment by segment (a fused ring's items, whose cost is mostly
    // their later steps, keep pairs)
    if (!P.sched || parts == 3) return cudaErrorInvalidValue;  // one work counter pair per launch
    // dK and dV through bulk tensor stores (32 x 32 boxes, 64-byte swizzle) when their
    // layouts allow a map (else row stores)
    CUtensorMap mdk, mdv;
    const bool dkv_map = encode_map(&mdk, P.dk, P.B, P.Hkv, P.N, P.D, P.sdk, P.rs, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) &&
                         encode_map(&mdv, P.dv, P.B, P.Hkv, P.N, P.D, P.sdv, P.rs, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!dkv_map) {
        memset(&mdk, 0, sizeof mdk);
        memset(&mdv, 0, sizeof mdv);
    }
    BwdParams Pq = P, Pk = P;
    Pq.single = Pk.single = (P.nseg == 1 && !P.ring_fused) ? 1 : 0;
    Pq.head_group = Pq.single ? bwd_head_group(P, 0) : 0;
    Pk.head_group = Pk.single ? bwd_head_group(P, 1) : 0;
    Pk.dkv_tma = dkv_map ? 1 : 0;
    const int64_t tq = Pq.single ? (int64_t)P.B * P.Hq * tps : (int64_t)P.B * P.Hq * P.nseg * np;
    const int64_t tkv = Pk.single ? (int64_t)P.B * P.Hkv * tps : (int64_t)P.B * P.Hkv * P.nseg * np;
    if (tq > 0x7fffffff || tkv > 0x7fffffff) return cudaErrorInvalidValue;
    const int gq = (int)std::min<int64_t>(tq, num_sms), gkv = (int)std::min<int64_t>(tkv, num_sms);
    if (parts & 1) {
        if (P.ring_fused)
            tcb::bwd_dq_tc_kernel<HD, true><<<gq, tcb::kThreads, C::SMEM_BYTES_DQ, stream>>>(mq, mk, mv, mdo, Pq, (int)tq,
                                                                                          wait_ns, err);
        else
            tcb::bwd_dq_tc_kernel<HD, false><<<gq, tcb::kThreads, C::SMEM_BYTES_DQ, stream>>>(mq, mk, mv, mdo, Pq,
                                                                                           (int)tq, wait_ns, err);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (parts & 2) {
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = dim3(gkv);
        cfg.blockDim = dim3(tcb::kThreads);
        cfg.dynamicSmemBytes = P.ring_fused ? C::SMEM_BYTES_FUSED : C::SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        if (after_dq || (parts & 1)) {  // overlaps the tail of the dQ kernel just launched (no data between them)
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        const int itkv = (int)tkv;
        cudaError_t e = P.ring_fused
                            ? cudaLaunchKernelEx(&cfg, tcb::bwd_dkdv_tc_kernel<HD, true>, mq, mk, mv, mdo, mdk, mdv, Pk, itkv,
                                                 wait_ns, err)
                            : cudaLaunchKernelEx(&cfg, tcb::bwd_dkdv_tc_kernel<HD, false>, mq, mk, mv, mdo, mdk, mdv, Pk, itkv,
                                                 wait_ns, err);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

// The dQ kernel (parts 1) or the dK/dV kernel (parts 2) over the segments in P (the D
// vector is computed before), taking its items from the work counter pair P.sched: one
// kernel per call, since each launch needs its own pair.
// after_dq: the launch directly follows a dQ kernel on `stream`, so the dK/dV kernel may
// start on the SMs the dQ grid frees (programmatic dependent launch).
cudaError_t launch_attn_bwd_tc(const BwdParams &P, int parts, int num_sms, int64_t wait_ns, int *err,
                               cudaStream_t stream, bool after_dq) {
    if (P.B <= 0 || P.Hq <= 0 || P.nseg <= 0 || P.flen <= 0) return cudaSuccess;
    if (P.D == 128) return launch_bwd_tc_hd<128>(P, parts, num_sms, wait_ns, err, stream, after_dq);
    if (P.D == 64) return launch_bwd_tc_hd<64>(P, parts, num_sms, wait_ns, err, stream, after_dq);
    return cudaErrorInvalidValue;
}

}  // namespace ra
