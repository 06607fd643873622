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
// Warp roles: warp 0 TMA producer, warp 1 MMA issuer and tensor-memory owner, warps 4-11
// the element-wise work and the epilogue: two warps per tensor-memory lane quarter, each
// owning 32 of a sub-tile's 64 columns (one warp per scheduler left the exponentials and
// the tensor-memory round trips exposed).  The streamed tile is handled as two 64-wide
// halves with their own S / dP buffers, so the tensor core computes one half's S / dP
// while the element-wise warps work on the other.  The bf16 P / dS overwrite the
// columns of the fp32 S / dP they came from once those are in registers; the MMA
// thread issues the next S / dP of a half after the products that read it (tcgen05 MMAs
// of a thread run in order).  Every wait is bounded like the forward kernel's.
//
// A launch covers the segments of one ring step (struct BSeg): the whole-sequence
// backward is one segment.  On a ring, the gradient of a range that earlier or later
// steps also write is carried between steps in fp32 running buffers (store_grad_chunk).
#include "tc_common.cuh"

namespace ra {
namespace tcb {

using namespace ra::tc;

constexpr int kT = 128;   // rows per tile (queries or keys)
constexpr int kSub = 64;  // a tile's streamed dimension is processed as two 64-wide halves
constexpr int kThreads = 384;
constexpr int kEwWarps = 8;
constexpr uint32_t kNegInfBits = 0xff800000u;  // -inf as fp32 bits  // warps 4-11: two groups of four, one per 32-column half of a sub-tile

// Tensor memory: for sub-tile u in {0, 1}, S_u at 128u (64 fp32 columns) and dP_u at
// 128u + 64.  Element-wise group g in {0, 1} reads columns [32g, 32g + 32) of S_u / dP_u
// and writes its 32 bf16 values (16 columns) of P_u / dS_u to columns 16 + 16g of them:
// inside what the group itself read, and clear of the other group's columns, so P_u and
// dS_u are 32 contiguous columns at 128u + 16 and 128u + 80.  Accumulators at 256 (dQ or
// dV) and 256 + HD (dK).
template <int HD>
struct BCfg {
    static constexpr int SLABS = HD / 64;
    static constexpr int TILE_BYTES = kT * HD * 2;
    static constexpr int SLAB_BYTES = 128 * 128;
    static constexpr int NST = (HD == 128) ? 2 : 4;  // stages of two tiles
    static constexpr uint32_t TM_A0 = 256, TM_A1 = 256 + HD;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int BAR_OFF = (2 + 2 * NST) * TILE_BYTES;
    static constexpr int SMEM_BYTES = 1024 + BAR_OFF + 256 + kEwWarps * 2 * 64 * 4;
};

struct BBars {
    uint64_t fix_full, fix_empty;  // the item's fixed pair (Q, dO) or (K, V)
    uint64_t full[4], empty[4];    // streamed pairs
    uint64_t s_full[2], o_full, drain;
    uint32_t tmem_base;
    int32_t abort;
    uint32_t p_count[2];
};
static_assert(sizeof(BBars) <= 256, "barrier block");

// Work items are pairs of tiles of one segment and one head: tile p and tile tps-1-p of
// the segment's fixed range.  Under causality the two costs add up to the same total,
// so every item of a segment costs the same; items are numbered segment (heaviest
// first, as the host orders them), then head, then pair, so the CTAs that run at the
// same time share the streamed tiles of a few heads in L2.  `sub` selects the pair's
// first (0) or second (1) tile; false when the pair has a single (middle) tile.
__device__ __forceinline__ int tile_pairs(int tps) { return (tps + 1) >> 1; }

// dQ sub-item: query tile of one segment and one (b, h).  Rows [r_lo, r_hi) of the
// segment's fixed range; streamed key tiles: n0 from the first range, then n - n0 from
// the second.
struct QItem {
    int b, h, hk, si, r_lo, r_hi, n0, n;
};
__device__ __forceinline__ bool decode_q(const BwdParams &P, int tps, int L, int sub, QItem &it) {
    const int BH = P.B * P.Hq;
    const int np = tile_pairs(tps);
    const int per_seg = BH * np;
    it.si = L / per_seg;
    const int rem = L - it.si * per_seg;
    const int bh = rem / np;
    const int pp = rem - bh * np;
    const int qi = sub ? pp : tps - 1 - pp;  // the later (heavier) query tile first
    if (sub && qi == tps - 1 - pp) return false;
    it.b = bh / P.Hq;
    it.h = bh - it.b * P.Hq;
    it.hk = it.h / (P.Hq / P.Hkv);
    const BSeg &S = P.seg[it.si];
    it.r_lo = S.f0 + qi * kT;
    it.r_hi = min(it.r_lo + kT, S.f1);
    it.n = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int a = S.s0[p];
        const int e = P.causal ? min(S.s1[p], it.r_hi - S.diag) : S.s1[p];
        const int np_ = e > a ? (e - a + kT - 1) / kT : 0;
        if (p == 0) it.n0 = np_;
        it.n += np_;
    }
    return true;
}

// Streamed key tile t of a dQ item: first key index and the end of its range.
__device__ __forceinline__ void q_tile(const BSeg &S, const QItem &it, int t, int &k0, int &klim) {
    const int p = t < it.n0 ? 0 : 1;
    k0 = p ? S.s0[1] + (t - it.n0) * kT : S.s0[0] + t * kT;
    klim = p ? S.s1[1] : S.s1[0];
}

// dK/dV sub-item: key tile of one segment and one (b, KV head), the earlier (heavier)
// tile of the pair first; it visits the visible query tiles of both streamed ranges for
// each of the G query heads: n = G * per.
struct KItem {
    int b, hk, si, c_lo, c_hi, t0[2], n0, per, n;
};
__device__ __forceinline__ bool decode_kv(const BwdParams &P, int tps, int L, int sub, KItem &it) {
    const int BHk = P.B * P.Hkv;
    const int np = tile_pairs(tps);
    const int per_seg = BHk * np;
    it.si = L / per_seg;
    const int rem = L - it.si * per_seg;
    const int bhk = rem / np;
    const int pp = rem - bhk * np;
    const int kj = sub ? tps - 1 - pp : pp;
    if (sub && kj == pp) return false;
    it.b = bhk / P.Hkv;
    it.hk = bhk - it.b * P.Hkv;
    const BSeg &S = P.seg[it.si];
    it.c_lo = S.f0 + kj * kT;
    it.c_hi = min(it.c_lo + kT, S.f1);
    it.per = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int a = P.causal ? max(S.s0[p], it.c_lo + S.diag) : S.s0[p];
        int np_ = 0, t0 = 0;
        if (a < S.s1[p]) {
            t0 = (a - S.s0[p]) / kT;
            np_ = (S.s1[p] - S.s0[p] + kT - 1) / kT - t0;
        }
        it.t0[p] = t0;
        if (p == 0) it.n0 = np_;
        it.per += np_;
    }
    it.n = (P.Hq / P.Hkv) * it.per;
    return true;
}

// Streamed query tile t of a dK/dV item: first query index, the end of its range, head.
__device__ __forceinline__ void kv_tile(const BSeg &S, const KItem &it, int G, int t, int &q0, int &qlim,
                                        int &g) {
    g = t / it.per;
    const int tt = t - g * it.per;
    const int p = tt < it.n0 ? 0 : 1;
    q0 = p ? S.s0[1] + (it.t0[1] + tt - it.n0) * kT : S.s0[0] + (it.t0[0] + tt) * kT;
    qlim = p ? S.s1[1] : S.s1[0];
    (void)G;
}

__device__ __forceinline__ int snake(int k) {
    const int G = gridDim.x;
    return k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
}

// ---------------------------------------------------------------- shared pieces

__device__ __forceinline__ void bwd_init(BBars *bars, int nst) {
    bars->abort = 0;
    bars->p_count[0] = bars->p_count[1] = 0;
    mbar_init(smem_u32(&bars->fix_full), 1);
    mbar_init(smem_u32(&bars->fix_empty), 1);
    for (int s = 0; s < nst; ++s) {
        mbar_init(smem_u32(&bars->full[s]), 1);
        mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full[0]), 1);
    mbar_init(smem_u32(&bars->s_full[1]), 1);
    mbar_init(smem_u32(&bars->o_full), 1);
    mbar_init(smem_u32(&bars->drain), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's lane: 16 bf16 pairs.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Producer: per item the fixed pair (fa, fb) at index f_row of rank f_rank of (fh, b), then
// `n` streamed pairs (sa, sb) at the index and head coords(t) gives, of rank s_rank.
// Shared by both kernels.
template <int HD, typename StreamCoords>
__device__ __forceinline__ bool produce_item(BBars *bars, uint32_t fix0, uint32_t st0, int &slot, uint32_t &ph,
                                             uint32_t &fcnt, uint32_t &issued, uint32_t &last_ph,
                                             const CUtensorMap *fa, const CUtensorMap *fb, int f_row, int f_rank,
                                             int fh, const CUtensorMap *sa, const CUtensorMap *sb, int s_rank,
                                             int n, int b,
                                             StreamCoords coords, volatile int32_t *abort_flag,
                                             int64_t limit, int *err) {
    using C = BCfg<HD>;
    if (!wait_phase(smem_u32(&bars->fix_empty), (fcnt & 1u) ^ 1u, abort_flag, limit, err)) return false;
    {
        const uint32_t bf = smem_u32(&bars->fix_full);
        mbar_expect_tx(bf, 2 * C::TILE_BYTES);
        for (int c = 0; c < C::SLABS; ++c) {
            tma_load_5d(fix0 + c * C::SLAB_BYTES, fa, bf, c * 64, f_rank, f_row, fh, b);
            tma_load_5d(fix0 + C::TILE_BYTES + c * C::SLAB_BYTES, fb, bf, c * 64, f_rank, f_row, fh, b);
        }
        ++fcnt;
    }
    for (int t = 0; t < n; ++t) {
        if (!wait_phase(smem_u32(&bars->empty[slot]), ph ^ 1u, abort_flag, limit, err)) return false;
        int row, head;
        coords(t, row, head);
        const uint32_t bf = smem_u32(&bars->full[slot]);
        mbar_expect_tx(bf, 2 * C::TILE_BYTES);
        const uint32_t a0 = st0 + (2 * slot) * C::TILE_BYTES;
        for (int c = 0; c < C::SLABS; ++c) {
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

// MMA issue for S_u = A B_u^T and dP_u = A' B'_u^T (N = 64 of the streamed tile's rows,
// K = HD): the fixed pair (fa, fb) against half u of the streamed pair (sa, sb).
template <int HD>
__device__ __forceinline__ void issue_sdp(uint32_t tmem, int u, uint32_t fa, uint32_t fb, uint32_t sa,
                                          uint32_t sb) {
    using C = BCfg<HD>;
    constexpr uint32_t ID = idesc_bf16(kT, kSub, false);
    const uint32_t half = u * kSub * 128;  // rows 64u.. of each 128-byte-wide slab
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::SLAB_BYTES + (kk & 3) * 32;
        mma_ss(tmem + 128 * u, sdesc_sw128(fa + off, 16, 1024), sdesc_sw128(sa + half + off, 16, 1024), ID,
               kk > 0);
        mma_ss(tmem + 128 * u + 64, sdesc_sw128(fb + off, 16, 1024),
               sdesc_sw128(sb + half + off, 16, 1024), ID, kk > 0);
    }
}

// acc += X_u B_u where X_u (bf16, 128 x 64) sits in tensor memory at column xcol and B_u
// is rows 64u.. of a streamed tile read as an MN-major operand (K = 64, N = HD).
template <int HD>
__device__ __forceinline__ void issue_acc(uint32_t tmem, uint32_t acc_col, uint32_t xcol, uint32_t bsrc, int u,
                                          bool accumulate) {
    using C = BCfg<HD>;
    constexpr uint32_t ID = idesc_bf16(kT, HD, true);
    for (int kk = 0; kk < kSub / 16; ++kk)
        mma_ts(tmem + acc_col, tmem + xcol + kk * 8,
               sdesc_sw128(bsrc + u * kSub * 128 + kk * 16 * 128, C::SLAB_BYTES, 1024), ID,
               (accumulate || kk > 0) ? 1u : 0u);
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

template <int HD>
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
    const uint32_t sSt = base + 2 * C::TILE_BYTES;  // stages of (K, V)
    BBars *bars = reinterpret_cast<BBars *>(base_ptr + C::BAR_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((int)blockIdx.x >= total) return;
    volatile int32_t *abort_flag = &bars->abort;
    const int tps = (P.flen + kT - 1) / kT;
    const float sl2 = P.scale_log2;

    if (threadIdx.x == 0) bwd_init(bars, C::NST);
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
            int slot = 0;
            uint32_t ph = 0, fcnt = 0, issued = 0, last_ph = 0;
            bool ok = true;
            for (int k2 = 0; (k2 >> 1) * (int)gridDim.x < total && ok; ++k2) {  // (item, tile of the pair)
                const int L = snake(k2 >> 1);
                if (L >= total) continue;
                QItem it;
                if (!decode_q(P, tps, L, k2 & 1, it)) continue;
                if (it.n == 0) continue;
                const BSeg &S = P.seg[it.si];
                const int hk = it.hk;
                auto coords = [=, &S](int t, int &row, int &head) {
                    int klim;
                    q_tile(S, it, t, row, klim);
                    head = hk;
                };
                ok = produce_item<HD>(bars, sQ, sSt, slot, ph, fcnt, issued, last_ph, &tm_q, &tm_do, it.r_lo,
                                      S.f_rank, it.h, &tm_k, &tm_v, S.s_rank, it.n, it.b, coords, abort_flag,
                                      limit, err);
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
            uint32_t ph = 0, fcnt = 0, pc[2] = {0u, 0u};
            bool ok = true;
            for (int k2 = 0; (k2 >> 1) * (int)gridDim.x < total && ok; ++k2) {  // (item, tile of the pair)
                const int L = snake(k2 >> 1);
                if (L >= total) continue;
                QItem it;
                if (!decode_q(P, tps, L, k2 & 1, it)) continue;
                const int n = it.n;
                if (n == 0) continue;
                ok = wait_phase(smem_u32(&bars->fix_full), fcnt & 1u, abort_flag, limit, err);
                ++fcnt;
                if (!ok) break;
                // S / dP of both halves of key tile 0
                ok = wait_phase(smem_u32(&bars->full[slot]), ph, abort_flag, limit, err);
                if (!ok) break;
                tc_fence_after();
                for (int u = 0; u < 2; ++u) {
                    const uint32_t kb = sSt + (2 * slot) * C::TILE_BYTES;
                    issue_sdp<HD>(tmem, u, sQ, sDo, kb, kb + C::TILE_BYTES);
                    mma_commit(smem_u32(&bars->s_full[u]));
                }
                if (n == 1) mma_commit(smem_u32(&bars->fix_empty));
                for (int t = 0; ok && t < n; ++t) {
                    const int cur = slot;
                    const uint32_t kb = sSt + (2 * cur) * C::TILE_BYTES;
                    int nslot = slot + 1;
                    uint32_t nph = ph;
                    if (nslot == C::NST) {
                        nslot = 0;
                        nph ^= 1u;
                    }
                    for (int u = 0; u < 2 && ok; ++u) {
                        ++pc[u];
                        ok = wait_count(&bars->p_count[u], (uint32_t)kEwWarps * pc[u], abort_flag, limit, err);
                        if (!ok) break;
                        tc_fence_after();
                        issue_acc<HD>(tmem, C::TM_A0, 128 * u + 80, kb, u, t > 0 || u > 0);  // dQ += dS_u K_u
                        if (t + 1 < n) {
                            if (u == 0) {
                                ok = wait_phase(smem_u32(&bars->full[nslot]), nph, abort_flag, limit, err);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            const uint32_t nb = sSt + (2 * nslot) * C::TILE_BYTES;
                            issue_sdp<HD>(tmem, u, sQ, sDo, nb, nb + C::TILE_BYTES);
                            mma_commit(smem_u32(&bars->s_full[u]));
                            if (u == 1 && t + 2 == n) mma_commit(smem_u32(&bars->fix_empty));
                        }
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&bars->empty[cur]));
                    if (t == n - 1) mma_commit(smem_u32(&bars->o_full));
                    slot = nslot;
                    ph = nph;
                }
            }
            mma_commit(smem_u32(&bars->drain));
            wait_phase_drain(smem_u32(&bars->drain), 0);
        }
    } else if (warp >= 4) {
        const int quarter = warp & 3;
        const int grp = (warp - 4) >> 2;  // which 32 columns of a sub-tile this warp owns
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t sc[2] = {0u, 0u}, ocnt = 0;
        bool ok = true;
        for (int k2 = 0; (k2 >> 1) * (int)gridDim.x < total && ok; ++k2) {  // (item, tile of the pair)
            const int L = snake(k2 >> 1);
            if (L >= total) continue;
            QItem it;
            if (!decode_q(P, tps, L, k2 & 1, it)) continue;
            const BSeg &S = P.seg[it.si];
            const int n = it.n, diag = S.diag;
            const int row = it.r_lo + quarter * 32 + lane;  // index in the fixed range
            const bool valid = row < it.r_hi;
            const int64_t pos = (int64_t)row * P.rs + S.f_rank;
            const int64_t lrow = ((int64_t)it.b * P.Hq + it.h) * P.N + pos;
            const float lse_l2 = valid ? P.lse[lrow] * kLog2e : 0.f;
            const float d_r = valid ? P.dvec[lrow] : 0.f;
            float *accp = P.acc_q + lrow * HD;
            if (valid && grp == 0 && !(S.flags & SEG_FIRST))
                for (int i = 0; i < HD * 4; i += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(
                                                          reinterpret_cast<const char *>(accp) + i));
            for (int t = 0; t < n && ok; ++t) {
                int kt0, klim;
                q_tile(S, it, t, kt0, klim);
                for (int u = 0; u < 2; ++u) {
                    ok = wait_phase(smem_u32(&bars->s_full[u]), sc[u] & 1u, abort_flag, limit, err);
                    ++sc[u];
                    if (!ok) break;
                    tc_fence_after();
                    const int k0 = kt0 + u * kSub + grp * 32;  // first key of this warp's columns
                    const bool mask = (k0 + 32 > klim) || (P.causal && k0 + 31 + diag > row) || !valid;
                    uint32_t pk[16];
                    {
                        uint32_t s[32], dp[32];
                        tmem_ld32(tmem + 128 * u + lane_off + grp * 32, s);
                        tmem_ld32(tmem + 128 * u + 64 + lane_off + grp * 32, dp);
                        tmem_ld_wait();
                        // invisible scores become -inf (P = 0, dS = 0) in a pass of their own,
                        // so the loop below has no branch and its iterations interleave
                        if (mask) {
                            const int lim = !valid ? 0 : (P.causal ? min(klim, row + 1 - diag) : klim) - k0;
#pragma unroll
                            for (int e = 0; e < 32; ++e) s[e] = e < lim ? s[e] : kNegInfBits;
                        }
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float p0 = ex2(fmaf(__uint_as_float(s[e]), sl2, -lse_l2));
                            const float p1 = ex2(fmaf(__uint_as_float(s[e + 1]), sl2, -lse_l2));
                            pk[e / 2] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - d_r),
                                                    p1 * (__uint_as_float(dp[e + 1]) - d_r));
                        }
                    }
                    // this warp's half of dS_u, inside the dP_u columns it has read
                    tmem_st16(tmem + 128 * u + 80 + 16 * grp + lane_off, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) count_release_add(&bars->p_count[u]);
                }
            }
            if (!ok) break;
            if (n > 0) {
                ok = wait_phase(smem_u32(&bars->o_full), ocnt & 1u, abort_flag, limit, err);
                ++ocnt;
                if (!ok) break;
                tc_fence_after();
            }
            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(P.dq) + (int64_t)it.b * P.sdq[0] +
                                  (int64_t)it.h * P.sdq[1] + pos * P.sdq[2];
            for (int c = grp * (HD / 64); c < (grp + 1) * (HD / 64); ++c) {  // this group's columns
                uint32_t o[32];
                if (n > 0) {
                    tmem_ld32(tmem + C::TM_A0 + lane_off + c * 32, o);
                    tmem_ld_wait();
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
}

// ---------------------------------------------------------------- dK / dV kernel

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ BwdParams P, int total, int64_t limit, int *err) {
    using C = BCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sK = base, sV = base + C::TILE_BYTES;
    const uint32_t sSt = base + 2 * C::TILE_BYTES;  // stages of (Q, dO)
    BBars *bars = reinterpret_cast<BBars *>(base_ptr + C::BAR_OFF);
    // per element-wise warp: the current query tile's LSE (log2 units) and D values
    float *s_stage = reinterpret_cast<float *>(base_ptr + C::BAR_OFF + 256);  // [8 warps][2][64]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((int)blockIdx.x >= total) return;
    volatile int32_t *abort_flag = &bars->abort;
    const int G = P.Hq / P.Hkv;
    const int tps = (P.flen + kT - 1) / kT;
    const float sl2 = P.scale_log2;

    if (threadIdx.x == 0) bwd_init(bars, C::NST);
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
            int slot = 0;
            uint32_t ph = 0, fcnt = 0, issued = 0, last_ph = 0;
            bool ok = true;
            for (int k2 = 0; (k2 >> 1) * (int)gridDim.x < total && ok; ++k2) {  // (item, tile of the pair)
                const int L = snake(k2 >> 1);
                if (L >= total) continue;
                KItem it;
                if (!decode_kv(P, tps, L, k2 & 1, it)) continue;
                if (it.n == 0) continue;
                const BSeg &S = P.seg[it.si];
                const int hk = it.hk;
                auto coords = [=, &S](int t, int &row, int &head) {
                    int qlim, g;
                    kv_tile(S, it, G, t, row, qlim, g);
                    head = hk * G + g;
                };
                ok = produce_item<HD>(bars, sK, sSt, slot, ph, fcnt, issued, last_ph, &tm_k, &tm_v, it.c_lo,
                                      S.f_rank, hk, &tm_q, &tm_do, S.s_rank, it.n, it.b, coords, abort_flag,
                                      limit, err);
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
            uint32_t ph = 0, fcnt = 0, pc[2] = {0u, 0u};
            bool ok = true;
            for (int k2 = 0; (k2 >> 1) * (int)gridDim.x < total && ok; ++k2) {  // (item, tile of the pair)
                const int L = snake(k2 >> 1);
                if (L >= total) continue;
                KItem it;
                if (!decode_kv(P, tps, L, k2 & 1, it)) continue;
                const int n = it.n;
                if (n == 0) continue;
                ok = wait_phase(smem_u32(&bars->fix_full), fcnt & 1u, abort_flag, limit, err);
                ++fcnt;
                if (!ok) break;
                ok = wait_phase(smem_u32(&bars->full[slot]), ph, abort_flag, limit, err);
                if (!ok) break;
                tc_fence_after();
                for (int u = 0; u < 2; ++u) {
                    const uint32_t qb = sSt + (2 * slot) * C::TILE_BYTES;
                    issue_sdp<HD>(tmem, u, sK, sV, qb, qb + C::TILE_BYTES);  // S^T_u, dP^T_u
                    mma_commit(smem_u32(&bars->s_full[u]));
                }
                if (n == 1) mma_commit(smem_u32(&bars->fix_empty));
                for (int t = 0; ok && t < n; ++t) {
                    const int cur = slot;
                    const uint32_t qb = sSt + (2 * cur) * C::TILE_BYTES;
                    int nslot = slot + 1;
                    uint32_t nph = ph;
                    if (nslot == C::NST) {
                        nslot = 0;
                        nph ^= 1u;
                    }
                    for (int u = 0; u < 2 && ok; ++u) {
                        ++pc[u];
                        ok = wait_count(&bars->p_count[u], (uint32_t)kEwWarps * pc[u], abort_flag, limit, err);
                        if (!ok) break;
                        tc_fence_after();
                        const bool accum = t > 0 || u > 0;
                        issue_acc<HD>(tmem, C::TM_A0, 128 * u + 16, qb + C::TILE_BYTES, u, accum);  // dV += P^T_u dO_u
                        issue_acc<HD>(tmem, C::TM_A1, 128 * u + 80, qb, u, accum);                  // dK += dS^T_u Q_u
                        if (t + 1 < n) {
                            if (u == 0) {
                                ok = wait_phase(smem_u32(&bars->full[nslot]), nph, abort_flag, limit, err);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            const uint32_t nb = sSt + (2 * nslot) * C::TILE_BYTES;
                            issue_sdp<HD>(tmem, u, sK, sV, nb, nb + C::TILE_BYTES);
                            mma_commit(smem_u32(&bars->s_full[u]));
                            if (u == 1 && t + 2 == n) mma_commit(smem_u32(&bars->fix_empty));
                        }
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&bars->empty[cur]));
                    if (t == n - 1) mma_commit(smem_u32(&bars->o_full));
                    slot = nslot;
                    ph = nph;
                }
            }
            mma_commit(smem_u32(&bars->drain));
            wait_phase_drain(smem_u32(&bars->drain), 0);
        }
    } else if (warp >= 4) {
        const int quarter = warp & 3;
        const int grp = (warp - 4) >> 2;  // which 32 columns of a sub-tile this warp owns
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float *lb = s_stage + (warp - 4) * 2 * 64;  // this warp's columns only: no cross-warp barrier
        float *db = lb + 64;
        uint32_t sc[2] = {0u, 0u}, ocnt = 0;
        bool ok = true;
        for (int k2 = 0; (k2 >> 1) * (int)gridDim.x < total && ok; ++k2) {  // (item, tile of the pair)
            const int L = snake(k2 >> 1);
            if (L >= total) continue;
            KItem it;
            if (!decode_kv(P, tps, L, k2 & 1, it)) continue;
            const BSeg &S = P.seg[it.si];
            const int n = it.n, diag = S.diag;
            const int key = it.c_lo + quarter * 32 + lane;  // index in the fixed range
            const bool kvalid = key < it.c_hi;
            const int64_t kpos = (int64_t)key * P.rs + S.f_rank;
            const int64_t arow = (((int64_t)it.b * P.Hkv + it.hk) * P.N + kpos) * HD;
            if (kvalid && grp == 0 && !(S.flags & SEG_FIRST))
                for (int i = 0; i < HD * 4; i += 128) {
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(P.acc_k + arow) + i));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(P.acc_v + arow) + i));
                }
            for (int t = 0; t < n && ok; ++t) {
                int q0, qlim, g;
                kv_tile(S, it, G, t, q0, qlim, g);
                const int h = it.hk * G + g;
                __syncwarp();  // every lane is done with the previous tile's values
#pragma unroll
                for (int r = 0; r < 2; ++r) {  // the queries of this warp's columns of both halves
                    const int qme = q0 + r * kSub + grp * 32 + lane;
                    const int64_t li = ((int64_t)it.b * P.Hq + h) * P.N + (int64_t)qme * P.rs + S.s_rank;
                    lb[r * 32 + lane] = qme < qlim ? P.lse[li] * kLog2e : 0.f;
                    db[r * 32 + lane] = qme < qlim ? P.dvec[li] : 0.f;
                }
                __syncwarp();
                for (int u = 0; u < 2; ++u) {
                    ok = wait_phase(smem_u32(&bars->s_full[u]), sc[u] & 1u, abort_flag, limit, err);
                    ++sc[u];
                    if (!ok) break;
                    tc_fence_after();
                    const int qa = q0 + u * kSub + grp * 32;  // first query of this warp's columns
                    const bool mask = (qa + 32 > qlim) || (P.causal && it.c_hi - 1 + diag > qa);
                    uint32_t pp[16], pd[16];
                    {
                        uint32_t s[32], dp[32];
                        tmem_ld32(tmem + 128 * u + lane_off + grp * 32, s);
                        tmem_ld32(tmem + 128 * u + 64 + lane_off + grp * 32, dp);
                        tmem_ld_wait();
                        const float *lu = lb + u * 32, *du = db + u * 32;
                        // invisible scores become -inf (P = 0, dS = 0) in a pass of their own,
                        // so the loop below has no branch and its iterations interleave
                        if (mask) {
                            const int lo = P.causal ? key + diag - qa : 0;  // first visible offset
                            const int hi = qlim - qa;                       // end of the range
#pragma unroll
                            for (int e = 0; e < 32; ++e) s[e] = (e >= lo && e < hi) ? s[e] : kNegInfBits;
                        }
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float p0 = ex2(fmaf(__uint_as_float(s[e]), sl2, -lu[e]));
                            const float p1 = ex2(fmaf(__uint_as_float(s[e + 1]), sl2, -lu[e + 1]));
                            pp[e / 2] = pack_bf16x2(p0, p1);
                            pd[e / 2] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - du[e]),
                                                    p1 * (__uint_as_float(dp[e + 1]) - du[e + 1]));
                        }
                    }
                    // this warp's halves of P_u and dS_u, inside the columns it has read
                    tmem_st16(tmem + 128 * u + 16 + 16 * grp + lane_off, pp);
                    tmem_st16(tmem + 128 * u + 80 + 16 * grp + lane_off, pd);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) count_release_add(&bars->p_count[u]);
                }
            }
            if (!ok) break;
            if (n > 0) {
                ok = wait_phase(smem_u32(&bars->o_full), ocnt & 1u, abort_flag, limit, err);
                ++ocnt;
                if (!ok) break;
                tc_fence_after();
            }
            __nv_bfloat16 *vrow = static_cast<__nv_bfloat16 *>(P.dv) + (int64_t)it.b * P.sdv[0] +
                                  (int64_t)it.hk * P.sdv[1] + kpos * P.sdv[2];
            __nv_bfloat16 *krow = static_cast<__nv_bfloat16 *>(P.dk) + (int64_t)it.b * P.sdk[0] +
                                  (int64_t)it.hk * P.sdk[1] + kpos * P.sdk[2];
            for (int which = 0; which < 2; ++which) {
                const float mul = which ? P.scale : 1.f;
                __nv_bfloat16 *dst = which ? krow : vrow;
                float *acc = (which ? P.acc_k : P.acc_v) + arow;
                const uint32_t col = which ? C::TM_A1 : C::TM_A0;
                for (int c = grp * (HD / 64); c < (grp + 1) * (HD / 64); ++c) {  // this group's columns
                    uint32_t o[32];
                    if (n > 0) {
                        tmem_ld32(tmem + col + lane_off + c * 32, o);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = 0u;
                    }
                    if (!kvalid) continue;
                    store_grad_chunk(dst + c * 32, acc + c * 32, o, mul, S.flags);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

}  // namespace tcb

template <int HD>
static cudaError_t launch_bwd_tc_hd(const BwdParams &P, int parts, int num_sms, int64_t wait_ns, int *err,
                                    cudaStream_t stream) {
    using C = tcb::BCfg<HD>;
    static int configured_mask = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(configured_mask & (1 << (dev & 31)))) {
        cudaError_t e = cudaFuncSetAttribute(tcb::bwd_dq_tc_kernel<HD>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tcb::bwd_dkdv_tc_kernel<HD>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured_mask |= 1 << (dev & 31);
    }
    CUtensorMap mq, mk, mv, mdo;
    if (!encode_map(&mq, P.q, P.B, P.Hq, P.N, P.D, P.sq, P.rs) ||
        !encode_map(&mk, P.k, P.B, P.Hkv, P.N, P.D, P.sk, P.rs) ||
        !encode_map(&mv, P.v, P.B, P.Hkv, P.N, P.D, P.sv, P.rs) ||
        !encode_map(&mdo, P.dout, P.B, P.Hq, P.N, P.D, P.sdo, P.rs))
        return cudaErrorInvalidValue;
    const int np = ((P.flen + tcb::kT - 1) / tcb::kT + 1) / 2;  // tile pairs per segment and head
    const int64_t tq = (int64_t)P.B * P.Hq * P.nseg * np, tkv = (int64_t)P.B * P.Hkv * P.nseg * np;
    if (tq > 0x7fffffff || tkv > 0x7fffffff) return cudaErrorInvalidValue;
    if (parts & 1) {
        tcb::bwd_dq_tc_kernel<HD><<<(int)std::min<int64_t>(tq, num_sms), tcb::kThreads, C::SMEM_BYTES, stream>>>(
            mq, mk, mv, mdo, P, (int)tq, wait_ns, err);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (parts & 2)
        tcb::bwd_dkdv_tc_kernel<HD><<<(int)std::min<int64_t>(tkv, num_sms), tcb::kThreads, C::SMEM_BYTES,
                                      stream>>>(mq, mk, mv, mdo, P, (int)tkv, wait_ns, err);
    return cudaGetLastError();
}

// The dQ kernel (parts & 1) and the dK/dV kernel (parts & 2) over the segments in P (the
// D vector is computed before).
cudaError_t launch_attn_bwd_tc(const BwdParams &P, int parts, int num_sms, int64_t wait_ns, int *err,
                               cudaStream_t stream) {
    if (P.B <= 0 || P.Hq <= 0 || P.nseg <= 0 || P.flen <= 0) return cudaSuccess;
    if (P.D == 128) return launch_bwd_tc_hd<128>(P, parts, num_sms, wait_ns, err, stream);
    if (P.D == 64) return launch_bwd_tc_hd<64>(P, parts, num_sms, wait_ns, err, stream);
    return cudaErrorInvalidValue;
}

}  // namespace ra
