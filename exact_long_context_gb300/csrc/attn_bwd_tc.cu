// attn_bwd_tc.cu - gradients of exact attention on the sm_103a tensor cores.
//
// The same quantities as attn_bwd_simt.cu (the recompute-from-LSE backward of the
// `ring_attention_backward` listing of "Ring Attention 论文解析"), as two persistent
// kernels with one writer per output element (no atomics):
//
//   dQ kernel   one CTA item = 128 query rows of one (b, h); for each visible key tile:
//                 S  = Q K^T,  dP = dO V^T          (tcgen05, A and B from shared memory)
//                 dS = P * (dP - D),  P = exp(S * scale - LSE)   (one thread per row)
//                 dQ += dS K                        (tcgen05, A = dS from tensor memory)
//   dK/dV kernel one CTA item = 128 keys of one (b, KV head); for each visible query tile
//                of every query head that reads the KV head:
//                 S^T = K Q^T,  dP^T = V dO^T
//                 P^T, dS^T                         (one thread per key)
//                 dV += P^T dO,  dK += dS^T Q       (A from tensor memory)
//
// Warp roles: warp 0 TMA producer, warp 1 MMA issuer and tensor-memory owner, warps 4-7
// the element-wise work and the epilogue.  The streamed tile is handled as two 64-wide
// halves with their own S / dP buffers, so the tensor core computes one half's S / dP
// while the element-wise warps work on the other.  The bf16 P / dS overwrite the
// columns of the fp32 S / dP they came from once those are in registers; the MMA
// thread issues the next S / dP of a half after the products that read it (tcgen05 MMAs
// of a thread run in order).  Every wait is bounded like the forward kernel's.
#include "tc_common.cuh"

namespace ra {
namespace tcb {

using namespace ra::tc;

constexpr int kT = 128;   // rows per tile (queries or keys)
constexpr int kSub = 64;  // a tile's streamed dimension is processed as two 64-wide halves
constexpr int kThreads = 256;

// Tensor memory: for sub-tile u in {0, 1}, S_u at 128u (64 fp32 columns) and dP_u at
// 128u + 64; the bf16 P_u / dS_u (32 columns) overwrite the leading columns of S_u / dP_u.
// Accumulators at 256 (dQ or dV) and 256 + HD (dK).
template <int HD>
struct BCfg {
    static constexpr int SLABS = HD / 64;
    static constexpr int TILE_BYTES = kT * HD * 2;
    static constexpr int SLAB_BYTES = 128 * 128;
    static constexpr int NST = (HD == 128) ? 2 : 4;  // stages of two tiles
    static constexpr uint32_t TM_A0 = 256, TM_A1 = 256 + HD;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int BAR_OFF = (2 + 2 * NST) * TILE_BYTES;
    static constexpr int SMEM_BYTES = 1024 + BAR_OFF + 256 + 4096;
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

// dQ item L: query tile of one (b, h), the heaviest (most key tiles under causality) first.
__device__ __forceinline__ void decode_q(const BwdParams &P, int nq, int L, int &b, int &h, int &hk,
                                         int &qi, int &n) {
    const int BH = P.B * P.Hq;
    const int w = L / BH;
    const int bh = L - w * BH;
    b = bh / P.Hq;
    h = bh - b * P.Hq;
    hk = h / (P.Hq / P.Hkv);
    qi = nq - 1 - w;
    n = P.causal ? min(qi + 1, nq) : nq;
}

// dK/dV item L: keys [kj*128, +128) of (b, hk), the heaviest (most query tiles) first; it
// visits query tiles q_first .. nq-1 of each of the G query heads, n = G (nq - q_first).
__device__ __forceinline__ void decode_kv(const BwdParams &P, int nq, int L, int &b, int &hk,
                                          int &kj, int &q_first, int &n) {
    const int BHk = P.B * P.Hkv;
    const int w = L / BHk;
    const int bhk = L - w * BHk;
    b = bhk / P.Hkv;
    hk = bhk - b * P.Hkv;
    kj = w;
    q_first = P.causal ? kj : 0;
    n = (P.Hq / P.Hkv) * (nq - q_first);
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

// Producer: per item the fixed pair (fa, fb) at rows f_row of (fh, b), then `n` streamed
// pairs (sa, sb) from rows_of(t) of heads_of(t).  Shared by both kernels.
template <int HD, typename StreamCoords>
__device__ __forceinline__ bool produce_item(BBars *bars, uint32_t fix0, uint32_t st0, int &slot, uint32_t &ph,
                                             uint32_t &fcnt, uint32_t &issued, uint32_t &last_ph,
                                             const CUtensorMap *fa, const CUtensorMap *fb, int f_row, int fh,
                                             const CUtensorMap *sa, const CUtensorMap *sb, int n, int b,
                                             StreamCoords coords, volatile int32_t *abort_flag,
                                             int64_t limit, int *err) {
    using C = BCfg<HD>;
    if (!wait_phase(smem_u32(&bars->fix_empty), (fcnt & 1u) ^ 1u, abort_flag, limit, err)) return false;
    {
        const uint32_t bf = smem_u32(&bars->fix_full);
        mbar_expect_tx(bf, 2 * C::TILE_BYTES);
        for (int c = 0; c < C::SLABS; ++c) {
            tma_load_5d(fix0 + c * C::SLAB_BYTES, fa, bf, c * 64, 0, f_row, fh, b);
            tma_load_5d(fix0 + C::TILE_BYTES + c * C::SLAB_BYTES, fb, bf, c * 64, 0, f_row, fh, b);
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
            tma_load_5d(a0 + c * C::SLAB_BYTES, sa, bf, c * 64, 0, row, head, b);
            tma_load_5d(a0 + C::TILE_BYTES + c * C::SLAB_BYTES, sb, bf, c * 64, 0, row, head, b);
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
    const int nq = (P.N + kT - 1) / kT;
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
            for (int k = 0; k * (int)gridDim.x < total && ok; ++k) {
                const int L = snake(k);
                if (L >= total) continue;
                int b, h, hk, qi, n;
                decode_q(P, nq, L, b, h, hk, qi, n);
                auto coords = [=](int t, int &row, int &head) {
                    row = t * kT;
                    head = hk;
                };
                ok = produce_item<HD>(bars, sQ, sSt, slot, ph, fcnt, issued, last_ph, &tm_q, &tm_do, qi * kT, h,
                                      &tm_k, &tm_v, n, b, coords, abort_flag, limit, err);
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
            for (int k = 0; k * (int)gridDim.x < total && ok; ++k) {
                const int L = snake(k);
                if (L >= total) continue;
                int b, h, hk, qi, n;
                decode_q(P, nq, L, b, h, hk, qi, n);
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
                        ok = wait_count(&bars->p_count[u], 4u * pc[u], abort_flag, limit, err);
                        if (!ok) break;
                        tc_fence_after();
                        issue_acc<HD>(tmem, C::TM_A0, 128 * u + 64, kb, u, t > 0 || u > 0);  // dQ += dS_u K_u
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
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t sc[2] = {0u, 0u}, ocnt = 0;
        bool ok = true;
        for (int k = 0; k * (int)gridDim.x < total && ok; ++k) {
            const int L = snake(k);
            if (L >= total) continue;
            int b, h, hk, qi, n;
            decode_q(P, nq, L, b, h, hk, qi, n);
            const int row = qi * kT + quarter * 32 + lane;
            const bool valid = row < P.N;
            const int64_t lrow = ((int64_t)b * P.Hq + h) * P.N + row;
            const float lse_l2 = valid ? P.lse[lrow] * kLog2e : 0.f;
            const float d_r = valid ? P.dvec[lrow] : 0.f;
            for (int t = 0; t < n && ok; ++t) {
                for (int u = 0; u < 2; ++u) {
                    ok = wait_phase(smem_u32(&bars->s_full[u]), sc[u] & 1u, abort_flag, limit, err);
                    ++sc[u];
                    if (!ok) break;
                    tc_fence_after();
                    const int k0 = t * kT + u * kSub;  // first key of this half
                    const bool mask = (k0 + kSub > P.N) || (P.causal && k0 + kSub - 1 > qi * kT) || !valid;
                    uint32_t pk[2][16];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t s[32], dp[32];
                        tmem_ld32(tmem + 128 * u + lane_off + c * 32, s);
                        tmem_ld32(tmem + 128 * u + 64 + lane_off + c * 32, dp);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float p0 = ex2(fmaf(__uint_as_float(s[e]), sl2, -lse_l2));
                            float p1 = ex2(fmaf(__uint_as_float(s[e + 1]), sl2, -lse_l2));
                            if (mask) {
                                const int key = k0 + c * 32 + e;
                                p0 = (valid && key < P.N && (!P.causal || key <= row)) ? p0 : 0.f;
                                p1 = (valid && key + 1 < P.N && (!P.causal || key + 1 <= row)) ? p1 : 0.f;
                            }
                            pk[c][e / 2] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - d_r),
                                                       p1 * (__uint_as_float(dp[e + 1]) - d_r));
                        }
                    }
                    // dS_u over the (already loaded) leading dP_u columns
                    tmem_st16(tmem + 128 * u + 64 + lane_off, pk[0]);
                    tmem_st16(tmem + 128 * u + 64 + 16 + lane_off, pk[1]);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) count_release_add(&bars->p_count[u]);
                }
            }
            if (!ok) break;
            ok = wait_phase(smem_u32(&bars->o_full), ocnt & 1u, abort_flag, limit, err);
            ++ocnt;
            if (!ok) break;
            tc_fence_after();
            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(P.dq) + (int64_t)b * P.sdq[0] +
                                  (int64_t)h * P.sdq[1] + (int64_t)row * P.sdq[2];
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + C::TM_A0 + lane_off + c * 32, o);
                tmem_ld_wait();
                if (!valid) continue;
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 v4;
                    v4.x = pack_bf16x2(P.scale * __uint_as_float(o[e]), P.scale * __uint_as_float(o[e + 1]));
                    v4.y = pack_bf16x2(P.scale * __uint_as_float(o[e + 2]), P.scale * __uint_as_float(o[e + 3]));
                    v4.z = pack_bf16x2(P.scale * __uint_as_float(o[e + 4]), P.scale * __uint_as_float(o[e + 5]));
                    v4.w = pack_bf16x2(P.scale * __uint_as_float(o[e + 6]), P.scale * __uint_as_float(o[e + 7]));
                    *reinterpret_cast<uint4 *>(orow + c * 32 + e) = v4;
                }
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
    float *s_stage = reinterpret_cast<float *>(base_ptr + C::BAR_OFF + 256);  // [4 warps][2][128]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((int)blockIdx.x >= total) return;
    volatile int32_t *abort_flag = &bars->abort;
    const int G = P.Hq / P.Hkv;
    const int nq = (P.N + kT - 1) / kT;
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
            for (int k = 0; k * (int)gridDim.x < total && ok; ++k) {
                const int L = snake(k);
                if (L >= total) continue;
                int b, hk, kj, q_first, n;
                decode_kv(P, nq, L, b, hk, kj, q_first, n);
                const int per = nq - q_first;
                auto coords = [=](int t, int &row, int &head) {
                    const int g = t / per;
                    row = (q_first + (t - g * per)) * kT;
                    head = hk * G + g;
                };
                ok = produce_item<HD>(bars, sK, sSt, slot, ph, fcnt, issued, last_ph, &tm_k, &tm_v, kj * kT, hk,
                                      &tm_q, &tm_do, n, b, coords, abort_flag, limit, err);
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
            for (int k = 0; k * (int)gridDim.x < total && ok; ++k) {
                const int L = snake(k);
                if (L >= total) continue;
                int b, hk, kj, q_first, n;
                decode_kv(P, nq, L, b, hk, kj, q_first, n);
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
                        ok = wait_count(&bars->p_count[u], 4u * pc[u], abort_flag, limit, err);
                        if (!ok) break;
                        tc_fence_after();
                        const bool accum = t > 0 || u > 0;
                        issue_acc<HD>(tmem, C::TM_A0, 128 * u, qb + C::TILE_BYTES, u, accum);  // dV += P^T_u dO_u
                        issue_acc<HD>(tmem, C::TM_A1, 128 * u + 64, qb, u, accum);             // dK += dS^T_u Q_u
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
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float *lb = s_stage + quarter * 2 * kT;  // this warp's copy, so no cross-warp barrier
        float *db = lb + kT;
        uint32_t sc[2] = {0u, 0u}, ocnt = 0;
        bool ok = true;
        for (int k = 0; k * (int)gridDim.x < total && ok; ++k) {
            const int L = snake(k);
            if (L >= total) continue;
            int b, hk, kj, q_first, n;
            decode_kv(P, nq, L, b, hk, kj, q_first, n);
            const int key = kj * kT + quarter * 32 + lane;
            const int per = nq - q_first;
            for (int t = 0; t < n && ok; ++t) {
                const int g = t / per;
                const int q0 = (q_first + (t - g * per)) * kT;
                const int h = hk * G + g;
                __syncwarp();  // every lane is done with the previous tile's values
#pragma unroll
                for (int r = 0; r < kT / 32; ++r) {
                    const int qme = q0 + r * 32 + lane;
                    const int64_t li = ((int64_t)b * P.Hq + h) * P.N + qme;
                    lb[r * 32 + lane] = qme < P.N ? P.lse[li] * kLog2e : 0.f;
                    db[r * 32 + lane] = qme < P.N ? P.dvec[li] : 0.f;
                }
                __syncwarp();
                for (int u = 0; u < 2; ++u) {
                    ok = wait_phase(smem_u32(&bars->s_full[u]), sc[u] & 1u, abort_flag, limit, err);
                    ++sc[u];
                    if (!ok) break;
                    tc_fence_after();
                    const int qa = q0 + u * kSub;  // first query of this half
                    const bool mask = (qa + kSub > P.N) || (P.causal && kj * kT + kT - 1 > qa);
                    uint32_t pp[2][16], pd[2][16];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t s[32], dp[32];
                        tmem_ld32(tmem + 128 * u + lane_off + c * 32, s);
                        tmem_ld32(tmem + 128 * u + 64 + lane_off + c * 32, dp);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const int qo = u * kSub + c * 32 + e;  // offset in the tile
                            float p0 = ex2(fmaf(__uint_as_float(s[e]), sl2, -lb[qo]));
                            float p1 = ex2(fmaf(__uint_as_float(s[e + 1]), sl2, -lb[qo + 1]));
                            if (mask) {
                                const int qq = q0 + qo;
                                p0 = (qq < P.N && (!P.causal || key <= qq)) ? p0 : 0.f;
                                p1 = (qq + 1 < P.N && (!P.causal || key <= qq + 1)) ? p1 : 0.f;
                            }
                            pp[c][e / 2] = pack_bf16x2(p0, p1);
                            pd[c][e / 2] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - db[qo]),
                                                       p1 * (__uint_as_float(dp[e + 1]) - db[qo + 1]));
                        }
                    }
                    tmem_st16(tmem + 128 * u + lane_off, pp[0]);
                    tmem_st16(tmem + 128 * u + 16 + lane_off, pp[1]);
                    tmem_st16(tmem + 128 * u + 64 + lane_off, pd[0]);
                    tmem_st16(tmem + 128 * u + 64 + 16 + lane_off, pd[1]);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) count_release_add(&bars->p_count[u]);
                }
            }
            if (!ok) break;
            ok = wait_phase(smem_u32(&bars->o_full), ocnt & 1u, abort_flag, limit, err);
            ++ocnt;
            if (!ok) break;
            tc_fence_after();
            const bool valid = key < P.N;
            __nv_bfloat16 *vrow = static_cast<__nv_bfloat16 *>(P.dv) + (int64_t)b * P.sdv[0] +
                                  (int64_t)hk * P.sdv[1] + (int64_t)key * P.sdv[2];
            __nv_bfloat16 *krow = static_cast<__nv_bfloat16 *>(P.dk) + (int64_t)b * P.sdk[0] +
                                  (int64_t)hk * P.sdk[1] + (int64_t)key * P.sdk[2];
            for (int which = 0; which < 2; ++which) {
                const float mul = which ? P.scale : 1.f;
                __nv_bfloat16 *dst = which ? krow : vrow;
                const uint32_t col = which ? C::TM_A1 : C::TM_A0;
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tmem + col + lane_off + c * 32, o);
                    tmem_ld_wait();
                    if (!valid) continue;
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v4;
                        v4.x = pack_bf16x2(mul * __uint_as_float(o[e]), mul * __uint_as_float(o[e + 1]));
                        v4.y = pack_bf16x2(mul * __uint_as_float(o[e + 2]), mul * __uint_as_float(o[e + 3]));
                        v4.z = pack_bf16x2(mul * __uint_as_float(o[e + 4]), mul * __uint_as_float(o[e + 5]));
                        v4.w = pack_bf16x2(mul * __uint_as_float(o[e + 6]), mul * __uint_as_float(o[e + 7]));
                        *reinterpret_cast<uint4 *>(dst + c * 32 + e) = v4;
                    }
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
static cudaError_t launch_bwd_tc_hd(const BwdParams &P, int num_sms, int64_t wait_ns, int *err,
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
    if (!encode_map(&mq, P.q, P.B, P.Hq, P.N, P.D, P.sq, 1) ||
        !encode_map(&mk, P.k, P.B, P.Hkv, P.N, P.D, P.sk, 1) ||
        !encode_map(&mv, P.v, P.B, P.Hkv, P.N, P.D, P.sv, 1) ||
        !encode_map(&mdo, P.dout, P.B, P.Hq, P.N, P.D, P.sdo, 1))
        return cudaErrorInvalidValue;
    const int nt = (P.N + tcb::kT - 1) / tcb::kT;
    const int64_t tq = (int64_t)P.B * P.Hq * nt, tkv = (int64_t)P.B * P.Hkv * nt;
    if (tq > 0x7fffffff || tkv > 0x7fffffff) return cudaErrorInvalidValue;
    tcb::bwd_dq_tc_kernel<HD><<<(int)std::min<int64_t>(tq, num_sms), tcb::kThreads, C::SMEM_BYTES, stream>>>(
        mq, mk, mv, mdo, P, (int)tq, wait_ns, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    tcb::bwd_dkdv_tc_kernel<HD><<<(int)std::min<int64_t>(tkv, num_sms), tcb::kThreads, C::SMEM_BYTES, stream>>>(
        mq, mk, mv, mdo, P, (int)tkv, wait_ns, err);
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd_tc(const BwdParams &P, int num_sms, int64_t wait_ns, int *err,
                               cudaStream_t stream) {
    if (P.B <= 0 || P.Hq <= 0 || P.N <= 0) return cudaSuccess;
    if (P.D == 128) return launch_bwd_tc_hd<128>(P, num_sms, wait_ns, err, stream);
    if (P.D == 64) return launch_bwd_tc_hd<64>(P, num_sms, wait_ns, err, stream);
    return cudaErrorInvalidValue;
}

}  // namespace ra
