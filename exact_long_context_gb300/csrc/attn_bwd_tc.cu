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
// the element-wise work and the epilogue.  The bf16 P / dS overwrite the columns of the
// fp32 S / dP they came from once those are in registers; the MMA thread issues the
// next S / dP after the products that read them (tcgen05 MMAs of a thread run in order).
// Every wait is bounded like the forward kernel's.
#include "tc_common.cuh"

namespace ra {
namespace tcb {

using namespace ra::tc;

constexpr int kT = 128;  // rows per tile (queries or keys)
constexpr int kThreads = 256;

template <int HD>
struct BCfg {
    static constexpr int SLABS = HD / 64;
    static constexpr int TILE_BYTES = kT * HD * 2;
    static constexpr int SLAB_BYTES = 128 * 128;
    static constexpr int NST = (HD == 128) ? 2 : 4;  // stages of two tiles
    static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_A0 = 256, TM_A1 = 256 + HD;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int SMEM_BYTES = 1024 + (2 + 2 * NST) * TILE_BYTES + 256;
};

struct BBars {
    uint64_t fix_full, fix_empty;  // the item's fixed pair (Q, dO) or (K, V)
    uint64_t full[4], empty[4];    // streamed pairs
    uint64_t s_full, o_full, drain;
    uint32_t tmem_base;
    int32_t abort;
    uint32_t p_count;
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

// ---------------------------------------------------------------- dQ kernel

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ BwdParams P, int total, int wait_ns_hi, int wait_ns_lo,
                     int *err) {
    using C = BCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sQ = base, sDo = base + C::TILE_BYTES;
    const uint32_t sSt = base + 2 * C::TILE_BYTES;  // stages of (K, V)
    BBars *bars = reinterpret_cast<BBars *>(base_ptr + (2 + 2 * C::NST) * C::TILE_BYTES);
    const int64_t limit = ((int64_t)wait_ns_hi << 32) | (uint32_t)wait_ns_lo;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((int)blockIdx.x >= total) return;
    volatile int32_t *abort_flag = &bars->abort;
    const int nq = (P.N + kT - 1) / kT;
    const float sl2 = P.scale_log2;

    if (threadIdx.x == 0) {
        bars->abort = 0;
        bars->p_count = 0;
        mbar_init(smem_u32(&bars->fix_full), 1);
        mbar_init(smem_u32(&bars->fix_empty), 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->o_full), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
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
                for (int t = -1; t < n && ok; ++t) {
                    if (t == -1) {  // the item's Q and dO
                        if (!wait_phase(smem_u32(&bars->fix_empty), (fcnt & 1u) ^ 1u, abort_flag, limit,
                                        err)) {
                            ok = false;
                            break;
                        }
                        const uint32_t bf = smem_u32(&bars->fix_full);
                        mbar_expect_tx(bf, 2 * C::TILE_BYTES);
                        for (int c = 0; c < C::SLABS; ++c) {
                            tma_load_5d(sQ + c * C::SLAB_BYTES, &tm_q, bf, c * 64, 0, qi * kT, h, b);
                            tma_load_5d(sDo + c * C::SLAB_BYTES, &tm_do, bf, c * 64, 0, qi * kT, h, b);
                        }
                        ++fcnt;
                        continue;
                    }
                    if (!wait_phase(smem_u32(&bars->empty[slot]), ph ^ 1u, abort_flag, limit, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bf = smem_u32(&bars->full[slot]);
                    mbar_expect_tx(bf, 2 * C::TILE_BYTES);
                    const uint32_t kb = sSt + (2 * slot) * C::TILE_BYTES;
                    const uint32_t vb = kb + C::TILE_BYTES;
                    for (int c = 0; c < C::SLABS; ++c) {
                        tma_load_5d(kb + c * C::SLAB_BYTES, &tm_k, bf, c * 64, 0, t * kT, hk, b);
                        tma_load_5d(vb + c * C::SLAB_BYTES, &tm_v, bf, c * 64, 0, t * kT, hk, b);
                    }
                    issued |= 1u << slot;
                    last_ph = (last_ph & ~(1u << slot)) | (ph << slot);
                    if (++slot == C::NST) {
                        slot = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (fcnt) wait_phase_drain(smem_u32(&bars->fix_full), (fcnt - 1u) & 1u);
                for (int s2 = 0; s2 < C::NST; ++s2)
                    if (issued & (1u << s2)) wait_phase_drain(smem_u32(&bars->full[s2]), (last_ph >> s2) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(kT, kT, false);
            constexpr uint32_t ID_Q = idesc_bf16(kT, HD, true);
            int slot = 0;
            uint32_t ph = 0, fcnt = 0, pcnt = 0;
            bool ok = true;
            for (int k = 0; k * (int)gridDim.x < total && ok; ++k) {
                const int L = snake(k);
                if (L >= total) continue;
                int b, h, hk, qi, n;
                decode_q(P, nq, L, b, h, hk, qi, n);
                ok = wait_phase(smem_u32(&bars->fix_full), fcnt & 1u, abort_flag, limit, err);
                ++fcnt;
                for (int t = 0; ok && t < n; ++t) {
                    ok = wait_phase(smem_u32(&bars->full[slot]), ph, abort_flag, limit, err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kb = sSt + (2 * slot) * C::TILE_BYTES;
                    const uint32_t vb = kb + C::TILE_BYTES;
                    for (int kk = 0; kk < HD / 16; ++kk) {  // S = Q K^T, dP = dO V^T
                        const uint32_t off = (kk >> 2) * C::SLAB_BYTES + (kk & 3) * 32;
                        mma_ss(tmem + C::TM_S, sdesc_sw128(sQ + off, 16, 1024),
                               sdesc_sw128(kb + off, 16, 1024), ID_S, kk > 0);
                        mma_ss(tmem + C::TM_DP, sdesc_sw128(sDo + off, 16, 1024),
                               sdesc_sw128(vb + off, 16, 1024), ID_S, kk > 0);
                    }
                    mma_commit(smem_u32(&bars->s_full));
                    if (t == n - 1) mma_commit(smem_u32(&bars->fix_empty));
                    ++pcnt;
                    ok = wait_count(&bars->p_count, 4u * pcnt, abort_flag, limit, err);
                    if (!ok) break;
                    tc_fence_after();
                    for (int kk = 0; kk < kT / 16; ++kk)  // dQ += dS K
                        mma_ts(tmem + C::TM_A0, tmem + C::TM_DP + kk * 8,
                               sdesc_sw128(kb + kk * 16 * 128, C::SLAB_BYTES, 1024), ID_Q,
                               (t > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&bars->empty[slot]));
                    if (t == n - 1) mma_commit(smem_u32(&bars->o_full));
                    if (++slot == C::NST) {
                        slot = 0;
                        ph ^= 1u;
                    }
                }
            }
            mma_commit(smem_u32(&bars->drain));
            wait_phase_drain(smem_u32(&bars->drain), 0);
        }
    } else if (warp >= 4) {
        const int quarter = warp & 3;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t scnt = 0, ocnt = 0;
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
            for (int t = 0; t < n; ++t) {
                ok = wait_phase(smem_u32(&bars->s_full), scnt & 1u, abort_flag, limit, err);
                ++scnt;
                if (!ok) break;
                tc_fence_after();
                const bool mask = (t * kT + kT > P.N) || (P.causal && t == qi) || !valid;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t s[32], dp[32];
                    tmem_ld32(tmem + C::TM_S + lane_off + c * 32, s);
                    tmem_ld32(tmem + C::TM_DP + lane_off + c * 32, dp);
                    tmem_ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float p0 = ex2(fmaf(__uint_as_float(s[e]), sl2, -lse_l2));
                        float p1 = ex2(fmaf(__uint_as_float(s[e + 1]), sl2, -lse_l2));
                        if (mask) {
                            const int key = t * kT + c * 32 + e;
                            const bool v0 = valid && key < P.N && (!P.causal || key <= row);
                            const bool v1 = valid && key + 1 < P.N && (!P.causal || key + 1 <= row);
                            p0 = v0 ? p0 : 0.f;
                            p1 = v1 ? p1 : 0.f;
                        }
                        const float ds0 = p0 * (__uint_as_float(dp[e]) - d_r);
                        const float ds1 = p1 * (__uint_as_float(dp[e + 1]) - d_r);
                        pk[e / 2] = pack_bf16x2(ds0, ds1);
                    }
                    // dS overwrites the already-loaded leading dP columns
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                            tmem + C::TM_DP + lane_off + c * 16),
                        "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]),
                        "r"(pk[6]), "r"(pk[7]), "r"(pk[8]), "r"(pk[9]), "r"(pk[10]), "r"(pk[11]),
                        "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15])
                        : "memory");
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) count_release_add(&bars->p_count);
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
                    uint4 u;
                    u.x = pack_bf16x2(P.scale * __uint_as_float(o[e]), P.scale * __uint_as_float(o[e + 1]));
                    u.y = pack_bf16x2(P.scale * __uint_as_float(o[e + 2]), P.scale * __uint_as_float(o[e + 3]));
                    u.z = pack_bf16x2(P.scale * __uint_as_float(o[e + 4]), P.scale * __uint_as_float(o[e + 5]));
                    u.w = pack_bf16x2(P.scale * __uint_as_float(o[e + 6]), P.scale * __uint_as_float(o[e + 7]));
                    *reinterpret_cast<uint4 *>(orow + c * 32 + e) = u;
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
                       const __grid_constant__ BwdParams P, int total, int wait_ns_hi, int wait_ns_lo,
                       int *err) {
    using C = BCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sK = base, sV = base + C::TILE_BYTES;
    const uint32_t sSt = base + 2 * C::TILE_BYTES;  // stages of (Q, dO)
    BBars *bars = reinterpret_cast<BBars *>(base_ptr + (2 + 2 * C::NST) * C::TILE_BYTES);
    const int64_t limit = ((int64_t)wait_ns_hi << 32) | (uint32_t)wait_ns_lo;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((int)blockIdx.x >= total) return;
    volatile int32_t *abort_flag = &bars->abort;
    const int G = P.Hq / P.Hkv;
    const int nq = (P.N + kT - 1) / kT;
    const float sl2 = P.scale_log2;

    if (threadIdx.x == 0) {
        bars->abort = 0;
        bars->p_count = 0;
        mbar_init(smem_u32(&bars->fix_full), 1);
        mbar_init(smem_u32(&bars->fix_empty), 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->o_full), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
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
                for (int t = -1; t < n && ok; ++t) {
                    if (t == -1) {  // the item's K and V
                        if (!wait_phase(smem_u32(&bars->fix_empty), (fcnt & 1u) ^ 1u, abort_flag, limit,
                                        err)) {
                            ok = false;
                            break;
                        }
                        const uint32_t bf = smem_u32(&bars->fix_full);
                        mbar_expect_tx(bf, 2 * C::TILE_BYTES);
                        for (int c = 0; c < C::SLABS; ++c) {
                            tma_load_5d(sK + c * C::SLAB_BYTES, &tm_k, bf, c * 64, 0, kj * kT, hk, b);
                            tma_load_5d(sV + c * C::SLAB_BYTES, &tm_v, bf, c * 64, 0, kj * kT, hk, b);
                        }
                        ++fcnt;
                        continue;
                    }
                    const int per = nq - q_first;
                    const int g = t / per;
                    const int qt = q_first + (t - g * per);
                    const int h = hk * G + g;
                    if (!wait_phase(smem_u32(&bars->empty[slot]), ph ^ 1u, abort_flag, limit, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bf = smem_u32(&bars->full[slot]);
                    mbar_expect_tx(bf, 2 * C::TILE_BYTES);
                    const uint32_t qb = sSt + (2 * slot) * C::TILE_BYTES;
                    const uint32_t db = qb + C::TILE_BYTES;
                    for (int c = 0; c < C::SLABS; ++c) {
                        tma_load_5d(qb + c * C::SLAB_BYTES, &tm_q, bf, c * 64, 0, qt * kT, h, b);
                        tma_load_5d(db + c * C::SLAB_BYTES, &tm_do, bf, c * 64, 0, qt * kT, h, b);
                    }
                    issued |= 1u << slot;
                    last_ph = (last_ph & ~(1u << slot)) | (ph << slot);
                    if (++slot == C::NST) {
                        slot = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (fcnt) wait_phase_drain(smem_u32(&bars->fix_full), (fcnt - 1u) & 1u);
                for (int s2 = 0; s2 < C::NST; ++s2)
                    if (issued & (1u << s2)) wait_phase_drain(smem_u32(&bars->full[s2]), (last_ph >> s2) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(kT, kT, false);
            constexpr uint32_t ID_G = idesc_bf16(kT, HD, true);
            int slot = 0;
            uint32_t ph = 0, fcnt = 0, pcnt = 0;
            bool ok = true;
            for (int k = 0; k * (int)gridDim.x < total && ok; ++k) {
                const int L = snake(k);
                if (L >= total) continue;
                int b, hk, kj, q_first, n;
                decode_kv(P, nq, L, b, hk, kj, q_first, n);
                ok = wait_phase(smem_u32(&bars->fix_full), fcnt & 1u, abort_flag, limit, err);
                ++fcnt;
                for (int t = 0; ok && t < n; ++t) {
                    ok = wait_phase(smem_u32(&bars->full[slot]), ph, abort_flag, limit, err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t qb = sSt + (2 * slot) * C::TILE_BYTES;
                    const uint32_t db = qb + C::TILE_BYTES;
                    for (int kk = 0; kk < HD / 16; ++kk) {  // S^T = K Q^T, dP^T = V dO^T
                        const uint32_t off = (kk >> 2) * C::SLAB_BYTES + (kk & 3) * 32;
                        mma_ss(tmem + C::TM_S, sdesc_sw128(sK + off, 16, 1024),
                               sdesc_sw128(qb + off, 16, 1024), ID_S, kk > 0);
                        mma_ss(tmem + C::TM_DP, sdesc_sw128(sV + off, 16, 1024),
                               sdesc_sw128(db + off, 16, 1024), ID_S, kk > 0);
                    }
                    mma_commit(smem_u32(&bars->s_full));
                    if (t == n - 1) mma_commit(smem_u32(&bars->fix_empty));
                    ++pcnt;
                    ok = wait_count(&bars->p_count, 4u * pcnt, abort_flag, limit, err);
                    if (!ok) break;
                    tc_fence_after();
                    for (int kk = 0; kk < kT / 16; ++kk) {  // dV += P^T dO, dK += dS^T Q
                        const uint32_t off = kk * 16 * 128;
                        mma_ts(tmem + C::TM_A0, tmem + C::TM_S + kk * 8,
                               sdesc_sw128(db + off, C::SLAB_BYTES, 1024), ID_G,
                               (t > 0 || kk > 0) ? 1u : 0u);
                        mma_ts(tmem + C::TM_A1, tmem + C::TM_DP + kk * 8,
                               sdesc_sw128(qb + off, C::SLAB_BYTES, 1024), ID_G,
                               (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&bars->empty[slot]));
                    if (t == n - 1) mma_commit(smem_u32(&bars->o_full));
                    if (++slot == C::NST) {
                        slot = 0;
                        ph ^= 1u;
                    }
                }
            }
            mma_commit(smem_u32(&bars->drain));
            wait_phase_drain(smem_u32(&bars->drain), 0);
        }
    } else if (warp >= 4) {
        const int quarter = warp & 3;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t scnt = 0, ocnt = 0;
        bool ok = true;
        for (int k = 0; k * (int)gridDim.x < total && ok; ++k) {
            const int L = snake(k);
            if (L >= total) continue;
            int b, hk, kj, q_first, n;
            decode_kv(P, nq, L, b, hk, kj, q_first, n);
            const int key = kj * kT + quarter * 32 + lane;
            const int per = nq - q_first;
            for (int t = 0; t < n; ++t) {
                const int g = t / per;
                const int qt = q_first + (t - g * per);
                const int h = hk * G + g;
                const int64_t lbase = ((int64_t)b * P.Hq + h) * P.N;
                ok = wait_phase(smem_u32(&bars->s_full), scnt & 1u, abort_flag, limit, err);
                ++scnt;
                if (!ok) break;
                tc_fence_after();
                const bool mask = (qt * kT + kT > P.N) || (P.causal && qt == kj);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t s[32], dp[32];
                    tmem_ld32(tmem + C::TM_S + lane_off + c * 32, s);
                    tmem_ld32(tmem + C::TM_DP + lane_off + c * 32, dp);
                    // this chunk's 32 queries: LSE (log2 units) and D, shared by the warp
                    const int qa = qt * kT + c * 32;
                    const int qme = qa + lane;
                    const float lse_me = qme < P.N ? P.lse[lbase + qme] * kLog2e : 0.f;
                    const float d_me = qme < P.N ? P.dvec[lbase + qme] : 0.f;
                    tmem_ld_wait();
                    uint32_t pp[16], pd[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float l0 = __shfl_sync(0xffffffffu, lse_me, e);
                        const float l1 = __shfl_sync(0xffffffffu, lse_me, e + 1);
                        const float d0 = __shfl_sync(0xffffffffu, d_me, e);
                        const float d1 = __shfl_sync(0xffffffffu, d_me, e + 1);
                        float p0 = ex2(fmaf(__uint_as_float(s[e]), sl2, -l0));
                        float p1 = ex2(fmaf(__uint_as_float(s[e + 1]), sl2, -l1));
                        if (mask) {
                            const int q0 = qa + e;
                            p0 = (q0 < P.N && (!P.causal || key <= q0)) ? p0 : 0.f;
                            p1 = (q0 + 1 < P.N && (!P.causal || key <= q0 + 1)) ? p1 : 0.f;
                        }
                        pp[e / 2] = pack_bf16x2(p0, p1);
                        pd[e / 2] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - d0),
                                                p1 * (__uint_as_float(dp[e + 1]) - d1));
                    }
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                            tmem + C::TM_S + lane_off + c * 16),
                        "r"(pp[0]), "r"(pp[1]), "r"(pp[2]), "r"(pp[3]), "r"(pp[4]), "r"(pp[5]),
                        "r"(pp[6]), "r"(pp[7]), "r"(pp[8]), "r"(pp[9]), "r"(pp[10]), "r"(pp[11]),
                        "r"(pp[12]), "r"(pp[13]), "r"(pp[14]), "r"(pp[15])
                        : "memory");
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                            tmem + C::TM_DP + lane_off + c * 16),
                        "r"(pd[0]), "r"(pd[1]), "r"(pd[2]), "r"(pd[3]), "r"(pd[4]), "r"(pd[5]),
                        "r"(pd[6]), "r"(pd[7]), "r"(pd[8]), "r"(pd[9]), "r"(pd[10]), "r"(pd[11]),
                        "r"(pd[12]), "r"(pd[13]), "r"(pd[14]), "r"(pd[15])
                        : "memory");
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) count_release_add(&bars->p_count);
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
                        uint4 u;
                        u.x = pack_bf16x2(mul * __uint_as_float(o[e]), mul * __uint_as_float(o[e + 1]));
                        u.y = pack_bf16x2(mul * __uint_as_float(o[e + 2]), mul * __uint_as_float(o[e + 3]));
                        u.z = pack_bf16x2(mul * __uint_as_float(o[e + 4]), mul * __uint_as_float(o[e + 5]));
                        u.w = pack_bf16x2(mul * __uint_as_float(o[e + 6]), mul * __uint_as_float(o[e + 7]));
                        *reinterpret_cast<uint4 *>(dst + c * 32 + e) = u;
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
    const int hi = (int)(wait_ns >> 32), lo = (int)(wait_ns & 0xffffffff);
    tcb::bwd_dq_tc_kernel<HD><<<(int)std::min<int64_t>(tq, num_sms), tcb::kThreads, C::SMEM_BYTES, stream>>>(
        mq, mk, mv, mdo, P, (int)tq, hi, lo, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    tcb::bwd_dkdv_tc_kernel<HD><<<(int)std::min<int64_t>(tkv, num_sms), tcb::kThreads, C::SMEM_BYTES, stream>>>(
        mq, mk, mv, mdo, P, (int)tkv, hi, lo, err);
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
