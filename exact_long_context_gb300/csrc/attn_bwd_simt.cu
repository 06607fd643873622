// attn_bwd_simt.cu - gradients of exact attention on the CUDA cores (float32 arithmetic).
//
// For L = sum(dO * O), with P_ij = exp(s_ij - LSE_i) recomputed from the forward's LSE
// (the recompute-from-LSE backward of the `ring_attention_backward` listing of
// "Ring Attention 论文解析"):
//   D_i   = sum_t dO[i,t] O[i,t]                      (bwd_rowdot_kernel)
//   dV_j  = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i   (bwd_dkdv_simt_kernel)
//   dQ_i  = scale sum_j dS_ij k_j                     (bwd_dq_simt_kernel)
//   with dS_ij = P_ij (dO_i . v_j - D_i).
// The dK/dV kernel owns a tile of keys of one KV head and walks every query row of the
// heads that read it (GQA); the dQ kernel owns query rows.  Each output element has one
// writer per launch, so no atomics are needed.  A launch covers the segments of one ring
// step (struct BSeg): the whole-sequence backward is one segment; on a ring, running
// sums carry dQ, dK and dV from step to step in fp32.
#include <algorithm>

#include "ra_internal.cuh"

namespace ra {

template <bool BF16>
__device__ __forceinline__ float bld(const void *base, int64_t idx) {
    if constexpr (BF16)
        return bf16_to_f32(static_cast<const uint16_t *>(base)[idx]);
    else
        return static_cast<const float *>(base)[idx];
}

template <bool BF16>
__device__ __forceinline__ void bst(void *base, int64_t idx, float x) {
    if constexpr (BF16)
        static_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
    else
        static_cast<float *>(base)[idx] = x;
}

__device__ __forceinline__ float bwarp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// D_i = sum_t dO[i,t] O[i,t]: one warp per row.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const __grid_constant__ BwdParams P) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)P.B * P.Hq * P.N;
    for (int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows;
         row += (int64_t)gridDim.x * 8) {
        const int64_t n = row % P.N, bh = row / P.N;
        const int64_t h = bh % P.Hq, b = bh / P.Hq;
        const int64_t oo = b * P.so[0] + h * P.so[1] + n * P.so[2];
        const int64_t od = b * P.sdo[0] + h * P.sdo[1] + n * P.sdo[2];
        float acc = 0.f;
        for (int d = lane; d < P.D; d += 32) acc += bld<BF16>(P.o, oo + d) * bld<BF16>(P.dout, od + d);
        acc = bwarp_sum(acc);
        if (lane == 0) P.dvec[row] = acc;
    }
}

// The same for bf16 rows of 16-byte multiples with 16-byte aligned starts: each lane
// reads 8 elements of O and of dO per load; a warp covers 256 elements of a row per
// pass (two rows of D = 128, four of D = 64), so every lane has work and the loads stay
// coalesced.  A warp takes kRowdotPasses passes at a time and issues all their loads
// before the first product, so each lane has 2 * kRowdotPasses 16-byte loads in flight.
// HBM-bound: 4 D bytes read per row.
constexpr int kRowdotPasses = 4;
__global__ void __launch_bounds__(256) bwd_rowdot_vec_kernel(const __grid_constant__ BwdParams P) {
    const int lane = threadIdx.x & 31;
    const int per_row = P.D / 8;                 // lanes per row (8 or 16)
    const int rows_per_warp = 32 / per_row;      // 4 or 2
    const int sub = lane / per_row, l = lane - sub * per_row;
    const int64_t rows = (int64_t)P.B * P.Hq * P.N;
    const int64_t span = (int64_t)rows_per_warp * kRowdotPasses;  // rows of one warp iteration
    const int64_t wstride = (int64_t)gridDim.x * 8 * span;
    for (int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * span; row0 < rows; row0 += wstride) {
        // (batch, head, position) of this lane's first row, then stepped: two divisions per
        // warp iteration instead of two 64-bit divisions per row (they made the pass
        // issue-bound)
        const int64_t first = row0 + sub;
        const int64_t bh0 = first / P.N;
        int n = (int)(first - bh0 * P.N);
        int64_t b = bh0 / P.Hq;
        int h = (int)(bh0 - b * P.Hq);
        uint4 x[kRowdotPasses], y[kRowdotPasses];
#pragma unroll
        for (int p = 0; p < kRowdotPasses; ++p) {
            if (p > 0) {
                n += rows_per_warp;
                while (n >= P.N) {
                    n -= P.N;
                    if (++h == P.Hq) {
                        h = 0;
                        ++b;
                    }
                }
            }
            const int64_t row = row0 + p * rows_per_warp + sub;
            x[p] = y[p] = make_uint4(0u, 0u, 0u, 0u);
            if (row < rows) {
                x[p] = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(P.o) + b * P.so[0] +
                                                              (int64_t)h * P.so[1] + (int64_t)n * P.so[2]) + l);
                y[p] = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(P.dout) + b * P.sdo[0] +
                                                              (int64_t)h * P.sdo[1] + (int64_t)n * P.sdo[2]) + l);
            }
        }
#pragma unroll
        for (int p = 0; p < kRowdotPasses; ++p) {
            const uint32_t xa[4] = {x[p].x, x[p].y, x[p].z, x[p].w}, ya[4] = {y[p].x, y[p].y, y[p].z, y[p].w};
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = fmaf(__uint_as_float(xa[i] << 16), __uint_as_float(ya[i] << 16), acc);
                acc = fmaf(__uint_as_float(xa[i] & 0xffff0000u), __uint_as_float(ya[i] & 0xffff0000u), acc);
            }
            // reduce within each row's group of lanes
            for (int o = per_row >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            const int64_t row = row0 + p * rows_per_warp + sub;
            if (l == 0 && row < rows) P.dvec[row] = acc;
        }
    }
}

// A gradient element of a ring step: the step's value plus the running value of earlier
// steps (unless the range is new this step), written to the gradient on the range's last
// step and to the fp32 running buffer otherwise.
template <bool BF16>
__device__ __forceinline__ void bwd_put(void *g, int64_t gi, float *acc, int64_t ai, float x, int flags) {
    if (!(flags & SEG_FIRST)) x += acc[ai];
    if (flags & SEG_FINAL)
        bst<BF16>(g, gi, x);
    else
        acc[ai] = x;
}

constexpr int kBwdKeysPerWarp = 2;
constexpr int kBwdWarps = 4;
constexpr int kBwdKeys = kBwdKeysPerWarp * kBwdWarps;  // keys per block

// dK, dV for kBwdKeys keys of one segment's fixed range and one (b, KV head); lanes own
// head dimensions (D <= 128).  blockIdx.y = segment * tiles + tile.
template <bool BF16>
__global__ void __launch_bounds__(128) bwd_dkdv_simt_kernel(const __grid_constant__ BwdParams P) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int bhk = blockIdx.x;
    const int b = bhk / P.Hkv, hk = bhk - (bhk / P.Hkv) * P.Hkv;
    const int G = P.Hq / P.Hkv;
    const int tps = (P.flen + kBwdKeys - 1) / kBwdKeys;
    const int si = blockIdx.y / tps;
    const BSeg &S = P.seg[si];
    const int j0 = S.f0 + (blockIdx.y - si * tps) * kBwdKeys + warp * kBwdKeysPerWarp;
    float kr[kBwdKeysPerWarp][4], vr[kBwdKeysPerWarp][4];
    float dka[kBwdKeysPerWarp][4], dva[kBwdKeysPerWarp][4];
#pragma unroll
    for (int t = 0; t < kBwdKeysPerWarp; ++t) {
        const int j = j0 + t;
        const int64_t jp = (int64_t)j * P.rs + S.f_rank;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            const bool in = j < S.f1 && d < P.D;
            kr[t][c] = in ? bld<BF16>(P.k, (int64_t)b * P.sk[0] + (int64_t)hk * P.sk[1] + jp * P.sk[2] + d)
                          : 0.f;
            vr[t][c] = in ? bld<BF16>(P.v, (int64_t)b * P.sv[0] + (int64_t)hk * P.sv[1] + jp * P.sv[2] + d)
                          : 0.f;
            dka[t][c] = 0.f;
            dva[t][c] = 0.f;
        }
    }
    for (int g = 0; g < G; ++g) {
        const int h = hk * G + g;
        const int64_t lbase = ((int64_t)b * P.Hq + h) * P.N;
        for (int pc = 0; pc < 2; ++pc) {
            const int first = P.causal ? max(S.s0[pc], j0 + S.diag) : S.s0[pc];
            for (int i = first; i < S.s1[pc]; ++i) {
                const int64_t ip = (int64_t)i * P.rs + S.s_rank;
                float qi[4], di[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int d = lane + 32 * c;
                    qi[c] = d < P.D ? bld<BF16>(P.q, (int64_t)b * P.sq[0] + (int64_t)h * P.sq[1] + ip * P.sq[2] + d)
                                    : 0.f;
                    di[c] = d < P.D ? bld<BF16>(P.dout,
                                                (int64_t)b * P.sdo[0] + (int64_t)h * P.sdo[1] + ip * P.sdo[2] + d)
                                    : 0.f;
                }
                const float lse_i = P.lse[lbase + ip];
                const float d_i = P.dvec[lbase + ip];
#pragma unroll
                for (int t = 0; t < kBwdKeysPerWarp; ++t) {
                    const int j = j0 + t;
                    float s = 0.f, dp = 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        s = fmaf(qi[c], kr[t][c], s);
                        dp = fmaf(di[c], vr[t][c], dp);
                    }
                    s = bwarp_sum(s);
                    dp = bwarp_sum(dp);
                    const bool vis = j < S.f1 && (!P.causal || j + S.diag <= i) && lse_i != -INFINITY;
                    const float p = vis ? exp2f(s * P.scale_log2 - lse_i * kLog2e) : 0.f;
                    const float ds = p * (dp - d_i);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        dva[t][c] = fmaf(p, di[c], dva[t][c]);
                        dka[t][c] = fmaf(ds, qi[c], dka[t][c]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kBwdKeysPerWarp; ++t) {
        const int j = j0 + t;
        if (j >= S.f1) continue;
        const int64_t jp = (int64_t)j * P.rs + S.f_rank;
        const int64_t arow = (((int64_t)b * P.Hkv + hk) * P.N + jp) * P.D;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d >= P.D) continue;
            bwd_put<BF16>(P.dk, (int64_t)b * P.sdk[0] + (int64_t)hk * P.sdk[1] + jp * P.sdk[2] + d, P.acc_k,
                          arow + d, P.scale * dka[t][c], S.flags);
            bwd_put<BF16>(P.dv, (int64_t)b * P.sdv[0] + (int64_t)hk * P.sdv[1] + jp * P.sdv[2] + d, P.acc_v,
                          arow + d, dva[t][c], S.flags);
        }
    }
}

constexpr int kDqRows = 8;   // query rows per block (2 per warp)
constexpr int kDqRowsPerWarp = kDqRows / 4;
constexpr int kDqKT = 32;    // keys per shared-memory tile

// dQ for kDqRows query rows of one segment's fixed range and one (b, h).
template <bool BF16>
__global__ void __launch_bounds__(128) bwd_dq_simt_kernel(const __grid_constant__ BwdParams P) {
    __shared__ float sK[kDqKT][129];
    __shared__ float sV[kDqKT][129];
    __shared__ float sQ[kDqRows][128];
    __shared__ float sDo[kDqRows][128];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x;
    const int b = bh / P.Hq, h = bh - (bh / P.Hq) * P.Hq;
    const int hk = h / (P.Hq / P.Hkv);
    const int tps = (P.flen + kDqRows - 1) / kDqRows;
    const int si = blockIdx.y / tps;
    const BSeg &S = P.seg[si];
    const int qa = S.f0 + (blockIdx.y - si * tps) * kDqRows;
    const int qb = min(qa + kDqRows, S.f1);
    const int D = P.D;
    for (int idx = tid; idx < kDqRows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx - (idx / D) * D;
        const int row = qa + r;
        const int64_t rp = (int64_t)row * P.rs + S.f_rank;
        sQ[r][d] = row < qb ? bld<BF16>(P.q, (int64_t)b * P.sq[0] + (int64_t)h * P.sq[1] + rp * P.sq[2] + d)
                            : 0.f;
        sDo[r][d] = row < qb
                        ? bld<BF16>(P.dout, (int64_t)b * P.sdo[0] + (int64_t)h * P.sdo[1] + rp * P.sdo[2] + d)
                        : 0.f;
    }
    const int64_t lbase = ((int64_t)b * P.Hq + h) * P.N;
    float lse_r[kDqRowsPerWarp], d_r[kDqRowsPerWarp], acc[kDqRowsPerWarp][4];
#pragma unroll
    for (int rr = 0; rr < kDqRowsPerWarp; ++rr) {
        const int row = qa + warp * kDqRowsPerWarp + rr;
        const int64_t rp = (int64_t)row * P.rs + S.f_rank;
        lse_r[rr] = row < qb ? P.lse[lbase + rp] : -INFINITY;
        d_r[rr] = row < qb ? P.dvec[lbase + rp] : 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[rr][c] = 0.f;
    }
    for (int pc = 0; pc < 2; ++pc) {
        const int klim = S.s1[pc];
        const int kend = P.causal ? min(klim, qb - S.diag) : klim;
        for (int t0 = S.s0[pc]; t0 < kend; t0 += kDqKT) {
            __syncthreads();
            for (int idx = tid; idx < kDqKT * D; idx += blockDim.x) {
                const int j = idx / D, d = idx - (idx / D) * D;
                const int key = t0 + j;
                const bool in = key < klim;
                const int64_t kp = (int64_t)key * P.rs + S.s_rank;
                sK[j][d] = in ? bld<BF16>(P.k, (int64_t)b * P.sk[0] + (int64_t)hk * P.sk[1] + kp * P.sk[2] + d)
                              : 0.f;
                sV[j][d] = in ? bld<BF16>(P.v, (int64_t)b * P.sv[0] + (int64_t)hk * P.sv[1] + kp * P.sv[2] + d)
                              : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int rr = 0; rr < kDqRowsPerWarp; ++rr) {
                const int lr = warp * kDqRowsPerWarp + rr;
                const int row = qa + lr;
                const int key = t0 + lane;
                float s = 0.f, dp = 0.f;
                for (int d = 0; d < D; ++d) {
                    s = fmaf(sQ[lr][d], sK[lane][d], s);
                    dp = fmaf(sDo[lr][d], sV[lane][d], dp);
                }
                const bool vis = key < klim && row < qb && (!P.causal || key + S.diag <= row) &&
                                 lse_r[rr] != -INFINITY;
                const float p = vis ? exp2f(s * P.scale_log2 - lse_r[rr] * kLog2e) : 0.f;
                const float ds = p * (dp - d_r[rr]);
                for (int j = 0; j < kDqKT; ++j) {
                    const float dsj = __shfl_sync(0xffffffffu, ds, j);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int d = lane + 32 * c;
                        if (d < D) acc[rr][c] = fmaf(dsj, sK[j][d], acc[rr][c]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kDqRowsPerWarp; ++rr) {
        const int row = qa + warp * kDqRowsPerWarp + rr;
        if (row >= qb) continue;
        const int64_t rp = (int64_t)row * P.rs + S.f_rank;
        const int64_t arow = (((int64_t)b * P.Hq + h) * P.N + rp) * D;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d < D)
                bwd_put<BF16>(P.dq, (int64_t)b * P.sdq[0] + (int64_t)h * P.sdq[1] + rp * P.sdq[2] + d, P.acc_q,
                              arow + d, P.scale * acc[rr][c], S.flags);
        }
    }
}

cudaError_t launch_bwd_rowdot(const BwdParams &P, int num_sms, cudaStream_t stream) {
    if (P.B <= 0 || P.Hq <= 0 || P.N <= 0) return cudaSuccess;
    const int64_t rows = (int64_t)P.B * P.Hq * P.N;
    const bool vec = P.bf16 && (P.D == 64 || P.D == 128) && P.so[0] % 8 == 0 && P.so[1] % 8 == 0 &&
                     P.so[2] % 8 == 0 && P.sdo[0] % 8 == 0 && P.sdo[1] % 8 == 0 && P.sdo[2] % 8 == 0 &&
                     reinterpret_cast<uintptr_t>(P.o) % 16 == 0 && reinterpret_cast<uintptr_t>(P.dout) % 16 == 0;
    if (vec) {
        const int64_t span = (int64_t)(256 / P.D) * kRowdotPasses;  // rows of one warp iteration
        const int64_t warps = (rows + span - 1) / span;                  // warps needed
        const int g = (int)std::min<int64_t>((warps + 7) / 8, (int64_t)num_sms * 8);
        bwd_rowdot_vec_kernel<<<g, 256, 0, stream>>>(P);
        return cudaGetLastError();
    }
    const int g0 = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms * 16);
    if (P.bf16)
        bwd_rowdot_kernel<true><<<g0, 256, 0, stream>>>(P);
    else
        bwd_rowdot_kernel<false><<<g0, 256, 0, stream>>>(P);
    return cudaGetLastError();
}

// The dQ kernel (parts & 1) and the dK/dV kernel (parts & 2) over the segments in P (the
// D vector is computed before).
cudaError_t launch_attn_bwd_simt(const BwdParams &P, int parts, cudaStream_t stream) {
    if (P.B <= 0 || P.Hq <= 0 || P.nseg <= 0 || P.flen <= 0) return cudaSuccess;
    const dim3 gkv(P.B * P.Hkv, P.nseg * ((P.flen + kBwdKeys - 1) / kBwdKeys));
    const dim3 gq(P.B * P.Hq, P.nseg * ((P.flen + kDqRows - 1) / kDqRows));
    if ((int64_t)P.nseg * ((P.flen + kDqRows - 1) / kDqRows) > 65535) return cudaErrorInvalidConfiguration;
    if (P.bf16) {
        if (parts & 2) bwd_dkdv_simt_kernel<true><<<gkv, 128, 0, stream>>>(P);
        if (parts & 1) bwd_dq_simt_kernel<true><<<gq, 128, 0, stream>>>(P);
    } else {
        if (parts & 2) bwd_dkdv_simt_kernel<false><<<gkv, 128, 0, stream>>>(P);
        if (parts & 1) bwd_dq_simt_kernel<false><<<gq, 128, 0, stream>>>(P);
    }
    return cudaGetLastError();
}

}  // namespace ra
