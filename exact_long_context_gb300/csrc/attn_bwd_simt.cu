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
// writer, so no atomics are needed.
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

constexpr int kBwdKeysPerWarp = 2;
constexpr int kBwdWarps = 4;
constexpr int kBwdKeys = kBwdKeysPerWarp * kBwdWarps;  // keys per block

// dK, dV for kBwdKeys keys of one (b, KV head); lanes own head dimensions (D <= 128).
template <bool BF16>
__global__ void __launch_bounds__(128) bwd_dkdv_simt_kernel(const __grid_constant__ BwdParams P) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int bhk = blockIdx.x;
    const int b = bhk / P.Hkv, hk = bhk - (bhk / P.Hkv) * P.Hkv;
    const int G = P.Hq / P.Hkv;
    const int j0 = blockIdx.y * kBwdKeys + warp * kBwdKeysPerWarp;
    float kr[kBwdKeysPerWarp][4], vr[kBwdKeysPerWarp][4];
    float dka[kBwdKeysPerWarp][4], dva[kBwdKeysPerWarp][4];
#pragma unroll
    for (int t = 0; t < kBwdKeysPerWarp; ++t) {
        const int j = j0 + t;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            const bool in = j < P.N && d < P.D;
            kr[t][c] = in ? bld<BF16>(P.k, (int64_t)b * P.sk[0] + (int64_t)hk * P.sk[1] +
                                                (int64_t)j * P.sk[2] + d)
                          : 0.f;
            vr[t][c] = in ? bld<BF16>(P.v, (int64_t)b * P.sv[0] + (int64_t)hk * P.sv[1] +
                                                (int64_t)j * P.sv[2] + d)
                          : 0.f;
            dka[t][c] = 0.f;
            dva[t][c] = 0.f;
        }
    }
    const int first_row = P.causal ? min(j0, P.N) : 0;
    for (int g = 0; g < G; ++g) {
        const int h = hk * G + g;
        const int64_t lbase = ((int64_t)b * P.Hq + h) * P.N;
        for (int i = first_row; i < P.N; ++i) {
            float qi[4], di[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int d = lane + 32 * c;
                qi[c] = d < P.D ? bld<BF16>(P.q, (int64_t)b * P.sq[0] + (int64_t)h * P.sq[1] +
                                                      (int64_t)i * P.sq[2] + d)
                                : 0.f;
                di[c] = d < P.D ? bld<BF16>(P.dout, (int64_t)b * P.sdo[0] + (int64_t)h * P.sdo[1] +
                                                         (int64_t)i * P.sdo[2] + d)
                                : 0.f;
            }
            const float lse_i = P.lse[lbase + i];
            const float d_i = P.dvec[lbase + i];
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
                const bool vis = j < P.N && (!P.causal || j <= i) && lse_i != -INFINITY;
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
#pragma unroll
    for (int t = 0; t < kBwdKeysPerWarp; ++t) {
        const int j = j0 + t;
        if (j >= P.N) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d >= P.D) continue;
            bst<BF16>(P.dk, (int64_t)b * P.sdk[0] + (int64_t)hk * P.sdk[1] + (int64_t)j * P.sdk[2] + d,
                      P.scale * dka[t][c]);
            bst<BF16>(P.dv, (int64_t)b * P.sdv[0] + (int64_t)hk * P.sdv[1] + (int64_t)j * P.sdv[2] + d,
                      dva[t][c]);
        }
    }
}

constexpr int kDqRows = 8;   // query rows per block (2 per warp)
constexpr int kDqRowsPerWarp = kDqRows / 4;
constexpr int kDqKT = 32;    // keys per shared-memory tile

// dQ for kDqRows query rows of one (b, h).
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
    const int qa = blockIdx.y * kDqRows;
    const int qb = min(qa + kDqRows, P.N);
    const int D = P.D;
    for (int idx = tid; idx < kDqRows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx - (idx / D) * D;
        const int row = qa + r;
        sQ[r][d] = row < qb ? bld<BF16>(P.q, (int64_t)b * P.sq[0] + (int64_t)h * P.sq[1] +
                                                  (int64_t)row * P.sq[2] + d)
                            : 0.f;
        sDo[r][d] = row < qb ? bld<BF16>(P.dout, (int64_t)b * P.sdo[0] + (int64_t)h * P.sdo[1] +
                                                      (int64_t)row * P.sdo[2] + d)
                             : 0.f;
    }
    const int64_t lbase = ((int64_t)b * P.Hq + h) * P.N;
    float lse_r[kDqRowsPerWarp], d_r[kDqRowsPerWarp], acc[kDqRowsPerWarp][4];
#pragma unroll
    for (int rr = 0; rr < kDqRowsPerWarp; ++rr) {
        const int row = qa + warp * kDqRowsPerWarp + rr;
        lse_r[rr] = row < qb ? P.lse[lbase + row] : -INFINITY;
        d_r[rr] = row < qb ? P.dvec[lbase + row] : 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[rr][c] = 0.f;
    }
    const int kend = P.causal ? qb : P.N;
    for (int t0 = 0; t0 < kend; t0 += kDqKT) {
        __syncthreads();
        for (int idx = tid; idx < kDqKT * D; idx += blockDim.x) {
            const int j = idx / D, d = idx - (idx / D) * D;
            const int key = t0 + j;
            const bool in = key < P.N;
            sK[j][d] = in ? bld<BF16>(P.k, (int64_t)b * P.sk[0] + (int64_t)hk * P.sk[1] +
                                               (int64_t)key * P.sk[2] + d)
                          : 0.f;
            sV[j][d] = in ? bld<BF16>(P.v, (int64_t)b * P.sv[0] + (int64_t)hk * P.sv[1] +
                                               (int64_t)key * P.sv[2] + d)
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
            const bool vis = key < P.N && row < qb && (!P.causal || key <= row) &&
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
#pragma unroll
    for (int rr = 0; rr < kDqRowsPerWarp; ++rr) {
        const int row = qa + warp * kDqRowsPerWarp + rr;
        if (row >= qb) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d < D)
                bst<BF16>(P.dq, (int64_t)b * P.sdq[0] + (int64_t)h * P.sdq[1] + (int64_t)row * P.sdq[2] + d,
                          P.scale * acc[rr][c]);
        }
    }
}

cudaError_t launch_bwd_rowdot(const BwdParams &P, int num_sms, cudaStream_t stream) {
    if (P.B <= 0 || P.Hq <= 0 || P.N <= 0) return cudaSuccess;
    const int64_t rows = (int64_t)P.B * P.Hq * P.N;
    const int g0 = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms * 16);
    if (P.bf16)
        bwd_rowdot_kernel<true><<<g0, 256, 0, stream>>>(P);
    else
        bwd_rowdot_kernel<false><<<g0, 256, 0, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd_simt(const BwdParams &P, int num_sms, cudaStream_t stream) {
    if (P.B <= 0 || P.Hq <= 0 || P.N <= 0) return cudaSuccess;
    const int64_t rows = (int64_t)P.B * P.Hq * P.N;
    const int g0 = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms * 16);
    const dim3 gkv(P.B * P.Hkv, (P.N + kBwdKeys - 1) / kBwdKeys);
    const dim3 gq(P.B * P.Hq, (P.N + kDqRows - 1) / kDqRows);
    if (gkv.y > 65535 || gq.y > 65535) return cudaErrorInvalidConfiguration;
    if (P.bf16) {
        bwd_rowdot_kernel<true><<<g0, 256, 0, stream>>>(P);
        bwd_dkdv_simt_kernel<true><<<gkv, 128, 0, stream>>>(P);
        bwd_dq_simt_kernel<true><<<gq, 128, 0, stream>>>(P);
    } else {
        bwd_rowdot_kernel<false><<<g0, 256, 0, stream>>>(P);
        bwd_dkdv_simt_kernel<false><<<gkv, 128, 0, stream>>>(P);
        bwd_dq_simt_kernel<false><<<gq, 128, 0, stream>>>(P);
    }
    return cudaGetLastError();
}

}  // namespace ra
