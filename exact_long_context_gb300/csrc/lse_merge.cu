// lse_merge.cu - standalone log-sum-exp merge of a block partial into a running partial.
//
// `update_out_and_lse` of "序列并行与 Ring Attention：超长上下文训练技术解析" (section
// "前向传播：ZigZag Ring FlashAttention") in max-shifted form:
//   L = max(a,b) + ln(1 + e^-|a-b|),  o <- e^(a-L) o_acc + e^(b-L) o_blk,  lse <- L.
// HBM-bound: lanes own contiguous 16-byte pieces of a row so every load and store is
// coalesced; a grid-stride loop over rows on a grid sized to the SMs.  For D <= 128 half
// a warp takes a row (two rows in flight per warp) and a row's loads are issued before
// the weights are computed, so a row costs one memory latency instead of two; otherwise
// one warp per row.
#include <algorithm>

#include "ra_internal.cuh"

namespace ra {

// D <= 128 with 16-byte aligned rows (P.half_warp): half a warp per row, so a warp has two rows in
// flight and each lane moves 32 bytes of o_acc and 16 (bf16) or 32 (fp32) of o_blk per row.
// Every load is issued before the weights are known (one memory latency per row); the
// values of an identity side are discarded by select, never used.
template <bool BF16>
__device__ __forceinline__ void merge_row_half_warp(const MergeParams &P, int64_t row, int hl) {
    const int64_t n = row % P.N;
    const int64_t bh = row / P.N;
    const int64_t h = bh % P.H, b = bh / P.H;
    float *acc = P.oacc + b * P.sa[0] + h * P.sa[1] + n * P.sa[2];
    const int64_t boff = b * P.sb[0] + h * P.sb[1] + n * P.sb[2];
    const int d = hl * 8;
    const bool in = d < P.D;  // D is a multiple of 4: a lane holds 8 or (at the tail) 4 values
    const bool full = d + 8 <= P.D;
    float x[8], y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = y[i] = 0.f;
    if (in) {
        const float4 x0 = __ldcs(reinterpret_cast<const float4 *>(acc + d));
        x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
        if (full) {
            const float4 x1 = __ldcs(reinterpret_cast<const float4 *>(acc + d + 4));
            x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
        }
        if constexpr (BF16) {
            const uint16_t *src = static_cast<const uint16_t *>(P.oblk) + boff + d;
            uint32_t u[4];
            if (full) {
                const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(src));
                u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
            } else {
                const uint2 v = __ldcs(reinterpret_cast<const uint2 *>(src));
                u[0] = v.x; u[1] = v.y; u[2] = u[3] = 0u;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                y[2 * i] = __uint_as_float(u[i] << 16);
                y[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
            }
        } else {
            const float *src = static_cast<const float *>(P.oblk) + boff + d;
            const float4 y0 = __ldcs(reinterpret_cast<const float4 *>(src));
            y[0] = y0.x; y[1] = y0.y; y[2] = y0.z; y[3] = y0.w;
            if (full) {
                const float4 y1 = __ldcs(reinterpret_cast<const float4 *>(src + 4));
                y[4] = y1.x; y[5] = y1.y; y[6] = y1.z; y[7] = y1.w;
            }
        }
    }
    const MergeW w = merge_weights(P.lse_acc[row], P.lse_blk[row]);
    const bool use_a = w.wa != 0.f, use_b = w.wb != 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = (use_a ? w.wa * x[i] : 0.f) + (use_b ? w.wb * y[i] : 0.f);
    if (in) {
        __stcs(reinterpret_cast<float4 *>(acc + d), make_float4(x[0], x[1], x[2], x[3]));
        if (full) __stcs(reinterpret_cast<float4 *>(acc + d + 4), make_float4(x[4], x[5], x[6], x[7]));
    }
    if (hl == 0) P.lse_acc[row] = w.L;
}

template <bool BF16>
__global__ void __launch_bounds__(256) lse_merge_kernel(const __grid_constant__ MergeParams P) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const bool vec = P.vec != 0;
    if (P.half_warp) {
        const int half = lane >> 4, hl = lane & 15;
        for (int64_t r2 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); 2 * r2 < P.rows;
             r2 += warps) {
            const int64_t row = 2 * r2 + half;
            if (row < P.rows) merge_row_half_warp<BF16>(P, row, hl);
        }
        return;
    }
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < P.rows;
         row += warps) {
        const int64_t n = row % P.N;
        const int64_t bh = row / P.N;
        const int64_t h = bh % P.H, b = bh / P.H;
        float *acc = P.oacc + b * P.sa[0] + h * P.sa[1] + n * P.sa[2];
        const int64_t boff = b * P.sb[0] + h * P.sb[1] + n * P.sb[2];
        const float a = P.lse_acc[row];
        const float bl = P.lse_blk[row];
        const MergeW w = merge_weights(a, bl);
        if (vec) {
            for (int d = lane * 4; d < P.D; d += 128) {
                float4 x = (w.wa != 0.f) ? *reinterpret_cast<const float4 *>(acc + d)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                float y0, y1, y2, y3;
                if constexpr (BF16) {
                    const uint2 u = *reinterpret_cast<const uint2 *>(
                        static_cast<const uint16_t *>(P.oblk) + boff + d);
                    y0 = __uint_as_float(u.x << 16);
                    y1 = __uint_as_float(u.x & 0xffff0000u);
                    y2 = __uint_as_float(u.y << 16);
                    y3 = __uint_as_float(u.y & 0xffff0000u);
                } else {
                    const float4 f = *reinterpret_cast<const float4 *>(
                        static_cast<const float *>(P.oblk) + boff + d);
                    y0 = f.x;
                    y1 = f.y;
                    y2 = f.z;
                    y3 = f.w;
                }
                if (w.wb == 0.f) y0 = y1 = y2 = y3 = 0.f;
                x.x = w.wa * x.x + w.wb * y0;
                x.y = w.wa * x.y + w.wb * y1;
                x.z = w.wa * x.z + w.wb * y2;
                x.w = w.wa * x.w + w.wb * y3;
                *reinterpret_cast<float4 *>(acc + d) = x;
            }
        } else {
            for (int d = lane; d < P.D; d += 32) {
                const float x = (w.wa != 0.f) ? acc[d] : 0.f;
                float y;
                if constexpr (BF16) {
                    y = bf16_to_f32(static_cast<const uint16_t *>(P.oblk)[boff + d]);
                } else {
                    y = static_cast<const float *>(P.oblk)[boff + d];
                }
                if (w.wb == 0.f) y = 0.f;
                acc[d] = w.wa * x + w.wb * y;
            }
        }
        __syncwarp();
        if (lane == 0) P.lse_acc[row] = w.L;
    }
}

// Rows [r0, r1) of every (b, h): O = 0 and LSE = -inf, the identity partial of a row
// that sees no key (padding rows of a packed batch).
__global__ void __launch_bounds__(256) fill_identity_kernel(void *o, int o_bf16, int64_t s0, int64_t s1,
                                                            int64_t s2, float *lse, int H, int N, int D,
                                                            int r0, int r1) {
    const int64_t rows = (int64_t)(r1 - r0);
    const int64_t total = (int64_t)gridDim.y * H * rows;  // gridDim.y = B
    const int b = blockIdx.y;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)H * rows * D;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int d = (int)(i % D);
        const int64_t hr = i / D;
        const int h = (int)(hr / rows);
        const int n = r0 + (int)(hr - (int64_t)h * rows);
        const int64_t off = (int64_t)b * s0 + (int64_t)h * s1 + (int64_t)n * s2 + d;
        if (o_bf16)
            static_cast<uint16_t *>(o)[off] = 0;
        else
            static_cast<float *>(o)[off] = 0.f;
        if (d == 0) lse[((int64_t)b * H + h) * N + n] = -INFINITY;
    }
    (void)total;
}

cudaError_t launch_fill_identity(void *o, int o_bf16, const int64_t *so, float *lse, int B, int H,
                                 int N, int D, int r0, int r1, int num_sms, cudaStream_t stream) {
    if (r1 <= r0 || B <= 0 || H <= 0 || D <= 0) return cudaSuccess;
    const int64_t work = (int64_t)H * (r1 - r0) * D;
    int gx = (int)std::min<int64_t>((work + 255) / 256, (int64_t)num_sms * 8);
    if (gx < 1) gx = 1;
    fill_identity_kernel<<<dim3(gx, B), 256, 0, stream>>>(o, o_bf16, so[0], so[1], so[2], lse, H, N, D,
                                                          r0, r1);
    return cudaGetLastError();
}

cudaError_t launch_lse_merge(const MergeParams &P, int num_sms, cudaStream_t stream) {
    if (P.rows <= 0) return cudaSuccess;
    const int threads = 256;
    const int64_t want = (P.rows + 7) / 8;
    const int64_t cap = (int64_t)num_sms * 8;  // 8 blocks of 8 warps per SM
    const int grid = (int)(want < cap ? want : cap);
    if (P.blk_bf16)
        lse_merge_kernel<true><<<grid, threads, 0, stream>>>(P);
    else
        lse_merge_kernel<false><<<grid, threads, 0, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace ra
