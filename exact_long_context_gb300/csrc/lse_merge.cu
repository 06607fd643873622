// lse_merge.cu - standalone log-sum-exp merge of a block partial into a running partial.
//
// `update_out_and_lse` of "序列并行与 Ring Attention：超长上下文训练技术解析" (section
// "前向传播：ZigZag Ring FlashAttention") in max-shifted form:
//   L = max(a,b) + ln(1 + e^-|a-b|),  o <- e^(a-L) o_acc + e^(b-L) o_blk,  lse <- L.
// HBM-bound: one warp per row, lanes own contiguous 16-byte pieces of the row so every
// load and store is coalesced; a grid-stride loop over rows on a grid sized to the SMs.
// For D <= 128 the row's loads are issued before the weights are computed, so a row
// costs one memory latency instead of two.
#include <algorithm>

#include "ra_internal.cuh"

namespace ra {

template <bool BF16>
__global__ void __launch_bounds__(256) lse_merge_kernel(const __grid_constant__ MergeParams P) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const bool vec = P.vec != 0;
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < P.rows;
         row += warps) {
        const int64_t n = row % P.N;
        const int64_t bh = row / P.N;
        const int64_t h = bh % P.H, b = bh / P.H;
        float *acc = P.oacc + b * P.sa[0] + h * P.sa[1] + n * P.sa[2];
        const int64_t boff = b * P.sb[0] + h * P.sb[1] + n * P.sb[2];
        if (vec && P.D <= 128) {
            // every load is issued before the weights are known (one memory latency per
            // row); the values of an identity side are discarded by select, never used
            const int d = lane * 4;
            const bool in = d < P.D;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            float y0 = 0.f, y1 = 0.f, y2 = 0.f, y3 = 0.f;
            if (in) {
                x = __ldcs(reinterpret_cast<const float4 *>(acc + d));
                if constexpr (BF16) {
                    const uint2 u = __ldcs(reinterpret_cast<const uint2 *>(
                        static_cast<const uint16_t *>(P.oblk) + boff + d));
                    y0 = __uint_as_float(u.x << 16);
                    y1 = __uint_as_float(u.x & 0xffff0000u);
                    y2 = __uint_as_float(u.y << 16);
                    y3 = __uint_as_float(u.y & 0xffff0000u);
                } else {
                    const float4 f = __ldcs(reinterpret_cast<const float4 *>(
                        static_cast<const float *>(P.oblk) + boff + d));
                    y0 = f.x;
                    y1 = f.y;
                    y2 = f.z;
                    y3 = f.w;
                }
            }
            const MergeW w = merge_weights(P.lse_acc[row], P.lse_blk[row]);
            if (w.wa == 0.f) x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (w.wb == 0.f) y0 = y1 = y2 = y3 = 0.f;
            if (in) {
                x.x = w.wa * x.x + w.wb * y0;
                x.y = w.wa * x.y + w.wb * y1;
                x.z = w.wa * x.z + w.wb * y2;
                x.w = w.wa * x.w + w.wb * y3;
                __stcs(reinterpret_cast<float4 *>(acc + d), x);
            }
            __syncwarp();
            if (lane == 0) P.lse_acc[row] = w.L;
            continue;
        }
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
