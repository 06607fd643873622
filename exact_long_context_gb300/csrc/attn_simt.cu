// attn_simt.cu - exact attention on the CUDA cores, float32 arithmetic.
//
// The path for float32 inputs (the 1e-5 tolerance case) and for shapes the tensor-core
// kernel does not take (head sizes other than 64/128, unaligned strides).  Same step
// contract as the tensor-core kernel: one launch covers every segment of a ring step,
// and the epilogue writes, or LSE-merges into, the running result.
//
// Per query row the loop is the online softmax of "Ring Attention explained"
// (guijiagi.com), section "在线 Softmax 算法": running max m, running sum l, running
// unnormalised output, each rescaled by 2^(m_old - m_new) when the max grows, with
// the normalisation deferred to the end ("第12章 FlashAttention原理与实现",
// FlashAttention-2 paragraph).  Scores are kept in log2 units (scale * log2 e folded
// into one multiply) so the exponentials are exp2.
#include "ra_internal.cuh"

namespace ra {

constexpr int kSimtRows = 16;   // query rows per block (4 per warp)
constexpr int kSimtKT = 32;     // keys per shared-memory tile (one per lane)
constexpr int kSimtDMax = 128;  // largest head size

template <bool BF16>
__device__ __forceinline__ float ld_elem(const void *base, int64_t idx) {
    if constexpr (BF16) {
        return bf16_to_f32(static_cast<const uint16_t *>(base)[idx]);
    } else {
        return static_cast<const float *>(base)[idx];
    }
}

template <bool BF16>
__device__ __forceinline__ void st_elem(void *base, int64_t idx, float x) {
    if constexpr (BF16) {
        static_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
    } else {
        static_cast<float *>(base)[idx] = x;
    }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <bool BF16>
__global__ void __launch_bounds__(128) attn_simt_kernel(const __grid_constant__ StepParams P) {
    __shared__ float sK[kSimtKT][kSimtDMax + 1];
    __shared__ float sV[kSimtKT][kSimtDMax];
    __shared__ float sQ[kSimtRows][kSimtDMax];

    const int bh = blockIdx.x;
    const int b = bh / P.Hq, h = bh - (bh / P.Hq) * P.Hq;
    int si, lb;
    decode_work(P, blockIdx.y, si, lb);
    const Seg &S = P.seg[si];
    const int qa = S.q0 + lb * kSimtRows;
    if (lb < 0 || qa >= S.q1) return;
    const int qb = min(qa + kSimtRows, S.q1);
    const int hk = h / (P.Hq / P.Hkv);
    const int D = P.D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int64_t qbase = (int64_t)b * P.sq[0] + (int64_t)h * P.sq[1];
    const int64_t kbase = (int64_t)b * P.sk[0] + (int64_t)hk * P.sk[1];
    const int64_t vbase = (int64_t)b * P.sv[0] + (int64_t)hk * P.sv[1];

    // segment indices map to sequence positions through the rank interleave
    const int64_t qs = (int64_t)P.rs * P.sq[2], ks_ = (int64_t)P.rs * P.sk[2], vs_ = (int64_t)P.rs * P.sv[2];
    const int64_t qoff = (int64_t)S.q_rank * P.sq[2];
    const int64_t koff = (int64_t)S.kv_rank * P.sk[2], voff = (int64_t)S.kv_rank * P.sv[2];
    for (int idx = tid; idx < kSimtRows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx - (idx / D) * D;
        const int row = qa + r;
        sQ[r][d] = row < qb ? ld_elem<BF16>(P.q, qbase + qoff + (int64_t)row * qs + d) : 0.f;
    }

    float m[4], l[4], acc[4][4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[rr][c] = 0.f;
    }

    for (int r = 0; r < 2; ++r) {
        const int ka = S.k0[r], kb = S.k1[r];
        const int kend = P.causal ? min(kb, qb - S.diag) : kb;  // row qb-1 sees keys <= qb-1-diag
        for (int t0 = ka; t0 < kend; t0 += kSimtKT) {
            __syncthreads();
            for (int idx = tid; idx < kSimtKT * D; idx += blockDim.x) {
                const int j = idx / D, d = idx - (idx / D) * D;
                const int key = t0 + j;
                const bool in = key < kb;
                sK[j][d] = in ? ld_elem<BF16>(P.k, kbase + koff + (int64_t)key * ks_ + d) : 0.f;
                sV[j][d] = in ? ld_elem<BF16>(P.v, vbase + voff + (int64_t)key * vs_ + d) : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int lr = warp * 4 + rr;
                const int row = qa + lr;
                const int key = t0 + lane;
                float s = 0.f;
                for (int d = 0; d < D; ++d) s = fmaf(sQ[lr][d], sK[lane][d], s);
                const bool vis = key < kb && row < qb && (!P.causal || key + S.diag <= row);
                const float x = vis ? s * P.scale_log2 : -INFINITY;
                const float mnew = fmaxf(m[rr], warp_max(x));
                const float muse = (mnew == -INFINITY) ? 0.f : mnew;
                const float p = exp2f(x - muse);
                const float alpha = exp2f(m[rr] - muse);
                l[rr] = l[rr] * alpha + warp_sum(p);
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[rr][c] *= alpha;
                for (int j = 0; j < kSimtKT; ++j) {
                    const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int d = lane + 32 * c;
                        if (d < D) acc[rr][c] = fmaf(pj, sV[j][d], acc[rr][c]);
                    }
                }
                m[rr] = mnew;
            }
        }
    }

    // Epilogue: normalise, then write or merge into the running result.
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int row = qa + warp * 4 + rr;
        if (row >= qb) continue;
        const int pos = row * P.rs + S.q_rank;  // position in the sequence
        const bool have = l[rr] > 0.f;
        const float lse_b = have ? (m[rr] + log2f(l[rr])) * kLn2 : -INFINITY;
        const float inv = have ? 1.f / l[rr] : 0.f;
        const int64_t lrow = ((int64_t)b * P.Hq + h) * P.N + pos;
        const int64_t orow = (int64_t)b * P.so[0] + (int64_t)h * P.so[1] + (int64_t)pos * P.so[2];
        float *accrow = P.oacc ? P.oacc + lrow * D : nullptr;
        if (S.flags & SEG_FIRST) {
            for (int c = 0; c < 4; ++c) {
                const int d = lane + 32 * c;
                if (d >= D) break;
                const float ob = acc[rr][c] * inv;
                if (S.flags & SEG_FINAL) st_elem<BF16>(P.o, orow + d, ob);
                else accrow[d] = ob;
            }
            if (lane == 0) P.lse[lrow] = lse_b;
        } else {
            const float a = P.lse[lrow];
            const MergeW w = merge_weights(a, lse_b);
            for (int c = 0; c < 4; ++c) {
                const int d = lane + 32 * c;
                if (d >= D) break;
                const float ob = acc[rr][c] * inv;
                const float prev = (w.wa != 0.f) ? accrow[d] : 0.f;
                const float on = w.wa * prev + w.wb * ob;
                if (S.flags & SEG_FINAL) st_elem<BF16>(P.o, orow + d, on);
                else accrow[d] = on;
            }
            __syncwarp();
            if (lane == 0) P.lse[lrow] = w.L;
        }
    }
}

cudaError_t launch_attn_simt(const StepParams &P, int blocks_y, cudaStream_t stream) {
    if (blocks_y <= 0 || P.B * P.Hq <= 0) return cudaSuccess;
    dim3 grid(P.B * P.Hq, blocks_y);
    if (P.in_bf16)
        attn_simt_kernel<true><<<grid, 128, 0, stream>>>(P);
    else
        attn_simt_kernel<false><<<grid, 128, 0, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace ra
