// ulysses.cu - the Ulysses all-to-all as a one-GPU layout transform.
//
// "序列并行与 Ring Attention：超长上下文训练技术解析", section "1. Ulysses (All-to-All)":
// before attention every rank holds a sequence shard with all heads; the all-to-all
// scatters the head axis and gathers the sequence axis, so each rank then holds the
// whole sequence for H/sp heads; after attention the inverse exchange restores the
// sequence shards.  With all ranks' buffers in one GPU's memory the exchange is a
// permutation of rows:
//
//   seq -> head:  out[r, s, j, :] = in[s / (S/sp), s % (S/sp), r * (H/sp) + j, :]
//   head -> seq:  the inverse.
//
// HBM-bound: when rows are 16-byte aligned a thread moves four 16-byte pieces (rows of a
// multiple of 64 bytes) or one, so the grid-stride loop keeps every lane busy whatever D
// is; otherwise one warp per row.
#include <algorithm>

#include "ra_internal.cuh"

namespace ra {

__device__ __forceinline__ void ulysses_offsets(const UlyssesParams &P, int64_t r, int64_t &src,
                                                int64_t &dst) {
    // head-sharded row r = (rank, s, j) <-> sequence-sharded row (s / Ss, s % Ss, rank * Hs + j)
    const int Ss = P.S / P.sp, Hs = P.H / P.sp;
    const int j = (int)(r % Hs);
    const int64_t t = r / Hs;
    const int s = (int)(t % P.S);
    const int rank = (int)(t / P.S);
    const int64_t *hs = P.to_heads ? P.so : P.si;
    const int64_t *ss = P.to_heads ? P.si : P.so;
    const int64_t hoff = (int64_t)rank * hs[0] + (int64_t)s * hs[1] + (int64_t)j * hs[2];
    const int64_t soff = (int64_t)(s / Ss) * ss[0] + (int64_t)(s % Ss) * ss[1] + (int64_t)(rank * Hs + j) * ss[2];
    src = P.to_heads ? soff : hoff;
    dst = P.to_heads ? hoff : soff;
}

// One thread per 16-byte piece of a row (aligned rows), else one warp per row.
__global__ void __launch_bounds__(256) ulysses_kernel(const __grid_constant__ UlyssesParams P) {
    const int64_t rows = (int64_t)P.sp * P.S * (P.H / P.sp);
    if (P.vec && (P.D * P.esize) % 64 == 0) {
        // four 16-byte pieces per thread: one offset computation per 64 bytes, four loads
        // in flight before the stores
        const int per4 = P.D * P.esize / 64;
        const int64_t total = rows * per4;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
             i += (int64_t)gridDim.x * blockDim.x) {
            const int64_t r = i / per4;
            const int c = (int)(i - r * per4) * 4;
            int64_t src, dst;
            ulysses_offsets(P, r, src, dst);
            const uint4 *ip = reinterpret_cast<const uint4 *>(static_cast<const char *>(P.in) + src * P.esize) + c;
            uint4 *op = reinterpret_cast<uint4 *>(static_cast<char *>(P.out) + dst * P.esize) + c;
            const uint4 v0 = __ldcs(ip), v1 = __ldcs(ip + 1), v2 = __ldcs(ip + 2), v3 = __ldcs(ip + 3);
            __stcs(op, v0);
            __stcs(op + 1, v1);
            __stcs(op + 2, v2);
            __stcs(op + 3, v3);
        }
        return;
    }
    if (P.vec) {
        const int per = P.D * P.esize / 16;  // pieces per row
        const int64_t total = rows * per;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
             i += (int64_t)gridDim.x * blockDim.x) {
            const int64_t r = i / per;
            const int c = (int)(i - r * per);
            int64_t src, dst;
            ulysses_offsets(P, r, src, dst);
            const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const char *>(P.in) + src * P.esize) + c);
            __stcs(reinterpret_cast<uint4 *>(static_cast<char *>(P.out) + dst * P.esize) + c, v);
        }
        return;
    }
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        int64_t src, dst;
        ulysses_offsets(P, r, src, dst);
        const char *ip = static_cast<const char *>(P.in) + src * P.esize;
        char *op = static_cast<char *>(P.out) + dst * P.esize;
        if (P.esize == 2) {
            for (int d = lane; d < P.D; d += 32)
                reinterpret_cast<uint16_t *>(op)[d] = reinterpret_cast<const uint16_t *>(ip)[d];
        } else {
            for (int d = lane; d < P.D; d += 32)
                reinterpret_cast<uint32_t *>(op)[d] = reinterpret_cast<const uint32_t *>(ip)[d];
        }
    }
}

cudaError_t launch_ulysses(const UlyssesParams &P, int num_sms, cudaStream_t stream) {
    const int64_t rows = (int64_t)P.sp * P.S * (P.H / P.sp);
    if (rows <= 0) return cudaSuccess;
    const int64_t work = P.vec ? rows * (P.D * P.esize / ((P.D * P.esize) % 64 == 0 ? 64 : 16)) / 256 + 1
                               : (rows + 7) / 8;
    const int grid = (int)std::min<int64_t>(work, (int64_t)num_sms * 16);
    ulysses_kernel<<<grid, 256, 0, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace ra
