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
// HBM-bound: one warp moves one D-element row with 16-byte accesses when aligned.
#include <algorithm>

#include "ra_internal.cuh"

namespace ra {

__global__ void __launch_bounds__(256) ulysses_kernel(const __grid_constant__ UlyssesParams P) {
    const int lane = threadIdx.x & 31;
    const int Ss = P.S / P.sp, Hs = P.H / P.sp;
    const int64_t rows = (int64_t)P.sp * P.S * Hs;  // rows of the head-sharded layout
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        // head-sharded coordinates (rank, s, j) <-> sequence-sharded (s / Ss, s % Ss, rank * Hs + j)
        const int j = (int)(r % Hs);
        const int64_t t = r / Hs;
        const int s = (int)(t % P.S);
        const int rank = (int)(t / P.S);
        const int64_t hoff = (int64_t)rank * (P.to_heads ? P.so[0] : P.si[0]) +
                             (int64_t)s * (P.to_heads ? P.so[1] : P.si[1]) +
                             (int64_t)j * (P.to_heads ? P.so[2] : P.si[2]);
        const int64_t* ss = P.to_heads ? P.si : P.so;
        const int64_t soff = (int64_t)(s / Ss) * ss[0] + (int64_t)(s % Ss) * ss[1] +
                             (int64_t)(rank * Hs + j) * ss[2];
        const int64_t src = P.to_heads ? soff : hoff;
        const int64_t dst = P.to_heads ? hoff : soff;
        const char *ip = static_cast<const char *>(P.in) + src * P.esize;
        char *op = static_cast<char *>(P.out) + dst * P.esize;
        const int bytes = P.D * P.esize;
        if (P.vec) {
            for (int o = lane * 16; o < bytes; o += 32 * 16)
                *reinterpret_cast<uint4 *>(op + o) = *reinterpret_cast<const uint4 *>(ip + o);
        } else if (P.esize == 2) {
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
    const int grid = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms * 16);
    ulysses_kernel<<<grid, 256, 0, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace ra
