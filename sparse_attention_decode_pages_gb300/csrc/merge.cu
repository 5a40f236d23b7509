// merge.cu -- log-sum-exp merge of split-K partial attention results
// (FlashDecoding-style split over pages): for each row,
//   lse = log sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) * o_s,
// skipping partials with lse_s = -inf.  One warp per row; lanes stride over D.
#include "common.cuh"
#include "kernels.h"

namespace spd {

__global__ void __launch_bounds__(256) lse_merge_kernel(int S, int rows, int D, const float* __restrict__ part_o,
                                                        const float* __restrict__ part_lse, bf16* __restrict__ o,
                                                        float* __restrict__ lse) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    if (warp >= rows) return;
    const float NEG_INF = __int_as_float(0xff800000);
    float M = NEG_INF;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, part_lse[(long long)s * rows + warp]);
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    if (M != NEG_INF)
        for (int s = lane; s < S; s += 32) L += __expf(part_lse[(long long)s * rows + warp] - M);
#pragma unroll
    for (int off = 16; off; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    const float lse_all = M == NEG_INF ? NEG_INF : M + __logf(L);
    for (int d = lane; d < D; d += 32) {
        float acc = 0.f;
        if (M != NEG_INF)
            for (int s = 0; s < S; ++s) {
                const float ls = part_lse[(long long)s * rows + warp];
                if (ls != NEG_INF) acc += __expf(ls - lse_all) * part_o[((long long)s * rows + warp) * D + d];
            }
        o[(long long)warp * D + d] = __float2bfloat16(acc);
    }
    if (lane == 0 && lse) lse[warp] = lse_all;
}

cudaError_t launch_lse_merge(int S, int rows, int D, const float* part_o, const float* part_lse, uint16_t* o,
                             float* lse, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const int warps_per_block = 8;
    const int blocks = (rows + warps_per_block - 1) / warps_per_block;
    return launch_pdl(lse_merge_kernel, dim3(blocks), dim3(32 * warps_per_block), 0, st, S, rows, D, part_o,
                      part_lse, reinterpret_cast<bf16*>(o), lse);
}

}  // namespace spd
