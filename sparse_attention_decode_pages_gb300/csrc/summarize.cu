// summarize.cu -- per-page key summaries: channel-wise min and max of the valid
// keys of each (sequence, logical page, KV head).  These are the page metadata
// that the Quest-style upper-bound score reads (Sparrow, "Control Study 2": the
// scoring term of the cost model reads one summary per generated page).  They
// are stored sequence-major, [B][H_kv][max_pages][2][D], so that scoring a
// (sequence, KV head) row reads one contiguous stream.
//
// One warp per (page, KV head).  The K tile is ps rows of D bf16 (contiguous);
// lanes read 16-byte chunks so one warp instruction covers 512 contiguous
// bytes, then lanes holding the same channels reduce with shuffles.  bf16
// min/max is exact, so the result is bit-identical to any exact reference.
#include "common.cuh"
#include "kernels.h"

namespace spd {

template <int D>
__global__ void __launch_bounds__(256) summarize_kernel(SummarizeArgs a) {
    constexpr int LPR = D * 2 / 16;  // lanes per row (16-byte chunks per row)
    constexpr int RPI = 32 / LPR;    // rows per warp instruction
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    pdl_wait();
    pdl_trigger();

    int slot;
    if (a.only_pages) {
        slot = a.only_pages[blockIdx.x];
        if (slot < 0 || slot >= a.B * a.max_pages) {
            raise_status(a.status, SPD_DEV_BAD_PAGE);
            return;
        }
    } else {
        slot = blockIdx.x;
    }
    const int b = slot / a.max_pages;
    const int p = slot - b * a.max_pages;
    const int len = a.seq_lens[b];
    if (p * a.ps >= len) return;  // past the sequence's last page
    const int valid = min(a.ps, len - p * a.ps);
    const long long phys = a.page_table[slot];
    if (phys < 0 || phys >= a.num_phys) {
        if (threadIdx.x == 0) raise_status(a.status, SPD_DEV_BAD_PAGE);
        return;
    }

    const int r0 = lane / LPR;
    const int ch = lane % LPR;
    for (int h = warp; h < a.H_kv; h += nwarps) {
        const uint4* tile = reinterpret_cast<const uint4*>(
            a.K + ((phys * a.H_kv + h) * a.ps) * (long long)D);
        __nv_bfloat162 mn[4], mx[4];
        const __nv_bfloat162 pinf = __floats2bfloat162_rn(__int_as_float(0x7f800000), __int_as_float(0x7f800000));
        const __nv_bfloat162 ninf = __floats2bfloat162_rn(__int_as_float(0xff800000), __int_as_float(0xff800000));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            mn[i] = pinf;
            mx[i] = ninf;
        }
#pragma unroll 4
        for (int t = r0; t < valid; t += RPI) {
            uint4 v = __ldg(tile + t * LPR + ch);
            const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mn[i] = __hmin2(mn[i], e[i]);
                mx[i] = __hmax2(mx[i], e[i]);
            }
        }
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t a_ = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<uint32_t*>(&mn[i]), off);
                uint32_t b_ = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<uint32_t*>(&mx[i]), off);
                mn[i] = __hmin2(mn[i], *reinterpret_cast<__nv_bfloat162*>(&a_));
                mx[i] = __hmax2(mx[i], *reinterpret_cast<__nv_bfloat162*>(&b_));
            }
        }
        if (r0 == 0) {
            uint4* out = reinterpret_cast<uint4*>(
                a.summ + (((long long)b * a.H_kv + h) * a.max_pages + p) * 2LL * D);
            out[ch] = *reinterpret_cast<uint4*>(mn);
            out[LPR + ch] = *reinterpret_cast<uint4*>(mx);
        }
    }
}

cudaError_t launch_summarize(const SummarizeArgs& a, cudaStream_t st) {
    const long long nblk = a.only_pages ? (long long)a.n_only : (long long)a.B * a.max_pages;
    if (nblk <= 0) return cudaSuccess;
    const int warps = a.H_kv < 8 ? a.H_kv : 8;
    dim3 grid((unsigned)nblk), block(32 * warps);
    if (a.D == 128)
        return launch_pdl(summarize_kernel<128>, grid, block, 0, st, a);
    return launch_pdl(summarize_kernel<64>, grid, block, 0, st, a);
}

}  // namespace spd
