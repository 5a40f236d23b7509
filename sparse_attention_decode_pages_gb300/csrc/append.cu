// append.cu -- writes the T newest tokens of every sequence into the paged KV
// cache and rewrites the key summaries of the pages they land in, in one
// kernel.  This is the per-step cache update that comes before scoring: a
// decode step appends one token (T = 1); a verification pass rewrites the T
// drafted tokens with the target's keys and values.  (KV pages and the
// per-step scoring read: S3R Figure 1(c); Sparrow, "Control Study 2".)
//
// One CTA per (sequence, touched page), one warp per KV head.  The page's rows
// are visited once: rows at positions >= len - T come from k_new / v_new and
// are stored into the cache, older rows are read from the cache; the warp
// reduces the channel-wise min / max of all valid rows as it goes, so the
// summary is exactly that of the page after the write, whatever the summary
// held before.  Reads and writes touch disjoint rows, so there is no hazard.
#include "common.cuh"
#include "kernels.h"

namespace spd {

template <int D>
__global__ void __launch_bounds__(256) append_refresh_kernel(AppendArgs a) {
    constexpr int LPR = D * 2 / 16;  // lanes per row (16-byte chunks per row)
    constexpr int RPI = 32 / LPR;    // rows per warp instruction
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int b = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    const int len = a.seq_lens[b];
    if (len < a.T || len > a.max_pages * a.ps) {
        if (threadIdx.x == 0 && blockIdx.y == 0) raise_status(a.status, SPD_DEV_BAD_LEN);
        return;
    }
    const int first = len - a.T;  // position of the first new token
    const int p = first / a.ps + (int)blockIdx.y;
    if (p * a.ps >= len) return;  // this sequence touches fewer pages
    const int valid = min(a.ps, len - p * a.ps);
    const long long phys = a.page_table[(long long)b * a.max_pages + p];
    if (phys < 0 || phys >= a.num_phys) {
        if (threadIdx.x == 0) raise_status(a.status, SPD_DEV_BAD_PAGE);
        return;
    }

    const int r0 = lane / LPR;
    const int ch = lane % LPR;
    const __nv_bfloat162 pinf = __floats2bfloat162_rn(__int_as_float(0x7f800000), __int_as_float(0x7f800000));
    const __nv_bfloat162 ninf = __floats2bfloat162_rn(__int_as_float(0xff800000), __int_as_float(0xff800000));
    for (int h = warp; h < a.H_kv; h += nwarps) {
        const long long row0 = (phys * a.H_kv + h) * a.ps;  // cache row of slot 0
        uint4* kt = reinterpret_cast<uint4*>(a.K + row0 * D);
        uint4* vt = reinterpret_cast<uint4*>(a.V + row0 * D);
        __nv_bfloat162 mn[4], mx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            mn[i] = pinf;
            mx[i] = ninf;
        }
        auto fold = [&](const uint4& k) {
            const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&k);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mn[i] = __hmin2(mn[i], e[i]);
                mx[i] = __hmax2(mx[i], e[i]);
            }
        };
        // rows t = r0, r0 + RPI, ... in order: the page's older rows (before the first
        // new token) with kAppendBatch loads in flight, then the new ones, which are
        // read from k_new / v_new and stored into the cache
        const int nold = min(valid, max(0, first - p * a.ps));
        for (int t0 = r0; t0 < nold; t0 += kAppendBatch * RPI) {
            uint4 kk[kAppendBatch];
#pragma unroll
            for (int u = 0; u < kAppendBatch; ++u)
                if (t0 + u * RPI < nold) kk[u] = kt[(t0 + u * RPI) * LPR + ch];
#pragma unroll
            for (int u = 0; u < kAppendBatch; ++u)
                if (t0 + u * RPI < nold) fold(kk[u]);
        }
        for (int t = nold + ((r0 - nold) % RPI + RPI) % RPI; t < valid; t += RPI) {
            const long long src = (((long long)b * a.T + (p * a.ps + t - first)) * a.H_kv + h) * (D / 8);
            const uint4 k = __ldg(reinterpret_cast<const uint4*>(a.k_new) + src + ch);
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.v_new) + src + ch);
            kt[t * LPR + ch] = k;
            vt[t * LPR + ch] = v;
            fold(k);
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

cudaError_t launch_append_refresh(const AppendArgs& a, cudaStream_t st) {
    if (a.B <= 0) return cudaSuccess;
    // pages positions first .. first + T - 1 can span
    const int touched = (a.T - 1 + a.ps - 1) / a.ps + 1;
    const int warps = a.H_kv < 8 ? a.H_kv : 8;
    dim3 grid((unsigned)a.B, (unsigned)touched), block(32 * warps);
    if (a.D == 128)
        return launch_pdl(append_refresh_kernel<128>, grid, block, 0, st, a);
    return launch_pdl(append_refresh_kernel<64>, grid, block, 0, st, a);
}

}  // namespace spd
