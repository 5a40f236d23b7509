// score_select.cu -- query-aware page scoring and budgeted top-k selection
// (Sparrow, "Control Study 2": a Top-k over KV pages under a KV budget B and a
// page size; "Control Study 1": a budget that grows with generation length).
//
// Score of page p for KV head h (a Quest-style upper bound of q.k over the
// page, maximised over the G query heads of the group):
//   UB_g(p) = sum_d max(q_gd * kmin_d, q_gd * kmax_d)
//           = sum_d min(q_gd, 0) * kmin_d + max(q_gd, 0) * kmax_d .
// The second form is a dot product of the page's 2D-long summary vector
// [kmin | kmax] with [min(q,0) | max(q,0)], so a tile of 16 pages times the G
// (<= 8) query heads is one m16n8 MMA tile per 16 summary channels.  The bf16
// products are exact in fp32; accumulation is fp32.
//
// Layout of the work: grid (chunks, H_kv, B); a CTA of 4 warps scores one
// chunk of pages of one (sequence, KV head).  Each warp streams 16-page tiles:
// every thread issues 16-byte loads straight from global memory (two pages,
// 2D/16 chunks each), and those registers are the MMA A operand directly --
// the summary channels are assigned to MMA k-slots in the order the loads
// deliver them, and the B operand (the signed query) uses the same order, so
// no shared-memory staging or shuffles are needed.  Scores go to global memory.
// The last CTA to finish a row (an atomic ticket; nobody waits) then selects
// that row's pages: mandatory pages, then a 4-pass radix select on
// order-preserving fp32 keys for the k-th best score, ties to lower page ids,
// and an ascending compaction into sel[].
#include "common.cuh"
#include "kernels.h"

namespace spd {

constexpr int kScoreWarps = 4;
constexpr int kScoreThreads = 32 * kScoreWarps;

// Exclusive prefix sum over the CTA; returns this thread's prefix and the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kScoreWarps; ++w) {
        if (w < warp) base += warp_tot[w];
        tot += warp_tot[w];
    }
    __syncthreads();
    total = tot;
    return base + x - v;
}

__device__ __forceinline__ long long budget_pages(const spd_budget_policy& pol, long long len,
                                                  long long ps) {
    if (pol.mode == SPD_BUDGET_FIXED_PAGES) return pol.fixed_pages;
    if (pol.mode == SPD_BUDGET_LINEAR_TOKENS) {
        long long lin = (len * pol.slope_num + pol.slope_den - 1) / pol.slope_den + pol.intercept;
        long long tok = lin > pol.min_tokens ? lin : pol.min_tokens;
        return (tok + ps - 1) / ps;
    }
    return (len * pol.frac_num + pol.frac_den * ps - 1) / (pol.frac_den * ps);
}

// Selection for one (sequence, KV head) row by the CTA that finished it last.
__device__ void select_row(const ScoreSelectArgs& a, int b, int h, int P, int len,
                           uint32_t* keys /* smem [max_pages] */) {
    __shared__ uint32_t hist[256];
    __shared__ int warp_tot[kScoreWarps];
    __shared__ uint32_t s_digit;
    __shared__ int s_rem;
    const int tid = threadIdx.x;
    const int sink = min(a.pol.sink_pages, P), local = min(a.pol.local_pages, P);
    const int nm = min(P, sink + local);
    long long k = budget_pages(a.pol, len, a.ps);
    if (k > a.k_max) k = a.k_max;
    if (k < nm) k = nm;
    if (k > P) k = P;
    const int kp = (int)k - nm;   // pages to pick among the non-mandatory ones
    const int ncand = P - nm;
    auto mand = [&](int p) { return p < sink || p >= P - local; };

    const float* sc = a.scores + ((long long)b * a.H_kv + h) * a.max_pages;
    for (int p = tid; p < P; p += kScoreThreads) keys[p] = float_key(__ldcg(sc + p));
    __syncthreads();

    uint32_t thr;
    int rem;
    if (kp <= 0) {
        thr = 0xffffffffu;
        rem = 0;
    } else if (kp >= ncand) {
        thr = 0u;
        rem = ncand;
    } else {
        uint32_t prefix = 0, mask = 0;
        rem = kp;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kScoreThreads) hist[i] = 0;
            __syncthreads();
            for (int p = tid; p < P; p += kScoreThreads) {
                if (mand(p)) continue;
                const uint32_t u = keys[p];
                if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (tid < 32) {
                // lane l owns bins 255-8l .. 248-8l, visited from the top.
                int cnt[8], local_sum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    cnt[i] = (int)hist[255 - 8 * tid - i];
                    local_sum += cnt[i];
                }
                int incl = local_sum;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    int y = __shfl_up_sync(0xffffffffu, incl, off);
                    if (tid >= off) incl += y;
                }
                const int excl = incl - local_sum;
                const unsigned hit = __ballot_sync(0xffffffffu, excl < rem && rem <= incl);
                if (tid == __ffs(hit) - 1) {
                    int cum = excl;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (cum + cnt[i] >= rem) {
                            s_digit = (uint32_t)(255 - 8 * tid - i);
                            s_rem = rem - cum;
                            break;
                        }
                        cum += cnt[i];
                    }
                }
            }
            __syncthreads();
            prefix |= s_digit << shift;
            mask |= 255u << shift;
            rem = s_rem;
            __syncthreads();
        }
        thr = prefix;
    }

    // Ascending compaction: mandatory pages, keys above the threshold, and the
    // first `rem` keys equal to it in page order.
    const int seg = (P + kScoreThreads - 1) / kScoreThreads;
    const int lo = min(P, tid * seg), hi = min(P, lo + seg);
    int n_eq = 0;
    for (int p = lo; p < hi; ++p)
        if (!mand(p) && keys[p] == thr) ++n_eq;
    int total;
    const int eq_base = block_exclusive_scan(n_eq, warp_tot, total);
    int n_take = 0;
    {
        int eq = eq_base;
        for (int p = lo; p < hi; ++p) {
            bool take = mand(p);
            if (!take) {
                const uint32_t u = keys[p];
                if (u == thr) take = (eq++ < rem);
                else take = u > thr;
            }
            n_take += take;
        }
    }
    const int out_base = block_exclusive_scan(n_take, warp_tot, total);
    int32_t* out = a.sel + ((long long)b * a.H_kv + h) * a.k_max;
    {
        int eq = eq_base, pos = out_base;
        for (int p = lo; p < hi; ++p) {
            bool take = mand(p);
            if (!take) {
                const uint32_t u = keys[p];
                if (u == thr) take = (eq++ < rem);
                else take = u > thr;
            }
            if (take) {
                if (pos < a.k_max) out[pos] = p;
                ++pos;
            }
        }
    }
    if (tid == 0) {
        if (total > a.k_max) raise_status(a.status, SPD_DEV_BAD_SEL);
        a.nsel[(long long)b * a.H_kv + h] = min(total, a.k_max);
    }
}

template <int D>
__global__ void __launch_bounds__(kScoreThreads) score_select_kernel(ScoreSelectArgs a, int chunk_pages) {
    extern __shared__ uint32_t keys[];
    __shared__ int s_last;
    constexpr int NSS = 2 * D / 32;  // 32-channel super-steps over [kmin | kmax]
    const int b = blockIdx.z, h = blockIdx.y, chunk = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int len = a.seq_lens[b];
    const int P = (len + a.ps - 1) / a.ps;
    const int nch = (P + chunk_pages - 1) / chunk_pages;
    if (chunk >= nch) {
        if (chunk == 0 && threadIdx.x == 0) a.nsel[(long long)b * a.H_kv + h] = 0;
        return;
    }
    const int G = a.H_q / a.H_kv;
    const int n = lane >> 2, c = lane & 3;  // B operand: query head n of the group, k-slot group c

    // B fragments: k-step 2j holds channels 32j+8c+{0,1 | 2,3}, k-step 2j+1 holds +{4,5 | 6,7}.
    uint32_t bq[NSS][4];
    {
        const bf16* qrow = reinterpret_cast<const bf16*>(a.q) + ((long long)b * a.H_q + h * G + n) * D;
#pragma unroll
        for (int j = 0; j < NSS; ++j) {
            float v[8];
            const int e0 = 32 * j + 8 * c;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + i;
                float qv = 0.f;
                if (n < G) qv = __bfloat162float(qrow[e < D ? e : e - D]);
                v[i] = e < D ? fminf(qv, 0.f) : fmaxf(qv, 0.f);
            }
            bq[j][0] = pack_bf16(v[0], v[1]);
            bq[j][1] = pack_bf16(v[2], v[3]);
            bq[j][2] = pack_bf16(v[4], v[5]);
            bq[j][3] = pack_bf16(v[6], v[7]);
        }
    }

    float* sc_row = a.scores + ((long long)b * a.H_kv + h) * a.max_pages;
    const int32_t* pt = a.page_table + (long long)b * a.max_pages;
    const int chunk_lo = chunk * chunk_pages;
    const int chunk_hi = min(P, chunk_lo + chunk_pages);
    const int r = lane >> 2;
    for (int p0 = chunk_lo + warp * 16; p0 < chunk_hi; p0 += kScoreWarps * 16) {
        const int pa = p0 + r, pb = p0 + r + 8;
        long long fa = pa < chunk_hi ? pt[pa] : -1;
        long long fb = pb < chunk_hi ? pt[pb] : -1;
        bool va = pa < chunk_hi, vb = pb < chunk_hi;
        if (va && (fa < 0 || fa >= a.num_phys)) {
            raise_status(a.status, SPD_DEV_BAD_PAGE);
            va = false;
        }
        if (vb && (fb < 0 || fb >= a.num_phys)) {
            raise_status(a.status, SPD_DEV_BAD_PAGE);
            vb = false;
        }
        uint4 ra[NSS], rb[NSS];
        const uint4* sa = reinterpret_cast<const uint4*>(a.summ + (fa * a.H_kv + h) * 2LL * D) + c;
        const uint4* sb = reinterpret_cast<const uint4*>(a.summ + (fb * a.H_kv + h) * 2LL * D) + c;
#pragma unroll
        for (int j = 0; j < NSS; ++j) {
            ra[j] = va ? __ldcs(sa + 4 * j) : make_uint4(0, 0, 0, 0);
            rb[j] = vb ? __ldcs(sb + 4 * j) : make_uint4(0, 0, 0, 0);
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < NSS; ++j) {
            const uint32_t a0[4] = {ra[j].x, rb[j].x, ra[j].y, rb[j].y};
            mma_bf16(acc, a0, bq[j][0], bq[j][1]);
            const uint32_t a1[4] = {ra[j].z, rb[j].z, ra[j].w, rb[j].w};
            mma_bf16(acc, a1, bq[j][2], bq[j][3]);
        }
        // acc: pages r / r+8 x query heads 2c, 2c+1.  Max over the group's heads.
        const float ninf = __int_as_float(0xff800000);
        const bool h0 = 2 * c < G, h1 = 2 * c + 1 < G;
        float s0 = fmaxf(h0 ? acc[0] : ninf, h1 ? acc[1] : ninf);
        float s1 = fmaxf(h0 ? acc[2] : ninf, h1 ? acc[3] : ninf);
        s0 = fmaxf(s0, __shfl_xor_sync(0xffffffffu, s0, 1));
        s1 = fmaxf(s1, __shfl_xor_sync(0xffffffffu, s1, 1));
        s0 = fmaxf(s0, __shfl_xor_sync(0xffffffffu, s0, 2));
        s1 = fmaxf(s1, __shfl_xor_sync(0xffffffffu, s1, 2));
        if (c == 0) {
            if (pa < chunk_hi) sc_row[pa] = va ? s0 : ninf;
            if (pb < chunk_hi) sc_row[pb] = vb ? s1 : ninf;
        }
    }

    // Ticket: the last CTA of this row selects.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int prev = atomicAdd(a.counters + (long long)b * a.H_kv + h, 1);
        s_last = (prev == nch - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    select_row(a, b, h, P, len, keys);
    if (threadIdx.x == 0) a.counters[(long long)b * a.H_kv + h] = 0;
}

int score_chunk_pages(int max_pages, int rows, int num_sms) {
    // Enough CTAs to cover the GPU several times over, 64..512 pages per CTA.
    long long target = 8LL * num_sms;
    long long per_row = (target + rows - 1) / (rows > 0 ? rows : 1);
    int cp = (int)((max_pages + per_row - 1) / (per_row > 0 ? per_row : 1));
    cp = ((cp + 63) / 64) * 64;
    if (cp < 64) cp = 64;
    if (cp > 512) cp = 512;
    return cp;
}

cudaError_t launch_score_select(const ScoreSelectArgs& a, int chunk_pages, cudaStream_t st) {
    if (a.B == 0) return cudaSuccess;
    const int nch = (a.max_pages + chunk_pages - 1) / chunk_pages;
    dim3 grid(nch, a.H_kv, a.B), block(kScoreThreads);
    const size_t smem = (size_t)a.max_pages * sizeof(uint32_t);
    cudaError_t e;
    if (a.D == 128) {
        e = cudaFuncSetAttribute(score_select_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        score_select_kernel<128><<<grid, block, smem, st>>>(a, chunk_pages);
    } else {
        e = cudaFuncSetAttribute(score_select_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        score_select_kernel<64><<<grid, block, smem, st>>>(a, chunk_pages);
    }
    return cudaGetLastError();
}

}  // namespace spd
