// score_select.cu -- query-aware page scoring and budgeted top-k selection
// (Sparrow, "Control Study 2": a Top-k over KV pages under a KV budget B and a
// page size; "Control Study 1": a budget that grows with generation length).
//
// Score of page p for KV head h (a Quest-style upper bound of q.k over the
// page, maximised over the G query heads of the group):
//   UB_g(p) = sum_d max(q_gd * kmin_d, q_gd * kmax_d)
//           = sum_d min(q_gd, 0) * kmin_d + max(q_gd, 0) * kmax_d .
// The second form is a dot product of the page's 2D-long summary vector
// [kmin | kmax] with [min(q,0) | max(q,0)], so 16 pages times the G (<= 8)
// query heads form one m16n8 MMA tile per 16 summary channels.  The bf16
// products are exact in fp32; accumulation is fp32.
//
// Work layout: grid (chunks, H_kv, B); a CTA of 4 warps scores one chunk of
// pages of one (sequence, KV head).  Every warp owns a ring of shared-memory
// slots, one 16-page tile each, filled by 1-D bulk copies (one 512-byte
// summary per lane, completion counted on the slot's mbarrier) several tiles
// ahead of the MMAs.  Pages sit at a padded stride so that the 16-byte
// fragment reads of a quarter-warp hit distinct banks.  The summary channels
// are assigned to MMA k-slots in the order each thread reads them and the
// query operand uses the same order (the contraction is a sum, so any common
// order is exact), so no shuffles or ldmatrix are needed.
//
// Selection: the last CTA to finish a row (an atomic ticket; nothing waits)
// selects that row's pages: the mandatory pages, then the k'-th best score is
// found by bisection over order-preserving uint32 keys (32 counting rounds,
// one barrier each), and pages above it plus the lowest-id pages equal to it
// are compacted in ascending order into sel[].
#include "common.cuh"
#include "kernels.h"

namespace spd {

constexpr int kScoreWarps = 4;
constexpr int kScoreThreads = 32 * kScoreWarps;
constexpr int kScoreStages = 3;

template <int D>
struct ScoreCfg {
    static constexpr int PAGE_BYTES = 2 * D * 2;      // [kmin | kmax] bf16
    static constexpr int STRIDE = PAGE_BYTES + 64;    // consecutive pages 16 banks apart
    static constexpr int TILE = 16 * STRIDE;
    static constexpr int RING = kScoreWarps * kScoreStages * TILE;
    static constexpr int BARS = kScoreWarps * kScoreStages * 8;
};

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

// CTA-wide count of non-mandatory keys satisfying `pred`, one barrier.
template <typename Pred>
__device__ __forceinline__ int count_keys(const uint32_t* keys, int P, int sink, int local, Pred pred,
                                          int (*red)[kScoreWarps], int buf) {
    int cnt = 0;
    for (int p = threadIdx.x; p < P; p += kScoreThreads)
        if (!(p < sink || p >= P - local) && pred(keys[p])) ++cnt;
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if ((threadIdx.x & 31) == 0) red[buf][threadIdx.x >> 5] = cnt;
    __syncthreads();
    int tot = 0;
#pragma unroll
    for (int w = 0; w < kScoreWarps; ++w) tot += red[buf][w];
    return tot;
}

// Selection for one (sequence, KV head) row by the CTA that finished it last.
__device__ void select_row(const ScoreSelectArgs& a, int b, int h, int P, int len, uint32_t* keys) {
    __shared__ int warp_tot[kScoreWarps];
    __shared__ int red[2][kScoreWarps];
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
        // Largest T with #{key >= T} >= kp: the kp-th largest key.
        uint32_t T = 0;
        int buf = 0;
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = T | (1u << bit);
            const int c = count_keys(keys, P, sink, local, [cand](uint32_t u) { return u >= cand; }, red, buf);
            buf ^= 1;
            if (c >= kp) T = cand;
        }
        const int gt = count_keys(keys, P, sink, local, [T](uint32_t u) { return u > T; }, red, buf);
        thr = T;
        rem = kp - gt;
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
    using C = ScoreCfg<D>;
    constexpr int NSS = 2 * D / 32;  // 32-channel super-steps over [kmin | kmax]
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_last;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

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

    const int32_t* pt = a.page_table + (long long)b * a.max_pages;
    const int chunk_lo = chunk * chunk_pages;
    const int chunk_hi = min(P, chunk_lo + chunk_pages);
    // this warp's tiles: p0 = chunk_lo + (warp + 4 t) * 16
    const int span = chunk_hi - chunk_lo;
    const int ntiles_all = (span + 15) / 16;
    const int ntile = ntiles_all > warp ? (ntiles_all - warp + kScoreWarps - 1) / kScoreWarps : 0;

    // [barriers (128 B)][this chunk's page ids][ring: warps x stages x tiles];
    // the selection keys reuse the ring.
    int* s_pt = reinterpret_cast<int*>(smem + 128);
    uint8_t* ring_base = smem + 128 + ((chunk_pages * 4 + 127) & ~127);
    uint8_t* ring = ring_base + warp * kScoreStages * C::TILE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + warp * kScoreStages;
    if (lane == 0) {
        for (int i = 0; i < kScoreStages; ++i) mbar_init(bars + i, 1);
        mbar_fence_init();
    }
    for (int i = threadIdx.x; i < span; i += kScoreThreads) s_pt[i] = pt[chunk_lo + i];
    __syncthreads();

    const uint16_t* summ_h = a.summ + (long long)h * 2 * D;
    // Issue tile t into its slot: lanes 0..15 copy one page each.  Returns the
    // mask of pages with a valid physical id.
    auto issue = [&](int t) -> unsigned {
        const int slot = t % kScoreStages;
        const int p = chunk_lo + (warp + kScoreWarps * t) * 16 + lane;
        bool ok = false;
        long long phys = 0;
        if (lane < 16 && p < chunk_hi) {
            phys = s_pt[p - chunk_lo];
            ok = phys >= 0 && phys < a.num_phys;
            if (!ok) raise_status(a.status, SPD_DEV_BAD_PAGE);
        }
        const unsigned vm = __ballot_sync(0xffffffffu, ok);
        if (lane == 0) mbar_arrive_expect_tx(bars + slot, __popc(vm) * C::PAGE_BYTES);
        if (ok)
            bulk_load(ring + slot * C::TILE + lane * C::STRIDE, summ_h + phys * a.H_kv * 2 * D, C::PAGE_BYTES,
                      bars + slot);
        return vm;
    };
    unsigned vmask[kScoreStages];
#pragma unroll
    for (int i = 0; i < kScoreStages; ++i) vmask[i] = (i < ntile) ? issue(i) : 0u;

    // B fragments: k-step 2j holds channels 32j+8c+{0,1 | 2,3}, k-step 2j+1 holds +{4,5 | 6,7}.
    uint32_t bq[NSS][4];
    {
        const bf16* qrow = reinterpret_cast<const bf16*>(a.q) + ((long long)b * a.H_q + h * G + (n < G ? n : 0)) * D;
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
    const int r = lane >> 2;
    const float ninf = __int_as_float(0xff800000);
    const bool h0 = 2 * c < G, h1 = 2 * c + 1 < G;
    for (int t = 0; t < ntile; ++t) {
        const int slot = t % kScoreStages;
        if (!mbar_wait_bounded(bars + slot, (uint32_t)((t / kScoreStages) & 1), a.status)) {
            // Let the copies still in flight land (bounded) before giving up on this chunk.
            for (int k2 = t + 1; k2 < ntile && k2 < t + kScoreStages; ++k2)
                mbar_wait_bounded(bars + (k2 % kScoreStages), (uint32_t)((k2 / kScoreStages) & 1), a.status);
            break;
        }
        const unsigned vm = vmask[slot];
        const uint8_t* tile = ring + slot * C::TILE;
        const uint8_t* ta = tile + r * C::STRIDE + 16 * c;
        const uint8_t* tb = ta + 8 * C::STRIDE;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < NSS; ++j) {
            const uint4 ra = *reinterpret_cast<const uint4*>(ta + 64 * j);
            const uint4 rb = *reinterpret_cast<const uint4*>(tb + 64 * j);
            const uint32_t a0[4] = {ra.x, rb.x, ra.y, rb.y};
            mma_bf16(acc, a0, bq[j][0], bq[j][1]);
            const uint32_t a1[4] = {ra.z, rb.z, ra.w, rb.w};
            mma_bf16(acc, a1, bq[j][2], bq[j][3]);
        }
        // acc: pages r / r+8 x query heads 2c, 2c+1.  Max over the group's heads.
        float s0 = fmaxf(h0 ? acc[0] : ninf, h1 ? acc[1] : ninf);
        float s1 = fmaxf(h0 ? acc[2] : ninf, h1 ? acc[3] : ninf);
        s0 = fmaxf(s0, __shfl_xor_sync(0xffffffffu, s0, 1));
        s1 = fmaxf(s1, __shfl_xor_sync(0xffffffffu, s1, 1));
        s0 = fmaxf(s0, __shfl_xor_sync(0xffffffffu, s0, 2));
        s1 = fmaxf(s1, __shfl_xor_sync(0xffffffffu, s1, 2));
        const int p0 = chunk_lo + (warp + kScoreWarps * t) * 16;
        if (c == 0) {
            if (p0 + r < chunk_hi) sc_row[p0 + r] = (vm >> r) & 1u ? s0 : ninf;
            if (p0 + r + 8 < chunk_hi) sc_row[p0 + r + 8] = (vm >> (r + 8)) & 1u ? s1 : ninf;
        }
        __syncwarp();  // the slot has been read by every lane
        if (t + kScoreStages < ntile) vmask[slot] = issue(t + kScoreStages);
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
    select_row(a, b, h, P, len, reinterpret_cast<uint32_t*>(ring_base));
    if (threadIdx.x == 0) a.counters[(long long)b * a.H_kv + h] = 0;
}

int score_chunk_pages(int max_pages, int rows, int num_sms) {
    // About two CTAs per SM resident; aim for ~3 waves, 128..1024 pages per CTA.
    long long target = 6LL * num_sms;
    long long per_row = (target + rows - 1) / (rows > 0 ? rows : 1);
    int cp = (int)((max_pages + per_row - 1) / (per_row > 0 ? per_row : 1));
    cp = ((cp + 63) / 64) * 64;
    if (cp < 128) cp = 128;
    if (cp > 1024) cp = 1024;
    return cp;
}

template <int D>
static cudaError_t launch_score_t(const ScoreSelectArgs& a, int chunk_pages, cudaStream_t st) {
    using C = ScoreCfg<D>;
    const int nch = (a.max_pages + chunk_pages - 1) / chunk_pages;
    dim3 grid(nch, a.H_kv, a.B), block(kScoreThreads);
    static_assert(C::BARS <= 128, "barriers must fit in front of the ring");
    const size_t keys = (size_t)a.max_pages * sizeof(uint32_t);
    const size_t smem = 128 /*alignment slack*/ + 128 /*barriers*/ + (((size_t)chunk_pages * 4 + 127) & ~(size_t)127) +
                        (keys > (size_t)C::RING ? keys : (size_t)C::RING);
    cudaError_t e = cudaFuncSetAttribute(score_select_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    score_select_kernel<D><<<grid, block, smem, st>>>(a, chunk_pages);
    return cudaGetLastError();
}

cudaError_t launch_score_select(const ScoreSelectArgs& a, int chunk_pages, cudaStream_t st) {
    if (a.B == 0) return cudaSuccess;
    return a.D == 128 ? launch_score_t<128>(a, chunk_pages, st) : launch_score_t<64>(a, chunk_pages, st);
}

}  // namespace spd
