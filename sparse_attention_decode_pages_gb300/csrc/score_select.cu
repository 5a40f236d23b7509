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
// Work layout: a persistent grid (three CTAs of 4 warps per SM).  All 16-page
// tiles of all (sequence, KV head) rows are numbered in one sequence (a row's
// from its last page down) and every warp takes an equal contiguous share, so
// the work is balanced to a tile; in the chained step the warps instead take
// 4-tile chunks from a counter in row order (single tiles at the end, so they
// finish within about a tile of each other) and count finished tiles per row.
// The summaries are stored sequence-major, so a tile is one contiguous 8 KB
// run: every warp owns a 2-slot ring of shared-memory slots filled by one 1-D
// bulk copy per tile (completion counted on the slot's mbarrier) ahead of the
// MMAs; many short rings stream better than a few deep ones.  The summary
// channels are assigned to MMA k-slots in the order each thread reads them and
// the query operand uses the same order (the contraction is a sum, so any
// common order is exact), so no shuffles or ldmatrix are needed.
//
// Selection (a second kernel; a 256-thread CTA per (sequence, KV head) row, or
// in the chained step two persistent 128-thread CTAs per SM taking the rows in
// order): the mandatory pages, then the k'-th best score by a radix select over
// order-preserving uint32 keys (shared-memory histogram).  The first digit is
// the 8 bits below those all candidates share (where their minimum and maximum
// agree), so it already spreads them; as soon as the digit being refined holds
// at most as many keys as the CTA has threads (after one pass, typically)
// those keys are ranked pairwise by (key desc, page asc) instead; otherwise the
// passes end on the exact k'-th key.  Pages above the boundary plus the
// boundary pages that rank (or, at an exact key, the lowest-id pages equal to
// it) are compacted in ascending order into sel[] with ballots.
#include "common.cuh"
#include "kernels.h"

namespace spd {

constexpr int kScoreWarps = 4;
constexpr int kScoreThreads = 32 * kScoreWarps;
constexpr int kScoreStages = 2;  // (the slots' tile locations are kept in registers for exactly two)
constexpr int kChunkTiles = 4;  // chained step: consecutive tiles a warp takes at a time
constexpr int kTailTiles = 2;   // chained step: tiles per warp handed out singly at the end

template <int D>
struct ScoreCfg {
    static constexpr int PAGE_BYTES = 2 * D * 2;      // [kmin | kmax] bf16
    static constexpr int TILE = 16 * PAGE_BYTES;
    static constexpr int RING = kScoreWarps * kScoreStages * TILE;
    static constexpr int BARS = kScoreWarps * kScoreStages * 8;
};

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

// Selection CTAs: 256 threads for one row after the scoring grid.  In the
// chained step the width follows the row count: 128 threads, two per SM beside
// the three scoring CTAs, when there are more rows than two per SM (the rows
// become ready over the scoring and their selection overlaps it); 256 threads
// for up to two rows per SM and 512 for up to one (few long rows, all ready at
// about the same time, with nothing else to overlap their selection).  Once the
// radix digit being refined holds at most kRankMax candidates, they are ranked
// directly (pairwise, a thread each) instead of refining further digits.
constexpr int kSelThreads = 256;
constexpr int kRankMax = 128;

__device__ __forceinline__ float key_float(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// Page weight on a 2^-31 grid: exp(score_scale * (score - max)) * 2^31, rounded.
__device__ __forceinline__ uint32_t page_weight(uint32_t key, float smax, float c2) {
    const float w = exp2f((key_float(key) - smax) * c2);
    return __float2uint_rn(w * 2147483648.0f);
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    unsigned long long t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    return t;
}

// Query-dependent budget: the number of non-mandatory pages that, taken in
// score order after the mandatory ones, bring the selected page weight to
// top_p of the total (all of them if none does).  Weights are integers on a
// 2^-31 grid, so every sum is exact; each page's weight is computed once (into
// wts).  The k'-th page is found by a radix descent over the keys in which each
// bin carries its count and its weight, starting below the bits all candidates
// share (kmin / kmax: their smallest and largest key).
template <int NT, class Mand>
__device__ int top_p_pages(const ScoreSelectArgs& a, const uint32_t* keys, int P, Mand mand,
                           uint32_t* hist, int& s_digit, int& s_rem, uint32_t kmin, uint32_t kmax,
                           uint32_t* wts) {
    typedef unsigned long long u64;
    __shared__ u64 mhist[256];
    __shared__ u64 red[NT / 32];
    __shared__ u64 s_mass;
    __shared__ uint32_t s_kmax;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ncand = P - min(P, min(a.pol.sink_pages, P) + min(a.pol.local_pages, P));
    if (tid == 0) s_kmax = 0;
    __syncthreads();
    uint32_t km = 0;
    for (int p = tid; p < P; p += NT) km = max(km, keys[p]);
#pragma unroll
    for (int off = 16; off; off >>= 1) km = max(km, __shfl_xor_sync(0xffffffffu, km, off));
    if (lane == 0) atomicMax(&s_kmax, km);
    __syncthreads();
    const float smax = key_float(s_kmax);
    const float c2 = a.pol.score_scale * 1.4426950408889634f;
    u64 tot = 0, man = 0;
    for (int p = tid; p < P; p += NT) {
        const uint32_t w = page_weight(keys[p], smax, c2);
        wts[p] = w;
        tot += w;
        if (mand(p)) man += w;
    }
    const u64 total = block_sum_u64(tot, red);
    const u64 held = block_sum_u64(man, red);
    // weight still to gather from the candidates: ceil(top_p * total) - held
    const u64 need = (u64)ceil((double)a.pol.top_p * (double)total);
    if (need <= held) return 0;
    u64 R = need - held;

    // bits above h are the same in every candidate
    int h = 31 - __clz((int)(kmin ^ kmax));  // -1 when all candidates are equal
    uint32_t pmask = h < 0 ? 0xffffffffu : (h >= 31 ? 0u : ~((2u << h) - 1u));
    uint32_t prefix = kmin & pmask;
    u64 above = 0;        // weight of the candidates above the current prefix
    int n_above = 0;      // and their count
    int eq_count = ncand; // candidates matching the prefix
    while (h >= 0) {
        const int wd = h + 1 < 8 ? h + 1 : 8;
        const int shift = h + 1 - wd;
        const uint32_t dmask = (1u << wd) - 1u;
        for (int i = tid; i < 256; i += NT) {
            hist[i] = 0;
            mhist[i] = 0;
        }
        __syncthreads();
        for (int p0 = 0; p0 < P; p0 += NT) {
            const int p = p0 + tid;
            bool in = false;
            uint32_t bin = 0, w = 0;
            if (p < P && !mand(p)) {
                const uint32_t u = keys[p];
                if ((u & pmask) == prefix) {
                    in = true;
                    bin = (u >> shift) & dmask;
                    w = wts[p];
                }
            }
            // neighbouring scores share bins: one pair of atomics per distinct bin in the
            // warp (a weight is < 2^32, so its two 16-bit halves sum without overflow)
            const unsigned act = __ballot_sync(0xffffffffu, in);
            if (in) {
                const unsigned same = __match_any_sync(act, bin);
                const unsigned hi = __reduce_add_sync(same, w >> 16);
                const unsigned lo = __reduce_add_sync(same, w & 0xffffu);
                if (lane == __ffs(same) - 1) {
                    atomicAdd(hist + bin, (uint32_t)__popc(same));
                    atomicAdd(mhist + bin, ((u64)hi << 16) + (u64)lo);
                }
            }
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 255-8l .. 248-8l, visited from the top
            u64 m[8], msum = 0;
            int c[8], csum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                m[i] = mhist[255 - 8 * lane - i];
                c[i] = (int)hist[255 - 8 * lane - i];
                msum += m[i];
                csum += c[i];
            }
            u64 mincl = msum;
            int cincl = csum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const u64 y = __shfl_up_sync(0xffffffffu, mincl, off);
                const int z = __shfl_up_sync(0xffffffffu, cincl, off);
                if (lane >= off) {
                    mincl += y;
                    cincl += z;
                }
            }
            const u64 mexcl = mincl - msum;
            const int cexcl = cincl - csum;
            const unsigned hit = __ballot_sync(0xffffffffu, above + mexcl < R && R <= above + mincl);
            if (hit == 0) {
                if (lane == 0) s_digit = -1;  // the candidates cannot reach top_p: take them all
            } else if (lane == __ffs(hit) - 1) {
                u64 cm = mexcl;
                int cc = cexcl;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (above + cm + m[i] >= R) {
                        s_digit = 255 - 8 * lane - i;
                        s_mass = cm;   // weight of the higher bins at this level
                        s_rem = cc;    // and their count
                        break;
                    }
                    cm += m[i];
                    cc += c[i];
                }
            }
        }
        __syncthreads();
        if (s_digit < 0) return ncand;
        above += s_mass;
        n_above += s_rem;
        eq_count = (int)hist[s_digit];
        prefix |= (uint32_t)s_digit << shift;
        pmask |= dmask << shift;
        h = shift - 1;
        __syncthreads();  // hist / s_* are rewritten by the next level
    }
    // every candidate whose key equals prefix has the same weight
    const u64 wt = page_weight(prefix, smax, c2);
    const u64 t = wt ? (R - above + wt - 1) / wt : (u64)eq_count;
    return n_above + (int)min((u64)eq_count, t);
}

// Chained step: copies the row's P keys from global (kg) into shared memory (ks),
// thread `me` of `NT` taking every NT-th key; the loads of a batch are issued
// back to back before any is used, and note(p, key) sees each key that is there.
// True if this thread saw a key still 0 (not yet written by the scoring).
template <int NT, class Note>
__device__ __forceinline__ bool gather_keys(const unsigned* kg, uint32_t* ks, int P, int me, Note note) {
    constexpr int BATCH = 8;
    bool missing = false;
    for (int p0 = 0; p0 < P; p0 += NT * BATCH) {
        unsigned u[BATCH];
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            const int p = p0 + i * NT + me;
            u[i] = p < P ? ld_relaxed(kg + p) : 1u;
        }
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            const int p = p0 + i * NT + me;
            if (p < P) {
                ks[p] = u[i];
                if (u[i] != 0u) note(p, u[i]);
            }
            missing |= (u[i] == 0u);
        }
    }
    return missing;
}

// Reads again the keys still 0 in shared memory (note(p, key) for each that has
// arrived); true if one still is.
template <class Note>
__device__ __forceinline__ bool repoll_keys(const unsigned* kg, uint32_t* ks, int P, int me, int nt, Note note) {
    bool missing = false;
    for (int p = me; p < P; p += nt) {
        if (ks[p] == 0u) {
            const unsigned u = ld_relaxed(kg + p);
            ks[p] = u;
            if (u != 0u) note(p, u);
            missing |= (u == 0u);
        }
    }
    return missing;
}

// Selection of one (sequence, KV head) row by a CTA of NT / 32 warps.  keys: the
// dynamic shared memory (the row's order-preserving score keys, then bit words).
template <int NT>
__device__ __forceinline__ void select_row_block(const ScoreSelectArgs& a, const int row, uint32_t* keys) {
    constexpr int NWARP = NT / 32;
    __shared__ uint32_t hist[256];
    __shared__ int s_digit, s_rem, s_cnt, s_ncol;
    __shared__ uint32_t s_kmin, s_kmax;
    __shared__ int w_eq[NWARP], w_take[NWARP];
    constexpr int RK = NT < kRankMax ? NT : kRankMax;  // candidates ranked directly
    __shared__ uint32_t col_key[RK];
    __shared__ int col_p[RK];
    // after the keys: boundary pages chosen by rank and the final decision (a bit
    // per page each), (top-p) the page weights, (chained step) the row's page table
    const int words = (a.max_pages + 31) / 32;
    uint32_t* s_chosen = keys + a.max_pages;
    uint32_t* s_take = s_chosen + words;
    int32_t* s_pt = reinterpret_cast<int32_t*>(s_take + words + (a.pol.mode == SPD_BUDGET_TOP_P ? a.max_pages : 0));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int b = row / a.H_kv;
    const int len = a.seq_lens[b];
    __shared__ int s_ok;
    // the candidate count, the key range and the first radix level's histogram
    // start clear (ordered before their use by the barriers in between; the
    // previous row's last use ended at the barrier between rows)
    if (tid == 0) {
        s_ncol = 0;
        s_kmin = 0xffffffffu;
        s_kmax = 0u;
    }
    for (int i = tid; i < 256; i += NT) hist[i] = 0;
    for (int w = tid; w < words; w += NT) s_chosen[w] = 0u;
    const int P = max(0, seq_pages(len, a.ps, a.max_pages));  // a bad length: empty (flagged by the scoring)
    const int sink = min(a.pol.sink_pages, P), local = min(a.pol.local_pages, P);
    const int nm = min(P, sink + local);
    const int ncand = P - nm;
    auto mand = [&](int p) { return p < sink || p >= P - local; };
    // the candidates' smallest and largest key (in the chained step taken while the
    // keys are gathered)
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    auto note = [&](int p, uint32_t u) {
        if (!mand(p)) {
            kmin = min(kmin, u);
            kmax = max(kmax, u);
        }
    };
    if (a.keys) {
        // chained step: wait for this row's tiles only, not for the whole scoring grid.
        // The count is a hint (an unordered add); each key is its own ready flag, so
        // the keys are gathered into shared memory and any still 0 is read again.
        const int P0 = P;  // as the scoring kernel counts
        // the row's page-table entries, copied while the keys are awaited (for the
        // physical page of each selected page)
        if (a.sel_phys)
            for (int p = tid; p < P0; p += NT) cp_async4(s_pt + p, a.page_table + (long long)b * a.max_pages + p);
        if (tid == 0) s_ok = count_wait_bounded(a.tiles_done + row, (unsigned)((P0 + 15) / 16), a.status, a.wait_ns);
        __syncthreads();
        if (!s_ok) return;
        unsigned* kg = a.keys + (long long)row * a.max_pages;
        const unsigned long long t0 = globaltimer_ns();
        bool missing = gather_keys<NT>(kg, keys, P0, tid, note);
        while (true) {
            if (!__syncthreads_or(missing)) break;
            if (tid == 0) {
                s_ok = globaltimer_ns() - t0 <= a.wait_ns;
                if (!s_ok) raise_status(a.status, SPD_DEV_TIMEOUT);
            }
            __syncthreads();
            if (!s_ok) return;
            __nanosleep(64);
            missing = repoll_keys(kg, keys, P0, tid, NT, note);
        }
        // acquire: the fused append's writes are released before the keys of its tile
        // (the row's last), so thread 0, which publishes the row below, reads the last
        // key again with acquire semantics before it is zeroed: from then on the
        // append is visible to it and, through its release, to the attention
        if (tid == 0 && P0 > 0) {
            (void)ld_acquire(kg + P0 - 1);
            kg[P0 - 1] = 0u;
        }
        for (int p = tid; p < P0 - 1; p += NT) kg[p] = 0u;  // zero again for the next call
        if (tid == 0) a.tiles_done[row] = 0u;                     // this row's count is consumed
    }
    // chained step: the row's selection is published to the attention kernel
    // (the barrier orders every thread's writes before thread 0's release, which is
    // cumulative over them: one release store publishes the whole row)
    auto publish = [&]() {
        if (!a.sel_done) return;
        __syncthreads();
        if (tid == 0) st_release(a.sel_done + row, 1u);
    };
    int32_t* out = a.sel + (long long)row * a.k_max;
    if (P <= 0) {
        if (tid == 0) {
            a.nsel[row] = 0;
            if (a.K) raise_status(a.status, SPD_DEV_BAD_LEN);  // no position for the fused append
        }
        publish();
        return;
    }

    // keys (chained step: already in shared memory, their range taken): each thread's
    // loads are independent and issued back to back; the range on the way
    if (!a.keys) {
        __syncthreads();  // (chained: the waits above ordered the clearing)
        const float* sc = a.scores + (long long)row * a.max_pages;
        for (int p0 = 0; p0 < P; p0 += NT * 4) {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int p = p0 + i * NT + tid;
                v[i] = p < P ? sc[p] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int p = p0 + i * NT + tid;
                if (p < P) {
                    const uint32_t u = float_key(v[i]);
                    keys[p] = u;
                    if (!mand(p)) {
                        kmin = min(kmin, u);
                        kmax = max(kmax, u);
                    }
                }
            }
        }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) {
        atomicMin(&s_kmin, kmin);
        atomicMax(&s_kmax, kmax);
    }
    __syncthreads();

    long long k;
    if (a.pol.mode == SPD_BUDGET_TOP_P)
        k = nm + top_p_pages<NT>(a, keys, P, mand, hist, s_digit, s_rem, s_kmin, s_kmax, s_take + words);
    else
        k = budget_pages(a.pol, len, a.ps);
    if (k > a.k_max) k = a.k_max;
    if (k < nm) k = nm;
    if (k > P) k = P;
    const int kp = (int)k - nm;  // pages to pick among the non-mandatory ones

    uint32_t thr;
    int rem;
    // ranked: the boundary digit's candidates were ranked; chosen ones are in s_chosen
    bool ranked = false;
    uint32_t prefix = 0, pmask = 0;
    if (kp <= 0) {
        thr = 0xffffffffu;
        rem = 0;
    } else if (kp >= ncand) {
        thr = 0u;
        rem = ncand;
    } else {
        rem = kp;
        // The bits above h are the same in every candidate (their minimum and maximum
        // agree there): the radix starts below them, so the first digit already
        // spreads the keys.  Digits of up to 8 bits until the boundary digit holds at
        // most RK keys (then ranked) or every bit is refined (an exact key).
        int h = 31 - __clz((int)(s_kmin ^ s_kmax));  // -1 when all candidates are equal
        pmask = h < 0 ? 0xffffffffu : (h >= 31 ? 0u : ~((2u << h) - 1u));
        prefix = s_kmin & pmask;
        int ncnt = ncand;
        bool clean = a.pol.mode != SPD_BUDGET_TOP_P;  // the first level's histogram is clear
        while (h >= 0 && ncnt > RK) {
            const int wd = h + 1 < 8 ? h + 1 : 8;
            const int shift = h + 1 - wd;
            const uint32_t dmask = (1u << wd) - 1u;
            if (!clean) {
                for (int i = tid; i < 256; i += NT) hist[i] = 0;
                __syncthreads();
            }
            clean = false;
            for (int p0 = 0; p0 < P; p0 += NT) {
                const int p = p0 + tid;
                bool in = false;
                uint32_t bin = 0;
                if (p < P && !mand(p)) {
                    const uint32_t u = keys[p];
                    in = (u & pmask) == prefix;
                    bin = (u >> shift) & dmask;
                }
                // below the bits every candidate shares the keys spread over the bins,
                // so a plain shared atomic per key rarely conflicts
                if (in) atomicAdd(hist + bin, 1u);
            }
            __syncthreads();
            if (warp == 0) {
                // lane l owns bins 255-8l .. 248-8l, visited from the top (bins past
                // the digit's width stay empty)
                uint32_t cnt[8];
                int sum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    cnt[i] = hist[255 - 8 * lane - i];
                    sum += (int)cnt[i];
                }
                int incl = sum;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += y;
                }
                const int excl = incl - sum;
                const unsigned hit = __ballot_sync(0xffffffffu, excl < rem && rem <= incl);
                if (lane == __ffs(hit) - 1) {
                    int cum = excl;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (cum + (int)cnt[i] >= rem) {
                            s_digit = 255 - 8 * lane - i;
                            s_rem = rem - cum;
                            s_cnt = (int)cnt[i];
                            break;
                        }
                        cum += (int)cnt[i];
                    }
                }
            }
            __syncthreads();
            prefix |= (uint32_t)s_digit << shift;
            pmask |= dmask << shift;
            rem = s_rem;
            ncnt = s_cnt;
            h = shift - 1;
        }
        ranked = ncnt <= RK;  // block-uniform
        thr = prefix;
    }
    if (ranked) {
        // The candidates whose key matches the refined prefix, ranked by (key desc,
        // page asc); the first `rem` of them are chosen.
        // (s_chosen and s_ncol were cleared at the start of the row)
        for (int p0 = 0; p0 < P; p0 += NT) {
            const int p = p0 + tid;
            uint32_t u = 0;
            const bool in = p < P && !mand(p) && ((u = keys[p]) & pmask) == prefix;
            const unsigned bm = __ballot_sync(0xffffffffu, in);
            int base = 0;
            if (bm && lane == 0) base = atomicAdd(&s_ncol, __popc(bm));  // one atomic per warp
            base = __shfl_sync(0xffffffffu, base, 0);
            if (in) {
                const int at = base + __popc(bm & lt_mask);  // < s_cnt <= RK
                col_key[at] = u;
                col_p[at] = p;
            }
        }
        __syncthreads();
        const int m = s_ncol;
        if (tid < m) {
            const uint32_t ki = col_key[tid];
            const int pi = col_p[tid];
            int r = 0;
            for (int j = 0; j < m; ++j) {
                const uint32_t kj = col_key[j];
                r += (kj > ki) || (kj == ki && col_p[j] < pi);
            }
            if (r < rem) atomicOr(&s_chosen[pi >> 5], 1u << (pi & 31));
        }
        __syncthreads();
    }

    // Ascending compaction: mandatory pages, keys above the threshold, and the
    // first `rem` keys equal to it in page order.  Warp w owns a contiguous
    // segment of pages; per-warp counts are scanned through shared memory.
    const int seg = ((P + NT - 1) / NT) * 32;
    const int lo = min(P, warp * seg), hi = min(P, lo + seg);
    auto pick = [&](int p, bool& m, bool& eq) -> bool {  // taken regardless of tie order?
        m = mand(p);
        eq = false;
        if (m) return true;
        const uint32_t u = keys[p];
        if (ranked) return (u & pmask) > prefix || ((s_chosen[p >> 5] >> (p & 31)) & 1u);
        eq = u == thr;
        return u > thr;
    };
    int eq_before = 0;
    if (!ranked) {  // ties at an exact key are taken in page order: count them per warp
        int n_eq = 0;
        for (int p0 = lo; p0 < hi; p0 += 32) {
            const int p = p0 + lane;
            bool m = false, eq = false;
            if (p < hi) pick(p, m, eq);
            n_eq += __popc(__ballot_sync(0xffffffffu, eq));
        }
        if (lane == 0) w_eq[warp] = n_eq;
        __syncthreads();
        for (int w = 0; w < warp; ++w) eq_before += w_eq[w];
    }
    // decide every page once; the decisions (one word per 32 pages) are kept for the write
    int n_take = 0;
    {
        int eqb = eq_before;
        for (int p0 = lo; p0 < hi; p0 += 32) {
            const int p = p0 + lane;
            bool m = false, eq = false, sure = false;
            if (p < hi) sure = pick(p, m, eq);
            const unsigned eb = __ballot_sync(0xffffffffu, eq);
            const bool take = sure || (eq && eqb + __popc(eb & lt_mask) < rem);
            const unsigned tb = __ballot_sync(0xffffffffu, take);
            if (lane == 0) s_take[p0 >> 5] = tb;
            n_take += __popc(tb);
            eqb += __popc(eb);
        }
    }
    if (a.sel_phys) cp_async_wait_all();  // this thread's page-table copies (the barrier: everyone's)
    if (lane == 0) w_take[warp] = n_take;
    __syncthreads();
    int pos = 0, total = 0;
    for (int w = 0; w < NWARP; ++w) {
        if (w < warp) pos += w_take[w];
        total += w_take[w];
    }
    for (int p0 = lo; p0 < hi; p0 += 32) {
        const unsigned tb = s_take[p0 >> 5];
        const int at = pos + __popc(tb & lt_mask);
        if (((tb >> lane) & 1u) && at < a.k_max) {
            out[at] = p0 + lane;
            if (a.sel_phys) a.sel_phys[(long long)row * a.k_max + at] = s_pt[p0 + lane];
        }
        pos += __popc(tb);
    }
    if (tid == 0) {
        if (total > a.k_max) raise_status(a.status, SPD_DEV_BAD_SEL);
        a.nsel[row] = min(total, a.k_max);
    }
    publish();
}

// One CTA per row, or (chained step) two CTAs per SM, each selecting rows
// blockIdx.x, blockIdx.x + gridDim.x, ... in order (used for the top-p budget
// and for rows too long for a warp's shared memory).
template <int NT>
__global__ void __launch_bounds__(NT) select_kernel(ScoreSelectArgs a) {
    extern __shared__ uint32_t keys[];
    __shared__ int s_next;
    if (a.tiles_done) {
        pdl_trigger();  // each row waits for its own tiles instead of the scoring grid
    } else {
        pdl_wait();
        pdl_trigger();
    }
    const int rows = a.B * a.H_kv;
    if (!a.sel_claims || (int)gridDim.x >= rows) {  // (every row its own CTA: nothing to claim)
        for (int row = blockIdx.x; row < rows; row += gridDim.x) {
            select_row_block<NT>(a, row, keys);
            __syncthreads();  // the shared state is reused by the next row
        }
        return;
    }
    // chained step: CTA i selects row i, then claims the next row in order as it
    // finishes one (rows become ready in order; the CTA free first takes the next),
    // until a claim fails.  The grid's claims total exactly `rows`: the one that
    // returns rows - 1 is the last, and resets the counter for the next call.
    for (int row = blockIdx.x; row < rows;) {
        select_row_block<NT>(a, row, keys);
        if (threadIdx.x == 0) {
            const unsigned v = atomicAdd(a.sel_claims, 1u);
            if (v == (unsigned)rows - 1u) *a.sel_claims = 0u;
            s_next = (int)gridDim.x + (int)v;
        }
        __syncthreads();  // s_next, and the shared state reused by the next row
        row = s_next;
        __syncthreads();  // every thread has read s_next
    }
}

// Fused append of the step's token for row (b, h): the token at position
// len - 1 is written into the K / V cache, the summary of its page is rebuilt
// from the page's valid rows (the older ones read from the cache) and stored
// both to global memory and into the shared-memory copy of the tile being
// scored (`entry`, which the bulk copy filled with the stale summary).  Warp-
// wide; the same arithmetic as kv_append_refresh, so the same bits.
template <int D>
__device__ void append_last_page(const ScoreSelectArgs& a, int b, int h, int len, int P, uint8_t* entry) {
    constexpr int LPR = D * 2 / 16;  // lanes per row (16-byte chunks per row)
    constexpr int RPI = 32 / LPR;    // rows per warp instruction
    const int lane = threadIdx.x & 31;
    const int lp = P - 1;
    const int valid = len - lp * a.ps;  // rows of the page, the new token last
    const long long phys = a.page_table[(long long)b * a.max_pages + lp];
    if (phys < 0 || phys >= a.num_phys) {
        if (lane == 0) raise_status(a.status, SPD_DEV_BAD_PAGE);
        return;
    }
    const long long row0 = (phys * a.H_kv + h) * a.ps;
    uint4* kt = reinterpret_cast<uint4*>(a.K + row0 * D);
    uint4* vt = reinterpret_cast<uint4*>(a.V + row0 * D);
    const int r0 = lane / LPR, ch = lane % LPR;
    const __nv_bfloat162 pinf = __floats2bfloat162_rn(__int_as_float(0x7f800000), __int_as_float(0x7f800000));
    const __nv_bfloat162 ninf = __floats2bfloat162_rn(__int_as_float(0xff800000), __int_as_float(0xff800000));
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
    // rows t = r0, r0 + RPI, ... in order: the older ones with kFusedAppendBatch loads
    // in flight, then (in its lanes) the new token's row, the page's last
    const int last = valid - 1;
    for (int t0 = r0; t0 < last; t0 += kFusedAppendBatch * RPI) {
        uint4 kk[kFusedAppendBatch];
#pragma unroll
        for (int u = 0; u < kFusedAppendBatch; ++u)
            if (t0 + u * RPI < last) kk[u] = kt[(t0 + u * RPI) * LPR + ch];
#pragma unroll
        for (int u = 0; u < kFusedAppendBatch; ++u)
            if (t0 + u * RPI < last) fold(kk[u]);
    }
    if (r0 == last % RPI) {
        const long long src = ((long long)b * a.H_kv + h) * (D / 8);
        const uint4 k = __ldg(reinterpret_cast<const uint4*>(a.k_new) + src + ch);
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.v_new) + src + ch);
        kt[last * LPR + ch] = k;
        vt[last * LPR + ch] = v;
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
        uint4* out = reinterpret_cast<uint4*>(a.summ_w + (((long long)b * a.H_kv + h) * a.max_pages + lp) * 2LL * D);
        out[ch] = *reinterpret_cast<uint4*>(mn);
        out[LPR + ch] = *reinterpret_cast<uint4*>(mx);
        reinterpret_cast<uint4*>(entry)[ch] = *reinterpret_cast<uint4*>(mn);
        reinterpret_cast<uint4*>(entry)[LPR + ch] = *reinterpret_cast<uint4*>(mx);
        // these generic writes precede the next bulk copy into the slot
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
}

template <int D>
__global__ void __launch_bounds__(kScoreThreads) score_select_kernel(ScoreSelectArgs a, int unused) {
    using C = ScoreCfg<D>;
    constexpr int NSS = 2 * D / 32;   // 32-channel super-steps over [kmin | kmax]
    constexpr int SLOT = C::TILE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = a.H_q / a.H_kv;
    const int n = lane >> 2, c = lane & 3;  // B operand: query head n of the group, k-slot group c

    // [barriers (128 B)][ring: warps x stages x tiles][tile prefix: B + 1 ints][pages: B ints]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + warp * kScoreStages;
    uint8_t* ring = smem + 128 + warp * kScoreStages * SLOT;
    int* pref = reinterpret_cast<int*>(smem + 128 + kScoreWarps * kScoreStages * SLOT);
    int* pages = pref + a.B + 1;
    if (lane == 0) {
        for (int i = 0; i < kScoreStages; ++i) mbar_init(bars + i, 1);
        mbar_fence_init();
    }
    pdl_wait();
    pdl_trigger();
    // pref[b] = H_kv * (16-page tiles of sequences 0..b-1); a sequence's tiles are
    // ordered (KV head, tile).
    for (int bb = threadIdx.x; bb < a.B; bb += kScoreThreads) {
        const int P = seq_pages(a.seq_lens[bb], a.ps, a.max_pages);
        if (P < 0 && blockIdx.x == 0) raise_status(a.status, SPD_DEV_BAD_LEN);
        pages[bb] = P < 0 ? 0 : P;  // a length the page table cannot hold: nothing to score
    }
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        for (int b0 = 0; b0 < a.B; b0 += 32) {
            const int bb = b0 + lane;
            const int t = bb < a.B ? (pages[bb] + 15) / 16 * a.H_kv : 0;
            int incl = t;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            if (bb < a.B) pref[bb] = run + incl - t;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) pref[a.B] = run;
    }
    __syncthreads();
    const long long total = pref[a.B];
    const long long nwarps = (long long)gridDim.x * kScoreWarps;
    const long long gw = (long long)blockIdx.x * kScoreWarps + warp;
    const long long g0 = total * gw / nwarps, g1 = total * (gw + 1) / nwarps;
    // The warp's t-th tile: its t-th of an equal contiguous share, or (chained step)
    // the next tiles in row order from shared counters, so that rows finish in order
    // and their selection can start while later rows are still scored.  Tiles
    // [0, T1) go out in chunks of kChunkTiles (the query is reused within a chunk;
    // warp gw's first chunk is chunk gw, with no round trip before its first copy),
    // the last kTailTiles per warp [T1, total) one at a time from a second counter,
    // so the warps finish within about a tile of each other.
    const long long T1 = max(0LL, (total - nwarps * kTailTiles) / kChunkTiles * kChunkTiles);
    int phase = 0;  // 0: first chunk, 1: chunks, 2: single tiles, 3: drained
    long long ch_cur = 0, ch_end = 0;
    auto grab = [&](int t) -> long long {
        if (!a.tiles_done) return g0 + t < g1 ? g0 + t : -1;
        if (ch_cur < ch_end) return ch_cur++;
        if (phase == 0) {
            phase = 1;
            const long long v0 = gw * kChunkTiles;
            if (v0 < T1) {
                ch_cur = v0 + 1;
                ch_end = min(v0 + kChunkTiles, T1);
                return v0;
            }
        }
        if (phase == 1) {
            unsigned long long v = 0;
            if (lane == 0)
                v = atomicAdd(a.tile_ctr, (unsigned long long)kChunkTiles) + (unsigned long long)(nwarps * kChunkTiles);
            v = __shfl_sync(0xffffffffu, v, 0);
            if ((long long)v < T1) {
                ch_cur = (long long)v + 1;
                ch_end = min((long long)v + kChunkTiles, T1);
                return (long long)v;
            }
            phase = 2;
        }
        if (phase == 2) {
            unsigned long long v = 0;
            if (lane == 0) {
                v = T1 + atomicAdd(a.tile_ctr + 1, 1ull);
                if ((long long)v >= total) {  // each warp runs out exactly once; the last one resets
                    if (atomicAdd(a.warps_done, 1u) == (unsigned)nwarps - 1) {
                        a.tile_ctr[0] = 0ull;
                        a.tile_ctr[1] = 0ull;
                        *a.warps_done = 0u;
                    }
                }
            }
            v = __shfl_sync(0xffffffffu, v, 0);
            if ((long long)v < total) return (long long)v;
            phase = 3;
        }
        return -1;
    };
    int pend_row = -1, pend_cnt = 0;  // tiles finished but not yet reported
    // The count only tells the selection when to start reading the row's keys (each
    // key is its own ready flag), so it is an unordered add: no fence per chunk.
    auto report = [&]() {
        if (pend_cnt == 0) return;
        if (lane == 0) red_relaxed_add(a.tiles_done + pend_row, (unsigned)pend_cnt);
        pend_cnt = 0;
    };

    // tile index -> (sequence, KV head, first page); shared-memory lookups only.  A
    // row's tiles are numbered from its last page down, so the tile with the step's
    // appended token comes first and its extra work does not delay the row's end.
    auto locate = [&](long long g, int& b, int& h, int& p0, int& P) {
        int lo = 0, hi = a.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pref[mid] <= g) lo = mid;
            else hi = mid - 1;
        }
        b = lo;
        P = pages[b];
        const int tb = (P + 15) / 16;
        const int local = (int)(g - pref[b]);
        h = local / tb;
        p0 = (tb - 1 - (local - h * tb)) * 16;
    };
    int issued_row = -1;
    // Each slot's tile as located at issue (read back when it is scored); a tile
    // that continues the previously issued one's row is its 16 pages further down.
    static_assert(kScoreStages == 2, "one register set per slot");
    int4 loc_s0 = make_int4(0, 0, 0, 0), loc_s1 = make_int4(0, 0, 0, 0);
    long long last_g = -2;
    int4 last_loc = make_int4(0, 0, 0, 0);  // {b, h, p0, P}
    auto issue = [&](int t, long long g) {
        if (g == last_g + 1 && last_loc.z >= 16) {
            last_loc.z -= 16;
        } else {
            int b_, h_, p0_, P_;
            locate(g, b_, h_, p0_, P_);
            last_loc = make_int4(b_, h_, p0_, P_);
        }
        last_g = g;
        const int b = last_loc.x, h = last_loc.y, p0 = last_loc.z, P = last_loc.w;
        if (t % kScoreStages == 0) loc_s0 = last_loc;
        else loc_s1 = last_loc;
        const int row = b * a.H_kv + h;
        const bool newq = row != issued_row;
        issued_row = row;
        if (lane == 0) {
            const int slot = t % kScoreStages;
            const uint32_t bytes = (uint32_t)(min(16, P - p0) * C::PAGE_BYTES);
            mbar_arrive_expect_tx(bars + slot, bytes);
            bulk_load(ring + slot * SLOT, a.summ + ((((long long)b * a.H_kv + h) * a.max_pages) + p0) * 2LL * D,
                      bytes, bars + slot);
        }
        // a new row's query heads are pulled into L2 now, read when the tile is consumed
        if (newq && lane * 128 < G * D * 2)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(a.q) +
                                                          ((long long)b * a.H_q + h * G) * D * 2 + lane * 128));
    };
    __syncwarp();
    long long gq[kScoreStages];
#pragma unroll
    for (int i = 0; i < kScoreStages; ++i) {
        gq[i] = grab(i);
        if (gq[i] >= 0) issue(i, gq[i]);
    }

    uint32_t bq[NSS][4];
    int cur_row = -1;
    const int r = lane >> 2;
    const float ninf = __int_as_float(0xff800000);
    const bool h0 = 2 * c < G, h1 = 2 * c + 1 < G;
    for (int t = 0;; ++t) {
        const int slot = t % kScoreStages;
        const long long g = gq[slot];
        if (g < 0) break;  // tiles are grabbed in order: every earlier one is done
        const int4 loc = slot == 0 ? loc_s0 : loc_s1;
        const int b = loc.x, h = loc.y, p0 = loc.z, P = loc.w;
        const int row = b * a.H_kv + h;
        if (!mbar_wait_bounded(bars + slot, (uint32_t)((t / kScoreStages) & 1), a.status, a.wait_ns)) {
            // Let the copies still in flight land (bounded) before giving up.
            for (int k2 = t + 1; k2 < t + kScoreStages; ++k2)
                if (gq[k2 % kScoreStages] >= 0)
                    mbar_wait_bounded(bars + (k2 % kScoreStages), (uint32_t)((k2 / kScoreStages) & 1), a.status, a.wait_ns);
            break;
        }
        const uint8_t* sl = ring + slot * SLOT;
        if (a.K && p0 <= P - 1 && P - 1 < p0 + 16) {  // this tile holds the row's last page
            append_last_page<D>(a, b, h, a.seq_lens[b], P, ring + slot * SLOT + (P - 1 - p0) * C::PAGE_BYTES);
            // chained step: the append's K / V / summary writes are released before
            // this tile's keys, which the selection acquires (and the attention after it)
            if (a.keys) fence_acq_rel_gpu();
            __syncwarp();
        }
        if (row != cur_row) {
            // B fragments of this row's query heads: k-step 2j holds channels
            // 32j+8c+{0,1 | 2,3}, k-step 2j+1 holds +{4,5 | 6,7}
            cur_row = row;
            const bf16* qrow = reinterpret_cast<const bf16*>(a.q) + ((long long)b * a.H_q + h * G + (n < G ? n : 0)) * D;
#pragma unroll
            for (int jj = 0; jj < NSS; ++jj) {
                float v[8];
                const int e0 = 32 * jj + 8 * c;
                const uint4 raw = *reinterpret_cast<const uint4*>(qrow + (e0 < D ? e0 : e0 - D));
                const bf16* rv = reinterpret_cast<const bf16*>(&raw);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float qv = n < G ? __bfloat162float(rv[i]) : 0.f;
                    v[i] = e0 < D ? fminf(qv, 0.f) : fmaxf(qv, 0.f);
                }
                bq[jj][0] = pack_bf16(v[0], v[1]);
                bq[jj][1] = pack_bf16(v[2], v[3]);
                bq[jj][2] = pack_bf16(v[4], v[5]);
                bq[jj][3] = pack_bf16(v[6], v[7]);
            }
        }
        const uint8_t* ta = sl + r * C::PAGE_BYTES + 16 * c;
        const uint8_t* tb = ta + 8 * C::PAGE_BYTES;
        // four independent accumulator chains over the super-steps
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
        for (int jj = 0; jj < NSS; ++jj) {
            const uint4 ra = *reinterpret_cast<const uint4*>(ta + 64 * jj);
            const uint4 rb = *reinterpret_cast<const uint4*>(tb + 64 * jj);
            const uint32_t a0[4] = {ra.x, rb.x, ra.y, rb.y};
            mma_bf16(acc[(2 * jj) & 3], a0, bq[jj][0], bq[jj][1]);
            const uint32_t a1[4] = {ra.z, rb.z, ra.w, rb.w};
            mma_bf16(acc[(2 * jj + 1) & 3], a1, bq[jj][2], bq[jj][3]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[0][e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
        // acc: pages r / r+8 x query heads 2c, 2c+1.  Max over the group's heads.
        float s0 = fmaxf(h0 ? acc[0][0] : ninf, h1 ? acc[0][1] : ninf);
        float s1 = fmaxf(h0 ? acc[0][2] : ninf, h1 ? acc[0][3] : ninf);
        s0 = fmaxf(s0, __shfl_xor_sync(0xffffffffu, s0, 1));
        s1 = fmaxf(s1, __shfl_xor_sync(0xffffffffu, s1, 1));
        s0 = fmaxf(s0, __shfl_xor_sync(0xffffffffu, s0, 2));
        s1 = fmaxf(s1, __shfl_xor_sync(0xffffffffu, s1, 2));
        if (c == 0) {
            if (a.keys) {  // chained step: order-preserving keys, 0 reserved for "not yet"
                unsigned* kr = a.keys + (long long)row * a.max_pages;
                if (p0 + r < P) st_relaxed(kr + p0 + r, max(float_key(s0), 1u));
                if (p0 + r + 8 < P) st_relaxed(kr + p0 + r + 8, max(float_key(s1), 1u));
            } else {
                float* sc_row = a.scores + (long long)row * a.max_pages;
                if (p0 + r < P) sc_row[p0 + r] = s0;
                if (p0 + r + 8 < P) sc_row[p0 + r + 8] = s1;
            }
        }
        __syncwarp();  // the slot has been read by every lane
        if (a.tiles_done) {
            if (row != pend_row) {
                report();
                pend_row = row;
            }
            ++pend_cnt;
            // end of a run of consecutive tiles (a chunk): the next tile in flight is not g + 1
            if (gq[(slot + 1) % kScoreStages] != g + 1) report();
        }
        gq[slot] = grab(t + kScoreStages);
        if (gq[slot] >= 0) issue(t + kScoreStages, gq[slot]);
    }
    if (a.tiles_done) report();
}

template <int D>
static cudaError_t launch_score_t(const ScoreSelectArgs& a, int grid, cudaStream_t st) {
    using C = ScoreCfg<D>;
    static_assert(C::BARS <= 128, "barriers must fit in front of the ring");
    const size_t ring = (size_t)kScoreWarps * kScoreStages * C::TILE;
    const size_t smem = 128 /*alignment slack*/ + 128 /*barriers*/ + ring + (2 * (size_t)a.B + 1) * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(score_select_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(score_select_kernel<D>, dim3(grid), dim3(kScoreThreads), smem, st, a, 0);
}

cudaError_t launch_score_select(const ScoreSelectArgs& a, int num_sms, cudaStream_t st) {
    if (a.B == 0) return cudaSuccess;
    // persistent: three CTAs per SM, each warp streams an equal share of all tiles
    const int grid = 3 * num_sms;
    cudaError_t e = a.D == 128 ? launch_score_t<128>(a, grid, st) : launch_score_t<64>(a, grid, st);
    if (e != cudaSuccess) return e;
    // selection: one CTA per row, the row's keys in shared memory
    // keys, chosen and decision bit words, (top-p) the page weights, (chained) the
    // page-table row
    const size_t smem = ((size_t)a.max_pages + 2 * (((size_t)a.max_pages + 31) / 32) +
                         (a.pol.mode == SPD_BUDGET_TOP_P ? (size_t)a.max_pages : 0) +
                         (a.sel_phys ? (size_t)a.max_pages : 0)) * sizeof(uint32_t);
    long long sgrid = (long long)a.B * a.H_kv;
    if (a.tiles_done) {
        // chained step: persistent CTAs taking the rows in order, launched right
        // behind the scoring grid (so the attention grid is launched early); the
        // width by row count (above)
        auto chained = [&](auto kern, int nt, long long per_sm) -> cudaError_t {
            cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e2 != cudaSuccess) return e2;
            if (sgrid > per_sm * num_sms) sgrid = per_sm * num_sms;
            return launch_pdl(kern, dim3((unsigned)sgrid), dim3(nt), smem, st, a);
        };
        if (sgrid <= num_sms) return chained(select_kernel<512>, 512, 1);
        if (sgrid <= 2LL * num_sms) return chained(select_kernel<256>, 256, 2);
        return chained(select_kernel<128>, 128, 2);
    }
    auto kern = select_kernel<kSelThreads>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((unsigned)sgrid), dim3(kSelThreads), smem, st, a);
}

}  // namespace spd
