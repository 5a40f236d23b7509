// spec.cu -- exact speculative sampling after dense verification: the
// accept / reject decisions over k drafted tokens and the draw of the token
// that follows them (S3R abstract: responses come from full-attention
// verification followed by exact speculative sampling).
//
// One cluster of kSpecCluster CTAs per sequence.  Each CTA's first warp
// decides the k drafts at once, a lane each (cheap; every CTA needs the
// outcome): draft x at position i is accepted iff u_acc * p_i(x) < q_i(x),
// the product of the two fp32 values formed exactly in fp64; the first
// rejection ends the run.
//
// The token that follows is drawn from integer weights on a 2^-40 grid:
// W(x) = max(0, F(q_j(x)) - F(p_j(x))) at the first rejection j (F(q_j(x))
// when that is zero everywhere), or F(q_k(x)) after k acceptances, with
// F(v) = floor(2^40 v).  The draw is the smallest x whose running sum exceeds
// floor(u_res * sum W).  Every sum is an exact 64-bit integer, so the order in
// which the GPU adds them does not matter (fp64 would be both order-dependent
// and slow: this part runs fp64 at a small fraction of its fp32 rate).
//
// The draw streams the row once.  Each CTA sums the 128-element tiles of its
// share of the row into its shared memory: rows whose length is a multiple of
// 4 arrive through a 3-deep ring of 16-tile chunks filled by bulk copies (each
// warp reads two tiles of each chunk into registers, frees the slot, then sums
// them); other rows through plain loads, a warp per tile.  Six 8-warp CTAs per
// sequence: at B = 64 the 384 CTAs spread over every SM, two or three each (with
// eight per sequence, four deep, they filled only ~128 SMs and took 8 % longer).
// After a cluster barrier every CTA reads the six shares' sums through distributed
// shared memory; the one CTA whose share holds the target block-scans its own
// tile sums, the one thread whose run of tiles holds it finds the crossing
// tile, and a warp scans that tile's 128 weights to find the element and
// writes the token (CTA 0 has written the other outputs at the start).  The
// barrier after the shares are read is split: each CTA arrives once it has read
// them and waits only before its own shared memory is rewritten or released, so
// the search holds no other CTA back.
//
// Most tiles hold only probabilities below 2^-10, whose grid values fit 30 bits:
// their weights are formed and summed in 32-bit arithmetic (a float-to-uint32
// conversion of v * 2^40), the rest in the exact 64-bit form below.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace spd {

constexpr int kSpecThreads = 256;
constexpr int kSpecTile = 128;
constexpr int kSpecCluster = 6;
constexpr int kSpecUnroll = 2;
// n % 4 == 0 rows stream through shared memory: chunks of 16 tiles (q and p),
// kSpecStages in flight per CTA, copied by the bulk-copy engine.
constexpr int kSpecChunk = 16 * kSpecTile;  // elements (a whole number of tiles per warp)
constexpr int kSpecStages = 3;
constexpr size_t kSpecRingBytes = (size_t)kSpecStages * 2 * kSpecChunk * sizeof(float);
static_assert(kSpecChunk / kSpecTile % (kSpecThreads / 32) == 0, "every warp sums the same number of tiles of a chunk");
typedef unsigned long long u64;

// floor(2^40 v) from the float's bits, in integer operations only (a 64-bit
// float-to-integer conversion is a slow instruction): for a normal v < 1,
// v = mant * 2^(E - 150), so 2^40 v = (mant << 40) >> (150 - E), a shift the
// PTX shr clamps to 0 past 64.  v >= 1 (and +inf) counts as 1; v <= 0, NaN and
// subnormals (far below the grid) give 0.
__device__ __forceinline__ u64 fixed40(float v) {
    const unsigned bits = __float_as_uint(v);
    const unsigned E = bits >> 23;  // with the sign bit: negative values give E >= 256
    const u64 x = (u64)((bits & 0x7fffffu) | 0x800000u) << 40;
    u64 w;
    asm("shr.b64 %0, %1, %2;" : "=l"(w) : "l"(x), "r"(150u - E));
    if (E - 1u >= 126u) {  // not a normal value in (0, 1)
        const bool one = E >= 127u && E <= 255u && !(E == 255u && (bits & 0x7fffffu));
        w = one ? (1ull << 40) : 0ull;
    }
    return w;
}

// floor(2^40 v) when it lies below 2^32: v * 2^40 is exact in fp32 (a power-of-two
// scaling that neither overflows nor leaves the normal range for a normal v below 2^-8),
// and the float-to-uint32 conversion truncates it, i.e. floors it.  The conversion
// saturates: 0 for a negative v or a NaN (as fixed40), 2^32 - 1 for a v of 2^-8 or more
// or +inf, so a result below 2^30 is always the exact floor(2^40 v).
__device__ __forceinline__ unsigned fixed40_u32(float v) { return __float2uint_rz(v * 1099511627776.0f); }

// The four weights of a lane's float4 pair in 32-bit arithmetic, and whether they are
// exact and their sum fits 32 bits (every converted value below 2^30).
__device__ __forceinline__ bool spec_w4_small(const float4& q4, const float4& p4, bool residual, unsigned& sum) {
    unsigned w[4] = {fixed40_u32(q4.x), fixed40_u32(q4.y), fixed40_u32(q4.z), fixed40_u32(q4.w)};
    unsigned any = w[0] | w[1] | w[2] | w[3];
    if (residual) {
        const unsigned v[4] = {fixed40_u32(p4.x), fixed40_u32(p4.y), fixed40_u32(p4.z), fixed40_u32(p4.w)};
        any |= v[0] | v[1] | v[2] | v[3];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = max(w[i], v[i]) - v[i];
    }
    sum = w[0] + w[1] + w[2] + w[3];
    return any < (1u << 30);
}

__device__ __forceinline__ u64 spec_w(float qv, float pv, bool residual) {
    const u64 a = fixed40(qv);
    if (!residual) return a;
    const u64 b = fixed40(pv);
    return a > b ? a - b : 0ull;
}

// floor(u * total) for a float u in [0, 1), exactly: u = m * 2^-shift
__device__ __forceinline__ u64 scaled_floor(float u, u64 total) {
    const unsigned bits = __float_as_uint(u);
    const unsigned E = (bits >> 23) & 0xffu;
    u64 m;
    int shift;
    if (E == 0) {
        m = bits & 0x7fffffu;
        shift = 149;
    } else {
        m = (bits & 0x7fffffu) | 0x800000u;
        shift = 150 - (int)E;
    }
    if (shift <= 0) return ~0ull;  // u >= 2^23: past any total
    const u64 lo = m * total, hi = __umul64hi(m, total);
    if (shift >= 128) return 0ull;
    if (shift >= 64) return hi >> (shift - 64);
    return (lo >> shift) | (hi << (64 - shift));
}

__device__ __forceinline__ u64 shfl_xor_u64(u64 v, int off) {
    return __shfl_xor_sync(0xffffffffu, v, off);
}

// Warp sum of one tile's lane sums (each < 4 * 2^40 = 2^42): the low and the high 21
// bits are summed separately, each by one warp-reduce instruction (32 lanes x 2^21 <
// 2^26 fits 32 bits), so the 64-bit total is exact.
__device__ __forceinline__ u64 tile_sum(u64 v) {
    const unsigned lo = __reduce_add_sync(0xffffffffu, (unsigned)(v & 0x1fffffull));
    const unsigned hi = __reduce_add_sync(0xffffffffu, (unsigned)(v >> 21));
    return ((u64)hi << 21) + lo;
}

template <bool VEC>
__global__ void __cluster_dims__(kSpecCluster, 1, 1) __launch_bounds__(kSpecThreads, 3)
    spec_accept_kernel(SpecArgs a) {
    // [VEC: ring of kSpecStages x {q, p} chunks][tpc own tile sums][VEC: bars]
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ int s_acc, s_bad, s_cross_tile;
    __shared__ u64 s_cross_run;
    __shared__ u64 s_warp[kSpecThreads / 32];
    __shared__ u64 s_chunk;  // this CTA's share of the total
    constexpr int NW = kSpecThreads / 32;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / kSpecCluster;
    const int k = a.k;
    const long long n = a.n;
    const int ntiles = (int)((n + kSpecTile - 1) / kSpecTile);
    const int tpc = (ntiles + kSpecCluster - 1) / kSpecCluster;  // tiles per CTA
    float* ring = reinterpret_cast<float*>(smem_raw);
    u64* tsum = reinterpret_cast<u64*>(smem_raw + (VEC ? kSpecRingBytes : 0));
    uint64_t* bars = reinterpret_cast<uint64_t*>(tsum + tpc);
    if (VEC && tid == 0) {
        for (int i = 0; i < kSpecStages; ++i) mbar_init(bars + i, 1);
        mbar_fence_init();
    }
    __syncthreads();
    unsigned chunks_done = 0;  // ring phases used so far (VEC)
    bool dead = false;         // a bounded wait ran out: skip the data, keep the protocol
    pdl_wait();
    pdl_trigger();

    // the k <= 32 decisions in parallel, one lane each; the first rejection ends the run
    if (warp == 0) {
        bool ok = false, bad = false;
        if (lane < k) {
            const int x = a.draft[(long long)b * k + lane];
            if (x < 0 || x >= n) {
                bad = true;
            } else {
                const double px = (double)a.p[((long long)b * k + lane) * n + x];
                const double qx = (double)a.q[((long long)b * (k + 1) + lane) * n + x];
                ok = (double)a.u_acc[(long long)b * k + lane] * px < qx;
            }
        }
        const unsigned fail = __ballot_sync(0xffffffffu, lane < k && !ok);
        const unsigned badm = __ballot_sync(0xffffffffu, bad);
        if (lane == 0) {
            const int j = fail ? __ffs((int)fail) - 1 : k;
            // a bad token at the first failing position invalidates the sequence
            s_acc = j;
            s_bad = (j < k && ((badm >> j) & 1u)) ? 1 : 0;
            if (s_bad && rank == 0) raise_status(a.status, SPD_DEV_BAD_TOKEN);
        }
    }
    __syncthreads();
    const int acc = s_acc;
    int32_t* out = a.tokens + (long long)b * (k + 1);
    if (s_bad) {  // the same on every CTA of the cluster: all leave before any barrier
        if (rank == 0) {
            for (int i = tid; i <= k; i += kSpecThreads) out[i] = -1;
            if (tid == 0) a.n_accepted[b] = 0;
        }
        return;
    }
    // CTA 0 writes the outputs now, the drawn token's slot as "none"; the CTA that finds
    // the token overwrites that slot (ordered after this write by the cluster barrier)
    if (rank == 0) {
        for (int i = tid; i <= k; i += kSpecThreads) out[i] = i < acc ? a.draft[(long long)b * k + i] : -1;
        if (tid == 0) a.n_accepted[b] = acc;
    }
    const float* qr = a.q + ((long long)b * (k + 1) + acc) * n;
    const float* pr = acc < k ? a.p + ((long long)b * k + acc) * n : qr;
    const int my0 = rank * tpc;
    const int my1 = min(ntiles, my0 + tpc);

    for (int attempt = 0; attempt < 2; ++attempt) {
        // attempt 0: the residual at a rejection, or the target row after k acceptances;
        // attempt 1 (after a rejection whose residual is zero everywhere): the target row
        const bool residual = (attempt == 0) && (acc < k);
        if (VEC) {
            const long long e0 = (long long)my0 * kSpecTile;
            const long long e1 = min((long long)my1 * kSpecTile, n);
            const int nchunks = e1 > e0 ? (int)((e1 - e0 + kSpecChunk - 1) / kSpecChunk) : 0;
            auto issue = [&](int c) {  // thread 0
                const int slot = (int)((chunks_done + c) % kSpecStages);
                const long long s0 = e0 + (long long)c * kSpecChunk;
                const uint32_t nb = (uint32_t)(min((long long)kSpecChunk, e1 - s0) * sizeof(float));
                float* dst = ring + (size_t)slot * 2 * kSpecChunk;
                mbar_arrive_expect_tx(bars + slot, residual ? 2 * nb : nb);
                bulk_load(dst, qr + s0, nb, bars + slot);
                if (residual) bulk_load(dst + kSpecChunk, pr + s0, nb, bars + slot);
            };
            if (tid == 0)
                for (int c = 0; c < kSpecStages && c < nchunks; ++c) issue(c);
            for (int c = 0; c < nchunks; ++c) {
                const int slot = (int)((chunks_done + c) % kSpecStages);
                if (!dead && !mbar_wait_bounded(bars + slot, ((chunks_done + c) / kSpecStages) & 1u, a.status, a.wait_ns))
                    dead = true;
                // warp w sums tiles w, w + NW, ... of the chunk: their values are read
                // into registers first, so the slot is refilled while they are summed
                constexpr int TPW = kSpecChunk / kSpecTile / NW;  // tiles per warp
                const long long s0 = e0 + (long long)c * kSpecChunk;
                float4 q4[TPW], p4[TPW];
#pragma unroll
                for (int u = 0; u < TPW; ++u) {
                    const int tw = warp + u * NW;
                    const long long x0 = s0 + (long long)tw * kSpecTile + lane * 4;
                    q4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    p4[u] = q4[u];
                    if (!dead && x0 < e1) {
                        const float* src = ring + (size_t)slot * 2 * kSpecChunk + tw * kSpecTile + lane * 4;
                        q4[u] = *reinterpret_cast<const float4*>(src);
                        if (residual) p4[u] = *reinterpret_cast<const float4*>(src + kSpecChunk);
                    }
                }
                __syncthreads();  // the slot has been read
                if (tid == 0 && c + kSpecStages < nchunks) issue(c + kSpecStages);
#pragma unroll
                for (int u = 0; u < TPW; ++u) {
                    // a tile of small values (the usual case) in 32-bit operations, others in 64
                    u64 sum;
                    unsigned s32;
                    if (__all_sync(0xffffffffu, spec_w4_small(q4[u], p4[u], residual, s32))) {
                        sum = s32;
                    } else {
                        sum = spec_w(q4[u].x, p4[u].x, residual) + spec_w(q4[u].y, p4[u].y, residual) +
                              spec_w(q4[u].z, p4[u].z, residual) + spec_w(q4[u].w, p4[u].w, residual);
                    }
                    sum = tile_sum(sum);
                    const int t = (int)((s0 - e0) / kSpecTile) + warp + u * NW;
                    if (lane == 0 && t < my1 - my0) tsum[t] = sum;
                }
            }
            chunks_done += nchunks;
        } else {
            for (int t = my0 + warp; t < my1; t += NW * kSpecUnroll) {
                float4 q4[kSpecUnroll], p4[kSpecUnroll];
#pragma unroll
                for (int u = 0; u < kSpecUnroll; ++u) {
                    const int tt = t + u * NW;
                    const long long x0 = (long long)tt * kSpecTile + lane * 4;
                    float qv[4] = {0.f, 0.f, 0.f, 0.f}, pv[4] = {0.f, 0.f, 0.f, 0.f};
                    if (tt < my1)
                        for (int j = 0; j < 4 && x0 + j < n; ++j) {
                            qv[j] = __ldg(qr + x0 + j);
                            if (residual) pv[j] = __ldg(pr + x0 + j);
                        }
                    q4[u] = make_float4(qv[0], qv[1], qv[2], qv[3]);
                    p4[u] = make_float4(pv[0], pv[1], pv[2], pv[3]);
                }
#pragma unroll
                for (int u = 0; u < kSpecUnroll; ++u) {
                    const int tt = t + u * NW;
                    if (tt >= my1) break;  // warp-uniform
                    u64 sum = spec_w(q4[u].x, p4[u].x, residual) + spec_w(q4[u].y, p4[u].y, residual) +
                              spec_w(q4[u].z, p4[u].z, residual) + spec_w(q4[u].w, p4[u].w, residual);
                    sum = tile_sum(sum);
                    if (lane == 0) tsum[tt - my0] = sum;
                }
            }
        }
        __syncthreads();
        if (warp == 0) {
            u64 c = 0;
            for (int t = lane; t < my1 - my0; t += 32) c += tsum[t];
#pragma unroll
            for (int off = 16; off; off >>= 1) c += shfl_xor_u64(c, off);
            if (lane == 0) s_chunk = c;
        }
        cluster.sync();  // every CTA's share is visible cluster-wide
        u64 total = 0, before = 0;  // the row's sum, and the sum of the shares before this CTA's
        for (int r = 0; r < kSpecCluster; ++r) {
            const u64 v = *cluster.map_shared_rank(&s_chunk, r);
            total += v;
            if (r < rank) before += v;
        }
        // done with the other CTAs' shared memory: arrive now, wait before this CTA's
        // shared memory is rewritten or released (so the search below holds nobody back)
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        if (total == 0) {
            asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
            if (acc == k) break;  // the target row itself is zero: no token
            continue;
        }
        const u64 target = scaled_floor(a.u_res[b], total);
        if (before <= target && target - before < s_chunk) {
            // this CTA's share holds the crossing: scan its tile sums in runs, a run per thread
            if (tid == 0) s_cross_tile = -1;
            const int nt = my1 - my0;
            const int per = (nt + kSpecThreads - 1) / kSpecThreads;
            const int t0 = tid * per;
            const int t1 = min(nt, t0 + per);
            u64 mine = 0;
            for (int t = t0; t < t1; ++t) mine += tsum[t];
            u64 incl = mine;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const u64 y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            if (lane == 31) s_warp[warp] = incl;
            __syncthreads();
            u64 bw = before;
            for (int w = 0; w < warp; ++w) bw += s_warp[w];
            const u64 excl = bw + incl - mine;
            if (excl <= target && target < excl + mine) {
                // the crossing lies in this thread's run: find its tile from the sums
                u64 run = excl;
                int t = t0;
                for (; t < t1 - 1; ++t) {
                    if (run + tsum[t] > target) break;
                    run += tsum[t];
                }
                s_cross_tile = my0 + t;
                s_cross_run = run;
            }
            __syncthreads();
            if (warp == 0 && s_cross_tile >= 0) {
                // the tile's 128 weights: 4 per lane, a warp scan of the lane sums
                const long long x0 = (long long)s_cross_tile * kSpecTile + lane * 4;
                u64 w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    w[j] = (x0 + j < n) ? spec_w(__ldg(qr + x0 + j), residual ? __ldg(pr + x0 + j) : 0.f, residual) : 0ull;
                const u64 lsum = w[0] + w[1] + w[2] + w[3];
                u64 incl_l = lsum;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const u64 y = __shfl_up_sync(0xffffffffu, incl_l, off);
                    if (lane >= off) incl_l += y;
                }
                u64 r = s_cross_run + (incl_l - lsum);
                int hit = -1;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    r += w[j];
                    if (hit < 0 && r > target) hit = (int)(x0 + j);
                }
                const unsigned m = __ballot_sync(0xffffffffu, hit >= 0);
                if (m && lane == __ffs((int)m) - 1) out[acc] = hit;
            }
        }
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // nobody reads the shares any more
        break;
    }
}

size_t spec_smem_bytes(long long n) {
    const long long ntiles = (n + kSpecTile - 1) / kSpecTile;
    const long long tpc = (ntiles + kSpecCluster - 1) / kSpecCluster;
    const size_t ring = n % 4 == 0 ? kSpecRingBytes : 0;
    return ring + (size_t)tpc * sizeof(u64) + kSpecStages * sizeof(uint64_t);
}

cudaError_t launch_spec_accept(const SpecArgs& a, cudaStream_t st) {
    if (a.B <= 0) return cudaSuccess;
    const size_t smem = spec_smem_bytes(a.n);
    const unsigned grid = (unsigned)a.B * kSpecCluster;
    cudaError_t e;
    if (a.n % 4 == 0) {
        e = cudaFuncSetAttribute(spec_accept_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(spec_accept_kernel<true>, dim3(grid), dim3(kSpecThreads), smem, st, a);
    } else {
        e = cudaFuncSetAttribute(spec_accept_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(spec_accept_kernel<false>, dim3(grid), dim3(kSpecThreads), smem, st, a);
    }
}

}  // namespace spd
