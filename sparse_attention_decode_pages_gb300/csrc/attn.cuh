// attn.cuh -- paged FlashDecoding kernel shared by sparse decode (attention over
// the selected pages: Sparrow's block-sparse rollout attention, the S3R sparse
// drafter) and dense causal verification (S3R "Verify (TV)": T drafted
// positions over the complete KV cache).
//
// One CTA per (sequence, KV head, split).  The CTA holds all R = T*G query
// rows of the KV head (padded to 16-row MMA tiles) so the G grouped heads and T
// positions share every page load.  Warps form NG page groups of NMT warps;
// group g takes every NG-th item of the CTA's page range and owns a ring of
// STAGES shared-memory slots.  For each page one lane issues TMA tensor loads
// (cp.async.bulk.tensor, 128-byte swizzle, mbarrier transaction counts) of the
// page's K and V tiles -- only the selected pages are ever fetched.  Compute
// per 16-token chunk: S = Q K^T and O += P V on the tensor cores (mma.sync
// m16n8k16 bf16 -> fp32; K and V tiles read with ldmatrix, conflict-free under
// the swizzle), online softmax in fp32 with exp2.  The page groups are merged
// in shared memory at the end.  With several splits per row the CTA writes a
// normalised partial (o, lse) to the workspace and the last CTA of the row to
// finish (atomic ticket; nothing waits) merges them with the log-sum-exp rule.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace spd {

template <int D, int PS, int NMT>
struct AttnCfg;

// Page groups and ring depth: about 64-96 KB of ring per CTA.
template <int D, int PS, int NMT>
struct AttnCfg {
    static constexpr int TILE = PS * D * 2;  // bytes of one K (or V) tile
    static constexpr int SLOT = 2 * TILE;
    static constexpr int NG_BASE = (SLOT <= 8192) ? 4 : (SLOT <= 16384 ? 2 : 1);
    static constexpr int NG = (NG_BASE / NMT) > 0 ? (NG_BASE / NMT) : 1;
    static constexpr int STAGES = (SLOT <= 4096) ? 4 : 3;
    static constexpr int THREADS = NG * NMT * 32;
    static constexpr int RP = NMT * 16;  // padded rows
    static constexpr int RING = NG * STAGES * SLOT;
    static constexpr int EPI = NG * RP * (D + 2) * 4;
    static constexpr int BODY = RING > EPI ? RING : EPI;
    static constexpr int SMEM = 1024 /*alignment slack*/ + BODY + NG * STAGES * 8;
};

template <int D, int PS, int NMT, bool SPARSE>
__global__ void __launch_bounds__(AttnCfg<D, PS, NMT>::THREADS)
    attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV) {
    using C = AttnCfg<D, PS, NMT>;
    constexpr int NG = C::NG, STAGES = C::STAGES, RP = C::RP;
    constexpr int KSTEPS = D / 16;
    constexpr int NT_O = D / 8;
    constexpr int HALVES = D / 64;
    constexpr int HALF_BYTES = PS * 128;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_last;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BODY);

    const int b = blockIdx.z, h = blockIdx.y, split = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = warp / NMT, mt = warp % NMT;
    const int G = a.H_q / a.H_kv;
    const int R = a.T * G;
    const int len = a.seq_lens[b];
    const int P = (len + PS - 1) / PS;

    int n_items;
    const int32_t* sel_row = nullptr;
    if (SPARSE) {
        sel_row = a.sel + ((long long)b * a.H_kv + h) * a.k_max;
        n_items = a.nsel[(long long)b * a.H_kv + h];
        if (n_items > a.k_max || n_items < 0) {
            if (tid == 0) raise_status(a.status, SPD_DEV_BAD_SEL);
            n_items = n_items < 0 ? 0 : a.k_max;
        }
    } else {
        n_items = P;
    }
    const int nsplit_row = (n_items + a.items_per_split - 1) / a.items_per_split;
    const long long row0 = ((long long)b * a.H_kv + h);  // (b, h) index

    // Output row r -> (t, g): o index ((b*T + t)*H_q + h*G + g)*D.
    auto out_index = [&](int r) -> long long {
        const int t = r / G, g = r - t * G;
        return ((long long)b * a.T + t) * a.H_q + h * G + g;
    };

    if (split >= nsplit_row) {
        if (split == 0) {  // empty row: o = 0, lse = -inf
            for (int i = tid; i < R * D; i += C::THREADS) {
                const int r = i / D, d = i - r * D;
                reinterpret_cast<bf16*>(a.o)[out_index(r) * D + d] = __float2bfloat16(0.f);
            }
            if (a.lse)
                for (int r = tid; r < R; r += C::THREADS) a.lse[out_index(r)] = __int_as_float(0xff800000);
        }
        return;
    }
    const int it_begin = split * a.items_per_split;
    const int it_end = min(n_items, it_begin + a.items_per_split);
    // items of this group: it_begin + grp + NG*j
    const int n_g = (it_end - it_begin - grp + NG - 1) / NG > 0 ? (it_end - it_begin - grp + NG - 1) / NG : 0;

    const bool producer = (mt == 0) && (lane == 0);
    uint8_t* ring = smem + grp * STAGES * C::SLOT;
    uint64_t* gbar = bars + grp * STAGES;

    if (tid == 0) {
        for (int i = 0; i < NG * STAGES; ++i) mbar_init(bars + i, 1);
        mbar_fence_init();
    }
    if (tid == 32 % C::THREADS) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    __syncthreads();

    // Item j of this group -> logical page and physical page; -1 (and the
    // status bit to raise) when the selection entry or the page id is bad.
    auto item_page = [&](int j, long long& phys, unsigned& err) -> int {
        const int it = it_begin + grp + NG * j;
        const int lp = SPARSE ? sel_row[it] : it;
        phys = -1;
        if (lp < 0 || lp >= P) {
            err = SPD_DEV_BAD_SEL;
            return -1;
        }
        const long long f = a.page_table[(long long)b * a.max_pages + lp];
        if (f < 0 || f >= a.num_phys) {
            err = SPD_DEV_BAD_PAGE;
            return -1;
        }
        phys = f;
        err = 0;
        return lp;
    };
    auto issue = [&](int j) {
        const int slot = j % STAGES;
        long long phys;
        unsigned err;
        const int lp = item_page(j, phys, err);
        uint8_t* dst = ring + slot * C::SLOT;
        if (lp < 0) {
            raise_status(a.status, err);
            mbar_arrive_expect_tx(gbar + slot, 0);  // completes the phase with no data
            return;
        }
        mbar_arrive_expect_tx(gbar + slot, C::SLOT);
        const int y = (int)((phys * a.H_kv + h) * PS);
#pragma unroll
        for (int hf = 0; hf < HALVES; ++hf) {
            tma_load_2d(dst + hf * HALF_BYTES, &tmK, hf * 64, y, gbar + slot);
            tma_load_2d(dst + C::TILE + hf * HALF_BYTES, &tmV, hf * 64, y, gbar + slot);
        }
    };
    if (producer) {
        for (int j = 0; j < n_g && j < STAGES; ++j) issue(j);
    }

    // Q fragments (A operand) for this warp's 16 rows.
    const int qr0 = mt * 16 + (lane >> 2), qr1 = qr0 + 8;
    const int c4 = lane & 3;
    uint32_t qa[KSTEPS][4];
    {
        const bf16* qb = reinterpret_cast<const bf16*>(a.q);
        const bf16* q0 = qr0 < R ? qb + out_index(qr0) * D : nullptr;
        const bf16* q1 = qr1 < R ? qb + out_index(qr1) * D : nullptr;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            const int d0 = kk * 16 + 2 * c4;
            qa[kk][0] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + d0) : 0u;
            qa[kk][1] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + d0) : 0u;
            qa[kk][2] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + d0 + 8) : 0u;
            qa[kk][3] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + d0 + 8) : 0u;
        }
    }
    // Last visible absolute position of each of this thread's rows.
    const int lim0 = qr0 < R ? len - a.T + qr0 / G : len - 1;
    const int lim1 = qr1 < R ? len - a.T + qr1 / G : len - 1;
    const int lim_min = len - a.T;  // smallest limit among real rows

    const float NEG_INF = __int_as_float(0xff800000);
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    float oacc[NT_O][4];
#pragma unroll
    for (int i = 0; i < NT_O; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

    bool ok = true;
    for (int j = 0; j < n_g; ++j) {
        const int slot = j % STAGES;
        const uint32_t parity = (uint32_t)((j / STAGES) & 1);
        bool got = ok && mbar_wait_bounded(gbar + slot, parity, a.status);
        long long phys;
        unsigned err;
        const int lp = item_page(j, phys, err);
        if (got && lp >= 0) {
            uint8_t* kt = ring + slot * C::SLOT;
            uint8_t* vt = kt + C::TILE;
            const int page_start = lp * PS;
            // Slots past the sequence end may hold anything (even NaN): zero them in V.
            const int valid = min(PS, len - page_start);
            if (valid < PS) {
                for (int i = lane; i < (PS - valid) * HALVES * 8; i += 32) {
                    const int rr = valid + i / (HALVES * 8);
                    const int rem = i % (HALVES * 8);
                    const int hf = rem / 8, ch = rem % 8;
                    *reinterpret_cast<uint4*>(vt + hf * HALF_BYTES + rr * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                }
                // order these generic-proxy writes before the slot's next TMA refill
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
            }
            const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
#pragma unroll
            for (int cc = 0; cc < PS / 16; ++cc) {
                float s[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
                {
                    const int mi = lane >> 3, rr = lane & 7;
                    const int tok = cc * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        const int chunk = 2 * kk + (mi & 1);
                        const uint32_t addr = kbase + (chunk >> 3) * HALF_BYTES + swz128(tok, chunk & 7);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(addr, b0, b1, b2, b3);
                        mma_bf16(s[0], qa[kk], b0, b1);
                        mma_bf16(s[1], qa[kk], b2, b3);
                    }
                }
                // scale to log2 units, mask, online softmax
                const int tok0 = page_start + cc * 16;
                const bool need_mask = tok0 + 15 > lim_min;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int pos = tok0 + nt * 8 + 2 * c4 + e;
                        float x0 = s[nt][e] * a.scale_log2;
                        float x1 = s[nt][2 + e] * a.scale_log2;
                        if (need_mask) {
                            if (pos > lim0) x0 = NEG_INF;
                            if (pos > lim1) x1 = NEG_INF;
                        }
                        s[nt][e] = x0;
                        s[nt][2 + e] = x1;
                    }
                }
                float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
                float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float base0 = mn0 == NEG_INF ? 0.f : mn0;
                const float base1 = mn1 == NEG_INF ? 0.f : mn1;
                const float al0 = fast_exp2(m0 - base0), al1 = fast_exp2(m1 - base1);
                m0 = mn0;
                m1 = mn1;
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    s[nt][0] = fast_exp2(s[nt][0] - base0);
                    s[nt][1] = fast_exp2(s[nt][1] - base0);
                    s[nt][2] = fast_exp2(s[nt][2] - base1);
                    s[nt][3] = fast_exp2(s[nt][3] - base1);
                    ps0 += s[nt][0] + s[nt][1];
                    ps1 += s[nt][2] + s[nt][3];
                }
                l0 = l0 * al0 + ps0;
                l1 = l1 * al1 + ps1;
#pragma unroll
                for (int i = 0; i < NT_O; ++i) {
                    oacc[i][0] *= al0;
                    oacc[i][1] *= al0;
                    oacc[i][2] *= al1;
                    oacc[i][3] *= al1;
                }
                const uint32_t pa[4] = {pack_bf16(s[0][0], s[0][1]), pack_bf16(s[0][2], s[0][3]),
                                        pack_bf16(s[1][0], s[1][1]), pack_bf16(s[1][2], s[1][3])};
                {
                    const int mi = lane >> 3, rr = lane & 7;
                    const int tok = cc * 16 + (mi & 1) * 8 + rr;
#pragma unroll
                    for (int np = 0; np < D / 16; ++np) {
                        const int chunk = 2 * np + (mi >> 1);
                        const uint32_t addr = vbase + (chunk >> 3) * HALF_BYTES + swz128(tok, chunk & 7);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(addr, b0, b1, b2, b3);
                        mma_bf16(oacc[2 * np], pa, b0, b1);
                        mma_bf16(oacc[2 * np + 1], pa, b2, b3);
                    }
                }
            }
        }
        // The whole group agrees on abort, and is done reading the slot.
        bool bad = !got;
        if (NMT == 1) {
            bad = __any_sync(0xffffffffu, bad);
        } else {
            uint32_t any;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                : "=r"(any)
                : "r"((uint32_t)bad), "r"(1 + grp), "r"(NMT * 32)
                : "memory");
            bad = any != 0;
        }
        if (bad) {
            ok = false;
            // Let the copies this group already issued land (bounded) before leaving.
            if (producer)
                for (int k2 = j + 1; k2 < n_g && k2 < j + STAGES; ++k2)
                    mbar_wait_bounded(gbar + (k2 % STAGES), (uint32_t)((k2 / STAGES) & 1), a.status);
            break;
        }
        if (producer && j + STAGES < n_g) issue(j + STAGES);
    }

    // Row sums over the quad.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    // Merge the page groups through shared memory (the ring is idle now).
    __syncthreads();
    float* eo = reinterpret_cast<float*>(smem);             // [NG][RP][D]
    float* em = eo + NG * RP * D;                            // [NG][RP]
    float* el = em + NG * RP;                                // [NG][RP]
    {
        float* eg = eo + (grp * RP) * D;
#pragma unroll
        for (int i = 0; i < NT_O; ++i) {
            const int d = i * 8 + 2 * c4;
            *reinterpret_cast<float2*>(eg + qr0 * D + d) = make_float2(oacc[i][0], oacc[i][1]);
            *reinterpret_cast<float2*>(eg + qr1 * D + d) = make_float2(oacc[i][2], oacc[i][3]);
        }
        if (c4 == 0) {
            em[grp * RP + qr0] = m0;
            em[grp * RP + qr1] = m1;
            el[grp * RP + qr0] = l0;
            el[grp * RP + qr1] = l1;
        }
    }
    __syncthreads();

    const bool final_out = (nsplit_row == 1);
    float* po = a.part_o + ((row0 * a.num_splits + split) * (long long)R) * D;
    float* pl = a.part_lse + (row0 * a.num_splits + split) * (long long)R;
    for (int i = tid; i < R * D; i += C::THREADS) {
        const int r = i / D, d = i - r * D;
        float M = NEG_INF;
#pragma unroll
        for (int g = 0; g < NG; ++g) M = fmaxf(M, em[g * RP + r]);
        float L = 0.f, acc = 0.f;
        if (M != NEG_INF) {
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const float w = fast_exp2(em[g * RP + r] - M);
                L += w * el[g * RP + r];
                acc += w * eo[(g * RP + r) * D + d];
            }
        }
        const float ov = L > 0.f ? acc / L : 0.f;
        const float lv = L > 0.f ? (M + __log2f(L)) * kLn2 : NEG_INF;
        if (final_out) {
            reinterpret_cast<bf16*>(a.o)[out_index(r) * D + d] = __float2bfloat16(ov);
            if (d == 0 && a.lse) a.lse[out_index(r)] = lv;
        } else {
            po[(long long)r * D + d] = ov;
            if (d == 0) pl[r] = lv;
        }
    }
    if (final_out) return;

    // Split-K: the last CTA of the row merges the partials.
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(a.counters + row0, 1);
        s_last = (prev == nsplit_row - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* pob = a.part_o + (row0 * a.num_splits) * (long long)R * D;
    const float* plb = a.part_lse + (row0 * a.num_splits) * (long long)R;
    for (int i = tid; i < R * D; i += C::THREADS) {
        const int r = i / D, d = i - r * D;
        float M = NEG_INF;
        for (int s2 = 0; s2 < nsplit_row; ++s2) M = fmaxf(M, __ldcg(plb + (long long)s2 * R + r));
        float ov = 0.f, lv = NEG_INF;
        if (M != NEG_INF) {
            float L = 0.f;
            for (int s2 = 0; s2 < nsplit_row; ++s2) L += __expf(__ldcg(plb + (long long)s2 * R + r) - M);
            const float lse_all = M + __logf(L);
            for (int s2 = 0; s2 < nsplit_row; ++s2) {
                const float ls = __ldcg(plb + (long long)s2 * R + r);
                if (ls != NEG_INF) ov += __expf(ls - lse_all) * __ldcg(pob + ((long long)s2 * R + r) * D + d);
            }
            lv = lse_all;
        }
        reinterpret_cast<bf16*>(a.o)[out_index(r) * D + d] = __float2bfloat16(ov);
        if (d == 0 && a.lse) a.lse[out_index(r)] = lv;
    }
    if (tid == 0) a.counters[row0] = 0;
}

template <int D, int PS, int NMT, bool SPARSE>
cudaError_t launch_attn_t(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          cudaStream_t st) {
    using C = AttnCfg<D, PS, NMT>;
    auto kern = attn_kernel<D, PS, NMT, SPARSE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(a.num_splits, a.H_kv, a.B), block(C::THREADS);
    kern<<<grid, block, C::SMEM, st>>>(a, tmK, tmV);
    return cudaGetLastError();
}

template <int D, int PS, int NMT, bool SPARSE>
int attn_ctas_per_sm_t() {
    using C = AttnCfg<D, PS, NMT>;
    int n = 0;
    // The answer depends on the kernel's dynamic shared-memory limit: set it first
    // so the split count is the same before and after the kernel's first launch.
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, PS, NMT, SPARSE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel<D, PS, NMT, SPARSE>, C::THREADS, C::SMEM);
    if (e != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

}  // namespace spd
