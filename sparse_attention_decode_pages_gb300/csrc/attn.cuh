// attn.cuh -- persistent, warp-specialised paged FlashDecoding kernel shared by
// sparse decode (attention over the selected pages only: Sparrow's
// block-sparse rollout attention, the S3R sparse drafter) and dense causal
// verification (S3R "Verify (TV)": T drafted positions over the complete KV
// cache).
//
// Work units.  A unit is a contiguous run of at most `items_per_split` pages
// ("items") of one (sequence, KV head) row: the selected pages (sparse) or all
// pages (dense).  A unit holds all R = T*G query rows of the KV head, padded to
// 16-row MMA tiles, so the G grouped heads and T positions share each page
// load.  Units are numbered row-major and handed out by an atomic queue.
//
// Workers.  A CTA is one worker: NMT consumer warps (one per 16-row tile) and
// one producer warp, running until the queue is empty (a persistent grid sized
// to the GPU).  The producer claims units, resolves 32 items at a time (the
// selection entries and page-table lookups of a batch are one round trip),
// and for each item waits for a free ring slot (an "empty" mbarrier the
// consumers arrive on) and issues TMA tensor loads (cp.async.bulk.tensor,
// 128-byte swizzle) of the page's K and V tiles; the first item of a unit also
// carries a bulk copy of the unit's Q rows.  The item's logical page and unit
// are written to shared memory before the producer arrives on the slot's
// "full" mbarrier, so the consumers issue no global loads in their main loop
// and the ring keeps streaming across unit boundaries while an epilogue runs.
// The end of the work is signalled through the ring itself.
//
// Compute per 16-token chunk: S = Q K^T and O += P V on the tensor cores
// (mma.sync m16n8k16 bf16 -> fp32, K / V read with ldmatrix, conflict-free
// under the swizzle), online softmax in fp32 with exp2.  A unit that is a
// whole row writes o / lse directly; otherwise it writes a normalised partial
// and the last unit of the row to finish (an atomic ticket; nothing waits)
// merges the partials with the log-sum-exp rule.  The producer making the grid's
// last unit claim resets the queue, so the workspace counters are zero again on
// exit.
// Every wait is bounded (SPD_DEV_TIMEOUT on expiry).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace spd {

struct UnitInfo {
    int row;     // b * H_kv + h
    int split;   // index of this unit within the row
    int start;   // first item
    int count;   // items
    int len;     // seq_lens[b]
    int nsplit;  // units of this row
};

template <int D, int PS, int NMT, bool SPARSE, int KS>
struct AttnCfg {
    static constexpr int TILE = PS * D * 2;  // bytes of one K (or V) tile
    static constexpr int SLOT = 2 * TILE;
    // ring depth: ~32-128 KB of K/V in flight per worker, a multiple of KS (two slots
    // per consumer group up to 32 KB slots: a group with one slot computes while
    // nothing lands for it)
    static constexpr int STAGES = KS == 1 ? (SLOT <= 8192 ? 4 : (SLOT <= 16384 ? 3 : 2))
                                          : (SLOT <= 32768 ? 2 * KS : KS);
    static constexpr int CONSUMERS = NMT * KS;            // KS groups of NMT warps
    static constexpr int THREADS = (CONSUMERS + 1) * 32;  // consumers + one producer warp
    static constexpr int RP = NMT * 16;                   // padded rows
    // A Q buffer holds the unit's R real rows (decode: R = G <= 8; verify:
    // R <= RP); padding rows are zero in registers.
    static constexpr int QROWS = SPARSE ? 8 : RP;
    static constexpr int QBYTES = QROWS * D * 2;
    // Q buffers (per group) and unit-info entries: double-buffered; the producer
    // reuses one only after every consumer warp has read it (the qempty barriers).
    static constexpr int NQ = 2;
    static constexpr int FIFO = NQ;
    // Sparse decode (one query position, the G <= 8 heads of a KV head in one
    // tile) computes the transposed products S^T = K Q^T and O^T += V^T P^T, so
    // the 16 tokens of a chunk fill the MMA rows and the heads its 8 columns:
    // half the MMAs of the head-row form, whose 16 rows would hold G heads.
    static constexpr bool TRS = SPARSE && NMT == 1;
    static constexpr int OT = TRS ? D / 16 : D / 8;  // O accumulator tiles per lane
    // Per consumer lane of groups 1..KS-1: its O fragments, then m0, m1, l0, l1.
    static constexpr int MERGE_FLOATS = 4 * OT + 4;
    static constexpr int MERGE = KS > 1 ? (KS - 1) * NMT * 32 * MERGE_FLOATS * 4 : 0;
    static constexpr int OFF_Q = STAGES * SLOT;
    static constexpr int OFF_MERGE = OFF_Q + NQ * KS * QBYTES;
    // full[STAGES], empty[STAGES], merge_full, merge_empty, qempty[NQ]
    static constexpr int OFF_BAR = OFF_MERGE + MERGE;
    static constexpr int OFF_FIFO = OFF_BAR + (2 * STAGES + 2 + NQ) * 8;
    static constexpr int OFF_META = OFF_FIFO + FIFO * (int)sizeof(UnitInfo);  // int2 per slot
    static constexpr int BODY = OFF_META + STAGES * 8;
    static constexpr int SMEM = 1024 /*alignment slack*/ + BODY;
    static_assert(STAGES % KS == 0, "each ring slot must belong to one consumer group");
};

constexpr int kEndOfWork = -2;  // slot_meta.x: no more items
constexpr float kRescale = 8.f;  // log2 headroom before the running max moves

template <int D, int PS, int NMT, bool SPARSE, int KS>
__global__ void __launch_bounds__(AttnCfg<D, PS, NMT, SPARSE, KS>::THREADS)
    attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV) {
    using C = AttnCfg<D, PS, NMT, SPARSE, KS>;
    constexpr int STAGES = C::STAGES;
    constexpr int KSTEPS = D / 16;
    constexpr int NT_O = C::OT;
    constexpr int HALVES = D / 64;
    constexpr int HALF_BYTES = PS * 128;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_flag;
    __shared__ int2 s_items[32];  // producer: the current batch's {logical page, physical page}

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint8_t* qbuf = smem + C::OFF_Q;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + STAGES;
    uint64_t* merge_full = empty + STAGES;  // groups 1..KS-1 have written their state
    uint64_t* merge_empty = merge_full + 1; // group 0 has read it
    uint64_t* qempty = merge_empty + 1;     // [NQ]: every consumer warp has read unit info and Q
    UnitInfo* fifo = reinterpret_cast<UnitInfo*>(smem + C::OFF_FIFO);
    int2* slot_meta = reinterpret_cast<int2*>(smem + C::OFF_META);  // {logical page or -1 / end, unit seq}

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.H_q / a.H_kv;
    const int R = a.T * G;
    const float NEG_INF = __int_as_float(0xff800000);

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, NMT);
        }
        if (KS > 1) {
            mbar_init(merge_full, (KS - 1) * NMT);
            mbar_init(merge_empty, NMT);
        }
        for (int i = 0; i < C::NQ; ++i) mbar_init(qempty + i, C::CONSUMERS);
        mbar_fence_init();
    }
    if (tid == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    __syncthreads();
    if (!a.sel_done) pdl_wait();  // chained step: each unit waits for its row's selection instead
    pdl_trigger();

    // Output row r of a (b, h) row -> index into o ([B][T][H_q]) and lse.
    auto out_index = [&](int bh, int r) -> long long {
        const int b = bh / a.H_kv, h = bh - b * a.H_kv;
        const int t = r / G, g = r - t * G;
        return ((long long)b * a.T + t) * a.H_q + h * G + g;
    };

    if (warp == C::CONSUMERS) {
        // ============================================================ producer warp
        const long long total_units = (long long)a.B * a.H_kv * a.num_splits;
        // [0..1] 64-bit unit counter: every producer claims units after its first until
        // a claim fails, so the counter takes exactly total_units claims in all
        int* queue = a.queue;
        long long j = 0;       // items issued
        int seq = 0;           // units issued
        bool ok = true;
        // Waits (lane 0) until slot j % STAGES is free; false if the wait ran out.
        auto slot_free = [&](long long jj) -> bool {
            bool r = true;
            if (lane == 0 && jj >= STAGES)
                r = mbar_wait_bounded(empty + (jj % STAGES), (uint32_t)(((jj / STAGES) - 1) & 1), a.status, a.wait_ns);
            return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
        };
        bool first_unit = true;
        while (ok) {
            // The first unit of CTA i is unit i (the grid never exceeds the units);
            // later ones come from the queue, which counts past the grid.
            unsigned long long u = blockIdx.x;
            if (!first_unit) {
                if (lane == 0) {
                    unsigned long long* ctr = reinterpret_cast<unsigned long long*>(queue);
                    u = gridDim.x + atomicAdd(ctr, 1ull);
                    // the grid's last claim: every other claim has been made, so the
                    // counter can be reset for the next call here
                    if ((long long)u == (long long)gridDim.x + total_units - 1) *ctr = 0ull;
                }
                u = __shfl_sync(0xffffffffu, u, 0);
            }
            first_unit = false;
            if ((long long)u >= total_units) break;
            const int row = (int)(u / a.num_splits), split = (int)(u % a.num_splits);
            const int b = row / a.H_kv, h = row - b * a.H_kv;
            const int start = split * a.items_per_split;
            if (SPARSE && a.sel_done) {
                // chained step: wait for the row's selection flag; then every lane
                // acquires it (so its own loads below are ordered after the
                // selection's writes) and the TMA issuer fences the async proxy
                bool okw = true;
                if (lane == 0) okw = flag_wait_bounded(a.sel_done + row, 1u, a.status, a.wait_ns);
                if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) {
                    ok = false;
                    break;
                }
                (void)ld_acquire(a.sel_done + row);
                __syncwarp();
                if (lane == 0) {
                    // each of the row's num_splits units reads the flag once (counting
                    // up from 1); the last reader clears it for the next call
                    if (atomicAdd(a.sel_done + row, 1u) == (unsigned)a.num_splits) a.sel_done[row] = 0u;
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
            }
            // The first 32 selection entries are loaded together with the length
            // and the count (one round trip instead of two).
            // (chained step: with their physical pages, so no page-table round trip follows)
            const bool phys_given = SPARSE && a.sel_phys != nullptr;
            int pre = -1, pre_ph = -1;
            if (SPARSE && start + lane < a.k_max) {
                pre = a.sel[(long long)row * a.k_max + start + lane];
                if (phys_given) pre_ph = a.sel_phys[(long long)row * a.k_max + start + lane];
            }
            const int len = a.seq_lens[b];
            int P = seq_pages(len, PS, a.max_pages);
            if (P < 0) {  // a length the page table cannot hold: the row is empty
                if (lane == 0) raise_status(a.status, SPD_DEV_BAD_LEN);
                P = 0;
            }
            int n_items;
            if (SPARSE) {
                n_items = a.nsel[row];
                if (n_items < 0 || n_items > a.k_max) {
                    if (lane == 0) raise_status(a.status, SPD_DEV_BAD_SEL);
                    n_items = n_items < 0 ? 0 : a.k_max;
                }
            } else {
                n_items = P;
            }
            const int count = min(a.items_per_split, n_items - start);
            if (count <= 0) {
                if (split == 0)  // empty row: o = 0, lse = -inf
                    for (int i = lane; i < R * (D / 8); i += 32) {
                        const int r = i / (D / 8), d = (i % (D / 8)) * 8;
                        const long long oi = out_index(row, r);
                        *reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(a.o) + oi * D + d) = make_uint4(0, 0, 0, 0);
                        if (d == 0 && a.lse) a.lse[oi] = NEG_INF;
                    }
                continue;
            }
            if (seq >= C::NQ) {  // the unit-info entry and Q buffer of unit seq - NQ must be free
                bool r = true;
                if (lane == 0)
                    r = mbar_wait_bounded(qempty + seq % C::NQ, (uint32_t)(((seq / C::NQ) - 1) & 1), a.status, a.wait_ns);
                if (!__shfl_sync(0xffffffffu, r ? 1 : 0, 0)) {
                    ok = false;
                    break;
                }
            }
            if (lane == 0) {
                UnitInfo info;
                info.row = row;
                info.split = split;
                info.start = start;
                info.count = count;
                info.len = len;
                info.nsplit = (n_items + a.items_per_split - 1) / a.items_per_split;
                fifo[seq % C::NQ] = info;  // published by the first item's arrive (release)
            }
            // Items are issued in multiples of KS (padding items carry no page), so
            // every unit starts on group 0 and each group sees each unit.
            const int cpad = (count + KS - 1) / KS * KS;
            // Items are resolved 32 at a time (lane i: item base + i).  The first batch's
            // page-table entries are read here; each later batch's selection entries and
            // page-table entries are read while the batch before it is being issued, so
            // the ring does not drain between batches.
            int lp_raw = -1;         // this lane's logical page in the current batch (unchecked)
            long long ph_raw = -1;   // and its page-table entry (read when lp_raw is in range)
            if (lane < count) {
                lp_raw = SPARSE ? pre : start + lane;
                if (lp_raw >= 0 && lp_raw < P)
                    ph_raw = phys_given ? pre_ph : a.page_table[(long long)b * a.max_pages + lp_raw];
            }
            for (int base = 0; base < cpad && ok; base += 32) {
                int lp = -1;
                long long phys = -1;
                if (base + lane < count) {
                    lp = lp_raw;
                    if (lp < 0 || lp >= P) {
                        raise_status(a.status, SPD_DEV_BAD_SEL);
                        lp = -1;
                    } else {
                        phys = ph_raw;
                        if (phys < 0 || phys >= a.num_phys) {
                            raise_status(a.status, SPD_DEV_BAD_PAGE);
                            lp = -1;
                        }
                    }
                }
                // the next batch: its logical pages now; its page-table entries while this
                // batch is issued (lane 0 reads its own after a few of its pages)
                const int nbase = base + 32;
                int lp_next = -1, ph_given = -1;
                long long ph_next = -1;
                if (nbase + lane < count) {
                    lp_next = SPARSE ? a.sel[(long long)row * a.k_max + start + nbase + lane] : start + nbase + lane;
                    if (phys_given) ph_given = a.sel_phys[(long long)row * a.k_max + start + nbase + lane];
                }
                auto read_next_page_table = [&]() {
                    if (nbase + lane < count && lp_next >= 0 && lp_next < P)
                        ph_next = phys_given ? ph_given : a.page_table[(long long)b * a.max_pages + lp_next];
                };
                // Lane 0 issues the batch from shared memory (no shuffles per item); the
                // other lanes read their next page-table entries meanwhile.
                s_items[lane] = make_int2(lp, (int)phys);
                __syncwarp();
                const int nb = min(32, cpad - base);
                if (lane == 0) {
                    for (int k = 0; k < nb; ++k) {
                        if (k == min(4, nb - 1)) read_next_page_table();
                        const int2 it = s_items[k];
                        const int slot = (int)(j % STAGES);
                        if (j >= STAGES &&
                            !mbar_wait_bounded(empty + slot, (uint32_t)(((j / STAGES) - 1) & 1), a.status, a.wait_ns)) {
                            ok = false;
                            break;
                        }
                        slot_meta[slot] = make_int2(it.x, seq);
                        // each group's first item of the unit carries that group's copy of Q
                        const bool first = (base + k < KS);
                        uint32_t bytes = it.x >= 0 ? (uint32_t)C::SLOT : 0u;
                        if (first) bytes += (uint32_t)(R * D * 2);
                        mbar_arrive_expect_tx(full + slot, bytes);
                        if (first) {  // the unit's Q rows: T runs of G*D contiguous bf16
                            uint8_t* qd = qbuf + ((seq % C::NQ) * KS + (base + k)) * C::QBYTES;
                            const bf16* qs = reinterpret_cast<const bf16*>(a.q);
                            for (int t = 0; t < a.T; ++t)
                                bulk_load(qd + t * G * D * 2, qs + (((long long)b * a.T + t) * a.H_q + h * G) * D,
                                          (uint32_t)(G * D * 2), full + slot);
                        }
                        if (it.x >= 0) {  // the page's K and V tiles: one 3-D box each
                            uint8_t* dst = ring + slot * C::SLOT;
                            const int y = (it.y * a.H_kv + h) * PS;
                            tma_load_3d(dst, &tmK, 0, y, 0, full + slot);
                            tma_load_3d(dst + C::TILE, &tmV, 0, y, 0, full + slot);
                        }
                        ++j;
                    }
                } else {
                    read_next_page_table();
                }
                __syncwarp();
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                j = __shfl_sync(0xffffffffu, j, 0);
                lp_raw = lp_next;
                ph_raw = ph_next;
            }
            ++seq;
        }
        // End of work, signalled through the ring (once per consumer group).
        for (int e = 0; e < KS && ok; ++e) {
            if (!slot_free(j)) break;
            if (lane == 0) {
                const int slot = (int)(j % STAGES);
                slot_meta[slot] = make_int2(kEndOfWork, seq);
                mbar_arrive_expect_tx(full + slot, 0);
            }
            ++j;
        }
        return;
    }

    // ============================================================ consumer warps
    // Group kg takes the items j = kg (mod KS) of every unit (page-parallel), warp
    // mt of the group the 16-row tile mt.  Groups 1..KS-1 hand their softmax
    // state to group 0 at the end of each unit, which finishes the unit.
    const int kg = warp / NMT;
    const int mt = warp - kg * NMT;
    const int qr0 = mt * 16 + (lane >> 2), qr1 = qr0 + 8;
    const int c4 = lane & 3;
    uint32_t qa[KSTEPS][4];
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    float oacc[NT_O][4];
    int lim0 = 0, lim1 = 0, lim_min = 0;
    UnitInfo cu;
    cu.count = 0;
    int cur_seq = -1, c_item = 0, g_items = 0;
    unsigned units_done = 0;  // units this warp has finished (merge barrier phases)
    // consumer-only barrier (the producer warp never joins it)
    auto consumers_sync = [&]() {
        if (NMT > 1)
            asm volatile("bar.sync 1, %0;" ::"r"(NMT * 32) : "memory");
        else
            __syncwarp();
    };

    for (long long j = kg;; j += KS) {
        const int slot = (int)(j % STAGES);
        if (!mbar_wait_bounded(full + slot, (uint32_t)((j / STAGES) & 1), a.status, a.wait_ns)) break;
        const int2 meta = slot_meta[slot];
        if (meta.x == kEndOfWork) break;
        if (meta.y != cur_seq) {
            // new unit: its info, Q fragments, fresh softmax state, row limits
            cur_seq = meta.y;
            cu = fifo[cur_seq % C::NQ];
            c_item = 0;
            g_items = (cu.count + KS - 1) / KS;
            const uint8_t* qsm = qbuf + ((cur_seq % C::NQ) * KS + kg) * C::QBYTES;
            if constexpr (C::TRS) {
                // B fragments of Q^T (k = channel, n = head lane/4): k-step kk holds
                // channels 16kk + 2(lane%4) + {0, 1} and the same + 8
                const int hn = lane >> 2;
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const int d0 = kk * 16 + 2 * c4;
                    qa[kk][0] = hn < R ? *reinterpret_cast<const uint32_t*>(qsm + (hn * D + d0) * 2) : 0u;
                    qa[kk][1] = hn < R ? *reinterpret_cast<const uint32_t*>(qsm + (hn * D + d0 + 8) * 2) : 0u;
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const int d0 = kk * 16 + 2 * c4;
                    qa[kk][0] = qr0 < R ? *reinterpret_cast<const uint32_t*>(qsm + (qr0 * D + d0) * 2) : 0u;
                    qa[kk][1] = qr1 < R ? *reinterpret_cast<const uint32_t*>(qsm + (qr1 * D + d0) * 2) : 0u;
                    qa[kk][2] = qr0 < R ? *reinterpret_cast<const uint32_t*>(qsm + (qr0 * D + d0 + 8) * 2) : 0u;
                    qa[kk][3] = qr1 < R ? *reinterpret_cast<const uint32_t*>(qsm + (qr1 * D + d0 + 8) * 2) : 0u;
                }
            }
            m0 = m1 = NEG_INF;
            l0 = l1 = 0.f;
#pragma unroll
            for (int i = 0; i < NT_O; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
            lim0 = qr0 < R ? cu.len - a.T + qr0 / G : cu.len - 1;
            lim1 = qr1 < R ? cu.len - a.T + qr1 / G : cu.len - 1;
            lim_min = cu.len - a.T;
            __syncwarp();
            if (lane == 0) mbar_arrive(qempty + cur_seq % C::NQ);  // done with unit info and Q
        }
        const int lp = meta.x;
        if (lp >= 0) {
            uint8_t* kt = ring + slot * C::SLOT;
            uint8_t* vt = kt + C::TILE;
            const int page_start = lp * PS;
            // Slots past the sequence end may hold anything (even NaN): zero them in V.
            const int valid = min(PS, cu.len - page_start);
            if (valid < PS) {
                for (int i = lane; i < (PS - valid) * HALVES * 8; i += 32) {
                    const int rr = valid + i / (HALVES * 8);
                    const int rem = i % (HALVES * 8);
                    *reinterpret_cast<uint4*>(vt + (rem / 8) * HALF_BYTES + rr * 128 + (rem % 8) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                // order these generic-proxy writes before the producer's next TMA into the slot
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
            }
            const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
            if constexpr (C::TRS) {
#pragma unroll
                for (int cc = 0; cc < PS / 16; ++cc) {
                    // S^T = K Q^T (rows: the chunk's 16 tokens; columns: heads), four
                    // independent MMA chains over the k-steps
                    float sc[4][4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
                    const int mi = lane >> 3, rr = lane & 7;
                    {
                        // A fragments of K: matrices (tokens 0-7 | 8-15) x (channels lo | hi)
                        const int tok = cc * 16 + (mi & 1) * 8 + rr;
#pragma unroll
                        for (int kk = 0; kk < KSTEPS; ++kk) {
                            const int chunk = 2 * kk + (mi >> 1);
                            uint32_t ka[4];
                            ldsm_x4(kbase + (chunk >> 3) * HALF_BYTES + swz128(tok, chunk & 7), ka[0], ka[1], ka[2], ka[3]);
                            mma_bf16(sc[kk & 3], ka, qa[kk][0], qa[kk][1]);
                        }
                    }
                    // lane: tokens g, g + 8 (g = lane/4) x heads 2c, 2c + 1 (c = lane%4)
                    const int tok0 = page_start + cc * 16 + (lane >> 2);
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[e] = ((sc[0][e] + sc[1][e]) + (sc[2][e] + sc[3][e])) * a.scale_log2;
                    if (tok0 > lim_min) x[0] = x[1] = NEG_INF;      // past the sequence end
                    if (tok0 + 8 > lim_min) x[2] = x[3] = NEG_INF;
                    // per-head maximum over the chunk's tokens (lanes with the same c)
                    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    // lazy rescaling, as in the head-row form (m0 / m1: heads 2c / 2c + 1)
                    const bool up0 = mx0 > m0 + kRescale, up1 = mx1 > m1 + kRescale;
                    if (__any_sync(0xffffffffu, up0 || up1)) {
                        const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
                        const float al0 = (m0 == NEG_INF) ? 0.f : fast_exp2(m0 - mn0);
                        const float al1 = (m1 == NEG_INF) ? 0.f : fast_exp2(m1 - mn1);
                        m0 = mn0;
                        m1 = mn1;
                        l0 *= al0;
                        l1 *= al1;
#pragma unroll
                        for (int i = 0; i < NT_O; ++i) {
                            oacc[i][0] *= al0;
                            oacc[i][1] *= al1;
                            oacc[i][2] *= al0;
                            oacc[i][3] *= al1;
                        }
                    }
                    const float base0 = m0 == NEG_INF ? 0.f : m0;
                    const float base1 = m1 == NEG_INF ? 0.f : m1;
                    x[0] = fast_exp2(x[0] - base0);
                    x[1] = fast_exp2(x[1] - base1);
                    x[2] = fast_exp2(x[2] - base0);
                    x[3] = fast_exp2(x[3] - base1);
                    l0 += x[0] + x[2];
                    l1 += x[1] + x[3];
                    // P^T as the B operand (k = token, n = head): each 8-token half of
                    // the accumulator is one 8x8 fragment, transposed in registers
                    const uint32_t pb0 = movmatrix_t(pack_bf16(x[0], x[1]));
                    const uint32_t pb1 = movmatrix_t(pack_bf16(x[2], x[3]));
                    {
                        // A fragments of V^T: transposed loads of V's (tokens 0-7 | 8-15)
                        // x (channels lo | hi) matrices
                        const int tok = cc * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
                        for (int np = 0; np < D / 16; ++np) {
                            const int chunk = 2 * np + (mi & 1);
                            uint32_t va[4];
                            ldsm_x4_t(vbase + (chunk >> 3) * HALF_BYTES + swz128(tok, chunk & 7), va[0], va[1], va[2], va[3]);
                            mma_bf16(oacc[np], va, pb0, pb1);
                        }
                    }
                }
            } else {
#pragma unroll
            for (int cc = 0; cc < PS / 16; ++cc) {
                // S = Q K^T: even and odd k-steps accumulate in separate chains (four
                // independent MMA chains instead of two), added at the end
                float s[2][4], s_odd[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
                    s_odd[i][0] = s_odd[i][1] = s_odd[i][2] = s_odd[i][3] = 0.f;
                }
                {
                    const int mi = lane >> 3, rr = lane & 7;
                    const int tok = cc * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        const int chunk = 2 * kk + (mi & 1);
                        const uint32_t addr = kbase + (chunk >> 3) * HALF_BYTES + swz128(tok, chunk & 7);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(addr, b0, b1, b2, b3);
                        float(*acc)[4] = (kk & 1) ? s_odd : s;
                        mma_bf16(acc[0], qa[kk], b0, b1);
                        mma_bf16(acc[1], qa[kk], b2, b3);
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int e = 0; e < 4; ++e) s[i][e] += s_odd[i][e];
                }
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
                // Lazy rescaling: the running max (the exponent base) only moves when a
                // logit exceeds it by more than 2^8 (kRescale in log2 units), so most
                // chunks skip rescaling O; terms stay <= 2^8, harmless in fp32.
                const bool up0 = mx0 > m0 + kRescale, up1 = mx1 > m1 + kRescale;
                float al0 = 1.f, al1 = 1.f;
                if (__any_sync(0xffffffffu, up0 || up1)) {
                    const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
                    al0 = (m0 == NEG_INF) ? 0.f : fast_exp2(m0 - mn0);
                    al1 = (m1 == NEG_INF) ? 0.f : fast_exp2(m1 - mn1);
                    m0 = mn0;
                    m1 = mn1;
                    l0 *= al0;
                    l1 *= al1;
#pragma unroll
                    for (int i = 0; i < NT_O; ++i) {
                        oacc[i][0] *= al0;
                        oacc[i][1] *= al0;
                        oacc[i][2] *= al1;
                        oacc[i][3] *= al1;
                    }
                }
                const float base0 = m0 == NEG_INF ? 0.f : m0;
                const float base1 = m1 == NEG_INF ? 0.f : m1;
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
                l0 += ps0;
                l1 += ps1;
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
        }
        // This warp is done with the slot.
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + slot);
        if (++c_item < g_items) continue;

        // ---------------------------------------------------------- unit epilogue
        if constexpr (KS > 1) {
            // Groups 1..KS-1 dump their state (same fragment layout lane for lane);
            // group 0 rescales everything to a common base and adds it up.  The
            // hand-over uses two mbarriers, so every wait in it is bounded.
            float* mb = reinterpret_cast<float*>(smem + C::OFF_MERGE);
            const uint32_t ph = units_done & 1u;
            ++units_done;
            if (kg > 0) {
                // the previous unit's state must have been read before it is overwritten
                if (units_done > 1 && !mbar_wait_bounded(merge_empty, ph ^ 1u, a.status, a.wait_ns)) break;
                float* dst = mb + ((long long)((kg - 1) * NMT + mt) * 32 + lane) * C::MERGE_FLOATS;
#pragma unroll
                for (int i = 0; i < NT_O; ++i)
                    *reinterpret_cast<float4*>(dst + 4 * i) = make_float4(oacc[i][0], oacc[i][1], oacc[i][2], oacc[i][3]);
                *reinterpret_cast<float4*>(dst + 4 * NT_O) = make_float4(m0, m1, l0, l1);
                __syncwarp();
                if (lane == 0) mbar_arrive(merge_full);
                continue;
            }
            if (!mbar_wait_bounded(merge_full, ph, a.status, a.wait_ns)) break;
#pragma unroll 1
            for (int g = 1; g < KS; ++g) {
                const float* src = mb + ((long long)((g - 1) * NMT + mt) * 32 + lane) * C::MERGE_FLOATS;
                const float4 st = *reinterpret_cast<const float4*>(src + 4 * NT_O);
                const float M0 = fmaxf(m0, st.x), M1 = fmaxf(m1, st.y);
                const float a0 = m0 == NEG_INF ? 0.f : fast_exp2(m0 - M0);
                const float a1 = m1 == NEG_INF ? 0.f : fast_exp2(m1 - M1);
                const float b0 = st.x == NEG_INF ? 0.f : fast_exp2(st.x - M0);
                const float b1 = st.y == NEG_INF ? 0.f : fast_exp2(st.y - M1);
#pragma unroll
                for (int i = 0; i < NT_O; ++i) {
                    const float4 v = *reinterpret_cast<const float4*>(src + 4 * i);
                    if constexpr (C::TRS) {  // elements 0, 2: head 2c; 1, 3: head 2c + 1
                        oacc[i][0] = oacc[i][0] * a0 + v.x * b0;
                        oacc[i][1] = oacc[i][1] * a1 + v.y * b1;
                        oacc[i][2] = oacc[i][2] * a0 + v.z * b0;
                        oacc[i][3] = oacc[i][3] * a1 + v.w * b1;
                    } else {  // elements 0, 1: row qr0; 2, 3: row qr1
                        oacc[i][0] = oacc[i][0] * a0 + v.x * b0;
                        oacc[i][1] = oacc[i][1] * a0 + v.y * b0;
                        oacc[i][2] = oacc[i][2] * a1 + v.z * b1;
                        oacc[i][3] = oacc[i][3] * a1 + v.w * b1;
                    }
                }
                l0 = l0 * a0 + st.z * b0;
                l1 = l1 * a1 + st.w * b1;
                m0 = M0;
                m1 = M1;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(merge_empty);
        }
        if constexpr (C::TRS) {  // a head's row sum is spread over the lanes of one c
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
        } else {
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        }
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
        const float lse0 = l0 > 0.f ? (m0 + __log2f(l0)) * kLn2 : NEG_INF;
        const float lse1 = l1 > 0.f ? (m1 + __log2f(l1)) * kLn2 : NEG_INF;
        if constexpr (C::TRS) {
            // lane: heads h0 = 2c, h1 = 2c + 1; channels 16i + g and 16i + g + 8
            const int h0 = 2 * c4, h1 = h0 + 1, g = lane >> 2;
            if (cu.nsplit == 1) {
                bf16* o0 = reinterpret_cast<bf16*>(a.o) + out_index(cu.row, h0 < R ? h0 : 0) * D + g;
                bf16* o1 = reinterpret_cast<bf16*>(a.o) + out_index(cu.row, h1 < R ? h1 : 0) * D + g;
#pragma unroll
                for (int i = 0; i < NT_O; ++i) {
                    if (h0 < R) {
                        o0[16 * i] = __float2bfloat16_rn(oacc[i][0] * inv0);
                        o0[16 * i + 8] = __float2bfloat16_rn(oacc[i][2] * inv0);
                    }
                    if (h1 < R) {
                        o1[16 * i] = __float2bfloat16_rn(oacc[i][1] * inv1);
                        o1[16 * i + 8] = __float2bfloat16_rn(oacc[i][3] * inv1);
                    }
                }
                if (g == 0 && a.lse) {
                    if (h0 < R) a.lse[out_index(cu.row, h0)] = lse0;
                    if (h1 < R) a.lse[out_index(cu.row, h1)] = lse1;
                }
                continue;
            }
            const long long pb = ((long long)cu.row * a.num_splits + cu.split) * R;
#pragma unroll
            for (int i = 0; i < NT_O; ++i) {
                if (h0 < R) {
                    a.part_o[(pb + h0) * D + 16 * i + g] = oacc[i][0] * inv0;
                    a.part_o[(pb + h0) * D + 16 * i + g + 8] = oacc[i][2] * inv0;
                }
                if (h1 < R) {
                    a.part_o[(pb + h1) * D + 16 * i + g] = oacc[i][1] * inv1;
                    a.part_o[(pb + h1) * D + 16 * i + g + 8] = oacc[i][3] * inv1;
                }
            }
            if (g == 0) {
                if (h0 < R) a.part_lse[pb + h0] = lse0;
                if (h1 < R) a.part_lse[pb + h1] = lse1;
            }
        } else {
          if (cu.nsplit == 1) {
#pragma unroll
            for (int i = 0; i < NT_O; ++i) {
                const int d = i * 8 + 2 * c4;
                if (qr0 < R)
                    *reinterpret_cast<uint32_t*>(reinterpret_cast<bf16*>(a.o) + out_index(cu.row, qr0) * D + d) =
                        pack_bf16(oacc[i][0] * inv0, oacc[i][1] * inv0);
                if (qr1 < R)
                    *reinterpret_cast<uint32_t*>(reinterpret_cast<bf16*>(a.o) + out_index(cu.row, qr1) * D + d) =
                        pack_bf16(oacc[i][2] * inv1, oacc[i][3] * inv1);
            }
            if (c4 == 0 && a.lse) {
                if (qr0 < R) a.lse[out_index(cu.row, qr0)] = lse0;
                if (qr1 < R) a.lse[out_index(cu.row, qr1)] = lse1;
            }
            continue;
        }
        const long long pbase = ((long long)cu.row * a.num_splits + cu.split) * R;
#pragma unroll
        for (int i = 0; i < NT_O; ++i) {
            const int d = i * 8 + 2 * c4;
            if (qr0 < R)
                *reinterpret_cast<float2*>(a.part_o + (pbase + qr0) * D + d) =
                    make_float2(oacc[i][0] * inv0, oacc[i][1] * inv0);
            if (qr1 < R)
                *reinterpret_cast<float2*>(a.part_o + (pbase + qr1) * D + d) =
                    make_float2(oacc[i][2] * inv1, oacc[i][3] * inv1);
        }
        if (c4 == 0) {
            if (qr0 < R) a.part_lse[pbase + qr0] = lse0;
            if (qr1 < R) a.part_lse[pbase + qr1] = lse1;
        }
        }
        // Ticket: the partial writes of every consumer lane are ordered before one
        // acq_rel atomic (barrier, then release at GPU scope); the last unit of
        // the row sees every other unit's partials through the acquire.
        consumers_sync();
        if (tid == 0) s_flag = (atomic_add_acq_rel(a.counters + cu.row, 1) == cu.nsplit - 1);
        consumers_sync();
        const bool last = s_flag != 0;
        consumers_sync();  // s_flag is reused by the next unit
        if (!last) continue;
        // Last unit of the row: merge the partials of this warp's rows.  Lane s
        // holds split s's lse; each lane owns D/32 consecutive channels.
        if constexpr (C::TRS && D == 128) {
            // Per output row one L2 round trip for the lse of every split (loaded
            // once, kept for the max, the sum and the weights), then one per batch
            // of SB splits' o; each lane owns 4 channels.  For pages of 32 tokens
            // or more (whose kernels are held to one to three CTAs per SM by shared
            // memory, not registers) eight splits at a time, the first eight issued
            // with the lse loads; for 16-token pages four, after them (issuing them
            // with the lse made the page loop of that kernel measurably slower).
            constexpr bool EARLY = PS >= 32;
            constexpr int SB = PS >= 32 ? 8 : 4;  // splits whose o loads are in flight together
            const long long rbase = (long long)cu.row * a.num_splits * R;
            const int ns = cu.nsplit;
            for (int r = mt * 16; r < min(R, mt * 16 + 16); ++r) {
                const float* lse_r = a.part_lse + rbase + r;                // split s: lse_r[s * R]
                const float4* o_r = reinterpret_cast<const float4*>(a.part_o + (rbase + r) * D) + lane;
                const long long o_step = (long long)R * D / 4;              // split s: o_r[s * o_step]
                float4 v[SB];
                if constexpr (EARLY) {
#pragma unroll
                    for (int k = 0; k < SB; ++k)
                        if (k < ns) v[k] = __ldcg(o_r + k * o_step);
                }
                const float ls0 = lane < ns ? __ldcg(lse_r + (long long)lane * R) : NEG_INF;
                float M = ls0;
                for (int s = 32 + lane; s < ns; s += 32) M = fmaxf(M, __ldcg(lse_r + (long long)s * R));
#pragma unroll
                for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                float L = 0.f;
                if (M != NEG_INF) {
                    if (lane < ns) L += __expf(ls0 - M);
                    for (int s = 32 + lane; s < ns; s += 32) L += __expf(__ldcg(lse_r + (long long)s * R) - M);
                }
#pragma unroll
                for (int off = 16; off; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
                const float lse_all = M == NEG_INF ? NEG_INF : M + __logf(L);
                const float wl0 = (lane < ns && ls0 != NEG_INF && M != NEG_INF) ? __expf(ls0 - lse_all) : 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M != NEG_INF) {
                    for (int s0 = 0; s0 < ns; s0 += SB) {
                        if (!EARLY || s0 > 0) {
#pragma unroll
                            for (int k = 0; k < SB; ++k)
                                if (s0 + k < ns) v[k] = __ldcg(o_r + (s0 + k) * o_step);
                        }
#pragma unroll
                        for (int k = 0; k < SB; ++k) {
                            const int s = s0 + k;
                            if (s >= ns) break;
                            float wk;
                            if (s < 32) {
                                wk = __shfl_sync(0xffffffffu, wl0, s);
                            } else {
                                const float ls = __ldcg(lse_r + (long long)s * R);
                                wk = ls == NEG_INF ? 0.f : __expf(ls - lse_all);
                            }
                            acc.x += wk * v[k].x;
                            acc.y += wk * v[k].y;
                            acc.z += wk * v[k].z;
                            acc.w += wk * v[k].w;
                        }
                    }
                }
                const long long oi = out_index(cu.row, r);
                *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(a.o) + oi * D + lane * 4) =
                    make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
                if (lane == 0 && a.lse) a.lse[oi] = lse_all;
            }
        } else {
            // The lse is read per phase (max, sum, weights) and the o loads of a
            // split are independent of each other.
            const long long rbase = (long long)cu.row * a.num_splits * R;
            constexpr int DPL = D / 32;  // channels per lane
            for (int r = mt * 16; r < min(R, mt * 16 + 16); ++r) {
                float M = NEG_INF;
                for (int s0 = 0; s0 < cu.nsplit; s0 += 32)
                    if (s0 + lane < cu.nsplit) M = fmaxf(M, __ldcg(a.part_lse + rbase + (long long)(s0 + lane) * R + r));
#pragma unroll
                for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                float L = 0.f;
                if (M != NEG_INF)
                    for (int s0 = 0; s0 < cu.nsplit; s0 += 32)
                        if (s0 + lane < cu.nsplit) L += __expf(__ldcg(a.part_lse + rbase + (long long)(s0 + lane) * R + r) - M);
#pragma unroll
                for (int off = 16; off; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
                const float lse_all = M == NEG_INF ? NEG_INF : M + __logf(L);
                float acc[DPL];
#pragma unroll
                for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
                if (M != NEG_INF) {
                    for (int s0 = 0; s0 < cu.nsplit; s0 += 32) {
                        const int ns = min(32, cu.nsplit - s0);
                        float wl = 0.f;
                        if (lane < ns) {
                            const float ls = __ldcg(a.part_lse + rbase + (long long)(s0 + lane) * R + r);
                            wl = ls == NEG_INF ? 0.f : __expf(ls - lse_all);
                        }
#pragma unroll 4
                        for (int k = 0; k < ns; ++k) {
                            const float wk = __shfl_sync(0xffffffffu, wl, k);
                            const float* src = a.part_o + (rbase + (long long)(s0 + k) * R + r) * D + lane * DPL;
                            if (DPL == 4) {
                                const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
                                acc[0] += wk * v.x;
                                acc[1 % DPL] += wk * v.y;
                                acc[2 % DPL] += wk * v.z;
                                acc[3 % DPL] += wk * v.w;
                            } else {
                                const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
                                acc[0] += wk * v.x;
                                acc[1 % DPL] += wk * v.y;
                            }
                        }
                    }
                }
                const long long oi = out_index(cu.row, r);
                bf16* dst = reinterpret_cast<bf16*>(a.o) + oi * D + lane * DPL;
                if (DPL == 4) {
                    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(acc[0], acc[1 % DPL]), pack_bf16(acc[2 % DPL], acc[3 % DPL]));
                } else {
                    *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0], acc[1 % DPL]);
                }
                if (lane == 0 && a.lse) a.lse[oi] = lse_all;
            }
        }
        if (tid == 0) a.counters[cu.row] = 0;
    }
}

template <int D, int PS, int NMT, bool SPARSE, int KS>
int attn_ctas_per_sm_t() {
    using C = AttnCfg<D, PS, NMT, SPARSE, KS>;
    int n = 0;
    // The answer depends on the kernel's dynamic shared-memory limit: set it first
    // so the launch shape is the same before and after the kernel's first launch.
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, PS, NMT, SPARSE, KS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel<D, PS, NMT, SPARSE, KS>, C::THREADS, C::SMEM);
    if (e != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

template <int D, int PS, int NMT, bool SPARSE, int KS>
cudaError_t launch_attn_t(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          cudaStream_t st) {
    using C = AttnCfg<D, PS, NMT, SPARSE, KS>;
    auto kern = attn_kernel<D, PS, NMT, SPARSE, KS>;
    const int per_sm = attn_ctas_per_sm_t<D, PS, NMT, SPARSE, KS>();
    const long long units = (long long)a.B * a.H_kv * a.num_splits;
    long long grid = (long long)a.num_sms * per_sm;
    if (grid > units) grid = units;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM, st, a, tmK, tmV);
}

}  // namespace spd
