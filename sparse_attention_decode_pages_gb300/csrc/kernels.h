// kernels.h -- host-side launch interface between the C-ABI layer (spd_api.cu)
// and the kernel translation units.  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spd.h"

#include <utility>

namespace spd {

// Launches a kernel of the library with programmatic stream serialisation
// allowed (see pdl_wait / pdl_trigger): the launch of a kernel overlaps the
// tail of the previous one on the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct SummarizeArgs {
    const uint16_t* K;
    const int32_t* page_table;
    const int32_t* seq_lens;
    const int32_t* only_pages;  // NULL = all pages
    int n_only;
    uint16_t* summ;
    int B, H_kv, D, ps, max_pages;
    long long num_phys;
    unsigned* status;
};
cudaError_t launch_summarize(const SummarizeArgs& a, cudaStream_t st);

struct AppendArgs {
    uint16_t* K;
    uint16_t* V;
    const int32_t* page_table;
    const int32_t* seq_lens;
    const uint16_t* k_new;  // [B][T][H_kv][D]
    const uint16_t* v_new;
    uint16_t* summ;         // [B][H_kv][max_pages][2][D]
    int B, T, H_kv, D, ps, max_pages;
    long long num_phys;
    unsigned* status;
};
cudaError_t launch_append_refresh(const AppendArgs& a, cudaStream_t st);

// Default limit of every bounded wait in the kernels (spd_set_wait_limit_ns).
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
// The limit the next launches pass to their kernels.
unsigned long long wait_limit_ns();

struct SpecArgs {
    const float* p;        // [B][k][n] drafter probabilities
    const float* q;        // [B][k+1][n] target probabilities
    const int32_t* draft;  // [B][k]
    const float* u_acc;    // [B][k]
    const float* u_res;    // [B]
    int32_t* n_accepted;   // [B]
    int32_t* tokens;       // [B][k+1]
    int B, k;
    long long n;
    unsigned* status;
    unsigned long long wait_ns;
};
cudaError_t launch_spec_accept(const SpecArgs& a, cudaStream_t st);
size_t spec_smem_bytes(long long n);

struct ScoreSelectArgs {
    const uint16_t* q;
    const uint16_t* summ;  // [B][H_kv][max_pages][2][D]
    const int32_t* seq_lens;
    spd_budget_policy pol;
    int32_t* sel;
    int32_t* nsel;
    int k_max;
    float* scores;    // [B][H_kv][max_pages]
    int B, H_q, H_kv, D, ps, max_pages;
    long long num_phys;
    unsigned* status;
    // Fused append (pages_append_score_select): the step's token, written into the
    // cache and into its page's summary by the warp that scores that page.
    uint16_t* K;  // NULL: no append
    uint16_t* V;
    const int32_t* page_table;
    const uint16_t* k_new;  // [B][H_kv][D]
    const uint16_t* v_new;
    uint16_t* summ_w;       // == summ
    // Chained step (sparse_decode_step): tiles are handed out in row order from
    // counters, each finished tile is counted per row, and the selection of a row
    // starts when its count is complete (instead of after the whole scoring grid).
    unsigned long long* tile_ctr;  // [2]: chunk and single-tile counters, zero on entry and on exit
    unsigned* warps_done;
    unsigned* sel_claims;          // chained step: the selection CTAs' row claims (zero on entry and on exit)
    unsigned* tiles_done;          // [B*H_kv] progress hints (NULL: not chained), zero on entry and on exit
    unsigned* sel_done;            // [B*H_kv]: set when a row's selection is written
    // [B*H_kv][max_pages] order-preserving score keys (never 0), zero on entry and
    // on exit: a key is its own ready flag, so the scoring warps need no fences
    unsigned* keys;
    // chained step: [B*H_kv][k_max] the physical page of each selected page (read by
    // the attention instead of the page table); NULL otherwise
    int32_t* sel_phys;
    unsigned long long wait_ns;  // limit of every bounded wait
};
// Scores every page (persistent grid sized to num_sms), then selects per row.
cudaError_t launch_score_select(const ScoreSelectArgs& a, int num_sms, cudaStream_t st);

struct AttnArgs {
    const uint16_t* q;  // [B][T][H_q][D] (T = 1 for decode)
    const int32_t* page_table;
    const int32_t* seq_lens;
    const int32_t* sel;   // sparse only
    const int32_t* nsel;  // sparse only
    int k_max;
    int B, H_q, H_kv, D, ps, max_pages, T;
    long long num_phys;
    int items_per_split, num_splits;
    float scale_log2;
    uint16_t* o;
    float* lse;
    float* part_o;    // [B*H_kv][num_splits][R][D]
    float* part_lse;  // [B*H_kv][num_splits][R]
    int* counters;    // [B*H_kv] split tickets, zero on entry and on exit
    int* queue;       // 16 bytes (8-aligned): the unit queue counter, zero on entry and exit
    int num_sms;
    unsigned* status;
    unsigned* sel_done;  // chained step: wait for the row's selection flag instead of the previous grid
    const int32_t* sel_phys;  // chained step: physical pages of sel (NULL: look them up in page_table)
    unsigned long long wait_ns;  // limit of every bounded wait
};
// Rows (T * G) handled per CTA, padded to 16-row MMA tiles.
inline int attn_mtiles(int T, int G) {
    int r = T * G;
    return r <= 16 ? 1 : (r <= 32 ? 2 : 4);
}
cudaError_t launch_sparse_attn(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               cudaStream_t st);
cudaError_t launch_dense_attn(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              cudaStream_t st);
// CTAs of the attention kernel that fit on one SM for this shape.
int occ_sparse_attn(int D, int ps);
int occ_dense_attn(int D, int ps, int mtiles);

// Host helpers of the C-ABI layer shared with round.cu.
spd_status device_ready();
spd_status set_error(spd_status s, const char* msg);

cudaError_t launch_lse_merge(int S, int rows, int D, const float* part_o, const float* part_lse,
                             uint16_t* o, float* lse, cudaStream_t st);

}  // namespace spd
