// round.cu -- one S3R round (k sparse draft steps, then dense verification and
// exact speculative sampling) captured once into two CUDA graphs and replayed
// with one launch each.  The pages' own accounting splits a round the same
// way: drafting runs under CUDA Graphs, "Draft (6Tq)" and "Verify (TV)" are
// timed apart (S3R Table 7).
//
// The graphs hold exactly the library's calls, made through the C ABI with
// the descriptor's buffers: per draft step s, the append + summary refresh
// of the step's token, scoring + selection with the step's query, and the
// sparse attention; then the rewrite of the k + 1 verified positions, the dense
// verification and (optionally) the accept / reject + draw.  Capture uses a
// private stream in relaxed mode; nothing in those calls allocates or
// synchronises, so the replay is the eager sequence without launch overhead.
#include <cstdlib>
#include <cstring>

#include "kernels.h"

#define SPD_API extern "C" __attribute__((visibility("default")))

struct spd_round_s {
    spd_round_desc d;
    cudaGraphExec_t exec[2];
};

namespace {

spd_status capture(const spd_round_desc& r, int part, cudaStream_t st) {
    const spd_dims* dims = &r.dims;
    const long long B = dims->B;
    const long long qrow = (long long)dims->H_q * dims->D;   // one query row set per sequence
    const long long kvrow = (long long)dims->H_kv * dims->D; // one token's K (or V) per sequence
    spd_status s = SPD_OK;
    if (part == 0) {
        for (int i = 0; i < r.k && s == SPD_OK; ++i) {
            const int32_t* lens = r.seq_lens + i * B;
            const spd_bf16* q = r.q_draft + i * B * qrow;
            s = kv_append_refresh(dims, 1, r.K, r.V, r.page_table, lens, r.k_draft + i * B * kvrow,
                                  r.v_draft + i * B * kvrow, r.summ, st);
            if (s == SPD_OK)
                s = pages_score_select(dims, q, r.summ, lens, &r.policy, r.sel, r.nsel, r.k_max, nullptr,
                                       r.ws_select, r.ws_select_bytes, st);
            if (s == SPD_OK)
                s = sparse_decode_attn(dims, q, r.K, r.V, r.page_table, lens, r.sel, r.nsel, r.k_max,
                                       r.sparse_splits, r.softmax_scale, r.o_draft + i * B * qrow,
                                       r.lse_draft ? r.lse_draft + i * B * dims->H_q : nullptr, r.ws_sparse,
                                       r.ws_sparse_bytes, st);
        }
    } else {
        const int T = r.k + 1;
        const int32_t* lens = r.seq_lens + (long long)r.k * B;
        s = kv_append_refresh(dims, T, r.K, r.V, r.page_table, lens, r.k_verify, r.v_verify, r.summ, st);
        if (s == SPD_OK)
            s = dense_verify_attn(dims, T, r.q_verify, r.K, r.V, r.page_table, lens, r.verify_splits,
                                  r.softmax_scale, r.o_verify, r.lse_verify, r.ws_verify, r.ws_verify_bytes, st);
        if (s == SPD_OK && r.n_vocab > 0)
            s = spec_accept(dims->B, r.k, r.n_vocab, r.p_draft, r.q_target, r.draft_tokens, r.u_acc, r.u_res,
                            r.n_accepted, r.tokens, st);
    }
    return s;
}

}  // namespace

SPD_API spd_status spd_round_create(const spd_round_desc* desc, spd_round** out) {
    using spd::set_error;
    if (!desc || !out) return set_error(SPD_ERR_INVALID_ARG, "NULL descriptor or output");
    *out = nullptr;
    const spd_round_desc& r = *desc;
    if (r.k < 1 || r.k > 32) return set_error(SPD_ERR_UNSUPPORTED, "k must be in [1, 32]");
    if (r.dims.B < 1) return set_error(SPD_ERR_INVALID_ARG, "a round needs B >= 1");
    if (!r.seq_lens || !r.q_draft || !r.k_draft || !r.v_draft || !r.q_verify || !r.k_verify || !r.v_verify ||
        !r.o_draft || !r.o_verify || !r.sel || !r.nsel)
        return set_error(SPD_ERR_INVALID_ARG, "NULL pointer in the round descriptor");
    if (r.n_vocab > 0 && (!r.p_draft || !r.q_target || !r.draft_tokens || !r.u_acc || !r.u_res ||
                          !r.n_accepted || !r.tokens))
        return set_error(SPD_ERR_INVALID_ARG, "NULL sampling buffer in the round descriptor");
    spd_status s = spd::device_ready();
    if (s != SPD_OK) return s;

    spd_round* h = static_cast<spd_round*>(calloc(1, sizeof(spd_round)));
    if (!h) return set_error(SPD_ERR_INVALID_ARG, "out of host memory");
    h->d = r;
    cudaStream_t st = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        free(h);
        return set_error(SPD_ERR_CUDA, cudaGetErrorString(e));
    }
    for (int part = 0; part < 2 && s == SPD_OK; ++part) {
        cudaGraph_t g = nullptr;
        e = cudaStreamBeginCapture(st, cudaStreamCaptureModeRelaxed);
        if (e != cudaSuccess) {
            s = set_error(SPD_ERR_CUDA, cudaGetErrorString(e));
            break;
        }
        s = capture(r, part, st);
        e = cudaStreamEndCapture(st, &g);  // always end the capture, even after a failed call
        if (s == SPD_OK && e != cudaSuccess) s = set_error(SPD_ERR_CUDA, cudaGetErrorString(e));
        if (s == SPD_OK) {
            e = cudaGraphInstantiate(&h->exec[part], g, 0);
            if (e != cudaSuccess) s = set_error(SPD_ERR_CUDA, cudaGetErrorString(e));
        }
        if (g) cudaGraphDestroy(g);
    }
    cudaStreamDestroy(st);
    if (s != SPD_OK) {
        for (int part = 0; part < 2; ++part)
            if (h->exec[part]) cudaGraphExecDestroy(h->exec[part]);
        free(h);
        return s;
    }
    *out = h;
    return SPD_OK;
}

SPD_API spd_status spd_round_launch(spd_round* r, int32_t part, void* stream) {
    using spd::set_error;
    if (!r) return set_error(SPD_ERR_INVALID_ARG, "NULL round");
    if (part < 0 || part > 2) return set_error(SPD_ERR_INVALID_ARG, "part must be 0, 1 or 2");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int p = 0; p < 2; ++p) {
        if (part != 2 && part != p) continue;
        cudaError_t e = cudaGraphLaunch(r->exec[p], st);
        if (e != cudaSuccess) return set_error(SPD_ERR_CUDA, cudaGetErrorString(e));
    }
    return SPD_OK;
}

SPD_API void spd_round_destroy(spd_round* r) {
    if (!r) return;
    for (int p = 0; p < 2; ++p)
        if (r->exec[p]) cudaGraphExecDestroy(r->exec[p]);
    free(r);
}
