// attn_dense.cu -- instantiations of the paged attention kernel for dense causal
// verification (T drafted positions, R = T*G rows in 1, 2 or 4 MMA row tiles)
// and dense decode (T = 1); items = every page of the sequence.
#include "attn.cuh"

namespace spd {

template <int D, int PS>
static cudaError_t dense_mt(const AttnArgs& a, const CUtensorMap& k, const CUtensorMap& v, cudaStream_t st) {
    switch (attn_mtiles(a.T, a.H_q / a.H_kv)) {
        case 1: return launch_attn_t<D, PS, 1, false, 1>(a, k, v, st);
        case 2: return launch_attn_t<D, PS, 2, false, 1>(a, k, v, st);
        default: return launch_attn_t<D, PS, 4, false, 1>(a, k, v, st);
    }
}

template <int D>
static cudaError_t dense_ps(const AttnArgs& a, const CUtensorMap& k, const CUtensorMap& v, cudaStream_t st) {
    switch (a.ps) {
        case 16: return dense_mt<D, 16>(a, k, v, st);
        case 32: return dense_mt<D, 32>(a, k, v, st);
        default: return dense_mt<D, 64>(a, k, v, st);
    }
}

cudaError_t launch_dense_attn(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              cudaStream_t st) {
    if (a.B == 0) return cudaSuccess;
    return a.D == 128 ? dense_ps<128>(a, tmK, tmV, st) : dense_ps<64>(a, tmK, tmV, st);
}

template <int D, int PS>
static int occ_mt(int mtiles) {
    switch (mtiles) {
        case 1: return attn_ctas_per_sm_t<D, PS, 1, false, 1>();
        case 2: return attn_ctas_per_sm_t<D, PS, 2, false, 1>();
        default: return attn_ctas_per_sm_t<D, PS, 4, false, 1>();
    }
}

template <int D>
static int occ_dense(int ps, int mtiles) {
    switch (ps) {
        case 16: return occ_mt<D, 16>(mtiles);
        case 32: return occ_mt<D, 32>(mtiles);
        default: return occ_mt<D, 64>(mtiles);
    }
}

int occ_dense_attn(int D, int ps, int mtiles) { return D == 128 ? occ_dense<128>(ps, mtiles) : occ_dense<64>(ps, mtiles); }

}  // namespace spd
