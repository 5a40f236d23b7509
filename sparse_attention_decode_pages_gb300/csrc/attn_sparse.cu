// attn_sparse.cu -- instantiations of the paged attention kernel for sparse
// decode: one query position, the G <= 8 grouped heads in one 16-row tile,
// items = the selected pages of each (sequence, KV head).
#include "attn.cuh"

namespace spd {

template <int D>
static cudaError_t sparse_ps(const AttnArgs& a, const CUtensorMap& k, const CUtensorMap& v, cudaStream_t st) {
    switch (a.ps) {
        case 16: return launch_attn_t<D, 16, 1, true, 2>(a, k, v, st);
        case 32: return launch_attn_t<D, 32, 1, true, 2>(a, k, v, st);
        default: return launch_attn_t<D, 64, 1, true, 2>(a, k, v, st);
    }
}

cudaError_t launch_sparse_attn(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               cudaStream_t st) {
    if (a.B == 0) return cudaSuccess;
    return a.D == 128 ? sparse_ps<128>(a, tmK, tmV, st) : sparse_ps<64>(a, tmK, tmV, st);
}

template <int D>
static int occ_sparse(int ps) {
    switch (ps) {
        case 16: return attn_ctas_per_sm_t<D, 16, 1, true, 2>();
        case 32: return attn_ctas_per_sm_t<D, 32, 1, true, 2>();
        default: return attn_ctas_per_sm_t<D, 64, 1, true, 2>();
    }
}

int occ_sparse_attn(int D, int ps) { return D == 128 ? occ_sparse<128>(ps) : occ_sparse<64>(ps); }

}  // namespace spd
