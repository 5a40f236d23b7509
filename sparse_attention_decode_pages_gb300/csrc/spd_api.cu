// spd_api.cu -- the C ABI of libspd (declared in include/spd.h): argument
// validation, workspace carving, TMA tensor-map encoding, launch-shape choice
// and dispatch to the kernels.  Nothing here allocates device memory or
// synchronises (except spd_device_status).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "kernels.h"

#define SPD_API extern "C" __attribute__((visibility("default")))

namespace spd {
namespace {

thread_local std::string g_err;

// Device status word (SPD_DEV_* bits), one per device that loads the library.
__device__ unsigned g_status;

spd_status fail(spd_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

spd_status cuda_fail(cudaError_t e, const char* what) {
    return fail(SPD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
constexpr float kLog2e = 1.4426950408889634f;

struct DevInfo {
    std::once_flag once;
    unsigned* status = nullptr;
    int sms = 0;
    cudaError_t err = cudaSuccess;
};
DevInfo g_dev[kMaxDevices];

DevInfo* dev_info(spd_status* st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *st = cuda_fail(e, "cudaGetDevice");
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *st = fail(SPD_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
        return nullptr;
    }
    DevInfo* d = &g_dev[dev];
    std::call_once(d->once, [d, dev]() {
        void* p = nullptr;
        d->err = cudaGetSymbolAddress(&p, g_status);
        if (d->err == cudaSuccess) d->status = static_cast<unsigned*>(p);
        if (d->err == cudaSuccess) d->err = cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, dev);
    });
    if (d->err != cudaSuccess) {
        *st = cuda_fail(d->err, "device set-up");
        return nullptr;
    }
    return d;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(spd_status* st) {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn) *st = fail(SPD_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable (%s)", cudaGetErrorString(err));
    return fn;
}

// 3-D view of a paged K or V cache: x = 64 channels (128 bytes), y = rows
// (num_phys * H_kv * ps of D bf16, stride 2D bytes), z = the D / 64 halves of a
// row (stride 128 bytes).  One box = a page's ps rows of one KV head, laid out
// in shared memory as [half][row][64] with the 128-byte swizzle.
spd_status kv_map(CUtensorMap* m, const void* base, const spd_dims* d) {
    spd_status st = SPD_OK;
    EncodeTiledFn fn = encode_fn(&st);
    if (!fn) return st;
    cuuint64_t gdim[3] = {64, (cuuint64_t)d->num_phys_pages * d->H_kv * d->page_size, (cuuint64_t)d->D / 64};
    cuuint64_t gstride[2] = {(cuuint64_t)d->D * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)d->page_size, (cuuint32_t)d->D / 64};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SPD_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return SPD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace {
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
}  // namespace

unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

// Per-device set-up of the current device (status word, SM count), done once.
spd_status device_ready() {
    spd_status st = SPD_OK;
    return dev_info(&st) ? SPD_OK : st;
}

spd_status set_error(spd_status s, const char* msg) { return fail(s, "%s", msg); }

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

spd_status check_dims(const spd_dims* d) {
    if (!d) return fail(SPD_ERR_INVALID_ARG, "dims is NULL");
    if (d->B < 0 || d->H_q <= 0 || d->H_kv <= 0 || d->max_pages_per_seq <= 0 || d->num_phys_pages < 0)
        return fail(SPD_ERR_INVALID_ARG, "bad dims (B=%d H_q=%d H_kv=%d max_pages=%d num_phys=%lld)", d->B,
                    d->H_q, d->H_kv, d->max_pages_per_seq, (long long)d->num_phys_pages);
    if (d->H_q % d->H_kv) return fail(SPD_ERR_INVALID_ARG, "H_q (%d) is not a multiple of H_kv (%d)", d->H_q, d->H_kv);
    if (d->H_q / d->H_kv > 8) return fail(SPD_ERR_UNSUPPORTED, "GQA group %d > 8", d->H_q / d->H_kv);
    if (d->D != 64 && d->D != 128) return fail(SPD_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", d->D);
    if (d->page_size != 16 && d->page_size != 32 && d->page_size != 64)
        return fail(SPD_ERR_UNSUPPORTED, "page size %d (supported: 16, 32, 64)", d->page_size);
    if ((long long)d->num_phys_pages * d->H_kv * d->page_size >= (1LL << 31))
        return fail(SPD_ERR_UNSUPPORTED, "num_phys_pages * H_kv * page_size must be < 2^31");
    if ((long long)d->B * d->max_pages_per_seq >= (1LL << 31))
        return fail(SPD_ERR_UNSUPPORTED, "B * max_pages_per_seq must be < 2^31");
    return SPD_OK;
}

int pages_per_split_floor(int ps) { return ps >= 64 ? 2 : (ps == 32 ? 4 : 8); }

// Splits per row.  Sparse rows are short and about equal (k_max pages), so a
// row is one unit unless there are too few rows to occupy the persistent
// workers (a whole-row unit needs no partials or merge).  Dense rows differ in
// length by up to 2x, so they are cut into about units_per_worker units per
// worker for the queue to balance.  Each unit keeps at least floor_items pages.
int splits_for(long long rows, int items, long long workers, int floor_items, int units_per_worker,
               int req) {
    int S = req;
    if (S <= 0) {
        S = 1;
        const long long want = units_per_worker * workers;
        if (rows > 0 && (units_per_worker > 1 ? rows < want : 2 * rows < want)) {
            S = (int)((want + rows - 1) / rows);
            const int max_s = (items + floor_items - 1) / floor_items;
            if (S > max_s) S = max_s;
        }
    }
    if (S > items) S = items;
    if (S < 1) S = 1;
    const int ips = (items + S - 1) / S;
    return (items + ips - 1) / ips;
}

int sparse_splits(const spd_dims* d, int k_max, int req, int sms) {
    const long long rows = (long long)d->B * d->H_kv;
    const long long workers = (long long)sms * occ_sparse_attn(d->D, d->page_size);
    return splits_for(rows, k_max, workers, pages_per_split_floor(d->page_size), 1, req);
}

int dense_splits(const spd_dims* d, int T, int req, int sms) {
    const long long rows = (long long)d->B * d->H_kv;
    const int mt = attn_mtiles(T, d->H_q / d->H_kv);
    const long long workers = (long long)sms * occ_dense_attn(d->D, d->page_size, mt);
    return splits_for(rows, d->max_pages_per_seq, workers, 2 * pages_per_split_floor(d->page_size), 4, req);
}

struct AttnWs {
    int* queue;
    int* counters;
    float* part_lse;
    float* part_o;
    size_t bytes;
};

// [queue: 16 B][row tickets][partial lse][partial o]; the first two must start zeroed.
// The scores of pages_score_select start after a prefix as long as the attention
// calls' counters (queue + tickets) and stay clear of it, so the prefix stays zero
// and one buffer can serve the calls of a step in turn.
static size_t score_ws_prefix(const spd_dims* dims) {
    return align256(16 + (size_t)dims->B * dims->H_kv * sizeof(int));
}

// Bytes of attn_ws_layout the kernel touches: with one unit per row (S = 1) only
// the queue and the tickets (no partials).
size_t attn_ws_needed(long long rows, int S, int R, int D);

AttnWs attn_ws_layout(void* ws, long long rows, int S, int R, int D) {
    AttnWs w;
    size_t off = 0;
    char* base = static_cast<char*>(ws);
    w.queue = reinterpret_cast<int*>(base);
    off += 16;
    w.counters = reinterpret_cast<int*>(base + off);
    off = align256(off + rows * sizeof(int));
    w.part_lse = reinterpret_cast<float*>(base + off);
    off += align256((size_t)rows * S * R * sizeof(float));
    w.part_o = reinterpret_cast<float*>(base + off);
    off += (size_t)rows * S * R * D * sizeof(float);
    w.bytes = off;
    return w;
}

size_t attn_ws_needed(long long rows, int S, int R, int D) {
    if (S == 1) return align256(16 + (size_t)rows * sizeof(int));
    return attn_ws_layout(nullptr, rows, S, R, D).bytes;
}

}  // namespace
}  // namespace spd

using namespace spd;

SPD_API int32_t spd_version(void) { return 100; }

SPD_API const char* spd_last_error(void) { return g_err.c_str(); }

SPD_API spd_status spd_set_wait_limit_ns(uint64_t ns) {
    if (ns == 0) return fail(SPD_ERR_INVALID_ARG, "wait limit 0");
    g_wait_ns.store(ns, std::memory_order_relaxed);
    return SPD_OK;
}

SPD_API uint64_t spd_wait_limit_ns(void) { return wait_limit_ns(); }

SPD_API spd_status spd_device_status(uint32_t* out, int32_t clear) {
    if (!out) return fail(SPD_ERR_INVALID_ARG, "out is NULL");
    spd_status st = SPD_OK;
    DevInfo* d = dev_info(&st);
    if (!d) return st;
    unsigned v = 0;
    cudaError_t e = cudaMemcpy(&v, d->status, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
    *out = v;
    if (clear) {
        e = cudaMemset(d->status, 0, sizeof(unsigned));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device status");
    }
    return SPD_OK;
}

SPD_API size_t spd_score_select_workspace_size(const spd_dims* dims) {
    if (check_dims(dims) != SPD_OK) return 0;
    return score_ws_prefix(dims) + (size_t)dims->B * dims->H_kv * dims->max_pages_per_seq * sizeof(float);
}

SPD_API size_t spd_sparse_decode_workspace_size(const spd_dims* dims, int32_t k_max, int32_t num_splits) {
    if (check_dims(dims) != SPD_OK) return 0;
    if (k_max < 1) {
        fail(SPD_ERR_INVALID_ARG, "k_max < 1");
        return 0;
    }
    spd_status st = SPD_OK;
    DevInfo* d = dev_info(&st);
    if (!d) return 0;
    const int S = sparse_splits(dims, k_max, num_splits, d->sms);
    return attn_ws_layout(nullptr, (long long)dims->B * dims->H_kv, S, dims->H_q / dims->H_kv, dims->D).bytes;
}

SPD_API size_t spd_dense_verify_workspace_size(const spd_dims* dims, int32_t T, int32_t num_splits) {
    if (check_dims(dims) != SPD_OK) return 0;
    if (T < 1 || T * (dims->H_q / dims->H_kv) > 64) {
        fail(SPD_ERR_UNSUPPORTED, "T=%d with G=%d (need 1 <= T and T*G <= 64)", T, dims->H_q / dims->H_kv);
        return 0;
    }
    spd_status st = SPD_OK;
    DevInfo* d = dev_info(&st);
    if (!d) return 0;
    const int S = dense_splits(dims, T, num_splits, d->sms);
    return attn_ws_layout(nullptr, (long long)dims->B * dims->H_kv, S, T * (dims->H_q / dims->H_kv), dims->D).bytes;
}

SPD_API spd_status pages_summarize(const spd_dims* dims, const spd_bf16* K, const int32_t* page_table,
                                   const int32_t* seq_lens, const int32_t* only_pages, int32_t n_only,
                                   spd_bf16* summ, void* stream) {
    spd_status st = check_dims(dims);
    if (st != SPD_OK) return st;
    if (dims->B == 0 || (only_pages && n_only == 0)) return SPD_OK;
    if (!K || !page_table || !seq_lens || !summ) return fail(SPD_ERR_INVALID_ARG, "NULL pointer argument");
    if (only_pages && n_only < 0) return fail(SPD_ERR_INVALID_ARG, "n_only < 0");
    if (!aligned16(K) || !aligned16(summ)) return fail(SPD_ERR_INVALID_ARG, "K and summ must be 16-byte aligned");
    DevInfo* d = dev_info(&st);
    if (!d) return st;
    SummarizeArgs a;
    a.K = K;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.only_pages = only_pages;
    a.n_only = n_only;
    a.summ = summ;
    a.B = dims->B;
    a.H_kv = dims->H_kv;
    a.D = dims->D;
    a.ps = dims->page_size;
    a.max_pages = dims->max_pages_per_seq;
    a.num_phys = dims->num_phys_pages;
    a.status = d->status;
    cudaError_t e = launch_summarize(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPD_OK : cuda_fail(e, "pages_summarize launch");
}

SPD_API spd_status kv_append_refresh(const spd_dims* dims, int32_t T, spd_bf16* K, spd_bf16* V,
                                     const int32_t* page_table, const int32_t* seq_lens,
                                     const spd_bf16* k_new, const spd_bf16* v_new, spd_bf16* summ,
                                     void* stream) {
    spd_status st = check_dims(dims);
    if (st != SPD_OK) return st;
    if (T < 1 || T > 4096) return fail(SPD_ERR_INVALID_ARG, "T = %d outside [1, 4096]", T);
    if (dims->B == 0) return SPD_OK;
    if (!K || !V || !page_table || !seq_lens || !k_new || !v_new || !summ)
        return fail(SPD_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(K) || !aligned16(V) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(summ))
        return fail(SPD_ERR_INVALID_ARG, "K, V, k_new, v_new and summ must be 16-byte aligned");
    DevInfo* d = dev_info(&st);
    if (!d) return st;
    AppendArgs a;
    a.K = K;
    a.V = V;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.k_new = k_new;
    a.v_new = v_new;
    a.summ = summ;
    a.B = dims->B;
    a.T = T;
    a.H_kv = dims->H_kv;
    a.D = dims->D;
    a.ps = dims->page_size;
    a.max_pages = dims->max_pages_per_seq;
    a.num_phys = dims->num_phys_pages;
    a.status = d->status;
    cudaError_t e = launch_append_refresh(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPD_OK : cuda_fail(e, "kv_append_refresh launch");
}

SPD_API spd_status spec_accept(int32_t B, int32_t k, int32_t n_vocab, const float* p_draft,
                               const float* q_target, const int32_t* draft, const float* u_acc,
                               const float* u_res, int32_t* n_accepted, int32_t* tokens, void* stream) {
    if (B < 0) return fail(SPD_ERR_INVALID_ARG, "B < 0");
    if (k < 1 || k > 32) return fail(SPD_ERR_UNSUPPORTED, "k = %d outside [1, 32]", k);
    if (n_vocab < 1 || n_vocab > (1 << 21)) return fail(SPD_ERR_UNSUPPORTED, "n_vocab = %d outside [1, 2^21]", n_vocab);
    if (B == 0) return SPD_OK;
    if (!p_draft || !q_target || !draft || !u_acc || !u_res || !n_accepted || !tokens)
        return fail(SPD_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(p_draft) || !aligned16(q_target))
        return fail(SPD_ERR_INVALID_ARG, "p_draft and q_target must be 16-byte aligned");
    spd_status st;
    DevInfo* d = dev_info(&st);
    if (!d) return st;
    SpecArgs a;
    a.p = p_draft;
    a.q = q_target;
    a.draft = draft;
    a.u_acc = u_acc;
    a.u_res = u_res;
    a.n_accepted = n_accepted;
    a.tokens = tokens;
    a.B = B;
    a.k = k;
    a.n = n_vocab;
    a.status = d->status;
    a.wait_ns = wait_limit_ns();
    cudaError_t e = launch_spec_accept(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPD_OK : cuda_fail(e, "spec_accept launch");
}

static spd_status score_select_setup(const spd_dims* dims, const spd_bf16* q, const spd_bf16* summ,
                                     const int32_t* seq_lens, const spd_budget_policy* policy, int32_t* sel,
                                     int32_t* nsel, int32_t k_max, float* scores, void* ws, size_t ws_bytes,
                                     ScoreSelectArgs& a, DevInfo** dev) {
    spd_status st = check_dims(dims);
    if (st != SPD_OK) return st;
    if (!policy) return fail(SPD_ERR_INVALID_ARG, "policy is NULL");
    const spd_budget_policy& p = *policy;
    if (p.mode < 0 || p.mode > 3) return fail(SPD_ERR_INVALID_ARG, "unknown budget mode %d", p.mode);
    if (p.mode == SPD_BUDGET_TOP_P &&
        (!(p.top_p >= 0.f && p.top_p <= 1.f) || !(p.score_scale > 0.f) || !(p.score_scale < 1e30f)))
        return fail(SPD_ERR_INVALID_ARG, "top_p must be in [0, 1] and score_scale > 0 and finite");
    if (p.sink_pages < 0 || p.local_pages < 0) return fail(SPD_ERR_INVALID_ARG, "negative sink/local pages");
    if (p.mode == SPD_BUDGET_FIXED_PAGES && p.fixed_pages < 0) return fail(SPD_ERR_INVALID_ARG, "fixed_pages < 0");
    if (p.mode == SPD_BUDGET_LINEAR_TOKENS && (p.slope_den <= 0 || p.slope_num < 0 || p.min_tokens < 0))
        return fail(SPD_ERR_INVALID_ARG, "bad linear budget parameters");
    if (p.mode == SPD_BUDGET_FRACTION && (p.frac_den <= 0 || p.frac_num < 0))
        return fail(SPD_ERR_INVALID_ARG, "bad fraction budget parameters");
    if (k_max < 1 || (long long)k_max < (long long)p.sink_pages + p.local_pages)
        return fail(SPD_ERR_INVALID_ARG, "k_max (%d) must be >= 1 and >= sink_pages + local_pages", k_max);
    if (dims->max_pages_per_seq > 32768)
        return fail(SPD_ERR_UNSUPPORTED, "max_pages_per_seq %d > 32768", dims->max_pages_per_seq);
    if (dims->B > 16384) return fail(SPD_ERR_UNSUPPORTED, "pages_score_select supports B <= 16384");
    if (dims->B == 0) return SPD_OK;
    if (!q || !summ || !seq_lens || !sel || !nsel)
        return fail(SPD_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(q) || !aligned16(summ)) return fail(SPD_ERR_INVALID_ARG, "q and summ must be 16-byte aligned");
    const size_t need = spd_score_select_workspace_size(dims);
    if (!ws || ws_bytes < need) return fail(SPD_ERR_WORKSPACE, "workspace %zu bytes < %zu", ws_bytes, need);
    if (!aligned16(ws)) return fail(SPD_ERR_INVALID_ARG, "ws must be 16-byte aligned");
    DevInfo* d = dev_info(&st);
    if (!d) return st;
    a = ScoreSelectArgs{};
    a.q = q;
    a.summ = summ;
    a.seq_lens = seq_lens;
    a.pol = p;
    a.sel = sel;
    a.nsel = nsel;
    a.k_max = k_max;
    a.scores = scores ? scores : reinterpret_cast<float*>(static_cast<char*>(ws) + score_ws_prefix(dims));
    a.B = dims->B;
    a.H_q = dims->H_q;
    a.H_kv = dims->H_kv;
    a.D = dims->D;
    a.ps = dims->page_size;
    a.max_pages = dims->max_pages_per_seq;
    a.num_phys = dims->num_phys_pages;
    a.status = d->status;
    a.wait_ns = wait_limit_ns();
    *dev = d;
    return SPD_OK;
}

SPD_API spd_status pages_score_select(const spd_dims* dims, const spd_bf16* q, const spd_bf16* summ,
                                      const int32_t* seq_lens,
                                      const spd_budget_policy* policy, int32_t* sel, int32_t* nsel, int32_t k_max,
                                      float* scores, void* ws, size_t ws_bytes, void* stream) {
    ScoreSelectArgs a;
    DevInfo* d = nullptr;
    spd_status st = score_select_setup(dims, q, summ, seq_lens, policy, sel, nsel, k_max, scores, ws, ws_bytes, a, &d);
    if (st != SPD_OK || dims->B == 0) return st;
    cudaError_t e = launch_score_select(a, d->sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPD_OK : cuda_fail(e, "pages_score_select launch");
}

SPD_API spd_status pages_append_score_select(const spd_dims* dims, spd_bf16* K, spd_bf16* V,
                                             const int32_t* page_table, const int32_t* seq_lens,
                                             const spd_bf16* k_new, const spd_bf16* v_new, const spd_bf16* q,
                                             spd_bf16* summ, const spd_budget_policy* policy, int32_t* sel,
                                             int32_t* nsel, int32_t k_max, float* scores, void* ws,
                                             size_t ws_bytes, void* stream) {
    ScoreSelectArgs a;
    DevInfo* d = nullptr;
    spd_status st = score_select_setup(dims, q, summ, seq_lens, policy, sel, nsel, k_max, scores, ws, ws_bytes, a, &d);
    if (st != SPD_OK || dims->B == 0) return st;
    if (!K || !V || !page_table || !k_new || !v_new) return fail(SPD_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(K) || !aligned16(V) || !aligned16(k_new) || !aligned16(v_new))
        return fail(SPD_ERR_INVALID_ARG, "K, V, k_new and v_new must be 16-byte aligned");
    a.K = K;
    a.V = V;
    a.page_table = page_table;
    a.k_new = k_new;
    a.v_new = v_new;
    a.summ_w = summ;
    cudaError_t e = launch_score_select(a, d->sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPD_OK : cuda_fail(e, "pages_append_score_select launch");
}

static spd_status attn_common(const spd_dims* dims, const spd_bf16* q, const spd_bf16* K, const spd_bf16* V,
                              const int32_t* page_table, const int32_t* seq_lens, spd_bf16* o) {
    if (!q || !K || !V || !page_table || !seq_lens || !o) return fail(SPD_ERR_INVALID_ARG, "NULL pointer argument");
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(o))
        return fail(SPD_ERR_INVALID_ARG, "q, K, V and o must be 16-byte aligned");
    if (dims->num_phys_pages < 1) return fail(SPD_ERR_INVALID_ARG, "num_phys_pages < 1");
    return SPD_OK;
}

// Validates and launches the sparse attention kernel with S units per row (S >= 1
// already chosen); sel_done != NULL chains it behind the selection of each row.
static spd_status sparse_attn_launch(const spd_dims* dims, const spd_bf16* q, const spd_bf16* K, const spd_bf16* V,
                                     const int32_t* page_table, const int32_t* seq_lens, const int32_t* sel,
                                     const int32_t* nsel, int32_t k_max, int S, float softmax_scale, spd_bf16* o,
                                     float* lse, void* ws, size_t ws_bytes, unsigned* sel_done,
                                     const int32_t* sel_phys, DevInfo* d, void* stream) {
    spd_status st;
    const int G = dims->H_q / dims->H_kv;
    const long long rows = (long long)dims->B * dims->H_kv;
    AttnWs w = attn_ws_layout(ws, rows, S, G, dims->D);
    const size_t need = attn_ws_needed(rows, S, G, dims->D);
    if (!ws || ws_bytes < need) return fail(SPD_ERR_WORKSPACE, "workspace %zu bytes < %zu", ws_bytes, need);
    if (!aligned16(ws)) return fail(SPD_ERR_INVALID_ARG, "ws must be 16-byte aligned");
    CUtensorMap tk, tv;
    if ((st = kv_map(&tk, K, dims)) != SPD_OK || (st = kv_map(&tv, V, dims)) != SPD_OK) return st;
    AttnArgs a{};
    a.q = q;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.sel = sel;
    a.nsel = nsel;
    a.k_max = k_max;
    a.B = dims->B;
    a.H_q = dims->H_q;
    a.H_kv = dims->H_kv;
    a.D = dims->D;
    a.ps = dims->page_size;
    a.max_pages = dims->max_pages_per_seq;
    a.T = 1;
    a.num_phys = dims->num_phys_pages;
    a.items_per_split = (k_max + S - 1) / S;
    a.num_splits = S;
    a.scale_log2 = softmax_scale * kLog2e;
    a.o = o;
    a.lse = lse;
    a.part_o = w.part_o;
    a.part_lse = w.part_lse;
    a.counters = w.counters;
    a.queue = w.queue;
    a.num_sms = d->sms;
    a.status = d->status;
    a.wait_ns = wait_limit_ns();
    a.sel_done = sel_done;
    a.sel_phys = sel_phys;
    cudaError_t e = launch_sparse_attn(a, tk, tv, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPD_OK : cuda_fail(e, "sparse attention launch");
}

SPD_API spd_status sparse_decode_attn(const spd_dims* dims, const spd_bf16* q, const spd_bf16* K,
                                      const spd_bf16* V, const int32_t* page_table, const int32_t* seq_lens,
                                      const int32_t* sel, const int32_t* nsel, int32_t k_max, int32_t num_splits,
                                      float softmax_scale, spd_bf16* o, float* lse, void* ws, size_t ws_bytes,
                                      void* stream) {
    spd_status st = check_dims(dims);
    if (st != SPD_OK) return st;
    if (k_max < 1) return fail(SPD_ERR_INVALID_ARG, "k_max < 1");
    if (num_splits < 0) return fail(SPD_ERR_INVALID_ARG, "num_splits < 0");
    if (dims->B == 0) return SPD_OK;
    if ((st = attn_common(dims, q, K, V, page_table, seq_lens, o)) != SPD_OK) return st;
    if (!sel || !nsel) return fail(SPD_ERR_INVALID_ARG, "NULL selection");
    DevInfo* d = dev_info(&st);
    if (!d) return st;
    return sparse_attn_launch(dims, q, K, V, page_table, seq_lens, sel, nsel, k_max,
                              sparse_splits(dims, k_max, num_splits, d->sms), softmax_scale, o, lse, ws, ws_bytes,
                              nullptr, nullptr, d, stream);
}

// The chained step's workspace: [score / select][chain: two tile counters, warps
// done, selection claims, tiles_done[rows], sel_done[rows], (256-aligned) keys[rows][max_pages],
// (256-aligned) sel_phys[rows][k_max]][attention].
struct StepWs {
    size_t score, chain, keys, phys, attn, bytes;
};

// The chained selection also writes each selected page's physical page (from a copy
// of the row's page table in shared memory) when that copy fits comfortably.
static bool step_sel_phys(const spd_dims* dims, const spd_budget_policy* policy) {
    const size_t words = ((size_t)dims->max_pages_per_seq + 31) / 32;
    const size_t per = (policy && policy->mode == SPD_BUDGET_TOP_P) ? 3 : 2;
    return ((size_t)dims->max_pages_per_seq * per + 2 * words) * sizeof(uint32_t) <= 96 * 1024;
}

static bool step_ws_layout(const spd_dims* dims, int32_t k_max, StepWs* w, DevInfo* d) {
    const long long rows = (long long)dims->B * dims->H_kv;
    const int S = sparse_splits(dims, k_max, 0, d->sms);
    w->score = align256(spd_score_select_workspace_size(dims));
    w->keys = align256(32 + 2 * (size_t)rows * sizeof(unsigned));  // offset of the keys in the chain part
    w->phys = w->keys + align256((size_t)rows * dims->max_pages_per_seq * sizeof(unsigned));
    w->chain = w->phys + align256((size_t)rows * k_max * sizeof(int32_t));
    w->attn = attn_ws_layout(nullptr, rows, S, dims->H_q / dims->H_kv, dims->D).bytes;
    w->bytes = w->score + w->chain + w->attn;
    return w->score != 0;
}

SPD_API size_t spd_sparse_decode_step_workspace_size(const spd_dims* dims, int32_t k_max) {
    if (check_dims(dims) != SPD_OK) return 0;
    if (k_max < 1) {
        fail(SPD_ERR_INVALID_ARG, "k_max < 1");
        return 0;
    }
    spd_status st = SPD_OK;
    DevInfo* d = dev_info(&st);
    if (!d) return 0;
    StepWs w;
    return step_ws_layout(dims, k_max, &w, d) ? w.bytes : 0;
}

SPD_API spd_status sparse_decode_step(const spd_dims* dims, spd_bf16* K, spd_bf16* V, const int32_t* page_table,
                                      const int32_t* seq_lens, const spd_bf16* k_new, const spd_bf16* v_new,
                                      const spd_bf16* q, spd_bf16* summ, const spd_budget_policy* policy,
                                      int32_t* sel, int32_t* nsel, int32_t k_max, float softmax_scale,
                                      spd_bf16* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
    spd_status st = check_dims(dims);
    if (st != SPD_OK) return st;
    if (k_max < 1) return fail(SPD_ERR_INVALID_ARG, "k_max < 1");
    if (dims->B == 0) return SPD_OK;
    if ((k_new == nullptr) != (v_new == nullptr)) return fail(SPD_ERR_INVALID_ARG, "k_new and v_new: both or neither");
    if ((st = attn_common(dims, q, K, V, page_table, seq_lens, o)) != SPD_OK) return st;
    DevInfo* d = dev_info(&st);
    if (!d) return st;
    StepWs w;
    if (!step_ws_layout(dims, k_max, &w, d)) return fail(SPD_ERR_INVALID_ARG, "bad dims");
    if (!ws || ws_bytes < w.bytes) return fail(SPD_ERR_WORKSPACE, "workspace %zu bytes < %zu", ws_bytes, w.bytes);
    if (!aligned16(ws)) return fail(SPD_ERR_INVALID_ARG, "ws must be 16-byte aligned");
    char* base = static_cast<char*>(ws);
    ScoreSelectArgs a;
    DevInfo* d2 = nullptr;
    st = score_select_setup(dims, q, summ, seq_lens, policy, sel, nsel, k_max, nullptr, base, w.score, a, &d2);
    if (st != SPD_OK) return st;
    if (k_new) {
        if (!aligned16(k_new) || !aligned16(v_new)) return fail(SPD_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
        a.K = K;
        a.V = V;
        a.page_table = page_table;
        a.k_new = k_new;
        a.v_new = v_new;
        a.summ_w = summ;
    }
    // Chained row by row: the selection of a row starts as soon as its tiles are
    // scored, and each of its attention units as soon as it is selected.
    const int S = sparse_splits(dims, k_max, 0, d->sms);
    char* chain = base + w.score;
    const long long rows = (long long)dims->B * dims->H_kv;
    a.tile_ctr = reinterpret_cast<unsigned long long*>(chain);
    a.warps_done = reinterpret_cast<unsigned*>(chain + 16);
    a.sel_claims = reinterpret_cast<unsigned*>(chain + 20);
    a.tiles_done = reinterpret_cast<unsigned*>(chain + 32);
    a.sel_done = a.tiles_done + rows;
    a.keys = reinterpret_cast<unsigned*>(chain + w.keys);
    if (step_sel_phys(dims, policy)) {
        a.page_table = page_table;
        a.sel_phys = reinterpret_cast<int32_t*>(chain + w.phys);
    }
    unsigned* sel_done = a.sel_done;
    cudaError_t e = launch_score_select(a, d->sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse_decode_step scoring launch");
    return sparse_attn_launch(dims, q, K, V, page_table, seq_lens, sel, nsel, k_max, S, softmax_scale, o, lse,
                              base + w.score + w.chain, w.attn, sel_done, a.sel_phys, d, stream);
}

SPD_API spd_status dense_verify_attn(const spd_dims* dims, int32_t T, const spd_bf16* q, const spd_bf16* K,
                                     const spd_bf16* V, const int32_t* page_table, const int32_t* seq_lens,
                                     int32_t num_splits, float softmax_scale, spd_bf16* o, float* lse, void* ws,
                                     size_t ws_bytes, void* stream) {
    spd_status st = check_dims(dims);
    if (st != SPD_OK) return st;
    const int G = dims->H_q / dims->H_kv;
    if (T < 1 || T * G > 64) return fail(SPD_ERR_UNSUPPORTED, "T=%d with G=%d (need 1 <= T and T*G <= 64)", T, G);
    if (num_splits < 0) return fail(SPD_ERR_INVALID_ARG, "num_splits < 0");
    if (dims->B == 0) return SPD_OK;
    if ((st = attn_common(dims, q, K, V, page_table, seq_lens, o)) != SPD_OK) return st;
    DevInfo* d = dev_info(&st);
    if (!d) return st;
    const int S = dense_splits(dims, T, num_splits, d->sms);
    const long long rows = (long long)dims->B * dims->H_kv;
    AttnWs w = attn_ws_layout(ws, rows, S, T * G, dims->D);
    if (!ws || ws_bytes < w.bytes) return fail(SPD_ERR_WORKSPACE, "workspace %zu bytes < %zu", ws_bytes, w.bytes);
    if (!aligned16(ws)) return fail(SPD_ERR_INVALID_ARG, "ws must be 16-byte aligned");
    CUtensorMap tk, tv;
    if ((st = kv_map(&tk, K, dims)) != SPD_OK || (st = kv_map(&tv, V, dims)) != SPD_OK) return st;
    AttnArgs a{};
    a.q = q;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.sel = nullptr;
    a.nsel = nullptr;
    a.k_max = 0;
    a.B = dims->B;
    a.H_q = dims->H_q;
    a.H_kv = dims->H_kv;
    a.D = dims->D;
    a.ps = dims->page_size;
    a.max_pages = dims->max_pages_per_seq;
    a.T = T;
    a.num_phys = dims->num_phys_pages;
    a.items_per_split = (dims->max_pages_per_seq + S - 1) / S;
    a.num_splits = S;
    a.scale_log2 = softmax_scale * kLog2e;
    a.o = o;
    a.lse = lse;
    a.part_o = w.part_o;
    a.part_lse = w.part_lse;
    a.counters = w.counters;
    a.queue = w.queue;
    a.num_sms = d->sms;
    a.status = d->status;
    a.wait_ns = wait_limit_ns();
    cudaError_t e = launch_dense_attn(a, tk, tv, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPD_OK : cuda_fail(e, "dense_verify_attn launch");
}

SPD_API spd_status lse_merge(int32_t S, int32_t rows, int32_t D, const float* part_o, const float* part_lse,
                             spd_bf16* o, float* lse, void* stream) {
    if (S < 1 || rows < 0) return fail(SPD_ERR_INVALID_ARG, "bad S (%d) or rows (%d)", S, rows);
    if (D != 64 && D != 128) return fail(SPD_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", D);
    if (rows == 0) return SPD_OK;
    if (!part_o || !part_lse || !o) return fail(SPD_ERR_INVALID_ARG, "NULL pointer argument");
    cudaError_t e = launch_lse_merge(S, rows, D, part_o, part_lse, o, lse, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPD_OK : cuda_fail(e, "lse_merge launch");
}

// ---------------------------------------------------------------------------
// sparse_decode_attn_noalloc: the same launch with its scratch in a fixed
// device array instead of a caller workspace (see include/spd.h).

namespace spd {
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SPD_NOALLOC_SCRATCH_BYTES];

struct NoAllocDev {
    std::once_flag once;
    void* ptr = nullptr;
    cudaError_t err = cudaSuccess;
};
NoAllocDev g_noalloc[kMaxDevices];

// Device address of the fixed scratch array for the current device (looked up
// once per device; in host code the array's name is only a host-side handle).
void* noalloc_scratch(spd_status* st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *st = cuda_fail(e, "cudaGetDevice");
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *st = fail(SPD_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
        return nullptr;
    }
    NoAllocDev* n = &g_noalloc[dev];
    std::call_once(n->once, [n]() { n->err = cudaGetSymbolAddress(&n->ptr, g_noalloc_scratch); });
    if (n->err != cudaSuccess || !n->ptr) {
        *st = cuda_fail(n->err, "looking up the fixed scratch array");
        return nullptr;
    }
    return n->ptr;
}

}  // namespace
}  // namespace spd

SPD_API spd_status sparse_decode_attn_noalloc(const spd_dims* dims, const spd_bf16* q, const spd_bf16* K,
                                              const spd_bf16* V, const int32_t* page_table, const int32_t* seq_lens,
                                              const int32_t* sel, const int32_t* nsel, int32_t k_max,
                                              int32_t num_splits, float softmax_scale, spd_bf16* o, float* lse,
                                              void* stream) {
    spd_status st = check_dims(dims);
    if (st != SPD_OK) return st;
    if (k_max < 1) return fail(SPD_ERR_INVALID_ARG, "k_max < 1");
    if (num_splits < 0) return fail(SPD_ERR_INVALID_ARG, "num_splits < 0");
    if (dims->B == 0) return SPD_OK;
    if ((st = attn_common(dims, q, K, V, page_table, seq_lens, o)) != SPD_OK) return st;
    if (!sel || !nsel) return fail(SPD_ERR_INVALID_ARG, "NULL selection");
    DevInfo* d = dev_info(&st);
    if (!d) return st;
    void* scratch = noalloc_scratch(&st);
    if (!scratch) return st;
    const int G = dims->H_q / dims->H_kv;
    const long long rows = (long long)dims->B * dims->H_kv;
    int S = sparse_splits(dims, k_max, num_splits, d->sms);
    if (num_splits == 0) {
        // automatic: the usual split count, or fewer until the partials fit
        while (S > 1 && attn_ws_needed(rows, S, G, dims->D) > SPD_NOALLOC_SCRATCH_BYTES)
            S = sparse_splits(dims, k_max, S - 1, d->sms);
    }
    const size_t need = attn_ws_needed(rows, S, G, dims->D);
    if (need > SPD_NOALLOC_SCRATCH_BYTES)
        return fail(SPD_ERR_UNSUPPORTED,
                    "sparse_decode_attn_noalloc needs %zu bytes of scratch for %d split(s); the fixed array holds %zu",
                    need, S, (size_t)SPD_NOALLOC_SCRATCH_BYTES);
    // the queue and the split tickets must start at zero
    const AttnWs w = attn_ws_layout(scratch, rows, S, G, dims->D);
    const size_t zero_bytes = reinterpret_cast<char*>(w.part_lse) - static_cast<char*>(scratch);
    cudaError_t e = cudaMemsetAsync(scratch, 0, zero_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the fixed scratch array");
    return sparse_attn_launch(dims, q, K, V, page_table, seq_lens, sel, nsel, k_max, S, softmax_scale, o, lse,
                              scratch, SPD_NOALLOC_SCRATCH_BYTES, nullptr, nullptr, d, stream);
}
