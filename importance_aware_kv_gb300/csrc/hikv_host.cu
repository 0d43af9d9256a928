// Host side of the hikv C ABI: argument checks, the exact host mirror of each
// unit's length and mapped pages, device allocation, and kernel launches.
// Nothing here synchronises the device except create/destroy/device_status.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <numeric>
#include <queue>
#include <string>
#include <vector>

#include "../../include/hikv.h"
#include "hikv_internal.cuh"

namespace hikv {
size_t window_smem_bytes(int d, int nqv);
}

using namespace hikv;

namespace {

// NVTX range around an entry point (seen by nsys / ncu timelines; a no-op
// when no tool is attached)
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

}  // namespace

namespace {

thread_local std::string g_err;

}  // namespace

namespace hikv {
// lets other translation units of the library report through hikv_last_error()
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace hikv

namespace {

hikv_status fail(hikv_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

hikv_status cuda_fail(cudaError_t e, const char* what) {
    return fail(HIKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kWindowChunk = 1024;   // tokens per CTA of the window-scoring kernels

// cuTensorMapEncodeTiled from the driver, found through the runtime (no
// link-time dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

struct hikv_cache {
    // configuration
    int L = 0, B = 0, Hq = 0, Hkv = 0, G = 0, d = 0, dtype = 0, esz = 0;
    int S = 0, W = 0, cap = 0, P = 0, page_shift = 0, max_pages = 0, max_wq = 0;
    int units = 0, per_layer = 0;
    int64_t pool_pages = 0;
    float scale = 0.f;
    std::vector<int32_t> budget_unit;   // [units]
    // device
    int device = 0, sm_count = 0;
    size_t smem_optin = 0;
    int max_smem_chunk = 0;             // decode smem path limit (tokens per CTA)
    int dec_occ = 2;                    // decode CTAs per SM
    View v{};
    int32_t* d_append_base = nullptr;
    float* d_logits = nullptr;          // long-chunk decode logits (may be null)
    unsigned long long* d_cand = nullptr;
    int32_t* d_cand_slot = nullptr;
    int32_t* d_holes = nullptr;
    int64_t* d_hole_off = nullptr;
    float* d_wpart = nullptr;
    int wchunks = 0;
    int32_t* d_order_all = nullptr;
    int32_t* d_order_layer = nullptr;
    std::vector<int32_t> order_all, order_layer;   // host copies: units by budget, descending
    // balanced unit-to-cluster assignment of ragged decode calls (device copy
    // [units] list + [clusters + 1] offsets), recomputed when its inputs change
    // Device layout: [units] lists (a call over units [u0, u0 + nu) keeps its
    // list at [u0, ...)) + per first layer of a call an offsets region, so the
    // per-layer calls of a step each keep theirs and re-upload nothing while
    // their lengths repeat.
    int32_t* d_assign = nullptr;        // clusters: [units] + [L][max clusters + 1]
    std::vector<int32_t> asg;
    std::vector<uint64_t> asg_key;      // [L]
    // the same for the warp-per-unit kernel's per-warp unit lists
    int32_t* d_sassign = nullptr;       // [units] + [L][4 * max CTAs + 1]
    std::vector<int32_t> sasg;
    std::vector<uint64_t> sasg_key;     // [L]
    int small_mode = 1;                 // HIKV_DECODE_SMALL (tuning): 0 never, 1 auto, 2 always when eligible
    int first_burst = 4;                // one tile per consumer warp first (HIKV_DECODE_BURST: tuning)
    int prefetch_override = -1;         // HIKV_DECODE_PREFETCH (tuning): L2 prefetch distance in tiles, -1 auto
    CUtensorMap tmap;                   // the pool as rows of d elements, 16 x 128-byte swizzled boxes
    std::vector<void*> allocs;
    // host mirror
    std::vector<int32_t> len, next_pos, mapped;
    std::vector<uint8_t> fresh;         // decode ran since the last state change
    int64_t pages_in_use = 0;
    int cs_override = 0;                // HIKV_DECODE_CS (tuning)
    int64_t launches = 0;               // kernels launched through this cache
    // the cluster launches of the latest decode call (at most two): units,
    // cluster size, clusters, logits in shared memory
    int32_t last_cfg[2][4] = {};
    int last_ncfg = 0;
    int pool_k = 0;                     // SnapKV pooling of the prompt scores (> 1: on)
    // HiKV Stage II element-level decode (elem > 0: on)
    int elem = 0;
    int elem_stride = 0;                // row stride of its order / logit buffers
    int32_t* d_eorder = nullptr;        // [units][elem_stride]
    float* d_elg = nullptr;             // [units][G][elem_stride]
    float* d_epart = nullptr;           // [units][max spans][G][d + 2]
    unsigned long long* d_erows = nullptr;   // V rows the element-level steps read
    float* d_eqmask = nullptr;          // [units][G][d]
    int32_t* d_edone = nullptr;         // [units]
    // HiKV banded prefill scores (band_scoring): one layer's per-query softmax statistics
    float2* d_band = nullptr;           // [per_layer][G][cap]
    // Programmatic dependent launch: the units [pdl_lo, pdl_hi) the latest
    // kernel this cache launched may write, and its stream (pdl_valid: that
    // latest launch is known); a decode launch on disjoint units of the same
    // stream may load its pages before waiting for it
    bool pdl_on = true;                 // HIKV_PDL=0 (tuning) turns it off
    bool pdl_valid = false;
    int pdl_lo = 0, pdl_hi = 0;
    hikv_stream_t pdl_stream = nullptr;
};

namespace {

// HIKV_FAULT_ALLOC_AT=n makes the n-th device allocation of a create (from
// 1) fail, to test the cleanup path without exhausting the device
int fault_alloc_at() {
    const char* e = std::getenv("HIKV_FAULT_ALLOC_AT");
    return e ? std::atoi(e) : 0;
}

template <class T>
cudaError_t dalloc(hikv_cache* c, T** p, size_t count) {
    *p = nullptr;
    if (count == 0) count = 1;
    if (fault_alloc_at() > 0 && (int)c->allocs.size() + 1 == fault_alloc_at()) return cudaErrorMemoryAllocation;
    cudaError_t e = cudaMalloc((void**)p, count * sizeof(T));
    if (e == cudaSuccess) c->allocs.push_back(*p);
    return e;
}

void free_all(hikv_cache* c) {
    for (void* p : c->allocs) cudaFree(p);
    c->allocs.clear();
}

// Programmatic dependent launch bookkeeping (see hikv_cache::pdl_*): a launch
// of units [lo, hi) on `stream`; pdl_forget() when an entry point launches
// kernels that do not record their units.
void pdl_record(hikv_cache* c, int lo, int hi, hikv_stream_t stream) {
    c->pdl_valid = true;
    c->pdl_lo = lo;
    c->pdl_hi = hi;
    c->pdl_stream = stream;
}
void pdl_forget(hikv_cache* c) { if (c) c->pdl_valid = false; }
bool pdl_disjoint(const hikv_cache* c, int lo, int hi, hikv_stream_t stream) {
    return c->pdl_on && c->pdl_valid && c->pdl_stream == stream && (hi <= c->pdl_lo || lo >= c->pdl_hi);
}

bool range_ok(const hikv_cache* c, int32_t layer0, int32_t nl) {
    return c && layer0 >= 0 && nl > 0 && layer0 + nl <= c->L;
}

int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

}  // namespace

extern "C" {

const char* hikv_last_error(void) { return g_err.c_str(); }

hikv_status hikv_create_cache(const hikv_config* cfg, hikv_cache** out) {
    g_err.clear();
    if (!cfg || !out) return fail(HIKV_ERR_INVALID_ARG, "create: null config or out pointer");
    *out = nullptr;
    const hikv_config& f = *cfg;
    if (f.num_layers <= 0 || f.batch <= 0 || f.num_q_heads <= 0 || f.num_kv_heads <= 0 ||
        f.head_dim <= 0 || f.max_tokens <= 0)
        return fail(HIKV_ERR_INVALID_ARG, "create: sizes must be positive");
    if (f.num_q_heads % f.num_kv_heads)
        return fail(HIKV_ERR_INVALID_ARG, "create: num_q_heads must be a multiple of num_kv_heads");
    const int G = f.num_q_heads / f.num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(HIKV_ERR_UNSUPPORTED, "create: group size %d not in {1,2,4,8}", G);
    if (f.head_dim != 64 && f.head_dim != 128)
        return fail(HIKV_ERR_UNSUPPORTED, "create: head_dim %d not in {64,128}", f.head_dim);
    if (f.dtype != HIKV_F32 && f.dtype != HIKV_BF16)
        return fail(HIKV_ERR_UNSUPPORTED, "create: dtype %d", f.dtype);
    if (f.num_sink < 0 || f.recent_window < 0)
        return fail(HIKV_ERR_INVALID_ARG, "create: negative sink or window");
    if (!f.budgets) return fail(HIKV_ERR_INVALID_ARG, "create: budgets is NULL");
    const int P = f.page_tokens ? f.page_tokens : 64;
    if (P < 16 || (P & (P - 1)))
        return fail(HIKV_ERR_INVALID_ARG, "create: page_tokens %d must be a power of two >= 16", P);
    if (f.pool_pages < 0) return fail(HIKV_ERR_INVALID_ARG, "create: negative pool_pages");
    if (f.max_window_queries < 0) return fail(HIKV_ERR_INVALID_ARG, "create: negative max_window_queries");
    if (!(f.scale >= 0.f) || !std::isfinite(f.scale)) return fail(HIKV_ERR_INVALID_ARG, "create: bad scale");
    if (f.importance_mode != 0 && f.importance_mode != 1)
        return fail(HIKV_ERR_INVALID_ARG, "create: importance_mode %d not in {0, 1}", f.importance_mode);
    if (f.element_budget < 0 || f.element_budget > f.head_dim)
        return fail(HIKV_ERR_INVALID_ARG, "create: element_budget %d not in [0, head_dim=%d]", f.element_budget,
                    f.head_dim);
    if (f.band_scoring != 0 && f.band_scoring != 1)
        return fail(HIKV_ERR_INVALID_ARG, "create: band_scoring %d not in {0, 1}", f.band_scoring);
    if (f.pool_kernel < 0 || f.pool_kernel > kMaxPoolKernel)
        return fail(HIKV_ERR_INVALID_ARG, "create: pool_kernel %d not in [0, %d]", f.pool_kernel, kMaxPoolKernel);
    const int64_t units64 = (int64_t)f.num_layers * f.batch * f.num_kv_heads;
    if (units64 > 65535) return fail(HIKV_ERR_UNSUPPORTED, "create: %lld units > 65535", (long long)units64);
    for (int i = 0; i < f.num_layers * f.num_kv_heads; ++i) {
        const int32_t b = f.budgets[i];
        if (b < 1 || b < f.num_sink + f.recent_window)
            return fail(HIKV_ERR_INVALID_ARG, "create: budget[%d]=%d must be >= max(1, S+W=%d)", i, b,
                        f.num_sink + f.recent_window);
    }

    hikv_cache* c = new hikv_cache();
    c->L = f.num_layers; c->B = f.batch; c->Hq = f.num_q_heads; c->Hkv = f.num_kv_heads;
    c->G = G; c->d = f.head_dim; c->dtype = f.dtype; c->esz = f.dtype == HIKV_BF16 ? 2 : 4;
    c->S = f.num_sink; c->W = f.recent_window; c->cap = f.max_tokens;
    c->P = P; c->page_shift = ilog2(P);
    c->max_pages = ceil_div(c->cap, P);
    c->max_wq = f.max_window_queries ? f.max_window_queries : 32;
    c->units = (int)units64;
    c->per_layer = c->B * c->Hkv;
    c->pool_pages = f.pool_pages ? f.pool_pages : (int64_t)c->units * c->max_pages;
    if (c->pool_pages > INT32_MAX) {
        delete c;
        return fail(HIKV_ERR_UNSUPPORTED, "create: pool of %lld pages too large", (long long)f.pool_pages);
    }
    c->scale = f.scale > 0.f ? f.scale : 1.0f / std::sqrt((float)c->d);
    c->pool_k = f.pool_kernel;
    c->elem = f.element_budget < f.head_dim ? f.element_budget : 0;
    c->budget_unit.resize(c->units);
    for (int u = 0; u < c->units; ++u)
        c->budget_unit[u] = f.budgets[(u / c->per_layer) * c->Hkv + u % c->Hkv];
    if (const char* e = std::getenv("HIKV_DECODE_CS")) c->cs_override = std::atoi(e);
    if (const char* e = std::getenv("HIKV_DECODE_SMALL")) c->small_mode = std::atoi(e);
    if (const char* e = std::getenv("HIKV_DECODE_BURST")) c->first_burst = std::atoi(e);
    if (const char* e = std::getenv("HIKV_DECODE_PREFETCH")) c->prefetch_override = std::atoi(e);
    if (const char* e = std::getenv("HIKV_PDL")) c->pdl_on = std::atoi(e) != 0;

    cudaError_t e = cudaGetDevice(&c->device);
    if (e != cudaSuccess) { delete c; return cuda_fail(e, "create: cudaGetDevice"); }
    cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device);
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
    c->smem_optin = (size_t)optin;
    // shared-memory logits path: chunks small enough for the decode occupancy
    // decode CTAs per SM, and the dynamic shared memory each may take at that
    // occupancy (228 KB per SM, 1 KB of it reserved per CTA)
    c->dec_occ = dec_occupancy(c->d * c->esz, c->G);
    c->max_smem_chunk = decode_max_smem_chunk(
        c->dtype, c->d, c->G, std::min<size_t>(c->smem_optin, (228 * 1024) / c->dec_occ - 1024));

    View& v = c->v;
    const int row_bytes = c->d * c->esz;
    v.row_bytes = row_bytes;
    v.page_bytes = 2LL * P * row_bytes;
    v.page_tokens = P; v.page_shift = c->page_shift; v.max_pages = c->max_pages; v.cap = c->cap;
    v.pool_pages = (int32_t)c->pool_pages; v.units = c->units;
    v.batch = c->B; v.hq = c->Hq; v.hkv = c->Hkv; v.group = G; v.d = c->d;
    v.sink = c->S; v.window = c->W;
    v.recent_only = f.importance_mode == 1;
    // Home pages: a pool that holds every unit's max_tokens at once (the
    // default) gives unit u the pages u * max_pages .. for good, so kernels
    // compute a slot's page instead of loading it, and appends and evictions
    // move no pages.  A smaller pool shares its pages through the free stack.
    v.home_pages = c->pool_pages >= (int64_t)c->units * c->max_pages ? 1 : 0;
    if (const char* e = std::getenv("HIKV_DEBUG")) v.debug = std::atoi(e) != 0 ? 1 : 0;

    const size_t U = (size_t)c->units;
    // hole lists: a unit cut from n <= cap to B leaves at most min(B, cap - B) holes
    std::vector<int64_t> hole_off(U);
    int64_t holes_total = 0;
    for (size_t u = 0; u < U; ++u) {
        hole_off[u] = holes_total;
        holes_total += std::max(0, std::min(c->budget_unit[u], c->cap - c->budget_unit[u]));
    }
    c->wchunks = ceil_div(c->cap, kWindowChunk);
    // the decode kernel's global logits (a CTA's chunk too large for shared
    // memory): always there (G floats a slot, 3-6 % of the K/V bytes at
    // d = 128 in bf16), so that the cluster size is chosen by cost, not by what fits
    // shared memory -- one CTA per unit with global logits beats two with
    // shared-memory logits on ragged budgets (HeadKV workload: 157 vs 183 us)
    const bool need_logits = true;

#define ALLOC(ptr, n)                                                       \
    if ((e = dalloc(c, &(ptr), (n))) != cudaSuccess) {                      \
        free_all(c);                                                        \
        delete c;                                                           \
        cudaGetLastError();                                                 \
        return fail(HIKV_ERR_OUT_OF_MEMORY, "create: cudaMalloc of " #ptr " failed: %s", cudaGetErrorString(e)); \
    }
    ALLOC(v.pool, (size_t)c->pool_pages * (size_t)v.page_bytes);
    ALLOC(v.page_table, U * c->max_pages);
    ALLOC(v.imp, U * c->cap);
    ALLOC(v.pos, U * c->cap);
    ALLOC(v.len, U);
    ALLOC(v.next_pos, U);
    ALLOC(v.mapped, U);
    ALLOC(v.victim, U);
    ALLOC(v.budget, U);
    ALLOC(v.free_stack, (size_t)c->pool_pages);
    ALLOC(v.free_top, 1);
    ALLOC(v.err, 8);   // [0] error bits, [1..5] where the first bounded wait gave up
    ALLOC(c->d_append_base, U);
    ALLOC(c->d_cand, U * kMaxCS);
    ALLOC(c->d_cand_slot, U * kMaxCS);
    ALLOC(c->d_holes, (size_t)holes_total);
    ALLOC(c->d_hole_off, U);
    ALLOC(c->d_wpart, U * c->wchunks * (size_t)c->max_wq * G * 2);
    ALLOC(c->d_order_all, U);
    ALLOC(c->d_order_layer, U);
    ALLOC(c->d_assign, U + (size_t)c->L * (c->dec_occ * c->sm_count + 1));
    ALLOC(c->d_sassign, U + (size_t)c->L * (kSmallWarps * c->dec_occ * c->sm_count + 1));
    c->asg_key.assign(c->L, 0);
    c->sasg_key.assign(c->L, 0);
    if (need_logits) ALLOC(c->d_logits, U * (size_t)c->cap * G);
    if (c->elem) {
        c->elem_stride = std::min(c->cap, elem_max_tokens());
        const int spans = ceil_div(c->elem_stride, elem_span_ranks());
        ALLOC(c->d_eorder, U * (size_t)c->elem_stride);
        ALLOC(c->d_elg, U * (size_t)G * c->elem_stride);
        ALLOC(c->d_epart, U * (size_t)spans * G * (c->d + 2));
        ALLOC(c->d_erows, 1);
        ALLOC(c->d_eqmask, U * (size_t)G * c->d);
        ALLOC(c->d_edone, U);
    }
    if (f.band_scoring) ALLOC(c->d_band, (size_t)c->per_layer * G * c->cap);
#undef ALLOC

    // TMA descriptor of the pool: [pool_pages * 2P rows][d elements], boxes of
    // 16 rows x 128 bytes with the 128-byte swizzle the decode kernel reads
    {
        const uint64_t rows = (uint64_t)c->pool_pages * 2 * P;
        auto enc = tensor_map_encoder();
        if (!enc || rows > 0xFFFFFFFFull) {
            free_all(c);
            delete c;
            return fail(enc ? HIKV_ERR_UNSUPPORTED : HIKV_ERR_CUDA,
                        enc ? "create: pool too large for one tensor map" : "create: cuTensorMapEncodeTiled unavailable");
        }
        cuuint64_t dims[2] = {(cuuint64_t)c->d, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
        cuuint32_t box[2] = {(cuuint32_t)(128 / c->esz), 16u};
        cuuint32_t estr[2] = {1u, 1u};
        CUresult r = enc(&c->tmap, c->dtype == HIKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                         2, v.pool, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            free_all(c);
            delete c;
            return fail(HIKV_ERR_CUDA, "create: cuTensorMapEncodeTiled failed (%d)", (int)r);
        }
    }

    // initial device state
    std::vector<int32_t> stack((size_t)c->pool_pages);
    std::iota(stack.begin(), stack.end(), 0);
    std::vector<int32_t> home_table, home_mapped;
    if (v.home_pages) {
        home_table.resize(U * (size_t)c->max_pages);
        std::iota(home_table.begin(), home_table.end(), 0);
        home_mapped.assign(U, c->max_pages);
    }
    std::vector<int32_t>& order_all = c->order_all;
    std::vector<int32_t>& order_layer = c->order_layer;
    order_all.resize(U);
    order_layer.resize(U);
    std::iota(order_all.begin(), order_all.end(), 0);
    std::stable_sort(order_all.begin(), order_all.end(),
                     [&](int a, int b) { return c->budget_unit[a] > c->budget_unit[b]; });
    for (int l = 0; l < c->L; ++l) {
        auto first = order_layer.begin() + (size_t)l * c->per_layer;
        std::iota(first, first + c->per_layer, l * c->per_layer);
        std::stable_sort(first, first + c->per_layer,
                         [&](int a, int b) { return c->budget_unit[a] > c->budget_unit[b]; });
    }
    const int32_t top = v.home_pages ? 0 : (int32_t)c->pool_pages;   // home pages: the stack stays empty
    const int32_t minus1 = -1;
    (void)minus1;
    bool ok = cudaMemset(v.page_table, 0xFF, U * c->max_pages * 4) == cudaSuccess &&
              cudaMemset(v.imp, 0, U * c->cap * 4) == cudaSuccess &&
              cudaMemset(v.pos, 0xFF, U * c->cap * 4) == cudaSuccess &&
              cudaMemset(v.len, 0, U * 4) == cudaSuccess &&
              cudaMemset(v.next_pos, 0, U * 4) == cudaSuccess &&
              cudaMemset(v.mapped, 0, U * 4) == cudaSuccess &&
              cudaMemset(v.victim, 0xFF, U * 4) == cudaSuccess &&
              cudaMemset(v.err, 0, 32) == cudaSuccess &&
              (!c->d_erows || cudaMemset(c->d_erows, 0, 8) == cudaSuccess) &&
              (!c->d_edone || cudaMemset(c->d_edone, 0, U * 4) == cudaSuccess) &&
              cudaMemcpy(v.budget, c->budget_unit.data(), U * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(v.free_stack, stack.data(), stack.size() * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(v.free_top, &top, 4, cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(c->d_hole_off, hole_off.data(), U * 8, cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(c->d_order_all, order_all.data(), U * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(c->d_order_layer, order_layer.data(), U * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
              (!v.home_pages ||
               (cudaMemcpy(v.page_table, home_table.data(), home_table.size() * 4, cudaMemcpyHostToDevice) ==
                    cudaSuccess &&
                cudaMemcpy(v.mapped, home_mapped.data(), U * 4, cudaMemcpyHostToDevice) == cudaSuccess)) &&
              cudaDeviceSynchronize() == cudaSuccess;
    if (ok && v.debug) {
        // debug mode: every slot starts dead -- NaN rows and importance
        const uint32_t nan_word = c->esz == 2 ? 0x7FC07FC0u : 0x7FC00000u;
        ok = launch_fill_u32(reinterpret_cast<uint32_t*>(v.pool), (size_t)c->pool_pages * v.page_bytes / 4, nan_word,
                             nullptr) == cudaSuccess &&
             launch_fill_u32(reinterpret_cast<uint32_t*>(v.imp), U * c->cap, 0x7FC00000u, nullptr) == cudaSuccess &&
             cudaDeviceSynchronize() == cudaSuccess;
    }
    if (!ok) {
        e = cudaGetLastError();
        free_all(c);
        delete c;
        return cuda_fail(e, "create: initialisation");
    }
    c->len.assign(U, 0);
    c->next_pos.assign(U, 0);
    c->mapped.assign(U, v.home_pages ? c->max_pages : 0);
    if (v.home_pages) c->pages_in_use = (int64_t)U * c->max_pages;
    c->fresh.assign(U, 0);
    *out = c;
    return HIKV_OK;
}

hikv_status hikv_destroy_cache(hikv_cache* c) {
    g_err.clear();
    if (!c) return HIKV_OK;
    cudaError_t e = cudaDeviceSynchronize();
    free_all(c);
    delete c;
    if (e != cudaSuccess) return cuda_fail(e, "destroy: synchronize");
    return HIKV_OK;
}

hikv_status hikv_append(hikv_cache* c, int32_t layer0, int32_t nl, int32_t ntok, const void* k,
                        const void* vv, hikv_stream_t stream) {
    g_err.clear();
    pdl_forget(c);
    NvtxRange nvtx("hikv_append");
    if (!range_ok(c, layer0, nl)) return fail(HIKV_ERR_INVALID_ARG, "append: bad cache or layer range");
    if (ntok < 0) return fail(HIKV_ERR_INVALID_ARG, "append: ntok < 0");
    if (ntok == 0) return HIKV_OK;
    if (!k || !vv) return fail(HIKV_ERR_INVALID_ARG, "append: null k or v");
    const int u0 = layer0 * c->per_layer, nu = nl * c->per_layer;
    int64_t new_pages = 0;
    for (int u = u0; u < u0 + nu; ++u) {
        if ((int64_t)c->len[u] + ntok > c->cap)
            return fail(HIKV_ERR_CAPACITY, "append: unit %d would hold %lld > max_tokens %d", u,
                        (long long)c->len[u] + ntok, c->cap);
        if ((int64_t)c->next_pos[u] + ntok > INT32_MAX)
            return fail(HIKV_ERR_CAPACITY, "append: positions of unit %d overflow int32", u);
        new_pages += std::max(0, ceil_div(c->len[u] + ntok, c->P) - c->mapped[u]);
    }
    if (c->pages_in_use + new_pages > c->pool_pages)
        return fail(HIKV_ERR_CAPACITY, "append: page pool exhausted (%lld in use + %lld > %lld)",
                    (long long)c->pages_in_use, (long long)new_pages, (long long)c->pool_pages);
    AppendArgs a{};
    a.v = c->v;
    a.u0 = u0;
    a.nunits = nu;
    a.ntok = ntok;
    a.k = (const uint8_t*)k;
    a.vv = (const uint8_t*)vv;
    a.base = c->d_append_base;
    cudaError_t e = launch_append(a, (cudaStream_t)stream);
    c->launches += ntok <= 64 ? 1 : 2;
    if (e != cudaSuccess) return cuda_fail(e, "append: launch");
    for (int u = u0; u < u0 + nu; ++u) {
        c->len[u] += ntok;
        c->next_pos[u] += ntok;
        c->mapped[u] = std::max(c->mapped[u], ceil_div(c->len[u], c->P));
        c->fresh[u] = 0;
    }
    c->pages_in_use += new_pages;
    return HIKV_OK;
}

hikv_status hikv_score_window(hikv_cache* c, int32_t layer0, int32_t nl, int32_t nq, const void* q,
                              hikv_stream_t stream) {
    g_err.clear();
    pdl_forget(c);
    NvtxRange nvtx("hikv_score_window");
    if (!range_ok(c, layer0, nl)) return fail(HIKV_ERR_INVALID_ARG, "score_window: bad cache or layer range");
    if (nq < 1 || nq > c->max_wq)
        return fail(HIKV_ERR_INVALID_ARG, "score_window: nq=%d not in [1, %d]", nq, c->max_wq);
    if (!q) return fail(HIKV_ERR_INVALID_ARG, "score_window: null q");
    if (window_smem_bytes(c->d, nq * c->G) > c->smem_optin)
        return fail(HIKV_ERR_UNSUPPORTED, "score_window: nq*G=%d query vectors exceed shared memory", nq * c->G);
    const int u0 = layer0 * c->per_layer, nu = nl * c->per_layer;
    int maxn = 0;
    for (int u = u0; u < u0 + nu; ++u) {
        if (c->next_pos[u] < nq || c->len[u] < 1)
            return fail(HIKV_ERR_STATE, "score_window: unit %d has fewer than nq=%d positions", u, nq);
        if (c->pool_k > 1 && c->len[u] != c->next_pos[u])
            return fail(HIKV_ERR_STATE, "score_window: pooling needs unit %d's prompt uncut", u);
        maxn = std::max(maxn, c->len[u]);
    }
    WindowArgs a{};
    a.v = c->v;
    a.u0 = u0;
    a.nunits = nu;
    a.layer0 = layer0;
    a.nq = nq;
    a.q = (const uint8_t*)q;
    a.qscale = c->scale * 1.4426950408889634f;
    a.part = c->d_wpart;
    a.nchunks_max = c->wchunks;
    a.nchunks_grid = ceil_div(maxn, kWindowChunk);
    a.chunk = kWindowChunk;
    const int nqv = nq * c->G;
    cudaError_t e = window_tc_supported(c->dtype, c->d, nqv)
                        ? launch_window_tc(a, c->tmap, c->d, nqv, (cudaStream_t)stream)
                        : launch_window(a, c->dtype, c->d, c->G, (cudaStream_t)stream);
    c->launches += 2;
    if (e == cudaSuccess && c->pool_k > 1) {
        e = launch_pool_importance(c->v, u0, nu, c->pool_k, (cudaStream_t)stream);
        c->launches += 1;
    }
    if (e != cudaSuccess) return cuda_fail(e, "score_window: launch");
    for (int u = u0; u < u0 + nu; ++u) c->fresh[u] = 0;
    return HIKV_OK;
}

hikv_status hikv_score_band(hikv_cache* c, int32_t layer0, int32_t nl, int32_t band, const void* q,
                            hikv_stream_t stream) {
    g_err.clear();
    pdl_forget(c);
    NvtxRange nvtx("hikv_score_band");
    if (!range_ok(c, layer0, nl)) return fail(HIKV_ERR_INVALID_ARG, "score_band: bad cache or layer range");
    if (band < 1) return fail(HIKV_ERR_INVALID_ARG, "score_band: band=%d < 1", band);
    if (!q) return fail(HIKV_ERR_INVALID_ARG, "score_band: null q");
    if (!c->d_band) return fail(HIKV_ERR_STATE, "score_band: the cache was created without band_scoring");
    const int u0 = layer0 * c->per_layer, nu = nl * c->per_layer;
    const int n = c->len[u0];
    for (int u = u0; u < u0 + nu; ++u) {
        if (c->len[u] != n)
            return fail(HIKV_ERR_STATE, "score_band: unit %d holds %d tokens, unit %d holds %d", u, c->len[u], u0, n);
        if (c->len[u] != c->next_pos[u])
            return fail(HIKV_ERR_STATE, "score_band: unit %d has been cut (needs the whole prompt)", u);
    }
    if (n < 1) return fail(HIKV_ERR_STATE, "score_band: empty units");
    cudaError_t e = cudaSuccess;
    for (int li = 0; li < nl && e == cudaSuccess; ++li) {
        e = launch_band(c->v, (layer0 + li) * c->per_layer, c->per_layer, li, (const uint8_t*)q, n, band,
                        c->scale * 1.4426950408889634f, c->d_band, c->dtype, (cudaStream_t)stream);
        c->launches += 2;
    }
    if (e != cudaSuccess) return cuda_fail(e, "score_band: launch");
    for (int u = u0; u < u0 + nu; ++u) c->fresh[u] = 0;
    return HIKV_OK;
}

}  // extern "C"

namespace {

// Launch the decode kernel over the units of [layer0, layer0 + nl).  With
// fused = 1 the kernel first appends one token per unit (rows new_k/new_v)
// and, with evict = 1, moves it into the victim's slot when the unit is over
// budget; the host mirror then already holds the post-append lengths.
// Deal `units` (sorted by size, largest first) to `bins` bins, each to the
// least-loaded bin (LPT); writes the bin-major list and bin offsets into
// out [units.size() + bins + 1].
void lpt_assign(const std::vector<int32_t>& units, const std::vector<int64_t>& load, int bins,
                std::vector<int32_t>& out) {
    const int n = (int)units.size();
    std::vector<int32_t> owner(n), count(bins, 0);
    std::priority_queue<std::pair<int64_t, int32_t>, std::vector<std::pair<int64_t, int32_t>>,
                        std::greater<std::pair<int64_t, int32_t>>> heap;
    for (int j = 0; j < bins; ++j) heap.push({0, j});
    for (int i = 0; i < n; ++i) {
        auto [l, j] = heap.top();
        heap.pop();
        owner[i] = j;
        ++count[j];
        heap.push({l + load[i], j});
    }
    out.assign((size_t)n + bins + 1, 0);
    int32_t* off = out.data() + n;
    for (int j = 0; j < bins; ++j) off[j + 1] = off[j] + count[j];
    std::vector<int32_t> fill(off, off + bins);
    for (int i = 0; i < n; ++i) out[fill[owner[i]]++] = units[i];   // largest first within a bin
}

uint64_t fnv_mix(uint64_t h, uint64_t x) { return (h ^ x) * 1099511628211ull; }

// The fixed per-unit work of the decode kernel, in tokens of streaming.
int64_t unit_cost_tokens(const hikv_cache* c) { return c->G == 8 ? 400 : 190; }

// CTAs per unit for a launch of nu units, the longest maxn tokens, total
// tokens in all (ragged: dealt by LPT).
int choose_cluster_size(const hikv_cache* c, int nu, int maxn, int64_t total, bool ragged) {
    // CTAs per unit (cluster size cs) by a cost model of the busiest cluster:
    // tokens per CTA plus a fixed per-unit cost (exchanges, importance pass,
    // victim) worth kUnitCostTokens tokens, a fit to the measured decode
    // times.  Equal units go round-robin, so the busiest cluster gets
    // ceil(units / clusters) of them; ragged ones are dealt by LPT, whose
    // busiest cluster is about max(average load, largest unit).  The logits
    // of a chunk too large for shared memory go to the global buffer, when
    // there is one.  With G = 8 the kernel's two head groups stream a CTA's
    // tokens faster, so the same per-unit work weighs more tokens (refit on
    // the 70B workload, 640 units of 4097 tokens: cluster size 2 took 466 us,
    // 3 496 us, 4 487 us, 8 552 us).
    const int64_t kUnitCostTokens = unit_cost_tokens(c);
    int cs = 1;
    if (c->cs_override > 0) {
        cs = std::min(c->cs_override, kMaxCS);
    } else {
        const int slots = c->dec_occ * c->sm_count;
        int64_t best = INT64_MAX;
        for (int k = 1; k <= std::min(kMaxCS, maxn); ++k) {
            const int ck = dec_chunk_max(maxn, k);
            const bool sp = ck <= c->max_smem_chunk;
            if (!sp && !c->d_logits) continue;
            const size_t smem = decode_smem_bytes(c->dtype, c->d, c->G, sp, sp ? ck : 0);
            int ncl = std::max(1, std::min(nu, slots / k));
            const int active = decode_active_clusters(c->dtype, c->d, c->G, sp, k, smem);
            if (active > 0) ncl = std::min(ncl, active);
            int64_t cost;
            if (!ragged) {
                cost = (int64_t)ceil_div(nu, ncl) * (ceil_div(maxn, k) + kUnitCostTokens);
            } else {
                const int64_t sum = (total + (int64_t)nu * (k - 1)) / k + (int64_t)nu * kUnitCostTokens;
                cost = std::max<int64_t>((sum + ncl - 1) / ncl, ceil_div(maxn, k) + kUnitCostTokens);
            }
            if (cost < best) {
                best = cost;
                cs = k;
            }
        }
    }
    return cs;
}

// Clusters resident at once for cluster size cs (the persistent grid).
int resident_clusters(const hikv_cache* c, int nu, int maxn, int cs) {
    const int chunk = dec_chunk_max(maxn, cs);
    const bool sp = chunk <= c->max_smem_chunk;
    const size_t smem = decode_smem_bytes(c->dtype, c->d, c->G, sp, sp ? chunk : 0);
    int ncl = std::max(1, std::min(nu, (c->dec_occ * c->sm_count) / cs));
    const int active = decode_active_clusters(c->dtype, c->d, c->G, sp, cs, smem);
    if (active > 0) ncl = std::min(ncl, active);
    return ncl;
}

// The cluster kernel over all units of the range (equal budgets: identity
// order; range_count >= 0 limits it to units [range_first, + range_count) of
// the range) or over `subset` (ragged: largest first, dealt by LPT).
hikv_status launch_clusters(hikv_cache* c, int32_t layer0, int32_t nl, const std::vector<int32_t>* subset,
                            bool uni_len, bool uni_b, bool uni_np, const void* q, void* out, int fused,
                            int evict, const void* new_k, const void* new_v, hikv_stream_t stream,
                            const char* who, int range_first = 0, int range_count = -1) {
    const int u0 = layer0 * c->per_layer + (subset ? 0 : range_first);
    const int nu = subset ? (int)subset->size() : (range_count >= 0 ? range_count : nl * c->per_layer);
    auto unit_at = [&](int i) { return subset ? (*subset)[i] : u0 + i; };
    int maxn = 0;
    int64_t total = 0;
    for (int i = 0; i < nu; ++i) {
        const int n = c->len[unit_at(i)] + fused;
        maxn = std::max(maxn, n);
        total += n;
    }
    int cs = choose_cluster_size(c, nu, maxn, total, subset != nullptr);
    cs = std::min(cs, std::max(1, maxn));
    const int chunk = dec_chunk_max(maxn, cs);   // most slots a CTA holds
    const bool smem_path = chunk <= c->max_smem_chunk;
    if (!smem_path && !c->d_logits)
        return fail(HIKV_ERR_UNSUPPORTED, "%s: %d tokens per CTA exceed shared memory", who, chunk);
    const size_t smem = decode_smem_bytes(c->dtype, c->d, c->G, smem_path, smem_path ? chunk : 0);
    // persistent clusters: at most one wave (the clusters that fit at once)
    int ncl = std::max(1, std::min(nu, (c->dec_occ * c->sm_count) / cs));
    {
        const int active = decode_active_clusters(c->dtype, c->d, c->G, smem_path, cs, smem);
        if (active > 0) ncl = std::min(ncl, active);
    }
    const int32_t* d_assign = nullptr;
    const int32_t* d_assign_off = nullptr;
    if (subset) {
        uint64_t key = 1469598103934665603ull;
        key = fnv_mix(key, (uint64_t)cs);
        key = fnv_mix(key, (uint64_t)ncl);
        key = fnv_mix(key, (uint64_t)fused);
        for (int i = 0; i < nu; ++i) {
            key = fnv_mix(key, (uint64_t)(uint32_t)(*subset)[i]);
            key = fnv_mix(key, (uint64_t)(uint32_t)c->len[(*subset)[i]]);
        }
        d_assign = c->d_assign + u0;
        d_assign_off = c->d_assign + c->units + (size_t)layer0 * (c->dec_occ * c->sm_count + 1);
        if (key != c->asg_key[layer0]) {
            std::vector<int64_t> load(nu);
            for (int i = 0; i < nu; ++i) load[i] = ceil_div(c->len[(*subset)[i]] + fused, cs) + unit_cost_tokens(c);
            lpt_assign(*subset, load, ncl, c->asg);
            // pageable sources: the copies are staged before the calls return
            cudaError_t e = cudaMemcpyAsync(const_cast<int32_t*>(d_assign), c->asg.data(), nu * sizeof(int32_t),
                                            cudaMemcpyHostToDevice, (cudaStream_t)stream);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(const_cast<int32_t*>(d_assign_off), c->asg.data() + nu,
                                    (ncl + 1) * sizeof(int32_t), cudaMemcpyHostToDevice, (cudaStream_t)stream);
            if (e != cudaSuccess) return cuda_fail(e, who);
            c->asg_key[layer0] = key;
        }
    }
    DecodeArgs a{};
    a.v = c->v;
    a.order = (nl == c->L) ? c->d_order_all : c->d_order_layer + u0;
    a.n_units = nu;
    a.layer0 = layer0;
    a.q = (const uint8_t*)q;
    a.out = (uint8_t*)out;
    a.qscale = c->scale * 1.4426950408889634f;
    a.logits = c->d_logits;
    a.cand = c->d_cand;
    a.cand_slot = c->d_cand_slot;
    a.cs = cs;
    a.chunk_cap = smem_path ? chunk : 0;
    a.uni_len = (!subset && uni_len) ? c->len[u0] + fused : -1;
    a.uni_budget = (!subset && uni_b) ? c->budget_unit[u0] : -1;
    a.uni_next_pos = (!subset && uni_np) ? c->next_pos[u0] + fused : -1;
    a.identity_u0 = subset ? -1 : u0;
    a.n_clusters = ncl;
    a.assign = d_assign;
    a.assign_off = d_assign_off;
    // small calls fit in L2: prefetch each CTA's tiles there ahead of the ring
    const int64_t call_bytes = total * 2 * c->d * c->esz;
    a.prefetch_tiles = c->prefetch_override >= 0 ? c->prefetch_override : (call_bytes <= (48ll << 20) ? 16 : 0);
    a.first_burst = c->first_burst;
    a.fused = fused;
    a.evict = evict;
    a.new_k = (const uint8_t*)new_k;
    a.new_v = (const uint8_t*)new_v;
    int ulo = u0, uhi = u0 + nu;   // the units this launch writes
    if (subset) {
        ulo = *std::min_element(subset->begin(), subset->end());
        uhi = *std::max_element(subset->begin(), subset->end()) + 1;
    }
    a.pdl_early = pdl_disjoint(c, ulo, uhi, stream) ? 1 : 0;
    cudaError_t e = launch_decode(a, c->tmap, c->dtype, c->d, c->G, smem_path, smem, (cudaStream_t)stream);
    c->launches += 1;
    pdl_record(c, ulo, uhi, stream);
    if (c->last_ncfg < 2) {
        int32_t* r = c->last_cfg[c->last_ncfg++];
        r[0] = nu;
        r[1] = cs;
        r[2] = ncl;
        r[3] = smem_path ? 1 : 0;
    }
    if (e != cudaSuccess) return cuda_fail(e, who);
    return HIKV_OK;
}

// The warp-per-unit kernel over `units` (largest first), dealt by LPT to
// four warps per CTA.
hikv_status launch_small(hikv_cache* c, int32_t layer0, const std::vector<int32_t>& units, const void* q,
                         void* out, int fused, int evict, const void* new_k, const void* new_v,
                         hikv_stream_t stream, const char* who) {
    constexpr int64_t kWarpUnitCostTokens = 48;   // per-unit cost of a warp (its epilogue), in tokens
    const int nu = (int)units.size();
    const int n_ctas = std::max(1, std::min(c->dec_occ * c->sm_count, ceil_div(nu, kSmallWarps)));
    const int warps = n_ctas * kSmallWarps;
    uint64_t key = 7809847782465536322ull;
    key = fnv_mix(key, (uint64_t)warps);
    key = fnv_mix(key, (uint64_t)fused);
    for (int i = 0; i < nu; ++i) {
        key = fnv_mix(key, (uint64_t)(uint32_t)units[i]);
        key = fnv_mix(key, (uint64_t)(uint32_t)c->len[units[i]]);
    }
    const int32_t u0 = layer0 * c->per_layer;
    int32_t* d_list = c->d_sassign + u0;
    int32_t* d_off = c->d_sassign + c->units + (size_t)layer0 * (kSmallWarps * c->dec_occ * c->sm_count + 1);
    if (key != c->sasg_key[layer0]) {
        std::vector<int64_t> load(nu);
        for (int i = 0; i < nu; ++i) load[i] = c->len[units[i]] + fused + kWarpUnitCostTokens;
        lpt_assign(units, load, warps, c->sasg);
        cudaError_t e = cudaMemcpyAsync(d_list, c->sasg.data(), nu * sizeof(int32_t), cudaMemcpyHostToDevice,
                                        (cudaStream_t)stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(d_off, c->sasg.data() + nu, (warps + 1) * sizeof(int32_t), cudaMemcpyHostToDevice,
                                (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, who);
        c->sasg_key[layer0] = key;
    }
    SmallArgs a{};
    a.v = c->v;
    a.list = d_list;
    a.warp_off = d_off;
    a.layer0 = layer0;
    a.q = (const uint8_t*)q;
    a.out = (uint8_t*)out;
    a.qscale = c->scale * 1.4426950408889634f;
    a.fused = fused;
    a.evict = evict;
    a.new_k = (const uint8_t*)new_k;
    a.new_v = (const uint8_t*)new_v;
    cudaError_t e = launch_decode_small(a, c->tmap, c->dtype, c->d, c->G, n_ctas, (cudaStream_t)stream);
    c->launches += 1;
    // (launched without programmatic serialisation: it starts after the
    // previous grid completes; a following decode launch may overlap it)
    pdl_record(c, *std::min_element(units.begin(), units.end()), *std::max_element(units.begin(), units.end()) + 1,
               stream);
    if (e != cudaSuccess) return cuda_fail(e, who);
    return HIKV_OK;
}

// Launch the decode kernels over the units of [layer0, layer0 + nl).  With
// fused = 1 they first append one token per unit (rows new_k/new_v) and,
// with evict = 1, move it into the victim's slot when the unit is over
// budget; the host mirror then already holds the post-append lengths.
// Equal budgets: one cluster-kernel launch.  Ragged budgets (group <= 4):
// units of at most small_unit_cap(G) tokens go to the warp-per-unit kernel,
// the others to the cluster kernel.
hikv_status launch_decode_call(hikv_cache* c, int32_t layer0, int32_t nl, const void* q, void* out,
                               int fused, int evict, const void* new_k, const void* new_v,
                               hikv_stream_t stream, const char* who) {
    const int u0 = layer0 * c->per_layer, nu = nl * c->per_layer;
    c->last_ncfg = 0;
    bool uni_len = true, uni_b = true, uni_np = true;
    for (int u = u0; u < u0 + nu; ++u) {
        const int n = c->len[u] + fused;
        if (n < 1) return fail(HIKV_ERR_STATE, "%s: unit %d is empty", who, u);
        uni_len &= c->len[u] == c->len[u0];
        uni_b &= c->budget_unit[u] == c->budget_unit[u0];
        uni_np &= c->next_pos[u] == c->next_pos[u0];
    }
    if (uni_b) {
        // Equal units go round-robin over the resident clusters.  When the
        // last round would keep at most 70 % of them busy, the full rounds go
        // in one launch and the rest in a second one, each with the cluster
        // size the cost model picks for it, so the rest spreads over the
        // whole GPU instead of a few clusters (70B workload, 640 units: 467 ->
        // 434 us as 608 units at cluster size 1 plus 32 at size 8; forcing
        // size 2 on the 608, the size the split was counted with, took 451;
        // its full cache, last round 65 % busy: 13.42 -> 13.15 ms).
        if (uni_len && c->cs_override <= 0) {
            const int n = c->len[u0] + fused;
            const int cs = choose_cluster_size(c, nu, n, (int64_t)n * nu, false);
            const int ncl = resident_clusters(c, nu, n, cs);
            const int rem = nu % ncl;
            if (nu > ncl && rem > 0 && 10 * rem <= 7 * ncl) {
                const int full = nu - rem;
                hikv_status st = launch_clusters(c, layer0, nl, nullptr, uni_len, uni_b, uni_np, q, out, fused, evict,
                                                 new_k, new_v, stream, who, 0, full);
                if (st != HIKV_OK) return st;
                return launch_clusters(c, layer0, nl, nullptr, uni_len, uni_b, uni_np, q, out, fused, evict, new_k,
                                       new_v, stream, who, full, rem);
            }
        }
        return launch_clusters(c, layer0, nl, nullptr, uni_len, uni_b, uni_np, q, out, fused, evict, new_k, new_v,
                               stream, who);
    }
    std::vector<int32_t> units(nu);
    std::iota(units.begin(), units.end(), u0);
    std::stable_sort(units.begin(), units.end(), [&](int x, int y) { return c->len[x] > c->len[y]; });
    // split only when the small units are enough to occupy the GPU by
    // themselves: each launch has a fixed latency of its own, and a call of
    // few units (one layer of a model) is better served by one launch
    std::vector<int32_t> big, small;
    bool split = c->G <= kSmallWarps && c->small_mode != 0 && c->cs_override <= 0;
    if (split && c->small_mode == 1) {
        int nsmall = 0;
        for (int32_t u : units) nsmall += c->len[u] + fused <= small_unit_cap(c->G);
        split = nsmall >= 2 * c->sm_count;
    }
    for (int32_t u : units) (split && c->len[u] + fused <= small_unit_cap(c->G) ? small : big).push_back(u);
    hikv_status st = HIKV_OK;
    if (!big.empty())
        st = launch_clusters(c, layer0, nl, &big, false, false, false, q, out, fused, evict, new_k, new_v, stream, who);
    if (st == HIKV_OK && !small.empty())
        st = launch_small(c, layer0, small, q, out, fused, evict, new_k, new_v, stream, who);
    return st;
}

}  // namespace

extern "C" {

// HiKV Stage II decode of the layer range: sort, span and merge kernels.
// fused = 1: the order kernel appends new_k / new_v first and, with evict, the
// merge drops the victim (the host checked that the new slots' pages are
// mapped and that no unit needs more than one eviction).
static hikv_status launch_elem_call(hikv_cache* c, int32_t layer0, int32_t nl, const void* q, void* out,
                                    hikv_stream_t stream, int fused = 0, int evict = 0,
                                    const void* new_k = nullptr, const void* new_v = nullptr) {
    pdl_forget(c);
    const int u0 = layer0 * c->per_layer, nu = nl * c->per_layer;
    int max_n = 0;
    for (int u = u0; u < u0 + nu; ++u) {
        const int n = c->len[u] + (fused ? 1 : 0);
        if (n <= 0) return fail(HIKV_ERR_STATE, "decode_step: unit %d is empty", u);
        if (n > c->elem_stride)
            return fail(HIKV_ERR_CAPACITY, "decode_step: unit %d holds %d tokens, more than the %d of an element-level step",
                        u, n, c->elem_stride);
        max_n = std::max(max_n, n);
    }
    ElemArgs a{};
    a.v = c->v;
    a.q = q;
    a.out = out;
    a.u0 = u0;
    a.nunits = nu;
    a.layer0 = layer0;
    a.b2 = c->elem;
    a.ostride = c->elem_stride;
    a.nsp = ceil_div(max_n, elem_span_ranks());
    a.qscale = c->scale * 1.4426950408889634f;
    a.order = c->d_eorder;
    a.lg = c->d_elg;
    a.part = c->d_epart;
    a.rows_loaded = c->d_erows;
    a.qmask = c->d_eqmask;
    a.done = c->d_edone;
    a.fused = fused;
    a.evict = evict;
    a.new_k = new_k;
    a.new_v = new_v;
    cudaError_t e = launch_elem_decode(a, c->dtype, c->d, max_n, (cudaStream_t)stream);
    c->launches += 2;
    if (e != cudaSuccess) return cuda_fail(e, "decode_step: element-level launch");
    return HIKV_OK;
}

hikv_status hikv_decode_step(hikv_cache* c, int32_t layer0, int32_t nl, const void* q, void* out,
                             hikv_stream_t stream) {
    g_err.clear();
    NvtxRange nvtx("hikv_decode_step");
    if (!range_ok(c, layer0, nl)) return fail(HIKV_ERR_INVALID_ARG, "decode_step: bad cache or layer range");
    if (!q || !out) return fail(HIKV_ERR_INVALID_ARG, "decode_step: null q or out");
    if (q == out) return fail(HIKV_ERR_INVALID_ARG, "decode_step: out aliases q");
    hikv_status st = c->elem ? launch_elem_call(c, layer0, nl, q, out, stream)
                             : launch_decode_call(c, layer0, nl, q, out, 0, 0, nullptr, nullptr, stream, "decode_step");
    if (st != HIKV_OK) return st;
    const int u0 = layer0 * c->per_layer, nu = nl * c->per_layer;
    for (int u = u0; u < u0 + nu; ++u) c->fresh[u] = 1;
    return HIKV_OK;
}

hikv_status hikv_decode_step_fused(hikv_cache* c, int32_t layer0, int32_t nl, const void* k, const void* v,
                                   const void* q, void* out, int32_t evict, hikv_stream_t stream) {
    g_err.clear();
    NvtxRange nvtx("hikv_decode_step_fused");
    if (!range_ok(c, layer0, nl)) return fail(HIKV_ERR_INVALID_ARG, "decode_step_fused: bad cache or layer range");
    if (!k || !v || !q || !out) return fail(HIKV_ERR_INVALID_ARG, "decode_step_fused: null pointer");
    if (q == out) return fail(HIKV_ERR_INVALID_ARG, "decode_step_fused: out aliases q");
    if (((uintptr_t)k | (uintptr_t)v) & 15)
        return fail(HIKV_ERR_INVALID_ARG, "decode_step_fused: k and v must be 16-byte aligned");
    const int u0 = layer0 * c->per_layer, nu = nl * c->per_layer;
    bool one_launch = true;
    for (int u = u0; u < u0 + nu && one_launch; ++u) {
        const int n = c->len[u] + 1;
        if (n > c->cap) return fail(HIKV_ERR_CAPACITY, "decode_step_fused: unit %d would exceed max_tokens", u);
        if ((int64_t)c->next_pos[u] + 1 > INT32_MAX) return fail(HIKV_ERR_CAPACITY, "decode_step_fused: positions overflow");
        // the single launch needs the new slot's page mapped, and at most one eviction
        if (ceil_div(n, c->P) > c->mapped[u]) one_launch = false;
        if (evict && n - c->budget_unit[u] > 1) one_launch = false;
    }
    if (!one_launch) {
        hikv_status st = hikv_append(c, layer0, nl, 1, k, v, stream);
        if (st == HIKV_OK) st = hikv_decode_step(c, layer0, nl, q, out, stream);
        if (st == HIKV_OK && evict) st = hikv_evict(c, layer0, nl, stream);
        return st;
    }
    hikv_status st = c->elem ? launch_elem_call(c, layer0, nl, q, out, stream, 1, evict ? 1 : 0, k, v)
                             : launch_decode_call(c, layer0, nl, q, out, 1, evict ? 1 : 0, k, v, stream, "decode_step_fused");
    if (st != HIKV_OK) return st;
    for (int u = u0; u < u0 + nu; ++u) {
        const bool cut = evict && c->len[u] + 1 > c->budget_unit[u];
        c->len[u] = cut ? c->budget_unit[u] : c->len[u] + 1;
        c->next_pos[u] += 1;
        c->fresh[u] = cut ? 0 : 1;
    }
    return HIKV_OK;
}

hikv_status hikv_evict(hikv_cache* c, int32_t layer0, int32_t nl, hikv_stream_t stream) {
    g_err.clear();
    pdl_forget(c);
    NvtxRange nvtx("hikv_evict");
    if (!range_ok(c, layer0, nl)) return fail(HIKV_ERR_INVALID_ARG, "evict: bad cache or layer range");
    const int u0 = layer0 * c->per_layer, nu = nl * c->per_layer;
    bool any = false, fast = true;
    for (int u = u0; u < u0 + nu; ++u) {
        const int over = c->len[u] - c->budget_unit[u];
        if (over <= 0) continue;
        any = true;
        if (over > 1 || !c->fresh[u]) fast = false;
    }
    if (!any) return HIKV_OK;
    EvictArgs a{};
    a.v = c->v;
    a.u0 = u0;
    a.nunits = nu;
    a.holes = c->d_holes;
    a.hole_off = c->d_hole_off;
    cudaError_t e = fast ? launch_evict_fast(a, (cudaStream_t)stream) : launch_evict_general(a, (cudaStream_t)stream);
    c->launches += 1;
    if (e != cudaSuccess) return cuda_fail(e, "evict: launch");
    for (int u = u0; u < u0 + nu; ++u) {
        const int Bu = c->budget_unit[u];
        if (c->len[u] > Bu) {
            c->len[u] = Bu;
            const int keep = pages_kept(Bu, c->P, c->max_pages);
            if (!c->v.home_pages && c->mapped[u] > keep) {
                c->pages_in_use -= c->mapped[u] - keep;
                c->mapped[u] = keep;
            }
        }
        c->fresh[u] = 0;
    }
    return HIKV_OK;
}

hikv_status hikv_gather_retained(hikv_cache* c, int32_t layer0, int32_t nl, int32_t cap, int32_t* lengths,
                                 int32_t* positions, float* importance, void* k_out, void* v_out,
                                 hikv_stream_t stream) {
    g_err.clear();
    pdl_forget(c);
    NvtxRange nvtx("hikv_gather_retained");
    if (!range_ok(c, layer0, nl)) return fail(HIKV_ERR_INVALID_ARG, "gather: bad cache or layer range");
    if (!lengths || !positions || !importance) return fail(HIKV_ERR_INVALID_ARG, "gather: null output");
    const int u0 = layer0 * c->per_layer, nu = nl * c->per_layer;
    for (int u = u0; u < u0 + nu; ++u)
        if (c->len[u] > cap) return fail(HIKV_ERR_INVALID_ARG, "gather: cap %d < length %d of unit %d", cap, c->len[u], u);
    GatherArgs a{};
    a.v = c->v;
    a.u0 = u0;
    a.nunits = nu;
    a.cap = cap;
    a.lengths = lengths;
    a.positions = positions;
    a.importance = importance;
    a.k_out = (uint8_t*)k_out;
    a.v_out = (uint8_t*)v_out;
    cudaError_t e = launch_gather(a, (cudaStream_t)stream);
    c->launches += 1;
    if (e != cudaSuccess) return cuda_fail(e, "gather: launch");
    return HIKV_OK;
}

hikv_status hikv_last_decode_config(const hikv_cache* c, int32_t* out_host) {
    g_err.clear();
    if (!c || !out_host) return fail(HIKV_ERR_INVALID_ARG, "last_decode_config: null cache or output");
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 4; ++j) out_host[i * 4 + j] = i < c->last_ncfg ? c->last_cfg[i][j] : 0;
    return HIKV_OK;
}

hikv_status hikv_element_rows(const hikv_cache* c, int64_t* rows_host) {
    g_err.clear();
    if (!c || !rows_host) return fail(HIKV_ERR_INVALID_ARG, "element_rows: null cache or output");
    *rows_host = 0;
    if (!c->d_erows) return HIKV_OK;
    unsigned long long r = 0;
    cudaError_t e = cudaMemcpy(&r, c->d_erows, 8, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "element_rows: read");
    *rows_host = (int64_t)r;
    return HIKV_OK;
}

hikv_status hikv_read_slot(const hikv_cache* c, int32_t unit, int32_t slot, void* k_host, void* v_host,
                           float* imp_host, int32_t* pos_host) {
    g_err.clear();
    if (!c || unit < 0 || unit >= c->units || slot < 0 || slot >= c->cap)
        return fail(HIKV_ERR_INVALID_ARG, "read_slot: bad cache, unit or slot");
    int32_t pg = -1;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(&pg, c->v.page_table + (int64_t)unit * c->max_pages + (slot >> c->page_shift), 4,
                       cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read_slot");
    if (pg < 0 || pg >= c->pool_pages) return fail(HIKV_ERR_STATE, "read_slot: slot %d of unit %d has no page", slot, unit);
    const uint8_t* kr = c->v.pool + (int64_t)pg * c->v.page_bytes + (int64_t)(slot & (c->P - 1)) * c->v.row_bytes;
    const int64_t m = (int64_t)unit * c->cap + slot;
    if ((k_host && (e = cudaMemcpy(k_host, kr, c->v.row_bytes, cudaMemcpyDeviceToHost)) != cudaSuccess) ||
        (v_host && (e = cudaMemcpy(v_host, kr + (int64_t)c->P * c->v.row_bytes, c->v.row_bytes,
                                   cudaMemcpyDeviceToHost)) != cudaSuccess) ||
        (imp_host && (e = cudaMemcpy(imp_host, c->v.imp + m, 4, cudaMemcpyDeviceToHost)) != cudaSuccess) ||
        (pos_host && (e = cudaMemcpy(pos_host, c->v.pos + m, 4, cudaMemcpyDeviceToHost)) != cudaSuccess))
        return cuda_fail(e, "read_slot");
    return HIKV_OK;
}

hikv_status hikv_get_lengths(const hikv_cache* c, int32_t layer0, int32_t nl, int32_t* lengths_host) {
    g_err.clear();
    if (!range_ok(c, layer0, nl) || !lengths_host) return fail(HIKV_ERR_INVALID_ARG, "get_lengths: bad arguments");
    std::memcpy(lengths_host, c->len.data() + (size_t)layer0 * c->per_layer, sizeof(int32_t) * nl * c->per_layer);
    return HIKV_OK;
}

int64_t hikv_kernel_launches(const hikv_cache* c) { return c ? c->launches : -1; }

hikv_status hikv_selftest_timeout(hikv_cache* c, int32_t limit_us, hikv_stream_t stream) {
    g_err.clear();
    pdl_forget(c);
    if (!c || limit_us < 1 || limit_us > 2000000)
        return fail(HIKV_ERR_INVALID_ARG, "selftest_timeout: bad cache or limit");
    cudaError_t e = launch_selftest_timeout(c->v, (uint64_t)limit_us * 1000u, (cudaStream_t)stream);
    c->launches += 1;
    if (e != cudaSuccess) return cuda_fail(e, "selftest_timeout: launch");
    return HIKV_OK;
}

hikv_status hikv_budgets_pyramid(int32_t num_layers, int32_t num_kv_heads, int32_t avg, int32_t min_budget,
                                 int32_t floor_budget, int32_t* out) {
    g_err.clear();
    if (num_layers < 1 || num_kv_heads < 1 || !out || min_budget < 0 || min_budget > avg || avg < 1 ||
        floor_budget < 0 || avg > (1 << 29))
        return fail(HIKV_ERR_INVALID_ARG, "budgets_pyramid: bad arguments");
    const int64_t cmax = 2 * (int64_t)avg - min_budget, cmin = min_budget, den = num_layers - 1;
    for (int32_t l = 0; l < num_layers; ++l) {
        int64_t c = avg;
        if (den > 0) {
            // round_half_up(cmax - l (cmax - cmin) / den) = floor((2 (cmax den - l (cmax - cmin)) + den) / (2 den))
            const int64_t num = 2 * (cmax * den - (int64_t)l * (cmax - cmin)) + den;
            c = num >= 0 ? num / (2 * den) : -((-num + 2 * den - 1) / (2 * den));
        }
        c = std::max<int64_t>(c, floor_budget);
        for (int32_t h = 0; h < num_kv_heads; ++h) out[(int64_t)l * num_kv_heads + h] = (int32_t)c;
    }
    return HIKV_OK;
}

hikv_status hikv_budgets_duo(int32_t num_layers, int32_t num_kv_heads, const uint8_t* retrieval,
                             int32_t full_budget, int32_t num_sink, int32_t recent_window, int32_t* out) {
    g_err.clear();
    if (num_layers < 1 || num_kv_heads < 1 || !retrieval || !out || num_sink < 0 || recent_window < 0 ||
        full_budget < num_sink + recent_window)
        return fail(HIKV_ERR_INVALID_ARG, "budgets_duo: bad arguments");
    for (int64_t i = 0; i < (int64_t)num_layers * num_kv_heads; ++i)
        out[i] = retrieval[i] ? full_budget : num_sink + recent_window;
    return HIKV_OK;
}

hikv_status hikv_device_status(hikv_cache* c) {
    g_err.clear();
    if (!c) return fail(HIKV_ERR_INVALID_ARG, "device_status: null cache");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "device_status: synchronize");
    uint32_t w[8] = {};
    e = cudaMemcpy(w, c->v.err, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "device_status: read");
    if (w[0] || w[1]) {
        cudaMemset(c->v.err, 0, sizeof(w));
        cudaDeviceSynchronize();
    }
    if (w[0] & DEVERR_TIMEOUT) {
        static const char* const sites[] = {"?", "producer q-free", "producer stage-free", "producer drain",
                                            "consumer q", "consumer tile", "cluster exchange", "victim exchange",
                                            "self-test"};
        return fail(HIKV_ERR_TIMEOUT,
                    "device: a bounded wait gave up (bits 0x%x; first: %s wait, cluster %u, CTA %u, index 0x%x, "
                    "after %u us)", w[0], sites[w[1] < 9 ? w[1] : 0], w[2], w[3], w[4], w[5]);
    }
    if (w[0]) return fail(HIKV_ERR_STATE, "device: inconsistent state recorded (bits 0x%x)", w[0]);
    return HIKV_OK;
}

}  // extern "C"
