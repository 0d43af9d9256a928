// HiKV Stage II: element-level decode attention (HiKV sec. III-C, Algorithm 1).
//
// An approximation of the decode step, switched on by an element budget
// 0 < B2 < d.  Per query head h of a unit:
//   * K side: only the B2 dimensions of q_h with the largest |q| (ties: the
//     lower index) enter the logits, s_j = scale * sum_{c in E_Q} q_h[c] k_j[c];
//   * the softmax P of those logits over every retained token feeds the
//     importance update unchanged (Algorithm 1 adds P_t to the scores);
//   * V side: P is cut into chunks of d entries in position order (rank by
//     position among the retained tokens); each chunk keeps its B2 largest
//     entries (ties: the lower position) and the output is the sum of those
//     p_j v_j, not renormalised.  A chunk of at most B2 entries keeps all.
// Selecting the largest p of a chunk is selecting its largest logits (exp is
// increasing and every entry of a head shares m and l), so the kernels select
// on the logits.
//
// Two kernels per call:
//   k_elem_order  one CTA per unit: the unit's slots in position order (a
//                 bucket count of the positions, then ranks within buckets),
//                 and each query head's q with all but its B2 largest-|q|
//                 dimensions zeroed (a radix select on the |q| bits);
//   k_elem_span   one CTA per (unit, span of kElemSpan ranks): masked-q
//                 logits of the span's rows (8 lanes per row), per-span
//                 softmax statistics, the top-B2 selection of each d-rank
//                 chunk and head (a radix select on the logit bits in one
//                 warp), then p.v over the rows that at least one head of
//                 the group selected -- V rows no head selected are not read.
//                 The unit's last span CTA to finish then merges the spans'
//                 (m, l, o), writes the output, adds sum_h 2^(s - m_h) / l_h to
//                 every retained token's importance (HiKV Stage I mode: the
//                 recent bank only) and records the eviction victim, as the
//                 exact decode kernel does.
// In a fused step (append + decode + evict in one call) k_elem_order first
// writes the new token into its slot, and the merging CTA moves it into the
// victim's slot when the unit is cut, so the step is these two launches.
//
// The K side reads whole rows: the pool stores token-major rows, so B2 of the
// d dimensions of a row lie in nearly every 32-byte sector (DRAM's unit), and
// under GQA the union of the group's dimension sets covers most of d anyway.
#include "hikv_internal.cuh"

namespace hikv {
namespace {

constexpr int kElemThreads = 256;
constexpr int kElemWarps = kElemThreads / 32;
constexpr int kElemSpan = 128;       // ranks per span CTA (a multiple of d)
constexpr int kElemMaxG = 8;
constexpr int kElemMaxSpans = 16384 / kElemSpan;
constexpr int kElemMaxPages = 16384 / 16;   // pages of a unit at the smallest page size
constexpr int kOrderThreads = 1024;

// N consecutive elements of type T at p (16-byte aligned when N*sizeof(T) >= 16,
// else N*sizeof(T)-aligned), widened to float.
template <typename T, int N>
__device__ __forceinline__ void load_vec(const uint8_t* p, float (&x)[N]) {
    constexpr int BYTES = N * (int)sizeof(T);
    if constexpr (BYTES >= 16) {
        static_assert(BYTES % 16 == 0, "vector width");
#pragma unroll
        for (int i = 0; i < BYTES / 16; ++i) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(p) + i);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if constexpr (sizeof(T) == 2) {
                    x[i * 8 + 2 * k] = __uint_as_float(ws[k] << 16);
                    x[i * 8 + 2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
                } else {
                    x[i * 4 + k] = __uint_as_float(ws[k]);
                }
            }
        }
    } else if constexpr (BYTES == 8) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
        if constexpr (sizeof(T) == 2) {
            x[0] = __uint_as_float(w.x << 16);
            x[1] = __uint_as_float(w.x & 0xFFFF0000u);
            x[2] = __uint_as_float(w.y << 16);
            x[3] = __uint_as_float(w.y & 0xFFFF0000u);
        } else {
            x[0] = __uint_as_float(w.x);
            x[1] = __uint_as_float(w.y);
        }
    } else {
        static_assert(BYTES == 4 && sizeof(T) == 2, "vector width");
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(p));
        x[0] = __uint_as_float(w << 16);
        x[1] = __uint_as_float(w & 0xFFFF0000u);
    }
}

// raw 16-byte words of N elements of T (N * sizeof(T) a multiple of 16), and their widening
template <typename T, int N>
struct RawVec {
    static constexpr int W = N * (int)sizeof(T) / 16;
    uint4 w[W];
    __device__ __forceinline__ void load(const uint8_t* p) {
#pragma unroll
        for (int i = 0; i < W; ++i) w[i] = __ldg(reinterpret_cast<const uint4*>(p) + i);
    }
    __device__ __forceinline__ void widen(float (&x)[N]) const {
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if constexpr (sizeof(T) == 2) {
                    x[i * 8 + 2 * k] = __uint_as_float(ws[k] << 16);
                    x[i * 8 + 2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
                } else {
                    x[i * 4 + k] = __uint_as_float(ws[k]);
                }
            }
        }
    }
};

__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// order-preserving map of a float's bits to an unsigned key
__device__ __forceinline__ uint32_t ord_key(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// address of slot s's K (or V) row in unit u, null (and the error bit) for an unmapped page
__device__ __forceinline__ uint8_t* elem_row(const View& v, int32_t u, int32_t s, bool is_v) {
    const int32_t pg = v.page_table[(int64_t)u * v.max_pages + (s >> v.page_shift)];
    if (pg < 0 || pg >= v.pool_pages) {
        atomicOr(v.err, DEVERR_PAGE);
        return nullptr;
    }
    return v.pool + (int64_t)pg * v.page_bytes +
           ((is_v ? (int64_t)v.page_tokens : 0) + (s & (v.page_tokens - 1))) * v.row_bytes;
}

// ---------------------------------------------------------------------------
// k_elem_order: slots of each unit in position order (positions are unique).
// Positions are binned into kOrderBuckets buckets of 2^shift consecutive
// positions; a slot's rank is the count of earlier buckets plus the members of
// its own bucket at a lower position (a bucket holds at most 2^shift tokens).
// ---------------------------------------------------------------------------
constexpr int kOrderBuckets = 4096;

__host__ __device__ inline size_t order_smem(int max_n) { return (size_t)(2 * kOrderBuckets + 2 * max_n + 32) * 4; }

__global__ void __launch_bounds__(kOrderThreads) k_elem_order(const ElemArgs a) {
    extern __shared__ int32_t osm[];
    int32_t* cur = osm;                        // [kOrderBuckets] counts, then cursors
    int32_t* start = cur + kOrderBuckets;      // [kOrderBuckets] exclusive prefix
    int32_t* wsum = start + kOrderBuckets;     // [32]
    int32_t* ps = wsum + 32;                   // [n] positions
    int32_t* mem = ps + a.ostride;             // [n] slots grouped by bucket
    const View& v = a.v;
    const int32_t uu = blockIdx.x, u = a.u0 + uu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t n0 = v.len[u], p0 = v.next_pos[u];
    // fused step: the new token enters slot n0 first (its page is mapped: the host checked)
    const int32_t n = a.fused ? n0 + 1 : n0;
    const int32_t t = a.fused ? p0 : p0 - 1;
    if (a.fused) {
        __syncthreads();   // every thread has read the old length and position
        const int vec = v.row_bytes / 16;
        if (tid < 2 * vec) {
            const bool isv = tid >= vec;
            const int c = isv ? tid - vec : tid;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(isv ? a.new_v : a.new_k) + (int64_t)uu * v.row_bytes;
            uint8_t* dst = elem_row(v, u, n0, isv);
            if (dst) reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(src)[c];
        }
        if (tid == 0) {
            v.pos[(int64_t)u * v.cap + n0] = p0;
            v.imp[(int64_t)u * v.cap + n0] = 0.f;
            v.len[u] = n;
            v.next_pos[u] = p0 + 1;
        }
        __syncthreads();   // the new slot's position is visible to the block
    }
    // q of this warp's head (warps < G), loaded first so its latency overlaps the ranking
    const int D = v.d, PERL = D / 32;   // PERL <= 4
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp < v.group) {
        const int per_layer = v.batch * v.hkv;
        const int li = u / per_layer - a.layer0, b = (u / v.hkv) % v.batch, gh = u % v.hkv;
        const int64_t qoff = (((int64_t)li * v.batch + b) * v.hq + (int64_t)gh * v.group + warp) * D;
        for (int k = 0; k < PERL; ++k) {
            const int c = k * 32 + lane;
            x[k] = v.row_bytes == D * 2 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.q)[qoff + c])
                                        : reinterpret_cast<const float*>(a.q)[qoff + c];
        }
    }
    int shift = 0;
    while ((((int64_t)t + 1 + (1ll << shift) - 1) >> shift) > kOrderBuckets) ++shift;
    for (int b = tid; b < kOrderBuckets; b += kOrderThreads) cur[b] = 0;
    __syncthreads();
    for (int j = tid; j < n; j += kOrderThreads) {
        int32_t p = v.pos[(int64_t)u * v.cap + j];
        if (p < 0 || p > t) {
            atomicOr(v.err, DEVERR_STATE);
            p = p < 0 ? 0 : t;
        }
        ps[j] = p;
        atomicAdd(&cur[p >> shift], 1);
    }
    __syncthreads();
    // exclusive scan of the counts: 4 consecutive buckets per thread
    constexpr int PER = kOrderBuckets / kOrderThreads;
    int32_t c[PER], run = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        c[k] = cur[tid * PER + k];
        run += c[k];
    }
    int32_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int32_t base = incl - run;
    for (int w = 0; w < warp; ++w) base += wsum[w];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        start[tid * PER + k] = base;
        cur[tid * PER + k] = base;
        base += c[k];
    }
    __syncthreads();
    for (int j = tid; j < n; j += kOrderThreads) mem[atomicAdd(&cur[ps[j] >> shift], 1)] = j;
    __syncthreads();
    int32_t* ord = a.order + (int64_t)uu * a.ostride;
    for (int j = tid; j < n; j += kOrderThreads) {
        const int32_t p = ps[j], b = p >> shift;
        const int32_t e = b + 1 < kOrderBuckets ? start[b + 1] : n;
        int32_t r = start[b];
        for (int k = start[b]; k < e; ++k) r += ps[mem[k]] < p;
        ord[r] = j;
    }
    // K side of the unit's query heads: warp h keeps the b2 dimensions of q_h
    // with the largest |q| (ties: the lower index) and zeroes the rest
    if (warp < v.group) {
        const int h = warp;
        uint32_t key[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) key[k] = __float_as_uint(fabsf(x[k]));   // |q| >= 0: bits order like values
        uint32_t thr = 0u;
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = thr | (1u << bit);
            int cntb = 0;
            for (int k = 0; k < PERL; ++k) cntb += __popc(__ballot_sync(0xffffffffu, key[k] >= cand));
            if (cntb >= a.b2) thr = cand;
        }
        int above = 0;
        for (int k = 0; k < PERL; ++k) above += __popc(__ballot_sync(0xffffffffu, key[k] > thr));
        const int need = a.b2 - above;
        int before = 0;
        float* qm = a.qmask + ((int64_t)uu * v.group + h) * D;
        for (int k = 0; k < PERL; ++k) {
            const unsigned eq = __ballot_sync(0xffffffffu, key[k] == thr);
            const int mine = before + __popc(eq & ((1u << lane) - 1u));
            const bool keep = key[k] > thr || (key[k] == thr && mine < need);
            qm[k * 32 + lane] = keep ? x[k] : 0.f;
            before += __popc(eq);
        }
    }
}

// ---------------------------------------------------------------------------
// merge of a unit's spans (run by its last span CTA): output, importance from
// the whole P, and the victim -- the smallest (imp, -pos) outside sinks and window
// ---------------------------------------------------------------------------
template <typename T, int D, int G>
__device__ void merge_unit(const ElemArgs& a, int32_t uu, int32_t u, int32_t n, float* scratch,
                           unsigned long long* wkey, int32_t* wslot) {
    const View& v = a.v;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsp = (n + kElemSpan - 1) / kElemSpan;
    float* mfin = scratch;                 // [G]
    float* linv = scratch + kElemMaxG;     // [G]
    float* wsp = scratch + 2 * kElemMaxG;  // [G][nsp]: span m, then merge weight
    float* lsp = wsp + G * nsp;            // [G][nsp]: span l
    const float* part = a.part + (int64_t)uu * a.nsp * G * (D + 2);
    // the importance pass's first loads go out first: they do not depend on the merge
    const float* lgu = a.lg + (int64_t)uu * G * a.ostride;
    constexpr int MB = G >= 8 ? 1 : 8 / G;   // slots per thread whose loads are issued together
    float lgv[MB][G], iv[MB];
    int32_t pv[MB];
    auto load_batch = [&](int j0) {
#pragma unroll
        for (int q = 0; q < MB; ++q) {
            const int j = j0 + q * kElemThreads;
            if (j >= n) continue;
            const int64_t mi = (int64_t)u * v.cap + j;
#pragma unroll
            for (int h = 0; h < G; ++h) lgv[q][h] = __ldcg(lgu + (int64_t)h * a.ostride + j);
            iv[q] = v.imp[mi];
            pv[q] = v.pos[mi];
        }
    };
    load_batch(tid);
    for (int e = tid; e < G * nsp; e += kElemThreads) {   // all spans' (m, l) in one round trip
        const int s = e / G, h = e - s * G;
        wsp[h * nsp + s] = __ldcg(part + (int64_t)e * (D + 2));
        lsp[h * nsp + s] = __ldcg(part + (int64_t)e * (D + 2) + 1);
    }
    __syncthreads();
    if (tid < G) {
        const int h = tid;
        float m = -INFINITY;
        for (int s = 0; s < nsp; ++s) m = fmaxf(m, wsp[h * nsp + s]);
        float l = 0.f;
        for (int s = 0; s < nsp; ++s) {
            const float ls = lsp[h * nsp + s];
            const float w = ls > 0.f ? exp2f(wsp[h * nsp + s] - m) : 0.f;
            wsp[h * nsp + s] = w;
            l += ls * w;
        }
        mfin[h] = m;
        linv[h] = 1.0f / l;
    }
    __syncthreads();
    const int per_layer = v.batch * v.hkv;
    const int li = u / per_layer - a.layer0, b = (u / v.hkv) % v.batch, gh = u % v.hkv;
    T* outg = reinterpret_cast<T*>(a.out) + (((int64_t)li * v.batch + b) * v.hq + (int64_t)gh * G) * D;
    for (int e = tid; e < G * D; e += kElemThreads) {
        const int h = e / D, c = e - h * D;
        float o = 0.f;
#pragma unroll 8
        for (int s = 0; s < nsp; ++s) o = fmaf(__ldcg(part + ((int64_t)s * G + h) * (D + 2) + 2 + c), wsp[h * nsp + s], o);
        store_out(outg + e, o * linv[h]);
    }
    const int32_t tnew = v.next_pos[u] - 1;
    const bool need_victim = n > v.budget[u];
    const int32_t lo = v.sink, hi = tnew - v.window;
    unsigned long long kmin = ~0ull;
    int32_t smin = -1;
    for (int j0 = tid; j0 < n; j0 += kElemThreads * MB) {
        if (j0 != tid) load_batch(j0);
#pragma unroll
        for (int q = 0; q < MB; ++q) {
            const int j = j0 + q * kElemThreads;
            if (j >= n) continue;
            float inc = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h) inc += exp2f(lgv[q][h] - mfin[h]) * linv[h];
            const int32_t p = pv[q];
            const bool grows = !v.recent_only || p >= tnew - v.window;
            const float nw = grows ? iv[q] + inc : iv[q];
            v.imp[(int64_t)u * v.cap + j] = nw;
            if (need_victim && p >= lo && p <= hi) {
                const unsigned long long key =
                    ((unsigned long long)__float_as_uint(nw) << 32) | (unsigned long long)(~(uint32_t)p);
                if (key < kmin) {
                    kmin = key;
                    smin = j;
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long ok = __shfl_xor_sync(0xffffffffu, kmin, o);
        const int32_t os = __shfl_xor_sync(0xffffffffu, smin, o);
        if (ok < kmin) {
            kmin = ok;
            smin = os;
        }
    }
    __syncthreads();   // the warp counts sharing this scratch are no longer read
    if (lane == 0) {
        wkey[warp] = kmin;
        wslot[warp] = smin;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned long long kk = ~0ull;
        int32_t sl = -1;
        for (int w = 0; w < kElemWarps; ++w)
            if (wkey[w] < kk) {
                kk = wkey[w];
                sl = wslot[w];
            }
        wslot[kElemWarps] = need_victim ? sl : -1;
    }
    __syncthreads();   // the victim, and every slot's new importance, are visible to the block
    const int32_t vs = wslot[kElemWarps];
    if (!a.fused) {
        if (tid == 0) v.victim[u] = vs;
        return;
    }
    // fused step: with evict, the appended token (last slot) moves into the victim's slot
    const bool cut = a.evict && vs >= 0;
    if (cut && vs != n - 1) {
        const int vec = v.row_bytes / 16;
        if (tid < 2 * vec) {
            const bool isv = tid >= vec;
            const int c = isv ? tid - vec : tid;
            const uint8_t* src = elem_row(v, u, n - 1, isv);
            uint8_t* dst = elem_row(v, u, vs, isv);
            if (src && dst) reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(src)[c];
        }
        if (tid == 0) {
            v.imp[(int64_t)u * v.cap + vs] = v.imp[(int64_t)u * v.cap + n - 1];
            v.pos[(int64_t)u * v.cap + vs] = v.pos[(int64_t)u * v.cap + n - 1];
        }
    }
    if (v.debug && cut) {
        __syncthreads();
        if (tid < 32) poison_slot(v, u, n - 1, tid, 32);   // the last slot is vacated
    }
    if (tid == 0) {
        v.victim[u] = cut ? -1 : vs;
        v.len[u] = cut ? n - 1 : n;
    }
}

// ---------------------------------------------------------------------------
// k_elem_span
// ---------------------------------------------------------------------------
template <int D>
struct SpanLayout {
    size_t sl, pt, qm, S, sel, ul, ml, op, cnt, total;
    __host__ __device__ SpanLayout(int G) {
        size_t o = 0;
        auto take = [&](size_t bytes) { size_t r = o; o += (bytes + 15) / 16 * 16; return r; };
        sl = take(kElemSpan * 4);                        // slot of each rank
        pt = take(kElemMaxPages * 4);                    // the unit's page table
        qm = take((size_t)G * D * 4);                    // q with the dropped dimensions zeroed
        S = take((size_t)G * kElemSpan * 4);             // logits, then p of the kept entries
        sel = take((size_t)G * kElemSpan);               // kept by head h
        ul = take(kElemSpan * 4);                        // ranks some head kept
        ml = take((size_t)2 * kElemMaxG * 4);            // span (m, l) per head
        op = take((size_t)kElemWarps * G * D * 4);       // per-warp output sums; merge weights
        cnt = take(kElemWarps * 16 + 16);                // warp counts / victim keys, last-CTA flag
        total = o;
    }
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kElemThreads, (G >= 8 || sizeof(T) == 4) ? 3 : 4) k_elem_span(const ElemArgs a) {
    constexpr int DK = D / 8;    // dimensions per lane in the q.k pass (8 lanes per row)
    constexpr int DV = D / 32;   // dimensions per lane in the p.v pass (a warp per row)
    extern __shared__ __align__(16) uint8_t esm[];
    const View& v = a.v;
    const SpanLayout<D> L(G);
    int32_t* sl = reinterpret_cast<int32_t*>(esm + L.sl);
    int32_t* pt = reinterpret_cast<int32_t*>(esm + L.pt);
    float* qm = reinterpret_cast<float*>(esm + L.qm);
    float* S = reinterpret_cast<float*>(esm + L.S);
    uint8_t* sel = esm + L.sel;
    int32_t* ul = reinterpret_cast<int32_t*>(esm + L.ul);
    float* ml = reinterpret_cast<float*>(esm + L.ml);
    float* op = reinterpret_cast<float*>(esm + L.op);
    int32_t* wcnt = reinterpret_cast<int32_t*>(esm + L.cnt);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t uu = blockIdx.y, u = a.u0 + uu, sp = blockIdx.x;
    // the length, this span's slots, the unit's page table and the masked q
    // are independent loads: all are issued before the length is used
    const int32_t r0 = sp * kElemSpan;
    const int32_t n = v.len[u];
    static_assert(kElemSpan <= kElemThreads, "one rank per thread");
    const int32_t* ord = a.order + (int64_t)uu * a.ostride;
    const int32_t my_slot = (tid < kElemSpan && r0 + tid < a.ostride) ? ord[r0 + tid] : 0;
    constexpr int PPT = kElemMaxPages / kElemThreads;
    const int npg = min(v.max_pages, (a.ostride + v.page_tokens - 1) >> v.page_shift);
    int32_t my_pg[PPT];
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int i = tid + k * kElemThreads;
        my_pg[k] = i < npg ? v.page_table[(int64_t)u * v.max_pages + i] : -1;
    }
    constexpr int QPT = (G * D + kElemThreads - 1) / kElemThreads;
    const float* qmg = a.qmask + (int64_t)uu * G * D;
    float my_q[QPT];
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
        const int e = tid + k * kElemThreads;
        my_q[k] = e < G * D ? qmg[e] : 0.f;
    }
    if (r0 >= n) return;
    const int32_t cnt = min(n - r0, kElemSpan);
    if (tid < cnt) sl[tid] = my_slot;
#pragma unroll
    for (int k = 0; k < PPT; ++k)
        if (tid + k * kElemThreads < npg) pt[tid + k * kElemThreads] = my_pg[k];
    // q staged interleaved by lane: the 4-float piece c4 of lane sub's DK
    // dimensions (sub * DK + 4 c4 ...) sits at (c4 * 8 + sub) * 4, so the 8
    // lanes of a row read 8 consecutive float4 (no bank conflicts)
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
        const int e = tid + k * kElemThreads;
        if (e >= G * D) break;
        const int h = e / D, c = e - h * D, sub = c / DK, rem = c - sub * DK;
        qm[h * D + ((rem >> 2) * 8 + sub) * 4 + (rem & 3)] = my_q[k];
    }
    __syncthreads();
    // row of a slot from the staged page table (slot < n <= ostride, so its page index is < npg)
    auto rowp = [&](int32_t slot, bool is_v) -> const uint8_t* {
        const int32_t pg = pt[slot >> v.page_shift];
        if (pg < 0 || pg >= v.pool_pages) {
            atomicOr(v.err, DEVERR_PAGE);
            return nullptr;
        }
        return v.pool + (int64_t)pg * v.page_bytes +
               ((is_v ? (int64_t)v.page_tokens : 0) + (slot & (v.page_tokens - 1))) * v.row_bytes;
    };

    // logits of the span's rows: 8 lanes per row, DK dimensions each
    {
        const int grp = lane >> 3, sub = lane & 7;
        float* lgu = a.lg + (int64_t)uu * G * a.ostride;
        // rows in flight per 8-lane group: about 32 registers of raw K words
        constexpr int RAW = DK * (int)sizeof(T) / 4;
        constexpr int UK = RAW <= 8 ? 4 : 2;
        for (int i0 = warp * 4; i0 < cnt; i0 += kElemWarps * 4 * UK) {
            RawVec<T, DK> kr[UK];
            bool ok[UK];
            int32_t slot[UK];
#pragma unroll
            for (int w = 0; w < UK; ++w) {
                const int i = i0 + w * kElemWarps * 4 + grp;
                ok[w] = i < cnt;
                slot[w] = ok[w] ? sl[i] : 0;
                const uint8_t* rp = ok[w] ? rowp(slot[w], false) : nullptr;
                ok[w] = ok[w] && rp;
                if (ok[w]) kr[w].load(rp + sub * DK * (int)sizeof(T));
            }
#pragma unroll
            for (int w = 0; w < UK; ++w) {
                const int i = i0 + w * kElemWarps * 4 + grp;
                float kx[1][DK];
                kr[w].widen(kx[0]);
                for (int h = 0; h < G; ++h) {
                    const float4* qv = reinterpret_cast<const float4*>(qm + h * D) + sub;
                    float acc = 0.f;
#pragma unroll
                    for (int c4 = 0; c4 < DK / 4; ++c4) {
                        const float4 qq = qv[c4 * 8];
                        if (ok[w]) {
                            acc = fmaf(qq.x, kx[0][4 * c4], acc);
                            acc = fmaf(qq.y, kx[0][4 * c4 + 1], acc);
                            acc = fmaf(qq.z, kx[0][4 * c4 + 2], acc);
                            acc = fmaf(qq.w, kx[0][4 * c4 + 3], acc);
                        }
                    }
                    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                    if (sub == 0 && i < cnt) {
                        const float s = ok[w] ? acc * a.qscale : -INFINITY;
                        S[h * kElemSpan + i] = s;
                        lgu[(int64_t)h * a.ostride + slot[w]] = s;
                    }
                }
            }
        }
    }
    __syncthreads();

    // per-head span statistics (warp h), then the chunk selections
    for (int h = warp; h < G; h += kElemWarps) {
        float m = -INFINITY;
        for (int i = lane; i < cnt; i += 32) m = fmaxf(m, S[h * kElemSpan + i]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        if (m > -INFINITY)
            for (int i = lane; i < cnt; i += 32) l += exp2f(S[h * kElemSpan + i] - m);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            ml[2 * h] = m;
            ml[2 * h + 1] = l;
        }
    }
    {
        constexpr int PER = D / 32;   // ranks of a chunk per lane: k * 32 + lane
        const int nch = (cnt + D - 1) / D;
        for (int task = warp; task < nch * G; task += kElemWarps) {
            const int ch = task / G, h = task - ch * G;
            const int base = ch * D;
            const int m_c = min(D, cnt - base);
            const float* Sh = S + h * kElemSpan + base;
            uint8_t* selh = sel + h * kElemSpan + base;
            if (m_c <= a.b2) {
                for (int k = lane; k < m_c; k += 32) selh[k] = 1;
                continue;
            }
            uint32_t key[PER];
            bool val[PER];
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int r = k * 32 + lane;
                val[k] = r < m_c;
                key[k] = val[k] ? ord_key(Sh[r]) : 0u;
            }
            // the B2-th largest key: set bits from the top while >= B2 keys reach
            uint32_t thr = 0u;
            for (int bit = 31; bit >= 0; --bit) {
                const uint32_t cand = thr | (1u << bit);
                int c = 0;
#pragma unroll
                for (int k = 0; k < PER; ++k) c += __popc(__ballot_sync(0xffffffffu, val[k] && key[k] >= cand));
                if (c >= a.b2) thr = cand;
            }
            int above = 0;
#pragma unroll
            for (int k = 0; k < PER; ++k) above += __popc(__ballot_sync(0xffffffffu, val[k] && key[k] > thr));
            // equal keys fill the rest, lower rank (position) first
            int need = a.b2 - above, before = 0;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const unsigned eq = __ballot_sync(0xffffffffu, val[k] && key[k] == thr);
                const int mine = before + __popc(eq & ((1u << lane) - 1u));
                const bool take = val[k] && (key[k] > thr || (key[k] == thr && mine < need));
                if (val[k]) selh[k * 32 + lane] = take ? 1 : 0;
                before += __popc(eq);
            }
        }
    }
    __syncthreads();

    // p of the kept entries (span-local reference), and the union of the heads' rows
    int keep_n = 0;
    {
        constexpr int RPT = (kElemSpan + kElemThreads - 1) / kElemThreads;   // ranks per thread
        int mine[RPT];
#pragma unroll
        for (int w = 0; w < RPT; ++w) {
            mine[w] = 0;
            const int r = tid + w * kElemThreads;
            if (r >= cnt) continue;
            int any = 0;
            for (int h = 0; h < G; ++h) {
                const bool k = sel[h * kElemSpan + r] != 0;
                const float p = k ? exp2f(S[h * kElemSpan + r] - ml[2 * h]) : 0.f;
                S[h * kElemSpan + r] = p;
                any |= k;
            }
            mine[w] = any;
        }
        // ordered compaction of the kept ranks (rank order; deterministic sums)
#pragma unroll
        for (int w = 0; w < RPT; ++w) {
            const unsigned m = __ballot_sync(0xffffffffu, mine[w]);
            if (lane == 0) wcnt[warp] = __popc(m);
            __syncthreads();
            int off = keep_n;
            for (int x = 0; x < warp; ++x) off += wcnt[x];
            for (int x = 0; x < kElemWarps; ++x) keep_n += wcnt[x];
            if (mine[w]) ul[off + __popc(m & ((1u << lane) - 1u))] = tid + w * kElemThreads;
            __syncthreads();
        }
    }

    if (tid == 0 && a.rows_loaded) atomicAdd(a.rows_loaded, (unsigned long long)keep_n);

    // p.v over the kept rows: a warp per row, DV dimensions per lane
    float acc[G][DV];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int c = 0; c < DV; ++c) acc[h][c] = 0.f;
    constexpr int UNR = G >= 4 ? 4 : 8;   // rows in flight per warp
    for (int j0 = warp; j0 < keep_n; j0 += kElemWarps * UNR) {
        float vx[UNR][DV];
        int rr[UNR];
        bool ok[UNR];
#pragma unroll
        for (int w = 0; w < UNR; ++w) {
            const int j = j0 + w * kElemWarps;
            ok[w] = j < keep_n;
            rr[w] = ok[w] ? ul[j] : 0;
            const uint8_t* rp = ok[w] ? rowp(sl[rr[w]], true) : nullptr;
            ok[w] = ok[w] && rp;
            if (ok[w]) load_vec<T, DV>(rp + lane * DV * (int)sizeof(T), vx[w]);
        }
#pragma unroll
        for (int w = 0; w < UNR; ++w) {
            if (!ok[w]) continue;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float p = S[h * kElemSpan + rr[w]];
#pragma unroll
                for (int c = 0; c < DV; ++c) acc[h][c] = fmaf(p, vx[w][c], acc[h][c]);
            }
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int c = 0; c < DV; ++c) op[((size_t)warp * G + h) * D + lane * DV + c] = acc[h][c];
    }
    __syncthreads();
    float* part = a.part + ((int64_t)uu * a.nsp + sp) * G * (D + 2);
    for (int e = tid; e < G * D; e += kElemThreads) {
        float s = 0.f;
        for (int w = 0; w < kElemWarps; ++w) s += op[(size_t)w * G * D + e];
        const int h = e / D, c = e - h * D;
        part[h * (D + 2) + 2 + c] = s;
    }
    if (tid < G) {
        part[tid * (D + 2)] = ml[2 * tid];
        part[tid * (D + 2) + 1] = ml[2 * tid + 1];
    }
    // the unit's last span CTA to finish merges them (no waiting: the others
    // have published their partials before counting themselves in)
    int32_t* last = wcnt + kElemWarps * 4;
    __threadfence();   // every thread's partial and logit stores, before the count
    __syncthreads();
    if (tid == 0) {
        const int32_t nsp_u = (n + kElemSpan - 1) / kElemSpan;
        *last = atomicAdd(&a.done[uu], 1) == nsp_u - 1;
    }
    __syncthreads();
    if (!*last) return;
    __threadfence();
    if (tid == 0) a.done[uu] = 0;   // ready for the next call
    merge_unit<T, D, G>(a, uu, u, n, op, reinterpret_cast<unsigned long long*>(wcnt), wcnt + kElemWarps * 2);
}

template <typename T, int D, int G>
cudaError_t launch_elem_t(const ElemArgs& a, int max_n, cudaStream_t s) {
    const size_t osmem = order_smem(a.ostride);
    const size_t ssmem = SpanLayout<D>(G).total;
    cudaError_t e0 = func_smem_optin(reinterpret_cast<const void*>(k_elem_order), osmem);
    if (e0 == cudaSuccess) e0 = func_smem_optin(reinterpret_cast<const void*>(k_elem_span<T, D, G>), ssmem);
    if (e0 != cudaSuccess) return e0;
    k_elem_order<<<a.nunits, kOrderThreads, osmem, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_elem_span<T, D, G><<<dim3(a.nsp, a.nunits), kElemThreads, ssmem, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_elem_g(const ElemArgs& a, int max_n, cudaStream_t s) {
    switch (a.v.group) {
        case 1: return launch_elem_t<T, D, 1>(a, max_n, s);
        case 2: return launch_elem_t<T, D, 2>(a, max_n, s);
        case 4: return launch_elem_t<T, D, 4>(a, max_n, s);
        case 8: return launch_elem_t<T, D, 8>(a, max_n, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int elem_span_ranks() { return kElemSpan; }
int elem_max_tokens() { return 16384; }

cudaError_t launch_elem_decode(const ElemArgs& a, int dtype, int d, int max_n, cudaStream_t s) {
    if (a.v.group > kElemMaxG || a.nsp > kElemMaxSpans || a.ostride > elem_max_tokens()) return cudaErrorInvalidValue;
    if (dtype == 0 && d == 64) return launch_elem_g<float, 64>(a, max_n, s);
    if (dtype == 0 && d == 128) return launch_elem_g<float, 128>(a, max_n, s);
    if (dtype == 1 && d == 64) return launch_elem_g<__nv_bfloat16, 64>(a, max_n, s);
    if (dtype == 1 && d == 128) return launch_elem_g<__nv_bfloat16, 128>(a, max_n, s);
    return cudaErrorInvalidValue;
}

}  // namespace hikv
