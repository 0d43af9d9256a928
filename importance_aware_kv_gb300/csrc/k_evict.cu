// Eviction: cut a unit holding n > B tokens to exactly B and compact it.
//
// Keep rule (blog sec. 3 "H2O" with StreamingLLM's sinks and window; per-head
// budgets B_u, HeadKV summary sec. 3.2): positions < S and > t - W are always
// kept; of the other "candidate" tokens keep the B - S - W with the largest
// (importance, -position), i.e. ties keep the lower position.
//
// Two kernels:
//   k_evict_fast     n == B + 1 right after a decode step: the decode kernel
//                    already found the single victim (fused argmin); the
//                    token in the last slot moves into the victim's slot.
//   k_evict_general  any n > B: a per-unit radix select over 64-bit keys
//                    (importance bits << 32 | ~position; importance >= 0 so
//                    the float bits order like the values) finds the
//                    (B-S-W)-th largest candidate key T; survivors are the
//                    protected tokens and candidates with key >= T (keys are
//                    unique, so exactly B survive).  Survivors sitting in
//                    slots >= B move into the dead slots < B, k-th with k-th
//                    in slot order, and whole pages past the unit's need go
//                    back to the pool (blog sec. 5.1: a compaction kernel
//                    coalescing survivors into dense blocks frees pages).
// HiKV's sorter and Kelle's systolic evictor do this selection in custom
// silicon; here it is a radix select in shared memory.
#include "hikv_internal.cuh"

namespace hikv {
namespace {

__device__ __forceinline__ unsigned long long mk_key(float imp, int32_t pos) {
    return ((unsigned long long)__float_as_uint(imp) << 32) | (unsigned long long)(~(uint32_t)pos);
}

__device__ void move_slot(const View& v, int32_t u, int32_t src, int32_t dst, int lane, int nlanes) {
    if (v.debug && (src < 0 || src >= v.cap || dst < 0 || dst >= v.cap)) {
        if (lane == 0) atomicOr(v.err, DEVERR_STATE);
        return;
    }
    const int32_t vec = v.row_bytes / 16;
    for (int32_t i = lane; i < 2 * vec; i += nlanes) {
        const bool isv = i >= vec;
        const int32_t c = isv ? i - vec : i;
        const uint8_t* s = row_ptr(v, u, src, isv);
        uint8_t* d = row_ptr(v, u, dst, isv);
        if (!s || !d) continue;
        reinterpret_cast<uint4*>(d)[c] = reinterpret_cast<const uint4*>(s)[c];
    }
    if (lane == 0) {
        const int64_t b = (int64_t)u * v.cap;
        v.imp[b + dst] = v.imp[b + src];
        v.pos[b + dst] = v.pos[b + src];
    }
}

// warp per unit
__global__ void k_evict_fast(EvictArgs a) {
    const int32_t w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= a.nunits) return;
    const View& v = a.v;
    const int32_t u = a.u0 + w;
    const int32_t n = v.len[u];
    const int32_t B = v.budget[u];
    if (n <= B) return;
    const int32_t vs = v.victim[u];
    if (n != B + 1 || vs < 0 || vs >= n) {
        if (lane == 0) atomicOr(v.err, DEVERR_STATE);
        return;
    }
    if (vs != n - 1) move_slot(v, u, n - 1, vs, lane, 32);
    __syncwarp();
    if (v.debug) {
        poison_slot(v, u, n - 1, lane, 32);   // the last slot is vacated
        __syncwarp();
    }
    if (lane == 0) {
        v.len[u] = B;
        v.victim[u] = -1;
    }
}

constexpr int kEvThreads = 256;
constexpr int kEvWarps = kEvThreads / 32;

// exclusive block scan of one flag per thread; returns this thread's rank,
// writes the block total to *total (all threads).
__device__ int32_t block_rank(bool flag, int32_t* wsum, int32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned m = __ballot_sync(0xffffffffu, flag);
    const int32_t in_warp = __popc(m & ((1u << lane) - 1u));
    if (lane == 0) wsum[warp] = __popc(m);
    __syncthreads();
    int32_t before = 0, all = 0;
    for (int i = 0; i < kEvWarps; ++i) {
        const int32_t x = wsum[i];
        before += i < warp ? x : 0;
        all += x;
    }
    __syncthreads();
    *total = all;
    return before + in_warp;
}

__global__ void __launch_bounds__(kEvThreads) k_evict_general(EvictArgs a) {
    const View& v = a.v;
    const int32_t u = a.u0 + blockIdx.x;
    const int32_t n = v.len[u];
    const int32_t B = v.budget[u];
    if (n <= B) return;
    const int32_t t = v.next_pos[u] - 1;
    const int32_t lo = v.sink, hi = t - v.window;
    const int32_t kmid = B - v.sink - v.window;
    const float* imp = v.imp + (int64_t)u * v.cap;
    const int32_t* pos = v.pos + (int64_t)u * v.cap;

    __shared__ uint32_t hist[kEvWarps][256];   // per-warp histograms
    __shared__ unsigned long long s_prefix, s_mask;
    __shared__ int32_t s_rem, s_done;
    __shared__ int32_t wsum[kEvWarps];
    __shared__ int32_t mv_src[kEvThreads], mv_dst[kEvThreads];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // --- radix select of the kmid-th largest candidate key, 8 bits a pass ---
    if (threadIdx.x == 0) {
        s_prefix = 0ull;
        s_mask = 0ull;
        s_rem = kmid;
        s_done = 0;
    }
    __syncthreads();
    if (kmid > 0) {
        for (int pass = 0; pass < 8; ++pass) {
            const int shift = 56 - 8 * pass;
            for (int i = threadIdx.x; i < kEvWarps * 256; i += kEvThreads) (&hist[0][0])[i] = 0;
            __syncthreads();
            const unsigned long long prefix = s_prefix, mask = s_mask;
            // keys of a candidate set share their high bits, so most fall in
            // a few bins: lanes with the same bin add once per warp
            for (int32_t s0 = 0; s0 < n; s0 += kEvThreads) {
                const int32_t s = s0 + threadIdx.x;
                uint32_t bin = 256u;   // no bin
                if (s < n) {
                    const int32_t p = pos[s];
                    if (p >= lo && p <= hi) {
                        const unsigned long long key = mk_key(imp[s], p);
                        if ((key & mask) == prefix) bin = (uint32_t)(key >> shift) & 255u;
                    }
                }
                const unsigned peers = __match_any_sync(0xffffffffu, bin);
                if (bin < 256u && lane == __ffs(peers) - 1) atomicAdd(&hist[warp][bin], (uint32_t)__popc(peers));
            }
            __syncthreads();
            if (warp == 0) {
                // lane l owns bins 8l .. 8l+7; find, from the top bin down, the
                // bin where the running count reaches rem
                uint32_t c[8];
                int32_t tot = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t x = 0;
                    for (int w = 0; w < kEvWarps; ++w) x += hist[w][8 * lane + j];
                    c[j] = x;
                    tot += (int32_t)x;
                }
                int32_t incl = tot;   // bins of lanes >= this one
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int32_t y = __shfl_down_sync(0xffffffffu, incl, o);
                    if (lane + o < 32) incl += y;
                }
                const int32_t above = incl - tot;   // bins of lanes > this one
                const int32_t rem = s_rem;
                if (above < rem && rem <= incl) {
                    int32_t cum = above, sel = 8 * lane, r = rem, csel = 0;
                    for (int j = 7; j >= 0; --j) {
                        if (cum + (int32_t)c[j] >= rem) {
                            sel = 8 * lane + j;
                            r = rem - cum;
                            csel = (int32_t)c[j];
                            break;
                        }
                        cum += (int32_t)c[j];
                    }
                    s_rem = r;
                    s_prefix = prefix | ((unsigned long long)sel << shift);
                    s_mask = mask | (255ull << shift);
                    // every key of the chosen bin survives: then the bin's
                    // lowest possible key (the prefix, low bits zero) already
                    // splits the kmid largest from the rest
                    s_done = r == csel;
                }
            }
            __syncthreads();
            if (s_done) break;
        }
    }
    const unsigned long long T = s_prefix;
    auto survives = [&](int32_t s) -> bool {
        const int32_t p = pos[s];
        if (p < lo || p > hi) return true;
        return kmid > 0 && mk_key(imp[s], p) >= T;
    };

    // --- holes: dead slots in [0, B), ascending ---
    int32_t* holes = a.holes + a.hole_off[u];
    const int32_t hole_cap = max(0, min(B, v.cap - B));   // size of this unit's hole list
    int32_t base = 0;
    for (int32_t s0 = 0; s0 < B; s0 += kEvThreads) {
        const int32_t s = s0 + threadIdx.x;
        const bool f = s < B && !survives(s);
        int32_t tot;
        const int32_t r = block_rank(f, wsum, &tot);
        if (f) {
            if (base + r < hole_cap) holes[base + r] = s;
            else atomicOr(v.err, DEVERR_STATE);
        }
        base += tot;
    }
    __syncthreads();
    const int32_t nholes = min(base, hole_cap);

    // --- movers: survivors in [B, n), ascending; k-th mover -> k-th hole.
    // Each batch of 256 slots lists its movers, then the warps copy them,
    // one 2-row move per warp (a lane per 16-byte chunk) ---
    base = 0;
    for (int32_t s0 = B; s0 < n; s0 += kEvThreads) {
        const int32_t s = s0 + threadIdx.x;
        const bool f = s < n && survives(s);
        int32_t tot;
        const int32_t r = block_rank(f, wsum, &tot);
        if (f) {
            if (base + r < nholes) {
                mv_src[r] = s;
                mv_dst[r] = holes[base + r];
            } else {
                atomicOr(v.err, DEVERR_STATE);
            }
        }
        __syncthreads();
        const int32_t cnt = min(tot, max(0, nholes - base));
        for (int32_t m = warp; m < cnt; m += kEvWarps) move_slot(v, u, mv_src[m], mv_dst[m], lane, 32);
        base += tot;
        __syncthreads();   // the mover list is rewritten by the next batch
    }
    __syncthreads();
    if (v.debug) {
        // every slot in [B, n) is vacated (moved down or evicted) ...
        for (int32_t s = B + warp; s < n; s += kEvWarps) poison_slot(v, u, s, lane, 32);
        // ... and every row of the pages about to return to a shared pool
        const int32_t keep = pages_kept(B, v.page_tokens, v.max_pages);
        const int32_t m = v.mapped[u];
        if (!v.home_pages && m > keep) {
            const uint32_t w = v.row_bytes == 2 * v.d ? 0x7FC07FC0u : 0x7FC00000u;
            const int64_t words = v.page_bytes / 16;
            for (int32_t k = keep; k < m; ++k) {
                const int32_t pg = v.page_table[(int64_t)u * v.max_pages + k];
                if (pg < 0 || pg >= v.pool_pages) continue;
                uint4* p = reinterpret_cast<uint4*>(v.pool + (int64_t)pg * v.page_bytes);
                for (int64_t i = threadIdx.x; i < words; i += kEvThreads) p[i] = make_uint4(w, w, w, w);
            }
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        if (base != nholes) atomicOr(v.err, DEVERR_STATE);
        v.len[u] = B;
        v.victim[u] = -1;
        // return whole pages past slot B (one spare slot kept for the next append)
        const int32_t keep = pages_kept(B, v.page_tokens, v.max_pages);
        const int32_t m = v.mapped[u];
        if (!v.home_pages && m > keep) {
            const int32_t cnt = m - keep;
            const int32_t old = atomicAdd(v.free_top, cnt);
            if (old + cnt > v.pool_pages) atomicOr(v.err, DEVERR_POOL);
            for (int32_t i = 0; i < cnt; ++i) {
                const int64_t e = (int64_t)u * v.max_pages + keep + i;
                if (old + i < v.pool_pages) v.free_stack[old + i] = v.page_table[e];
                v.page_table[e] = -1;
            }
            v.mapped[u] = keep;
        }
    }
}

}  // namespace

cudaError_t launch_evict_fast(const EvictArgs& a, cudaStream_t s) {
    if (a.nunits <= 0) return cudaSuccess;
    const int threads = 128;
    k_evict_fast<<<ceil_div(a.nunits * 32, threads), threads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_evict_general(const EvictArgs& a, cudaStream_t s) {
    if (a.nunits <= 0) return cudaSuccess;
    k_evict_general<<<a.nunits, kEvThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hikv
