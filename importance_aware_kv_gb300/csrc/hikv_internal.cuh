// Internal definitions shared by the hikv kernels and the host cache manager.
//
// Memory layout in HBM (one cache):
//   pool        [pool_pages] pages; a page holds P consecutive slots of one
//               unit: K rows [P][d] then V rows [P][d], row = d * elem bytes.
//   page_table  [units][max_pages] int32 page ids (-1 = unmapped); slot s of
//               unit u lives in page page_table[u][s / P], row s % P.
//   imp, pos    [units][cap] fp32 importance and int32 original position of
//               every slot; slots [0, len[u]) are live, densely packed.
//   len, next_pos, mapped, victim   [units] int32 per-unit state.
//   free_stack  [pool_pages] ids of free pages, free_stack[0, *free_top).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace hikv {

// device error word bits
enum : uint32_t {
    DEVERR_TIMEOUT = 1u,     // a bounded mbarrier wait gave up
    DEVERR_PAGE = 2u,        // page id out of range / unmapped page touched
    DEVERR_POOL = 4u,        // free stack under/overflow
    DEVERR_STATE = 8u,       // inconsistent per-unit state
};

struct View {
    uint8_t* pool;
    int32_t* page_table;
    float* imp;
    int32_t* pos;
    int32_t* len;
    int32_t* next_pos;
    int32_t* mapped;
    int32_t* victim;
    int32_t* budget;      // [units]
    int32_t* free_stack;
    int32_t* free_top;
    uint32_t* err;
    int64_t page_bytes;   // 2 * P * row_bytes
    int32_t row_bytes;    // d * elem
    int32_t page_tokens;  // P (power of two)
    int32_t page_shift;   // log2(P)
    int32_t max_pages;    // per unit
    int32_t cap;          // slots per unit (metadata row stride)
    int32_t pool_pages;
    int32_t units;
    int32_t batch, hq, hkv, group, d;
    int32_t sink, window;
    int32_t recent_only;  // HiKV Stage I: decode steps add mass only to pos >= t - window
    int32_t home_pages;   // 1: page k of unit u is u * max_pages + k, mapped at create for good
                          // (the pool holds every unit's max_tokens); 0: pages from the free stack
    int32_t debug;        // 1: vacated slots and freed pages are overwritten with NaN, slot
                          // indices taken from data are range-checked (HIKV_DEBUG at create)
};

#ifndef HIKV_G8_GROUPS
#define HIKV_G8_GROUPS 2
#endif
constexpr int kMaxCS = 16;   // most CTAs (cluster size) per unit in the decode kernel

// Slots [t0, t1) of CTA c of a cs-CTA cluster for a unit of n tokens:
// chunks of ceil((n - 1) / cs) rounded up to whole 16-slot tiles, the last
// CTA taking the rest.  With n = 16k + 1 (a budget of whole tiles plus the
// new token) every CTA holds whole tiles and the last one a single extra
// row, so no tile is loaded by two CTAs and the tile counts balance.
__host__ __device__ inline int32_t dec_chunk(int32_t n, int32_t cs) {
    const int32_t m = n > 1 ? n - 1 : 1;
    return ((m + cs - 1) / cs + 15) / 16 * 16;
}
__host__ __device__ inline void dec_range(int32_t n, int32_t cs, int32_t c, int32_t& t0, int32_t& t1) {
    const int32_t ch = dec_chunk(n, cs);
    t0 = c * ch < n ? c * ch : n;
    t1 = c == cs - 1 ? n : (t0 + ch < n ? t0 + ch : n);
}
// most slots a CTA holds (the last CTA's chunk plus one)
__host__ __device__ inline int32_t dec_chunk_max(int32_t n, int32_t cs) {
    const int32_t ch = dec_chunk(n, cs);
    return ch + 1 < n ? ch + 1 : n;
}

// Pages a unit keeps after being cut to its budget B: room for B + kKeepSlack
// tokens, so the appends of up to kKeepSlack steps before the next eviction
// (a batched eviction interval) never need a page.
constexpr int kKeepSlack = 16;
__host__ __device__ inline int32_t pages_kept(int32_t B, int32_t page_tokens, int32_t max_pages) {
    const int32_t k = (B + kKeepSlack + page_tokens - 1) / page_tokens;
    return k < max_pages ? k : max_pages;
}

// Shape of the decode kernel for a K/V row of `row_bytes` and group size
// `group`: CTAs resident per SM (its register cap and the host's grid sizing
// follow it), consumer warps per CTA, and ring stages (tiles of 16 K + 16 V
// rows).  Two CTAs of four consumer warps (three CTAs of three warps measured
// slower on every workload).  Two stages per consumer warp: the stage count
// must be a multiple of the consumer warps, so that the same warp consumes
// successive fills of a stage -- a consumer waits on a stage by phase parity,
// which is only sound when it has itself seen the stage's previous phase
// complete.
__host__ __device__ constexpr int dec_occupancy(int /*row_bytes*/, int /*group*/) { return 2; }
// consumer warps of one head group
__host__ __device__ constexpr int dec_consumer_warps(int /*row_bytes*/, int /*group*/) { return 4; }
// Tensor-core decode (HIKV_DECODE_TC=1 at compile time): groups of eight
// query heads on bf16 rows of d = 128 run q.k and p.v as mma.sync m16n8k16
// (the eight heads in one warp's n = 8), with one head group.  Measured on
// the 70B shape (640 units of 4,097 tokens): 312 us against 404 us for the
// two CUDA-core head groups.  Off by default: on that shape's heavy-hitter
// logits it failed the one-ulp bf16 output check in one full test run of
// three (two-ulp errors on outputs of the first head of a group) with the
// same code and data that passed the other two: not deterministic, so more
// likely a race in this path than the mma's accumulation precision; the
// cause was not found.  With four heads the CUDA-core row-split path is as
// fast.
#ifndef HIKV_DECODE_TC
#define HIKV_DECODE_TC 0
#endif
__host__ __device__ constexpr bool dec_tc(int elem_bytes, int d, int group) {
    return HIKV_DECODE_TC != 0 && elem_bytes == 2 && d == 128 && group == 8;
}
// Head groups of a decode CTA: with G = 8 each tile is consumed by two warps,
// one per half of the group's query heads (two sets of dec_consumer_warps
// warps rotating over the same tiles), so a warp carries the state of four
// heads and twice the warps hide the tile loop's latency.
__host__ __device__ constexpr int dec_head_groups(int group, bool tc) { return group == 8 && !tc ? HIKV_G8_GROUPS : 1; }
__host__ __device__ constexpr int dec_stages(int /*row_bytes*/, int /*group*/) { return 8; }

__host__ __device__ inline int32_t ceil_div(int32_t a, int32_t b) { return (a + b - 1) / b; }

// Page id of slot s of unit u: computed for home pages (no memory access),
// else read from the page table.
__device__ __forceinline__ int32_t unit_page(const View& v, int32_t u, int32_t s) {
    return v.home_pages ? u * v.max_pages + (s >> v.page_shift)
                        : v.page_table[(int64_t)u * v.max_pages + (s >> v.page_shift)];
}

// Debug mode: overwrite slot s of unit u -- its K and V rows with NaN, its
// importance with NaN, its position with -1 -- so that a kernel that reads
// a dead slot poisons the outputs it feeds.  Lanes [0, nlanes) share it.
__device__ __forceinline__ void poison_slot(const View& v, int32_t u, int32_t s, int lane, int nlanes) {
    if (s < 0 || s >= v.cap) {
        if (lane == 0) atomicOr(v.err, DEVERR_STATE);
        return;
    }
    const int32_t pg = v.home_pages ? u * v.max_pages + (s >> v.page_shift)
                                    : v.page_table[(int64_t)u * v.max_pages + (s >> v.page_shift)];
    if (pg >= 0 && pg < v.pool_pages) {
        const uint32_t w = v.row_bytes == 2 * v.d ? 0x7FC07FC0u : 0x7FC00000u;   // bf16 pair / fp32 NaN
        const int32_t vec = v.row_bytes / 16;
        uint8_t* kr = v.pool + (int64_t)pg * v.page_bytes + (int64_t)(s & (v.page_tokens - 1)) * v.row_bytes;
        for (int32_t i = lane; i < 2 * vec; i += nlanes) {
            uint8_t* row = i < vec ? kr : kr + (int64_t)v.page_tokens * v.row_bytes;
            reinterpret_cast<uint4*>(row)[i < vec ? i : i - vec] = make_uint4(w, w, w, w);
        }
    }
    if (lane == 0) {
        v.imp[(int64_t)u * v.cap + s] = __int_as_float(0x7FC00000);
        v.pos[(int64_t)u * v.cap + s] = -1;
    }
}

// Address of the K (or V) row of slot s of unit u; nullptr if the page is bad.
__device__ __forceinline__ uint8_t* row_ptr(const View& v, int32_t u, int32_t s, bool is_v) {
    int32_t pg = v.page_table[(int64_t)u * v.max_pages + (s >> v.page_shift)];
    if (pg < 0 || pg >= v.pool_pages) {
        atomicOr(v.err, DEVERR_PAGE);
        return nullptr;
    }
    int32_t r = s & (v.page_tokens - 1);
    return v.pool + (int64_t)pg * v.page_bytes +
           ((is_v ? (int64_t)v.page_tokens : 0) + r) * v.row_bytes;
}

// ---------------------------------------------------------------------------
// PTX wrappers (sm_90+ mbarrier / bulk copy / cluster; used on sm_103a)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the thread may sleep up to `ns` inside
// the instruction until the phase completes, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// try_wait with cluster-scope acquire: completes the wait for data that CTAs
// of the same cluster stored into this CTA's shared memory before arriving
// (remotely) on the barrier with release semantics.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}


// Arrive on the mbarrier at shared::cluster address `addr` (possibly in
// another CTA of the cluster), releasing this thread's prior writes -- and
// those ordered before them -- at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

__device__ __forceinline__ void prefetch_global_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Where the first bounded wait of a launch sequence gave up: err[1] = site
// (a kWait* code), err[2] = blockIdx.y, err[3] = blockIdx.x, err[4] = a
// site-specific index, err[5] = microseconds waited.
enum : uint32_t {
    kWaitQEmpty = 1, kWaitEmpty = 2, kWaitDrain = 3, kWaitQFull = 4, kWaitFull = 5, kWaitXchg = 6,
    kWaitVictim = 7, kWaitSelftest = 8
};
__device__ __forceinline__ void record_timeout(uint32_t* err, uint32_t site, uint32_t extra, uint64_t waited_ns) {
    atomicOr(err, DEVERR_TIMEOUT);
    if (atomicCAS(err + 1, 0u, site) == 0u) {
        err[2] = blockIdx.y;
        err[3] = blockIdx.x;
        err[4] = extra;
        const uint64_t us = waited_ns / 1000u;
        err[5] = us > 0xffffffffull ? 0xffffffffu : (uint32_t)us;
    }
}

// Bounded waits: give up after about two seconds (global timer; at most 2^24
// tries of a ~1 us suspend each, should the timer not advance), record where
// and return false.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t site,
                                                  uint32_t extra, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait_hint(bar, parity, 1000u)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        if (mbar_try_wait_hint(bar, parity, 1000u)) return true;
        if ((i & 63u) == 63u && global_ns() - t0 > limit_ns) break;
    }
    record_timeout(err, site, extra, global_ns() - t0);
    return false;
}
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity, uint32_t* err,
                                                          uint32_t site, uint32_t extra) {
    if (mbar_try_wait_cluster(bar, parity, 1000u)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        if (mbar_try_wait_cluster(bar, parity, 1000u)) return true;
        if ((i & 63u) == 63u && global_ns() - t0 > kWaitLimitNs) break;
    }
    record_timeout(err, site, extra, global_ns() - t0);
    return false;
}

// Start pulling `bytes` at `src` from HBM into L2 (no destination, no wait).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled TMA load of box {x, y} of `tmap` into shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tmap, int32_t x, int32_t y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// packed fp32 pair FMA (two lanes of a float2 at once)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(*reinterpret_cast<unsigned long long*>(&d))
        : "l"(*reinterpret_cast<const unsigned long long*>(&a)),
          "l"(*reinterpret_cast<const unsigned long long*>(&b)),
          "l"(*reinterpret_cast<const unsigned long long*>(&c)));
    return d;
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
// mma.sync m16n8k16, bf16 operands, fp32 accumulate: D = A * B + D with A
// 16 x 16 row-major (4 registers), B 16 x 8 column-major (2 registers).
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices from shared memory: lane l gives the address of row
// (l mod 8) of matrix l / 8 (16 contiguous bytes); register i receives
// matrix i, each lane holding row lane / 4, columns 2 (lane mod 4) and + 1.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr));
}
// the same, each matrix transposed: lane l receives column l / 4, rows
// 2 (l mod 4) and + 1 of the stored matrix
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr));
}

// two floats as a bf16 pair (round to nearest even), the first in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}

// x0, x1 as three bf16 pairs whose sums give back their fp32 values: hi =
// x rounded to bf16, mid = the remainder (exact in fp32) rounded, lo = what
// is left of it rounded; 3 x 8 significant bits cover fp32's 24
__device__ __forceinline__ void split3_bf16(float x0, float x1, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
    const float h0 = __bfloat162float(__float2bfloat16_rn(x0)), h1 = __bfloat162float(__float2bfloat16_rn(x1));
    const float r0 = x0 - h0, r1 = x1 - h1;
    const float m0 = __bfloat162float(__float2bfloat16_rn(r0)), m1 = __bfloat162float(__float2bfloat16_rn(r1));
    hi = pack_bf16x2(h0, h1);
    mid = pack_bf16x2(m0, m1);
    lo = pack_bf16x2(r0 - m0, r1 - m1);
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// the two halves of cluster_sync_all, for work between them (whole warps)
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// arrive without release semantics: for signalling that this CTA's mbarriers
// are initialised, whose fence.mbarrier_init already released them at
// cluster scope (a release here would also wait for this thread's copies)
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Programmatic dependent launch: wait until the grid this one depends on
// (the previous kernel in the stream, when launched with programmatic stream
// serialisation) has completed and its memory is visible -- a no-op
// otherwise; and let the next grid in the stream be scheduled early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// shared::cluster address of `p` in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float dsmem_ld_f32_nv(uint32_t addr) {
    float v;
    asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void dsmem_st_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_u64(uint32_t addr, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_s32(uint32_t addr, int32_t v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// element conversion
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
    __device__ __forceinline__ static float to_f(float x) { return x; }
    __device__ __forceinline__ static float from_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    __device__ __forceinline__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// widen EPL consecutive elements held in raw registers
template <typename T, int EPL> struct Widen;
template <> struct Widen<__nv_bfloat16, 4> {   // 8 bytes
    __device__ __forceinline__ static void run(const uint2 r, float* f) {
        f[0] = __uint_as_float(r.x << 16);
        f[1] = __uint_as_float(r.x & 0xFFFF0000u);
        f[2] = __uint_as_float(r.y << 16);
        f[3] = __uint_as_float(r.y & 0xFFFF0000u);
    }
};
template <> struct Widen<__nv_bfloat16, 8> {   // 16 bytes
    __device__ __forceinline__ static void run(const uint4 r, float* f) {
        f[0] = __uint_as_float(r.x << 16);
        f[1] = __uint_as_float(r.x & 0xFFFF0000u);
        f[2] = __uint_as_float(r.y << 16);
        f[3] = __uint_as_float(r.y & 0xFFFF0000u);
        f[4] = __uint_as_float(r.z << 16);
        f[5] = __uint_as_float(r.z & 0xFFFF0000u);
        f[6] = __uint_as_float(r.w << 16);
        f[7] = __uint_as_float(r.w & 0xFFFF0000u);
    }
};
template <> struct Widen<__nv_bfloat16, 2> {   // 4 bytes
    __device__ __forceinline__ static void run(const uint32_t r, float* f) {
        f[0] = __uint_as_float(r << 16);
        f[1] = __uint_as_float(r & 0xFFFF0000u);
    }
};
template <> struct Widen<float, 2> {           // 8 bytes
    __device__ __forceinline__ static void run(const uint2 r, float* f) {
        f[0] = __uint_as_float(r.x);
        f[1] = __uint_as_float(r.y);
    }
};
template <> struct Widen<float, 4> {           // 16 bytes
    __device__ __forceinline__ static void run(const uint4 r, float* f) {
        f[0] = __uint_as_float(r.x);
        f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z);
        f[3] = __uint_as_float(r.w);
    }
};

// raw lane vector type: EPL * sizeof(T) bytes
template <int BYTES> struct RawVec;
template <> struct RawVec<4> { using type = uint32_t; };
template <> struct RawVec<8> { using type = uint2; };
template <> struct RawVec<16> { using type = uint4; };

// ---------------------------------------------------------------------------
// launchers (defined in the kernel files)
// ---------------------------------------------------------------------------
struct AppendArgs {
    View v;
    int32_t u0, nunits, ntok;
    const uint8_t* k;
    const uint8_t* vv;
    int32_t* base;   // scratch [units]: first slot of this append per unit
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);

struct DecodeArgs {
    View v;
    const int32_t* order;   // [n_units] absolute unit ids, launch order
    int32_t n_units;
    int32_t layer0;
    const uint8_t* q;
    uint8_t* out;
    float qscale;           // scale * log2(e)
    float* logits;          // global logit scratch [units][cap][G] (long path) or null
    unsigned long long* cand; // [units][16] local argmin keys
    int32_t* cand_slot;     // [units][16]
    int32_t cs;             // CTAs per unit (cluster size)
    int32_t chunk_cap;      // max tokens per CTA handled by the smem path
    // values the host mirror knows to be the same for every unit of the call
    // (-1: read per unit from device memory); they spare the kernel a chain of
    // dependent loads before its first copy can be issued
    int32_t uni_len, uni_budget, uni_next_pos;
    int32_t identity_u0;    // >= 0: unit of list index i is identity_u0 + i (order unused)
    // when set, cluster j takes the units assign[assign_off[j] .. assign_off[j+1])
    // (a balanced assignment) instead of every n_clusters-th of the launch order
    const int32_t* assign;
    const int32_t* assign_off;
    int32_t prefetch_tiles; // L2 prefetch distance in tiles (0: off)
    int32_t first_burst;    // tiles queued before waiting for the first to land (0: no wait); with
                            // every CTA queueing its whole ring at once, a CTA's first tile
                            // waits behind the others' (measured: 4 saves ~0.6 us of 25)
    int32_t n_clusters;     // persistent clusters launched; cluster y handles list indices y, y + n_clusters, ...
    // fused step (append + decode + one-token evict in one launch): fused = 1,
    // new_k/new_v the appended rows [units of the call][d]; evict = 1 moves
    // the new token into the victim's slot when the unit is over budget
    int32_t fused, evict;
    const uint8_t* new_k;
    const uint8_t* new_v;
    // programmatic dependent launch: 1 when the grid this launch may overlap
    // (the previous one in the stream) writes none of this launch's units, so
    // the kernel may load their pages before waiting for it; 0: wait first
    int32_t pdl_early;
};
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmap, int dtype, int d, int group,
                          bool smem_path, size_t smem_bytes, cudaStream_t s);
size_t decode_smem_bytes(int dtype, int d, int group, bool smem_path, int chunk_cap);
int decode_max_smem_chunk(int dtype, int d, int group, size_t smem_limit);
// clusters of `cs` decode CTAs of `smem_bytes` each that fit on the GPU at once
int decode_active_clusters(int dtype, int d, int group, bool smem_path, int cs, size_t smem_bytes);

// Small-unit decode: one consumer warp per unit (units of at most
// small_unit_cap(G) tokens; group sizes up to 4), same arithmetic as k_decode.
constexpr int kSmallWarps = 4;              // consumer warps per CTA (one unit each)
constexpr int kSmallLogitFloats = 1536;     // logits kept per warp: tokens x G
__host__ __device__ constexpr int small_unit_cap(int G) { return kSmallLogitFloats / G; }
struct SmallArgs {
    View v;
    const int32_t* list;      // unit ids, warp-major
    const int32_t* warp_off;  // [n_warps + 1]: warp i takes list[warp_off[i] .. warp_off[i+1])
    int32_t layer0;
    const uint8_t* q;
    uint8_t* out;
    float qscale;             // scale * log2(e)
    int32_t fused, evict;     // as in DecodeArgs
    const uint8_t* new_k;
    const uint8_t* new_v;
};
cudaError_t launch_decode_small(const SmallArgs& a, const CUtensorMap& tmap, int dtype, int d, int group,
                                int n_ctas, cudaStream_t s);

struct EvictArgs {
    View v;
    int32_t u0, nunits;
    int32_t* holes;          // scratch: per unit hole lists
    const int64_t* hole_off; // [units] offset of each unit's hole list
};
cudaError_t launch_evict_fast(const EvictArgs& a, cudaStream_t s);
cudaError_t launch_evict_general(const EvictArgs& a, cudaStream_t s);

struct WindowArgs {
    View v;
    int32_t u0, nunits, layer0, nq;
    const uint8_t* q;
    float qscale;
    float* part;        // [units][nchunks_max][G*nq][2] partial (m, l)
    int32_t nchunks_max; // per-unit stride of `part` in chunks
    int32_t nchunks_grid;// chunks launched (covers the longest unit of the call)
    int32_t chunk;      // tokens per CTA
};
cudaError_t launch_window(const WindowArgs& a, int dtype, int d, int group, cudaStream_t s);
// SnapKV pooling of the prompt scores of units [u0, u0 + nu) (slots must be
// in position order: nothing removed yet)
constexpr int kMaxPoolKernel = 64;
cudaError_t launch_pool_importance(const View& v, int32_t u0, int32_t nu, int k, cudaStream_t s);
// the tensor-core variant (bf16 K/V, at most 128 query vectors G*nq)
bool window_tc_supported(int dtype, int d, int nqv);
cudaError_t launch_window_tc(const WindowArgs& a, const CUtensorMap& tmap, int d, int nqv, cudaStream_t s);

// HiKV banded prefill scores of the units [u0, u0 + units) of one layer
// (k_band.cu): q is the call's [nl][B][Hq][n][d] with this layer at index
// li; stats the [units][G][n] (m, 1/l) work buffer.
cudaError_t launch_band(const View& v, int32_t u0, int32_t units, int32_t li, const uint8_t* q, int32_t n,
                        int32_t band, float qscale, float2* stats, int dtype, cudaStream_t s);

struct GatherArgs {
    View v;
    int32_t u0, nunits, cap;
    int32_t* lengths;
    int32_t* positions;
    float* importance;
    uint8_t* k_out;
    uint8_t* v_out;
};
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s);
cudaError_t launch_selftest_timeout(const View& v, uint64_t limit_ns, cudaStream_t s);
// fill n 32-bit words at p with `word` (debug mode's NaN pool at create)
cudaError_t launch_fill_u32(uint32_t* p, size_t n, uint32_t word, cudaStream_t s);

// HiKV Stage II element-level decode (k_elem.cu): sort, span and merge kernels.
struct ElemArgs {
    View v;
    const void* q;         // [nl][B][Hq][d]
    void* out;             // [nl][B][Hq][d]
    int32_t u0, nunits, layer0;
    int32_t b2;            // element budget, 0 < b2 < d
    int32_t ostride;       // row stride of order / lg (>= every unit's length)
    int32_t nsp;           // span CTAs per unit in the grid
    float qscale;          // scale * log2(e)
    int32_t* order;        // [nunits][ostride] slots in position order
    float* lg;             // [nunits][G][ostride] logits by slot (log2 domain)
    float* part;           // [nunits][nsp][G][d + 2] span (m, l, o)
    float* qmask;          // [nunits][G][d] q with the dropped dimensions zeroed
    int32_t* done;         // [nunits] span CTAs finished (0 between calls)
    int32_t fused, evict;  // fused step: append new_k / new_v first; with evict, drop the victim at the end
    const void* new_k;     // [nunits][d] (fused)
    const void* new_v;
    unsigned long long* rows_loaded;   // += V rows read (may be null)
};
int elem_span_ranks();
int elem_max_tokens();
cudaError_t launch_elem_decode(const ElemArgs& a, int dtype, int d, int max_n, cudaStream_t s);

// Per-(kernel, device) attribute settings and occupancy queries, thread-safe (func_attr.cu).
cudaError_t func_smem_optin(const void* func, size_t bytes);
cudaError_t func_allow_nonportable_clusters(const void* func);
int func_active_clusters(const void* func, int cs, const cudaLaunchConfig_t& cfg);

}  // namespace hikv
