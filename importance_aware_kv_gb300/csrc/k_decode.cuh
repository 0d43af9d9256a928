// Fused decode attention + importance update + victim argmin.
//
// Method: decode attention P = softmax(q K^T), O = P V over the retained
// tokens (HiKV sec. II-A; Kelle summary sec. 2.2); every retained token's
// importance accumulates P summed over the G query heads of its KV group
// (blog sec. 3 "H2O", sec. 5.2); the victim is the least important token that
// is neither a sink nor in the recent window, ties evicting the higher
// position (blog sec. 3 "H2O"/"StreamingLLM").  The fused argmin plays the
// role of the min-search that Kelle's systolic evictor runs alongside
// attention (Kelle summary sec. 5.3) and of HiKV's min-heap (sec. III-B).
//
// Persistent clusters: cluster y of CS CTAs processes the units of the launch
// list at indices y, y + n_clusters, ...; for each unit, CTA c takes the c-th
// of CS equal chunks of the unit's n live slots.  Per CTA:
//   producer warp   for unit after unit: copies the unit's q (1-D TMA bulk
//                   copy into a double buffer), loads the chunk's page ids,
//                   and streams 16-slot tiles, K rows and V rows together,
//                   with 2-D TMA tensor copies (128-byte swizzle) into an
//                   NSTAGE ring (mbarrier full/empty pairs, bounded waits).  It
//                   runs ahead into the next unit while the consumers finish
//                   the current one.
//   consumer warps  tile i of a unit belongs to warp i % 4, which keeps a
//                   private online softmax (reference m_w, sum l_w,
//                   unnormalised O_w; m_w follows the running max lazily,
//                   moving only when a logit exceeds it by 2^8).  With G = 8
//                   there are two such groups of four warps: both take tile
//                   i, one for heads 0-3 and one for heads 4-7, and a stage
//                   is released once each group's warp has arrived:
//     q.k   lane (row = lane % 16, half = lane / 16) owns half a K row: the
//           swizzle makes those 16-byte reads conflict-free and lets q be a
//           shared-memory broadcast; packed f32x2 FMAs, one shuffle joins the
//           halves; logits (scaled by log2 e) are kept for the importance pass;
//     p.v   lane owns d/32 output elements, packed f32x2 FMAs over the tile's
//           V rows with p broadcast from shared memory.
//   Per unit, the warp states merge per CTA, then each CTA stores its
//   (m_c, l_c) into every partner's shared memory and its output slices into
//   their owners' (DSMEM), and arrives remotely on their exchange mbarriers:
//     m = max_c m_c, l = sum_c l_c 2^(m_c - m); out_h = sum_c O_c[h] 2^(m_c - m) / l;
//     importance imp_j += sum_h 2^(s'_hj - m_h) / l_h (fp32 add, heads
//     ascending); each CTA's smallest eligible (imp, -pos) goes to CTA 0 the
//     same way, which records the unit's victim.  Exchange buffers are double
//     buffered by unit parity; no cluster barrier sits inside the unit loop.
#pragma once

#include "hikv_internal.cuh"

namespace hikv {

// threads of a decode CTA: the consumer warps and one producer warp
template <typename T, int D, int G>
constexpr int dec_threads() {
    return (dec_consumer_warps(D * (int)sizeof(T), G) * dec_head_groups(G, dec_tc((int)sizeof(T), D, G)) + 1) * 32;
}
constexpr int kDecTR = 16;                       // slots per tile
constexpr float kDecLazy = 8.f;                  // softmax reference slack (log2 units)
constexpr int kDecMaxPg = 256;                   // page ids cached in shared memory

struct DecSmem {
    // byte offsets into dynamic shared memory, from a 1024-aligned base
    uint32_t ring, bars, qraw, nrow, q, ps, red, xbuf, vbuf, small, pg, S, total;
    uint32_t xbuf_bytes;
};

template <typename T, int D, int G>
__host__ __device__ inline DecSmem dec_layout(bool smem_s, int chunk_cap) {
    constexpr uint32_t RB = D * sizeof(T);
    constexpr int kDecNGW = dec_consumer_warps(RB, G);   // warps per head group
    DecSmem L{};
    uint32_t off = 0;
    L.ring = off;                                 // K,V tiles
    off += dec_stages(RB, G) * 2 * kDecTR * RB;
    L.bars = off;                                 // full, empty [NST]; qfull, qempty, xbar, vbar [2]
    off += (2 * dec_stages(RB, G) + 8) * 8;
    off = (off + 127) & ~127u;
    L.qraw = off;                                 // q of the unit as stored, [2][G][D]
    off += 2 * G * D * sizeof(T);
    L.nrow = off;                                 // fused step: the new K and V rows, [2][2][D]
    off += 2 * 2 * RB;
    off = (off + 15) & ~15u;
    L.q = off;                                    // q * scale * log2 e, fp32 [G][D]
    off += G * D * 4;
    L.ps = off;                                   // per-warp p of the tile [NCW * HG][16][G / HG]
    // (= NCW * HG * 16 * G / HG; on the tensor cores [NCW][16][8], the heads padded to the mma's n = 8)
    off += kDecNGW * kDecTR * (dec_tc((int)sizeof(T), D, G) ? 8 : G) * 4;
    L.red = off;                                  // warp O partials [NGW][G][D]
    off += kDecNGW * G * D * 4;
    // exchange buffer per unit parity: m [kMaxCS][G], l [kMaxCS][G], O slices [G*D + kMaxCS]
    L.xbuf_bytes = (2 * kMaxCS * G + G * D + kMaxCS) * 4;
    L.xbuf = off;
    off += 2 * L.xbuf_bytes;
    L.vbuf = off;                                 // [2] x (keys [kMaxCS] u64, slots [kMaxCS] i32, new imp f32)
    off += 2 * (kMaxCS * 12 + 16);
    off = (off + 15) & ~15u;
    L.small = off;
    off += 2048;
    L.pg = off;                                   // page ids of the chunk
    off += kDecMaxPg * 4;
    L.S = off;
    if (smem_s) off += (uint32_t)chunk_cap * G * 4;
    L.total = ((off + 127) & ~127u) + 1024;       // + slack to align the base to 1024
    return L;
}

// byte offset of 16-byte chunk c of tile row r in a tile laid out as 128-byte
// swizzled boxes [c / 8][r][(c % 8) ^ (r % 8)]
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)((c >> 3) * (kDecTR * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// byte offset of 16-byte chunk c of row r in a tile of the cluster kernel:
// rows of RBYTES bytes in order, as one 1-D bulk copy of a page's
// consecutive rows lays them down (a warp reading whole rows, chunk by lane,
// reads contiguous bytes: no bank conflicts without a swizzle)
template <int RBYTES>
__device__ __forceinline__ uint32_t lin(int r, int c) {
    return (uint32_t)(r * RBYTES + (c << 4));
}

// Queue the copies of one tile -- 16 K rows and the 16 V rows P slots after
// them, starting at slot s0 of page pg -- into a ring stage (K at dst, V at
// dst + TB), completing on `bar`: two 1-D bulk copies of the contiguous rows
// (row-split path), or 2-D TMA boxes of 16 rows x 128 bytes that lay the
// rows down 128-byte swizzled (half-row path).
template <bool RS, int NBOX, int ESZ, int RB, int TB>
__device__ __forceinline__ void dec_load_tile(uint8_t* dst, const View& v, int32_t pg, int32_t s0,
                                              const CUtensorMap* tmap, uint64_t* bar) {
    if constexpr (RS) {
        const uint8_t* kb = v.pool + (int64_t)pg * v.page_bytes + (int64_t)(s0 & (v.page_tokens - 1)) * RB;
        bulk_g2s(dst, kb, (uint32_t)TB, bar);
        bulk_g2s(dst + TB, kb + (int64_t)v.page_tokens * RB, (uint32_t)TB, bar);
    } else {
        const int32_t yk = pg * 2 * v.page_tokens + (s0 & (v.page_tokens - 1));
#pragma unroll
        for (int bx = 0; bx < NBOX; ++bx) {
            tma_load_2d(dst + bx * (16 * 128), tmap, bx * (128 / ESZ), yk, bar);
            tma_load_2d(dst + TB + bx * (16 * 128), tmap, bx * (128 / ESZ), yk + v.page_tokens, bar);
        }
    }
}

// Reduce-scatter of v[0, N) over the lanes that differ in the bits of M,
// M / 2, ..., 1: at each level a lane keeps the half of its values that its
// bit selects (upper half when set) and adds the partner's copy of that
// half.  Afterwards v[0] holds, complete, the value whose index the lane's
// bits spell out (most significant level first); once one value is left,
// the remaining levels only sum it, so lanes differing in those bits hold
// the same total.  Values of different indices are never added together.
template <int M, int N>
__device__ __forceinline__ void qk_reduce(float* v, int lane) {
    if constexpr (M >= 1) {
        if constexpr (N > 1) {
            constexpr int H = N / 2;
            const bool up = (lane & M) != 0;
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const float send = up ? v[j] : v[j + H];
                const float keep = up ? v[j + H] : v[j];
                v[j] = keep + __shfl_xor_sync(0xffffffffu, send, M);
            }
            qk_reduce<M / 2, H>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
            qk_reduce<M / 2, 1>(v, lane);
        }
    }
}

// G consecutive floats (a row of p or logits, 4G-byte aligned), vectorised
template <int G>
__device__ __forceinline__ void store_group(float* dst, const float (&x)[G]) {
    if constexpr (G % 4 == 0) {
#pragma unroll
        for (int h = 0; h < G; h += 4)
            *reinterpret_cast<float4*>(dst + h) = make_float4(x[h], x[h + 1], x[h + 2], x[h + 3]);
    } else if constexpr (G == 2) {
        *reinterpret_cast<float2*>(dst) = make_float2(x[0], x[1]);
    } else {
#pragma unroll
        for (int h = 0; h < G; ++h) dst[h] = x[h];
    }
}

struct DecUnit {
    int32_t u, n, Bu, tnew;
};

// In a fused step the device length and position counters still describe the
// cache before the append; the unit then holds one more token, the new one,
// in slot n - 1 at position tnew.  (Uniform values from the host already
// include the append.)
__device__ __forceinline__ DecUnit dec_unit(const DecodeArgs& a, int32_t idx) {
    DecUnit r;
    r.u = a.assign ? a.assign[idx] : (a.identity_u0 >= 0 ? a.identity_u0 + idx : a.order[idx]);
    r.n = a.uni_len >= 0 ? a.uni_len : a.v.len[r.u] + a.fused;
    r.Bu = a.uni_budget >= 0 ? a.uni_budget : a.v.budget[r.u];
    r.tnew = (a.uni_next_pos >= 0 ? a.uni_next_pos : a.v.next_pos[r.u] + a.fused) - 1;
    return r;
}

template <typename T, int D, int G, bool SMEM_S>
__global__ void __launch_bounds__(dec_threads<T, D, G>(), dec_occupancy(D * sizeof(T), G))
    k_decode(const DecodeArgs a, const __grid_constant__ CUtensorMap tmap) {
    constexpr int ESZ = (int)sizeof(T);
    constexpr int kDecNGW = dec_consumer_warps(D * ESZ, G);   // warps of a head group (the tile rotation)
    constexpr bool kTC = dec_tc(ESZ, D, G);                      // q.k and p.v on the tensor cores
    constexpr int kHG = dec_head_groups(G, kTC);              // head groups
    constexpr int kDecNCW = kDecNGW * kHG;                    // consumer warps
    constexpr int GW = G / kHG;                               // query heads of a warp
    constexpr int RB = D * ESZ;              // row bytes: 128, 256 or 512
    constexpr int NBOX = RB / 128;           // 128-byte TMA boxes per row
    constexpr int TB = kDecTR * RB;          // K (or V) tile bytes
    constexpr int CPR = RB / 16;             // 16-byte chunks per row
    constexpr int EPC = 16 / ESZ;            // elements per chunk
    constexpr int EPL = D / 32;              // p.v: elements per lane
    constexpr int LB = EPL * ESZ;            // p.v: bytes per lane
    constexpr int NCT = kDecNCW * 32;        // consumer threads
    constexpr uint32_t QB = G * D * ESZ;     // bytes of one unit's q
    constexpr int kDecStages = dec_stages(RB, G);
    static_assert(kDecStages % kDecNGW == 0, "each stage must always be consumed by the same warp of each group");
    // q.k mapping: QK_LPR lanes share a K row, each taking one 16-byte chunk
    // of it against the same dimensions of q, which the lane keeps in
    // registers; a warp step covers QK_RPW rows.  A tile's QK_STEPS steps
    // run in QK_NSUB sub-blocks of QK_SUB steps, whose QK_NV = QK_SUB * GW
    // (row, head) partial sums are reduce-scattered over the row's lanes:
    // every lane ends each sub-block holding one finished logit, of one
    // fixed head (QK_DUP lanes hold the same one when QK_NV < QK_LPR).  The
    // per-tile shared-memory reads are then the K tile itself, not q again
    // for every row.
    // G = 8 runs two head groups of four warps at 96 registers, where the
    // q registers above do not fit: its warps keep the half-row mapping
    // (lane = tile row and half of it, q read from shared memory) over
    // 128-byte-swizzled tiles that 2-D TMA boxes lay down
    constexpr bool kRS = kHG == 1;
    // tiles laid down as plain rows by 1-D bulk copies (the row-split CUDA-
    // core path), else as 128-byte-swizzled 2-D TMA boxes (the half-row path,
    // and the tensor cores, whose ldmatrix row reads then hit distinct banks)
    constexpr bool kLin = kRS && !kTC;
    constexpr int CPL = CPR / 2;             // half-row q.k: chunks per lane
    constexpr int QK_LPR = RB / 16;
    constexpr int QK_RPW = 32 / QK_LPR;
    constexpr int QK_STEPS = kDecTR / QK_RPW;
    constexpr int QK_EPL = 16 / ESZ;
    constexpr int QK_SUB = (QK_LPR / GW) > QK_STEPS ? QK_STEPS : (QK_LPR / GW);
    constexpr int QK_NSUB = QK_STEPS / QK_SUB;
    constexpr int QK_NV = QK_SUB * GW;
    constexpr int QK_DUP = QK_LPR / QK_NV;
    static_assert(QK_SUB >= 1 && QK_STEPS % QK_SUB == 0 && QK_LPR % QK_NV == 0, "one logit per lane and sub-block");
    static_assert(EPL % 2 == 0 && EPC % 2 == 0, "pairs");
    using Raw = typename RawVec<LB>::type;

    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const View& v = a.v;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    const DecSmem L = dec_layout<T, D, G>(SMEM_S, a.chunk_cap);
    uint8_t* ring = smem + L.ring;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + kDecStages;
    uint64_t* qfull = empty + kDecStages;     // [2]
    uint64_t* qempty = qfull + 2;             // [2]
    uint64_t* xbar = qempty + 2;              // [2]
    uint64_t* vbar = xbar + 2;                // [2]
    float* q_s = reinterpret_cast<float*>(smem + L.q);
    float* ps_all = reinterpret_cast<float*>(smem + L.ps);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* sm = reinterpret_cast<float*>(smem + L.small);
    static_assert(kDecNGW * G <= 32, "warp state arrays");
    static_assert(kMaxCS * G <= NCT, "one consumer thread per (CTA, head) of the exchange");
    float* mw_s = sm;                          // [NGW][G]     (32)
    float* lw_s = sm + 32;                     // [NGW][G]     (32)
    float* wsc = sm + 64;                      // [NGW][G]     (32)
    float* mfin = sm + 96;                     // [G]
    float* linv = sm + 104;                    // [G]
    float* m_c = sm + 112;                     // [G]
    float* l_c = sm + 120;                     // [G]
    float* beta = sm + 128;                    // [kMaxCS][G]  (128)
    unsigned long long* wkey = reinterpret_cast<unsigned long long*>(sm + 256);  // [NCW]
    int32_t* wslot = reinterpret_cast<int32_t*>(wkey + kDecNCW);                 // [NCW]
    volatile int32_t* abort_flag = wslot + kDecNCW;
    float* new_imp_s = sm + 288;               // fused: the new token's final importance
    static_assert(256 + 3 * kDecNCW + 1 <= 288, "victim slots overlap");
    int32_t* pg_s = reinterpret_cast<int32_t*>(smem + L.pg);
    float* S_smem = reinterpret_cast<float*>(smem + L.S);

    const int32_t c = (int32_t)cluster_ctarank();
    const int32_t CS = (int32_t)cluster_nctarank();

    // this cluster's units: list indices it0, it0 + istep, ... < it1
    const int32_t it0 = a.assign_off ? a.assign_off[blockIdx.y] : (int32_t)blockIdx.y;
    const int32_t it1 = a.assign_off ? a.assign_off[blockIdx.y + 1] : a.n_units;
    const int32_t istep = a.assign_off ? 1 : a.n_clusters;

    // Programmatic dependent launch: this grid may start while the previous
    // one in the stream runs.  Unless the host found that one to write none
    // of this launch's units, wait for it before touching anything; else the
    // first tiles (this launch's own units) are queued before the wait, and
    // the caller's inputs (q, new rows) are read and `out` written after it.
    if (!a.pdl_early) griddep_wait();

    // producer: the first unit's page ids, loaded while the barriers are set up
    int32_t pre_pg = -1;
    if (warp == kDecNCW && it0 < it1) {
        const DecUnit du = dec_unit(a, it0);
        int32_t t0, t1;
        dec_range(du.n, CS, c, t0, t1);
        const int32_t pg0 = t0 >> v.page_shift;
        const int32_t npg = t1 > t0 ? ((t1 - 1) >> v.page_shift) - pg0 + 1 : 0;
        if (lane < npg && !v.home_pages) pre_pg = v.page_table[(int64_t)du.u * v.max_pages + pg0 + lane];
    }

    // The producer's lane 0 sets up the barriers and then queues the first
    // unit's q (and new rows) and, with home pages (tile addresses need no
    // lookup), its first tiles before the CTA-wide sync: those copies are the
    // launch's critical path.
    int32_t pre_issued = 0;
    bool pre_q = false;
    if (warp == kDecNCW && lane == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], (uint32_t)kHG);   // one warp of each head group releases the stage
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&qfull[b], 1);
            mbar_init(&qempty[b], 1);
            mbar_init(&xbar[b], (uint32_t)CS);
            mbar_init(&vbar[b], (uint32_t)CS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        if (v.home_pages && it0 < it1) {
            const DecUnit du = dec_unit(a, it0);
            int32_t t0, t1;
            dec_range(du.n, CS, c, t0, t1);
            const int32_t cnt = t1 - t0;
            const int32_t first_blk = t0 / kDecTR;
            const bool tail = cnt > 1 && (cnt - 1) % kDecTR == 0;
            const int32_t nt = tail ? (cnt - 1) / kDecTR : (cnt > 0 ? (t1 - 1) / kDecTR - first_blk + 1 : 0);
            const int32_t burst = min(nt, a.first_burst > 0 ? min(a.first_burst, kDecStages) : kDecStages);
            for (int i = 0; i < burst; ++i) {
                const int32_t s0 = (first_blk + i) * kDecTR;
                const int32_t pg = du.u * v.max_pages + (s0 >> v.page_shift);
                if (pg < 0 || pg >= v.pool_pages) {
                    atomicOr(v.err, DEVERR_PAGE);
                    *abort_flag = 1;
                    mbar_arrive(&full[i]);   // complete the stage without data
                    break;
                }
                uint8_t* dst = ring + i * 2 * TB;
                mbar_arrive_expect_tx(&full[i], 2 * TB);
                dec_load_tile<kLin, NBOX, ESZ, RB, TB>(dst, v, pg, s0, &tmap, &full[i]);
                pre_issued = i + 1;
            }
        }
        if (a.pdl_early) griddep_wait();   // q and the new rows may come from the previous grid
        if (it0 < it1) {
            const DecUnit du = dec_unit(a, it0);
            const int32_t per_layer = v.batch * v.hkv;
            const int32_t li = du.u / per_layer - a.layer0;
            const int64_t qbase = (((int64_t)li * v.batch + (du.u / v.hkv) % v.batch) * v.hq +
                                   (int64_t)(du.u % v.hkv) * G) * D;
            mbar_arrive_expect_tx(&qfull[0], QB + (a.fused ? 2 * RB : 0));
            bulk_g2s(smem + L.qraw, a.q + qbase * ESZ, QB, &qfull[0]);
            if (a.fused) {
                const int64_t ui = (int64_t)du.u - (int64_t)a.layer0 * per_layer;
                bulk_g2s(smem + L.nrow, a.new_k + ui * RB, RB, &qfull[0]);
                bulk_g2s(smem + L.nrow + RB, a.new_v + ui * RB, RB, &qfull[0]);
            }
            pre_q = true;
        }
    }
    __syncthreads();
    // every thread is now past the wait (the producer's lane 0 waited before
    // the sync): the next grid may start, and overlaps at most this one
    griddep_launch_dependents();
    // every CTA's barriers must be initialised before any partner arrives on
    // them: arrive here, wait before this CTA's first remote access (the
    // CTA-local ring starts at once)
    cluster_arrive_relaxed();
    bool cluster_ready = false;

    if (warp == kDecNCW) {
        // ======================= producer =======================
        if (!kLin && lane == 0) prefetch_tensormap(&tmap);
        int gi = pre_issued;   // running tile counter of this CTA (lane 0's copy is authoritative)
        for (int k = 0, idx = it0; idx < it1; ++k, idx += istep) {
            if (*abort_flag) break;
            const DecUnit du = dec_unit(a, idx);
            const int32_t per_layer = v.batch * v.hkv;
            const int32_t li = du.u / per_layer - a.layer0;
            const int32_t b = (du.u / v.hkv) % v.batch;
            const int32_t g = du.u % v.hkv;
            int32_t t0, t1;
            dec_range(du.n, CS, c, t0, t1);
            const int32_t cnt = t1 - t0;
            const int32_t first_blk = t0 / kDecTR;
            // a single row alone in the last tile is not loaded: a consumer
            // warp folds it in as one row (see the consumers)
            const bool tail = cnt > 1 && (cnt - 1) % kDecTR == 0;
            const int32_t nt = tail ? (cnt - 1) / kDecTR : (cnt > 0 ? (t1 - 1) / kDecTR - first_blk + 1 : 0);
            const int32_t pg0 = t0 >> v.page_shift;
            const int32_t npg = cnt > 0 ? ((t1 - 1) >> v.page_shift) - pg0 + 1 : 0;
            const int32_t* ptab = v.page_table + (int64_t)du.u * v.max_pages;
            const int qb = k & 1;
            if (lane == 0 && !(k == 0 && pre_q)) {
                // q of this unit into its half of the double buffer
                if (!*abort_flag && mbar_wait_bounded(&qempty[qb], ((uint32_t)(k >> 1) & 1u) ^ 1u, v.err, kWaitQEmpty, (uint32_t)k)) {
                    const int64_t qbase = (((int64_t)li * v.batch + b) * v.hq + (int64_t)g * G) * D;
                    mbar_arrive_expect_tx(&qfull[qb], QB + (a.fused ? 2 * RB : 0));
                    bulk_g2s(smem + L.qraw + qb * QB, a.q + qbase * ESZ, QB, &qfull[qb]);
                    if (a.fused) {   // the appended token's rows, for the tile patch and the evict move
                        const int64_t ui = (int64_t)du.u - (int64_t)a.layer0 * per_layer;
                        bulk_g2s(smem + L.nrow + qb * 2 * RB, a.new_k + ui * RB, RB, &qfull[qb]);
                        bulk_g2s(smem + L.nrow + qb * 2 * RB + RB, a.new_v + ui * RB, RB, &qfull[qb]);
                    }
                } else {
                    *abort_flag = 1;
                }
            }
            if (!v.home_pages)
                for (int j = lane; j < min(npg, kDecMaxPg); j += 32) pg_s[j] = (k == 0 && j < 32) ? pre_pg : ptab[pg0 + j];
            __syncwarp();
            auto page_of = [&](int32_t s0) -> int32_t {
                if (v.home_pages) return du.u * v.max_pages + (s0 >> v.page_shift);
                const int32_t pk = (s0 >> v.page_shift) - pg0;
                return pk < kDecMaxPg ? pg_s[pk] : ptab[pg0 + pk];
            };
            auto prefetch_tile = [&](int j) {
                const int32_t s0 = (first_blk + j) * kDecTR;
                const int32_t pg = page_of(s0);
                if (pg < 0 || pg >= v.pool_pages) return;
                const uint8_t* kb = v.pool + (int64_t)pg * v.page_bytes + (int64_t)(s0 & (v.page_tokens - 1)) * RB;
                prefetch_l2(kb, (uint32_t)TB);
                prefetch_l2(kb + (int64_t)v.page_tokens * RB, (uint32_t)TB);
            };
            const int pf = a.prefetch_tiles;
            for (int j = lane; j < min(nt, pf); j += 32) prefetch_tile(j);
            if (lane == 0) {
                for (int i = k == 0 ? pre_issued : 0; i < nt; ++i, ++gi) {
                    if (*abort_flag) break;
                    // the CTA's first tiles jump the DRAM queue: past the first
                    // burst, wait until tile 0 has landed before queueing more
                    if (gi == a.first_burst && a.first_burst > 0 &&
                        !mbar_wait_bounded(&full[0], 0u, v.err, kWaitFull, 0u)) {
                        *abort_flag = 1;
                        break;
                    }
                    const int st = gi % kDecStages;
                    if (!mbar_wait_bounded(&empty[st], ((uint32_t)(gi / kDecStages) & 1u) ^ 1u, v.err, kWaitEmpty,
                                           (uint32_t)gi)) {
                        *abort_flag = 1;
                        break;
                    }
                    const int32_t s0 = (first_blk + i) * kDecTR;       // 16-aligned: never crosses a page
                    const int32_t pg = page_of(s0);
                    if (pg < 0 || pg >= v.pool_pages) {
                        atomicOr(v.err, DEVERR_PAGE);
                        *abort_flag = 1;
                        mbar_arrive(&full[st]);   // complete the stage without data
                        break;
                    }
                    if (pf > 0 && i + pf < nt) prefetch_tile(i + pf);
                    uint8_t* dst = ring + st * 2 * TB;
                    mbar_arrive_expect_tx(&full[st], 2 * TB);
                    dec_load_tile<kLin, NBOX, ESZ, RB, TB>(dst, v, pg, s0, &tmap, &full[st]);
                }
            }
            gi = __shfl_sync(0xffffffffu, gi, 0);
            __syncwarp();
        }
        if (lane == 0 && *abort_flag) {
            // let copies already in flight land before the CTA can exit
            for (int j = max(0, gi - kDecStages); j < gi; ++j)
                mbar_wait_bounded(&full[j % kDecStages], (uint32_t)(j / kDecStages) & 1u, v.err, kWaitDrain, (uint32_t)j);
        }
        __syncwarp();
        cluster_wait();
        cluster_sync_all();
        return;
    }

    // ======================= consumers =======================
    const int ctid = tid;  // consumer thread 0 .. NCT-1
    const int wg = warp / kDecNGW, wi = warp % kDecNGW;   // head group, place in the tile rotation
    const int h0 = wg * GW;                               // this warp's heads: h0 .. h0 + GW - 1
    float* ps = ps_all + warp * (kDecTR * (kTC ? 8 : GW));   // [16][GW] p of the tile ([16][8] on the tensor cores)
    const int qr = lane & 15;                       // half-row q.k: tile row of this lane
    const int qh = lane >> 4;                       //               half of the row
    const int qk_c = lane % QK_LPR;                 // q.k: chunk of the row this lane reads
    const int qk_rg = lane / QK_LPR;                // q.k: row of the warp step
    const int qk_k = qk_c / QK_DUP;                 // q.k: index of the logit this lane ends with
    const int qk_step = qk_k / GW;                  //      its step within the sub-block
    const int hk = qk_k % GW;                       //      its head (of this warp's GW)
    const bool qk_own = (qk_c % QK_DUP) == 0;       //      the lane that records it
    const int pv_chunk = (lane * LB) >> 4, pv_in = (lane * LB) & 15;
    // byte offset of 16-byte chunk c of tile row r in a ring stage
    auto toff = [](int r, int c) -> uint32_t {
        if constexpr (kLin) return lin<RB>(r, c);
        else return swz(r, c);
    };
    // tensor-core fragments: this lane's row group (token or d offset) and
    // column pair (heads 2 tc_t, 2 tc_t + 1)
    const int tc_g = lane >> 2, tc_t = lane & 3;
    const int tc_hA = 2 * tc_t, tc_hB = tc_hA + 1;
    int gi_base = 0;

    for (int k = 0, idx = it0; idx < it1; ++k, idx += istep) {
        const DecUnit du = dec_unit(a, idx);
        const int32_t u = du.u;
        const int32_t n = du.n;
        const int32_t per_layer = v.batch * v.hkv;
        const int32_t li = u / per_layer - a.layer0;
        const int32_t b = (u / v.hkv) % v.batch;
        const int32_t g = u % v.hkv;
        const bool need_victim = n > du.Bu;
        int32_t t0, t1;
        dec_range(n, CS, c, t0, t1);
        const int32_t cnt = t1 - t0;
        if (SMEM_S && cnt > a.chunk_cap && ctid == 0) atomicOr(v.err, DEVERR_STATE);   // the host sizes chunk_cap
        const int32_t first_blk = t0 / kDecTR;
        // a single row alone in the CTA's last tile (t0 is tile-aligned) is
        // folded in by the warp next in the tile rotation instead of being
        // loaded as a tile: with a budget of whole tiles this is the new
        // token, and the warps' tile counts stay equal
        const bool tail = cnt > 1 && (cnt - 1) % kDecTR == 0;
        const int32_t ts = t1 - 1;   // the tail slot
        const int32_t nt = tail ? (cnt - 1) / kDecTR : (cnt > 0 ? (t1 - 1) / kDecTR - first_blk + 1 : 0);
        const int tail_warp = nt % kDecNGW;
        const int64_t qbase = (((int64_t)li * v.batch + b) * v.hq + (int64_t)g * G) * D;
        const int32_t per = ceil_div(G * D, CS);   // output elements finalised per CTA
        const int xb = k & 1;
        const uint32_t xpar = (uint32_t)(k >> 1) & 1u;
        float* m_recv = reinterpret_cast<float*>(smem + L.xbuf + xb * L.xbuf_bytes);   // [kMaxCS][G]
        float* l_recv = m_recv + kMaxCS * G;                                             // [kMaxCS][G]
        float* orecv = l_recv + kMaxCS * G;                                              // [CS][per]
        unsigned long long* akey = reinterpret_cast<unsigned long long*>(smem + L.vbuf + xb * (kMaxCS * 12 + 16));
        int32_t* aslot = reinterpret_cast<int32_t*>(akey + kMaxCS);
        float* aimp = reinterpret_cast<float*>(aslot + kMaxCS);     // final importance of the new token
        const uint8_t* nrow = smem + L.nrow + xb * 2 * RB;           // fused: new K row, new V row
        const int32_t sn = n - 1;                                    // fused: the new token's slot
        const bool owns_new = a.fused && cnt > 0 && sn >= t0 && sn < t1;
        float* Sb = SMEM_S ? S_smem : a.logits + ((int64_t)u * v.cap) * G;
        const int32_t s_off = SMEM_S ? t0 : 0;   // S index of slot s = (s - s_off) * G
        const float* impg = v.imp + (int64_t)u * v.cap;
        const int32_t* posg = v.pos + (int64_t)u * v.cap;

        // the tail row's K and V: the staged rows when it is the new token,
        // else this lane's share read from the pool now (used after the tiles)
        const bool tail_here = tail && wi == tail_warp;   // one warp of each head group
        const bool tail_staged = a.fused && ts == sn;
        Raw tail_k{}, tail_v{};
        if (tail_here && !tail_staged) {
            const int32_t pg = unit_page(v, u, ts);
            if (pg >= 0 && pg < v.pool_pages) {
                const uint8_t* kr = v.pool + (int64_t)pg * v.page_bytes + (int64_t)(ts & (v.page_tokens - 1)) * RB;
                tail_k = *reinterpret_cast<const Raw*>(kr + lane * LB);
                tail_v = *reinterpret_cast<const Raw*>(kr + (int64_t)v.page_tokens * RB + lane * LB);
            } else if (lane == 0) {
                atomicOr(v.err, DEVERR_PAGE);
            }
        }
        // the importance pass reads these at the end of the unit: start them towards L2 now
        for (int j = ctid * 32; j < cnt; j += NCT * 32) {
            prefetch_global_l2(impg + t0 + j);
            prefetch_global_l2(posg + t0 + j);
        }
        // q of this unit
        if (*abort_flag || !mbar_wait_bounded(&qfull[xb], xpar, v.err, kWaitQFull, (uint32_t)k)) *abort_flag = 1;
        {
            const T* qraw = reinterpret_cast<const T*>(smem + L.qraw + xb * QB);
            for (int i = ctid; i < G * D; i += NCT) q_s[i] = Elem<T>::to_f(qraw[i]) * a.qscale;
        }
        named_bar_sync(1, NCT);

        // q of this warp's heads at this lane's chunk, in registers
        float2 qreg[(kRS && !kTC) ? GW : 1][QK_EPL / 2];
        // tensor cores: q as the B operand of S = K q^T (k = dimension, n =
        // head), this lane's head tc_g and dimensions 16 ks + 2 tc_t (+ 1, + 8,
        // + 9) of each k-step, split into three bf16 parts (hi + mid + lo
        // carries q's 24-bit mantissa; K is bf16, so each partial product is
        // exact and the logits keep fp32 accuracy)
        uint32_t qb[kTC ? 3 : 1][kTC ? D / 16 : 1][2];
        if constexpr (kTC) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int d0 = ks * 16 + 2 * tc_t + 8 * r;
                    const float x0 = tc_g < G ? q_s[tc_g * D + d0] : 0.f;
                    const float x1 = tc_g < G ? q_s[tc_g * D + d0 + 1] : 0.f;
                    split3_bf16(x0, x1, qb[0][ks][r], qb[1][ks][r], qb[2][ks][r]);
                }
        } else if constexpr (kRS) {
#pragma unroll
            for (int h = 0; h < GW; ++h)
#pragma unroll
                for (int e = 0; e < QK_EPL / 2; ++e)
                    qreg[h][e] = *reinterpret_cast<const float2*>(q_s + (h0 + h) * D + qk_c * QK_EPL + 2 * e);
        }
        // softmax state: the reference m_w of every head (the same in all
        // lanes), this lane's share of its head's row sum, and the tail row's
        // share of each head's (lane 0)
        float m_w[GW], l_tail[GW];
        float l_row[GW];   // half-row path: this lane's row sums of every head
        float m_own = -INFINITY, l_own = 0.f;
        float2 o2[kTC ? 1 : GW][EPL / 2];
        // tensor cores: the reference and this lane's row-sum share of heads
        // tc_hA, tc_hB, and O^T in the mma's C layout (d-block mb: d = 16 mb +
        // tc_g (+ 8), heads tc_hA, tc_hB)
        float tc_m[2] = {-INFINITY, -INFINITY}, tc_l[2] = {0.f, 0.f};
        float tc_o[kTC ? D / 16 : 1][4];
#pragma unroll
        for (int mb = 0; mb < (kTC ? D / 16 : 1); ++mb) tc_o[mb][0] = tc_o[mb][1] = tc_o[mb][2] = tc_o[mb][3] = 0.f;
#pragma unroll
        for (int h = 0; h < GW; ++h) {
            m_w[h] = -INFINITY;
            l_tail[h] = 0.f;
            l_row[h] = 0.f;
            if constexpr (!kTC) {
#pragma unroll
                for (int e = 0; e < EPL / 2; ++e) o2[h][e] = make_float2(0.f, 0.f);
            }
        }

        for (int i = wi; i < nt; i += kDecNGW) {
            if (*abort_flag) break;
            const int gi = gi_base + i;
            const int st = gi % kDecStages;
            if (!mbar_wait_bounded(&full[st], (uint32_t)(gi / kDecStages) & 1u, v.err, kWaitFull,
                                   (uint32_t)(gi | (warp << 24)))) {
                *abort_flag = 1;
                break;
            }
            const int32_t s0 = (first_blk + i) * kDecTR;
            uint8_t* ktile = ring + st * 2 * TB;
            uint8_t* vtile = ktile + TB;
            const int32_t lo_r = max(0, t0 - s0), hi_r = min(kDecTR, t1 - s0);   // valid rows [lo_r, hi_r)
            if (owns_new && sn >= s0 && sn < s0 + kDecTR) {
                // the pool slot of the appended token was loaded stale: put the
                // new rows into the landed tile, and into the pool for later steps
                const int r = sn - s0;
                const Raw nk = *reinterpret_cast<const Raw*>(nrow + lane * LB);
                const Raw nv = *reinterpret_cast<const Raw*>(nrow + RB + lane * LB);
                *reinterpret_cast<Raw*>(ktile + toff(r, pv_chunk) + pv_in) = nk;
                *reinterpret_cast<Raw*>(vtile + toff(r, pv_chunk) + pv_in) = nv;
                fence_proxy_async_smem();   // the stage is refilled by TMA later
                // (both head groups' warps patch the landed tile with the same
                // bytes before reading it; one of them writes the pool)
                const int32_t pg = wg == 0 ? unit_page(v, u, sn) : -1;
                if (pg >= 0 && pg < v.pool_pages) {
                    uint8_t* kd = v.pool + (int64_t)pg * v.page_bytes + (int64_t)(sn & (v.page_tokens - 1)) * RB;
                    *reinterpret_cast<Raw*>(kd + lane * LB) = nk;
                    *reinterpret_cast<Raw*>(kd + (int64_t)v.page_tokens * RB + lane * LB) = nv;
                }
                __syncwarp();
            }

            if constexpr (kTC) {
            // ---- S = K q^T on the tensor cores: m = the tile's 16 tokens,
            // n = the group's heads (padded to 8), k = d; q in three parts ----
            // Each mma sums from zero and the partial sums are added in fp32
            // (round to nearest): chaining the accumulator through the mma
            // would round every step toward zero, a bias that large logits
            // turn into a visible error in p
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
            {
                const uint32_t kb = smem_u32(ktile);
                const int mi = lane >> 3;
                const int row = (mi & 1) * 8 + (lane & 7);   // ldmatrix: this lane's row of matrix mi
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint32_t af[4];
                    ldmatrix_x4(af, kb + swz(row, 2 * ks + (mi >> 1)));
#pragma unroll
                    for (int pt = 0; pt < 3; ++pt) {
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_bf16_16816(acc, af, qb[pt][ks][0], qb[pt][ks][1]);
#pragma unroll
                        for (int j = 0; j < 4; ++j) sc[j] += acc[j];
                    }
                }
            }
            // sc: (token tc_g, head tc_hA), (tc_g, tc_hB), (tc_g + 8, tc_hA), (tc_g + 8, tc_hB)
            const bool r0v = tc_g >= lo_r && tc_g < hi_r, r1v = tc_g + 8 >= lo_r && tc_g + 8 < hi_r;
            const bool vA = tc_hA < G, vB = tc_hB < G;
            float s4[4];
            s4[0] = (r0v && vA) ? sc[0] : -INFINITY;
            s4[1] = (r0v && vB) ? sc[1] : -INFINITY;
            s4[2] = (r1v && vA) ? sc[2] : -INFINITY;
            s4[3] = (r1v && vB) ? sc[3] : -INFINITY;
            // ---- online softmax over this tile, lazily rescaled (as below) ----
            const bool big = fmaxf(s4[0], s4[2]) > tc_m[0] + kDecLazy || fmaxf(s4[1], s4[3]) > tc_m[1] + kDecLazy;
            if (__any_sync(0xffffffffu, big)) {
                float mA = fmaxf(s4[0], s4[2]), mB = fmaxf(s4[1], s4[3]);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {   // over the lanes of the same heads
                    mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, o));
                    mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, o));
                }
                const float nA = fmaxf(tc_m[0], mA), nB = fmaxf(tc_m[1], mB);
                // 1 when unchanged, 0 from -inf; a head without a logit yet stays at -inf
                const float sA = nA == -INFINITY ? 1.f : exp2f(tc_m[0] - nA);
                const float sB = nB == -INFINITY ? 1.f : exp2f(tc_m[1] - nB);
                tc_m[0] = nA;
                tc_m[1] = nB;
                tc_l[0] *= sA;
                tc_l[1] *= sB;
#pragma unroll
                for (int mb = 0; mb < D / 16; ++mb) {
                    tc_o[mb][0] *= sA;
                    tc_o[mb][2] *= sA;
                    tc_o[mb][1] *= sB;
                    tc_o[mb][3] *= sB;
                }
            }
            float p4[4];
            p4[0] = s4[0] == -INFINITY ? 0.f : exp2f(s4[0] - tc_m[0]);
            p4[1] = s4[1] == -INFINITY ? 0.f : exp2f(s4[1] - tc_m[1]);
            p4[2] = s4[2] == -INFINITY ? 0.f : exp2f(s4[2] - tc_m[0]);
            p4[3] = s4[3] == -INFINITY ? 0.f : exp2f(s4[3] - tc_m[1]);
            tc_l[0] += p4[0] + p4[2];
            tc_l[1] += p4[1] + p4[3];
            auto keep_s = [&](int r, int h, float x) {   // for the importance pass
                if (r >= lo_r && r < hi_r && h < G && (!SMEM_S || s0 + r - s_off < a.chunk_cap))
                    Sb[(int64_t)(s0 + r - s_off) * G + h] = x;
            };
            keep_s(tc_g, tc_hA, sc[0]);
            keep_s(tc_g, tc_hB, sc[1]);
            keep_s(tc_g + 8, tc_hA, sc[2]);
            keep_s(tc_g + 8, tc_hB, sc[3]);
            // ---- P into the B layout of O^T += V^T P (k = token, n = head)
            // through this warp's [16][8] scratch, in three bf16 parts ----
            *reinterpret_cast<float2*>(ps + tc_g * 8 + tc_hA) = make_float2(p4[0], p4[1]);
            *reinterpret_cast<float2*>(ps + (tc_g + 8) * 8 + tc_hA) = make_float2(p4[2], p4[3]);
            __syncwarp();
            uint32_t pb[3][2];
            split3_bf16(ps[(2 * tc_t) * 8 + tc_g], ps[(2 * tc_t + 1) * 8 + tc_g], pb[0][0], pb[1][0], pb[2][0]);
            split3_bf16(ps[(2 * tc_t + 8) * 8 + tc_g], ps[(2 * tc_t + 9) * 8 + tc_g], pb[0][1], pb[1][1], pb[2][1]);
            if (lo_r > 0 || hi_r < kDecTR) {
                // a partial tile's other rows hold stale bytes (any bit
                // pattern, which p = 0 would not cancel): zero their V
                for (int i = lane; i < kDecTR * CPR; i += 32) {
                    const int r = i / CPR;
                    if (r < lo_r || r >= hi_r) *reinterpret_cast<uint4*>(vtile + swz(r, i % CPR)) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();   // the stage is refilled by TMA later
                __syncwarp();
            }
            {
                const uint32_t vb = smem_u32(vtile);
                const int mi = lane >> 3;
                const int trow = (mi >> 1) * 8 + (lane & 7);   // ldmatrix: this lane's token row of matrix mi
                // likewise every mma from zero, added to O in fp32
#pragma unroll
                for (int mb = 0; mb < D / 16; ++mb) {
                    uint32_t af[4];
                    ldmatrix_x4_trans(af, vb + swz(trow, 2 * mb + (mi & 1)));
#pragma unroll
                    for (int pt = 0; pt < 3; ++pt) {
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_bf16_16816(acc, af, pb[pt][0], pb[pt][1]);
#pragma unroll
                        for (int j = 0; j < 4; ++j) tc_o[mb][j] += acc[j];
                    }
                }
            }
            } else {   // CUDA cores
            if constexpr (kRS) {
            // ---- q.k: per sub-block, each lane's chunk of QK_SUB rows against
            // q in registers, then the partial sums reduce-scattered ----
            float sv[QK_NSUB];
#pragma unroll
            for (int sb = 0; sb < QK_NSUB; ++sb) {
                float part[QK_NV];
#pragma unroll
                for (int j = 0; j < QK_SUB; ++j) {
                    const int r = (sb * QK_SUB + j) * QK_RPW + qk_rg;
                    const uint4 raw = *reinterpret_cast<const uint4*>(ktile + toff(r, qk_c));
                    float x[QK_EPL];
                    Widen<T, QK_EPL>::run(raw, x);
#pragma unroll
                    for (int h = 0; h < GW; ++h) {
                        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < QK_EPL / 2; ++e)
                            acc = ffma2(make_float2(x[2 * e], x[2 * e + 1]), qreg[h][e], acc);
                        part[j * GW + h] = acc.x + acc.y;
                    }
                }
                qk_reduce<QK_LPR / 2, QK_NV>(part, lane);
                const int r = (sb * QK_SUB + qk_step) * QK_RPW + qk_rg;
                sv[sb] = (r >= lo_r && r < hi_r) ? part[0] : -INFINITY;   // invalid rows: -inf
            }
            // ---- online softmax over this tile, lazily rescaled: the
            // reference m_w moves (to the tile max) only when a logit exceeds
            // it by more than kDecLazy, so p <= 2^kDecLazy; row sums stay
            // per lane until the unit's merge ----
            bool big = false;
#pragma unroll
            for (int sb = 0; sb < QK_NSUB; ++sb) big |= sv[sb] > m_own + kDecLazy;
            if (__any_sync(0xffffffffu, big)) {
                float tmax = sv[0];
#pragma unroll
                for (int sb = 1; sb < QK_NSUB; ++sb) tmax = fmaxf(tmax, sv[sb]);
#pragma unroll
                for (int h = 0; h < GW; ++h) {
                    float mt = hk == h ? tmax : -INFINITY;
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                    const float mn = fmaxf(m_w[h], mt);
                    const float scl = exp2f(m_w[h] - mn);   // 1 when unchanged, 0 from -inf
                    m_w[h] = mn;
                    l_tail[h] *= scl;
                    if (hk == h) {
                        l_own *= scl;
                        m_own = mn;
                    }
#pragma unroll
                    for (int e = 0; e < EPL / 2; ++e) {
                        o2[h][e].x *= scl;
                        o2[h][e].y *= scl;
                    }
                }
            }
#pragma unroll
            for (int sb = 0; sb < QK_NSUB; ++sb) {
                const int r = (sb * QK_SUB + qk_step) * QK_RPW + qk_rg;
                const bool rv = sv[sb] > -INFINITY;
                const float p = rv ? exp2f(sv[sb] - m_own) : 0.f;
                if (qk_own) {
                    l_own += p;
                    ps[r * GW + hk] = p;
                    if (rv && (!SMEM_S || s0 + r - s_off < a.chunk_cap))
                        Sb[(int64_t)(s0 + r - s_off) * G + h0 + hk] = sv[sb];   // for the importance pass
                }
            }
            } else {
            // ---- q.k: this lane's half row (q from shared memory) ----
            float2 acc[GW];
#pragma unroll
            for (int h = 0; h < GW; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int cidx = 2 * j + qh;   // halves interleave: their q reads fall in different banks
                const uint4 raw = *reinterpret_cast<const uint4*>(ktile + swz(qr, cidx));
                float x[EPC];
                Widen<T, EPC>::run(raw, x);
#pragma unroll
                for (int h = 0; h < GW; ++h) {
                    const float* qp = q_s + (h0 + h) * D + cidx * EPC;
#pragma unroll
                    for (int e = 0; e < EPC; e += 4) {
                        const float4 q4 = *reinterpret_cast<const float4*>(qp + e);
                        acc[h] = ffma2(make_float2(x[e], x[e + 1]), make_float2(q4.x, q4.y), acc[h]);
                        acc[h] = ffma2(make_float2(x[e + 2], x[e + 3]), make_float2(q4.z, q4.w), acc[h]);
                    }
                }
            }
            const bool rv = qr >= lo_r && qr < hi_r;
            float sh[GW];
#pragma unroll
            for (int h = 0; h < GW; ++h) {
                float t = acc[h].x + acc[h].y;
                t += __shfl_xor_sync(0xffffffffu, t, 16);
                sh[h] = rv ? t : -INFINITY;
            }
            // ---- online softmax, lazily rescaled (as above, per head) ----
            bool big = false;
#pragma unroll
            for (int h = 0; h < GW; ++h) big |= sh[h] > m_w[h] + kDecLazy;   // invalid rows: -inf
            if (__any_sync(0xffffffffu, big)) {
#pragma unroll
                for (int h = 0; h < GW; ++h) {
                    float mt = sh[h];
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                    const float mn = fmaxf(m_w[h], mt);
                    const float scl = exp2f(m_w[h] - mn);   // 1 when unchanged, 0 from -inf
                    m_w[h] = mn;
                    l_row[h] *= scl;
#pragma unroll
                    for (int e = 0; e < EPL / 2; ++e) {
                        o2[h][e].x *= scl;
                        o2[h][e].y *= scl;
                    }
                }
            }
            float p[GW];
#pragma unroll
            for (int h = 0; h < GW; ++h) {
                p[h] = rv ? exp2f(sh[h] - m_w[h]) : 0.f;
                l_row[h] += p[h];   // this lane's row; both halves of a row hold the same p
            }
            if (qh == 0) {
                store_group<GW>(ps + qr * GW, p);
                if (rv && (!SMEM_S || s0 + qr - s_off < a.chunk_cap))
                    store_group<GW>(Sb + (int64_t)(s0 + qr - s_off) * G + h0, sh);   // this group's heads of the row
            }
            }   // half-row path
            __syncwarp();
            // ---- p.v over the tile's valid rows (unrolled; invalid rows skipped, their
            // stale V bytes may hold any bit pattern).  A full tile, the common
            // case, has no per-row test, so all of its loads can be issued ahead ----
            auto pv_row = [&](int r) {
                const Raw raw = *reinterpret_cast<const Raw*>(vtile + toff(r, pv_chunk) + pv_in);
                float x[EPL];
                Widen<T, EPL>::run(raw, x);
                const float* pr = ps + r * GW;
                float2 pp[GW];
                if constexpr (GW % 4 == 0) {
#pragma unroll
                    for (int h = 0; h < GW; h += 4) {
                        const float4 t4 = *reinterpret_cast<const float4*>(pr + h);
                        pp[h] = make_float2(t4.x, t4.x);
                        pp[h + 1] = make_float2(t4.y, t4.y);
                        pp[h + 2] = make_float2(t4.z, t4.z);
                        pp[h + 3] = make_float2(t4.w, t4.w);
                    }
                } else if constexpr (GW == 2) {
                    const float2 t2 = *reinterpret_cast<const float2*>(pr);
                    pp[0] = make_float2(t2.x, t2.x);
                    pp[1] = make_float2(t2.y, t2.y);
                } else {
#pragma unroll
                    for (int h = 0; h < GW; ++h) pp[h] = make_float2(pr[h], pr[h]);
                }
#pragma unroll
                for (int h = 0; h < GW; ++h) {
#pragma unroll
                    for (int e = 0; e < EPL / 2; ++e)
                        o2[h][e] = ffma2(make_float2(x[2 * e], x[2 * e + 1]), pp[h], o2[h][e]);
                }
            };
            if (lo_r == 0 && hi_r == kDecTR) {
#pragma unroll
                for (int r = 0; r < kDecTR; ++r) pv_row(r);
            } else {
#pragma unroll
                for (int r = 0; r < kDecTR; ++r)
                    if (r >= lo_r && r < hi_r) pv_row(r);
            }
            }   // CUDA cores
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        gi_base += nt;
        if (tail_here && !*abort_flag) {
            // the tail row as a rank-1 update of this warp's state; a lane owns
            // d/32 of its dimensions, so q.k is a warp sum
            if (tail_staged) {
                tail_k = *reinterpret_cast<const Raw*>(nrow + lane * LB);
                tail_v = *reinterpret_cast<const Raw*>(nrow + RB + lane * LB);
            }
            float xk[EPL], xv[EPL];
            Widen<T, EPL>::run(tail_k, xk);
            Widen<T, EPL>::run(tail_v, xv);
            float s[GW];
            bool big = false;
#pragma unroll
            for (int h = 0; h < GW; ++h) {
                float t = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) t = fmaf(q_s[(h0 + h) * D + lane * EPL + e], xk[e], t);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                s[h] = t;
                big |= t > m_w[h] + kDecLazy;
            }
            if constexpr (kTC) {
                // this lane's heads tc_hA, tc_hB in the mma's C layout (each
                // head's reference moves on its own: the result does not depend
                // on the reference); V through this warp's scratch as floats
                float sA = -INFINITY, sB = -INFINITY;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    if (h == tc_hA) sA = s[h];
                    if (h == tc_hB) sB = s[h];
                }
                if (sA > tc_m[0] + kDecLazy) {
                    const float sc_ = exp2f(tc_m[0] - sA);
                    tc_m[0] = sA;
                    tc_l[0] *= sc_;
#pragma unroll
                    for (int mb = 0; mb < D / 16; ++mb) {
                        tc_o[mb][0] *= sc_;
                        tc_o[mb][2] *= sc_;
                    }
                }
                if (sB > tc_m[1] + kDecLazy) {
                    const float sc_ = exp2f(tc_m[1] - sB);
                    tc_m[1] = sB;
                    tc_l[1] *= sc_;
#pragma unroll
                    for (int mb = 0; mb < D / 16; ++mb) {
                        tc_o[mb][1] *= sc_;
                        tc_o[mb][3] *= sc_;
                    }
                }
                const float pA = sA == -INFINITY ? 0.f : exp2f(sA - tc_m[0]);
                const float pB = sB == -INFINITY ? 0.f : exp2f(sB - tc_m[1]);
                if (tc_g == 0) {   // the tail row, once in the warp's row sums
                    tc_l[0] += pA;
                    tc_l[1] += pB;
                }
#pragma unroll
                for (int e = 0; e < EPL; ++e) ps[lane * EPL + e] = xv[e];
                __syncwarp();
#pragma unroll
                for (int mb = 0; mb < D / 16; ++mb) {
                    const float v0 = ps[mb * 16 + tc_g], v1 = ps[mb * 16 + tc_g + 8];
                    tc_o[mb][0] = fmaf(pA, v0, tc_o[mb][0]);
                    tc_o[mb][1] = fmaf(pB, v0, tc_o[mb][1]);
                    tc_o[mb][2] = fmaf(pA, v1, tc_o[mb][2]);
                    tc_o[mb][3] = fmaf(pB, v1, tc_o[mb][3]);
                }
                __syncwarp();
            } else {
            if (big) {   // warp-uniform: s is
#pragma unroll
                for (int h = 0; h < GW; ++h) {
                    const float mn = fmaxf(m_w[h], s[h]);
                    const float scl = exp2f(m_w[h] - mn);
                    m_w[h] = mn;
                    if constexpr (kRS) {
                        l_tail[h] *= scl;
                        if (hk == h) {
                            l_own *= scl;
                            m_own = mn;
                        }
                    } else {
                        l_row[h] *= scl;
                    }
#pragma unroll
                    for (int e = 0; e < EPL / 2; ++e) {
                        o2[h][e].x *= scl;
                        o2[h][e].y *= scl;
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < GW; ++h) {
                const float p = exp2f(s[h] - m_w[h]);
                if (lane == 0) {   // the tail row, once in the warp's row sums
                    if constexpr (kRS) l_tail[h] += p;
                    else l_row[h] += p;
                }
#pragma unroll
                for (int e = 0; e < EPL / 2; ++e)
                    o2[h][e] = ffma2(make_float2(xv[2 * e], xv[2 * e + 1]), make_float2(p, p), o2[h][e]);
            }
            }   // CUDA cores
            if (lane == 0 && (!SMEM_S || ts - s_off < a.chunk_cap)) store_group<GW>(Sb + (int64_t)(ts - s_off) * G + h0, s);
            if (tail_staged && wg == 0) {   // the new token's rows into the pool for later steps
                const int32_t pg = unit_page(v, u, sn);
                if (pg >= 0 && pg < v.pool_pages) {
                    uint8_t* kd = v.pool + (int64_t)pg * v.page_bytes + (int64_t)(sn & (v.page_tokens - 1)) * RB;
                    *reinterpret_cast<Raw*>(kd + lane * LB) = tail_k;
                    *reinterpret_cast<Raw*>(kd + (int64_t)v.page_tokens * RB + lane * LB) = tail_v;
                }
            }
        }

        // the importance pass's first loads, issued now so that they land
        // during the merge and the cluster exchange
        constexpr int kIP = 8;
        float iv[kIP];
        int32_t pv[kIP];
        auto load_imp = [&](int j0) {
#pragma unroll
            for (int q = 0; q < kIP; ++q) {
                const int j = j0 + q * NCT + ctid;
                const bool fresh_slot = a.fused && t0 + j == sn;   // the new token: importance 0
                iv[q] = (j < cnt && !fresh_slot) ? impg[t0 + j] : 0.f;
                pv[q] = fresh_slot ? du.tnew : (((need_victim || v.recent_only) && j < cnt) ? posg[t0 + j] : 0);
            }
        };
        load_imp(0);

        // ---- CTA merge of the warp states ----
        // (state of head h0 + h of rotation place wi at [wi][h0 + h]: a head's
        // partials come from the kDecNGW warps of its head group)
        if constexpr (kTC) {
            float lA = tc_l[0], lB = tc_l[1];
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {   // over the lanes of the same heads
                lA += __shfl_xor_sync(0xffffffffu, lA, o);
                lB += __shfl_xor_sync(0xffffffffu, lB, o);
            }
            if (tc_g == 0) {
                if (tc_hA < G) {
                    mw_s[wi * G + tc_hA] = tc_m[0];
                    lw_s[wi * G + tc_hA] = lA;
                }
                if (tc_hB < G) {
                    mw_s[wi * G + tc_hB] = tc_m[1];
                    lw_s[wi * G + tc_hB] = lB;
                }
            }
#pragma unroll
            for (int mb = 0; mb < D / 16; ++mb)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int h = (j & 1) ? tc_hB : tc_hA;
                    if (h < G) red[(wi * G + h) * D + mb * 16 + tc_g + (j >> 1) * 8] = tc_o[mb][j];
                }
        } else {
        float l_w[GW];   // each head's row sum over this warp's rows
#pragma unroll
        for (int h = 0; h < GW; ++h) {
            float t;
            if constexpr (kRS) t = ((qk_own && hk == h) ? l_own : 0.f) + (lane == 0 ? l_tail[h] : 0.f);
            else t = lane < 16 ? l_row[h] : 0.f;   // lanes 16-31 hold the same rows
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            l_w[h] = t;
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < GW; ++h) {
                mw_s[wi * G + h0 + h] = m_w[h];
                lw_s[wi * G + h0 + h] = l_w[h];
            }
        }
#pragma unroll
        for (int h = 0; h < GW; ++h)
#pragma unroll
            for (int e = 0; e < EPL / 2; ++e)
                *reinterpret_cast<float2*>(&red[(wi * G + h0 + h) * D + lane * EPL + 2 * e]) = o2[h][e];
        }   // CUDA cores
        named_bar_sync(1, NCT);
        if (ctid < G) {
            float m = -INFINITY;
            for (int w = 0; w < kDecNGW; ++w) m = fmaxf(m, mw_s[w * G + ctid]);
            float l = 0.f;
            for (int w = 0; w < kDecNGW; ++w) {
                const float mw = mw_s[w * G + ctid];
                const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - m);
                wsc[w * G + ctid] = f;
                l += lw_s[w * G + ctid] * f;
            }
            m_c[ctid] = m;
            l_c[ctid] = l;
            if (CS == 1) {   // a one-CTA unit's state is final
                mfin[ctid] = m;
                linv[ctid] = 1.0f / l;
            }
        }
        named_bar_sync(1, NCT);
        if (CS == 1) {
            // no partners: the output straight from the merged warp partials
            // (the general path's values: its weights are exactly 1 here)
            T* outp = reinterpret_cast<T*>(a.out) + qbase;
            for (int e = ctid; e < G * D; e += NCT) {
                const int h = e / D;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kDecNGW; ++w) sum += red[w * G * D + e] * wsc[w * G + h];
                outp[e] = Elem<T>::from_f(sum * linv[h]);
            }
        } else {
        if (!cluster_ready) {   // partners' barriers are initialised from here on
            cluster_wait();
            cluster_ready = true;
        }
        // store (m_c, l_c) into every CTA of the cluster, O_c slices into their owners
        if (ctid < CS * G) {
            const int cc = ctid / G, h = ctid % G;
            dsmem_st_f32(dsmem_addr(&m_recv[c * G + h], (uint32_t)cc), m_c[h]);
            dsmem_st_f32(dsmem_addr(&l_recv[c * G + h], (uint32_t)cc), l_c[h]);
        }
        for (int e = ctid; e < G * D; e += NCT) {
            const int h = e / D;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kDecNGW; ++w) sum += red[w * G * D + e] * wsc[w * G + h];
            const int owner = e / per, loc = e - owner * per;
            dsmem_st_f32(dsmem_addr(&orecv[c * per + loc], (uint32_t)owner), sum);
        }
        named_bar_sync(1, NCT);   // every remote store of this CTA is issued
        if (ctid < CS) mbar_arrive_remote(dsmem_addr(&xbar[xb], (uint32_t)ctid));
        if (*abort_flag || !mbar_wait_cluster_bounded(&xbar[xb], xpar, v.err, kWaitXchg, (uint32_t)k)) *abort_flag = 1;

        if (ctid < G) {
            float m = -INFINITY;
            for (int cc = 0; cc < CS; ++cc) m = fmaxf(m, m_recv[cc * G + ctid]);
            float l = 0.f;
            for (int cc = 0; cc < CS; ++cc)
                if (l_recv[cc * G + ctid] > 0.f) l += l_recv[cc * G + ctid] * exp2f(m_recv[cc * G + ctid] - m);
            mfin[ctid] = m;
            linv[ctid] = 1.0f / l;
        }
        named_bar_sync(1, NCT);
        if (ctid < CS * G) {
            const int h = ctid % G;
            beta[ctid] = (l_recv[ctid] > 0.f) ? exp2f(m_recv[ctid] - mfin[h]) * linv[h] : 0.f;
        }
        named_bar_sync(1, NCT);

        // output slice owned by this CTA
        {
            T* outp = reinterpret_cast<T*>(a.out) + qbase;
            for (int loc = ctid; loc < per; loc += NCT) {
                const int e = c * per + loc;
                if (e >= G * D) break;
                const int h = e / D;
                float sum = 0.f;
                for (int cc = 0; cc < CS; ++cc) sum += orecv[cc * per + loc] * beta[cc * G + h];
                outp[e] = Elem<T>::from_f(sum);
            }
        }
        }   // CS > 1
        // importance update + local victim
        unsigned long long kmin = ~0ull;
        int32_t smin = -1;
        {
            float mf[G], li_[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                mf[h] = mfin[h];
                li_[h] = linv[h];
            }
            const int32_t lo = v.sink, hi = du.tnew - v.window;
            // the loads of each batch are issued together (one L2 round trip); the
            // first batch's were issued before the exchanges
            for (int j0 = 0; j0 < cnt; j0 += kIP * NCT) {
                if (j0 > 0) load_imp(j0);
#pragma unroll
                for (int q = 0; q < kIP; ++q) {
                    const int j = j0 + q * NCT + ctid;
                    if (j >= cnt) continue;
                    const int32_t slot = t0 + j;
                    const float* srow = Sb + (int64_t)(slot - s_off) * G;
                    float inc = 0.f;
#pragma unroll
                    for (int h = 0; h < G; ++h) inc += exp2f(srow[h] - mf[h]) * li_[h];
                    // HiKV Stage I: only the recent bank (and the token leaving it)
                    // accumulates; older scores stay frozen
                    const bool grows = !v.recent_only || pv[q] >= du.tnew - v.window;
                    const float nw = grows ? iv[q] + inc : iv[q];
                    v.imp[(int64_t)u * v.cap + slot] = nw;
                    if (a.fused && slot == sn) {
                        v.pos[(int64_t)u * v.cap + slot] = du.tnew;
                        *new_imp_s = nw;
                    }
                    if (need_victim && pv[q] >= lo && pv[q] <= hi) {
                        const unsigned long long key =
                            ((unsigned long long)__float_as_uint(nw) << 32) | (unsigned long long)(~(uint32_t)pv[q]);
                        if (key < kmin) {
                            kmin = key;
                            smin = slot;
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
            if (lane == 0) {
                wkey[warp] = kmin;
                wslot[warp] = smin;
            }
        }
        named_bar_sync(1, NCT);
        if (ctid == 0) {
            unsigned long long kk = ~0ull;
            int32_t sl = -1;
            for (int w = 0; w < kDecNCW; ++w)
                if (wkey[w] < kk) {
                    kk = wkey[w];
                    sl = wslot[w];
                }
            if (CS > 1) {
                dsmem_st_u64(dsmem_addr(&akey[c], 0u), kk);
                dsmem_st_s32(dsmem_addr(&aslot[c], 0u), sl);
                if (owns_new) dsmem_st_f32(dsmem_addr(aimp, 0u), *new_imp_s);
                mbar_arrive_remote(dsmem_addr(&vbar[xb], 0u));
            } else if (owns_new) {
                *aimp = *new_imp_s;
            }
            if (c == 0) {
                int32_t vs = -1;
                if (CS == 1) {
                    vs = sl;
                } else if (!*abort_flag &&
                           mbar_wait_cluster_bounded(&vbar[xb], xpar, v.err, kWaitVictim, (uint32_t)k)) {
                    unsigned long long best = ~0ull;
                    for (int cc = 0; cc < CS; ++cc)
                        if (akey[cc] < best) {
                            best = akey[cc];
                            vs = aslot[cc];
                        }
                } else {
                    *abort_flag = 1;
                }
                vs = need_victim ? vs : -1;
                wslot[0] = vs;   // for the fused evict below
                if (!a.fused) {
                    v.victim[u] = vs;
                } else {
                    const bool cut = a.evict && vs >= 0;
                    v.victim[u] = cut ? -1 : vs;
                    v.len[u] = cut ? n - 1 : n;
                    v.next_pos[u] = du.tnew + 1;
                }
            }
        }
        named_bar_sync(1, NCT);
        // fused evict: the appended token (last slot) moves into the victim's
        // slot: rows from the stash, final importance from the exchange
        if (a.fused && a.evict && c == 0 && warp == 0) {
            const int32_t vs = wslot[0];
            if (vs >= 0 && vs != sn) {
                const int32_t pd = unit_page(v, u, vs);
                if (pd >= 0 && pd < v.pool_pages) {
                    uint8_t* kd = v.pool + (int64_t)pd * v.page_bytes + (int64_t)(vs & (v.page_tokens - 1)) * RB;
                    *reinterpret_cast<Raw*>(kd + lane * LB) = *reinterpret_cast<const Raw*>(nrow + lane * LB);
                    *reinterpret_cast<Raw*>(kd + (int64_t)v.page_tokens * RB + lane * LB) =
                        *reinterpret_cast<const Raw*>(nrow + RB + lane * LB);
                } else if (lane == 0) {
                    atomicOr(v.err, DEVERR_PAGE);
                }
                if (lane == 0) {
                    v.imp[(int64_t)u * v.cap + vs] = *aimp;
                    v.pos[(int64_t)u * v.cap + vs] = du.tnew;
                }
            }
            if (v.debug && vs >= 0) {
                if (vs > sn && lane == 0) atomicOr(v.err, DEVERR_STATE);   // a victim past the new slot
                __syncwarp();
                poison_slot(v, u, sn, lane, 32);   // the last slot is vacated
            }
        }
        named_bar_sync(1, NCT);   // shared buffers of this unit are free for the next
        if (ctid == 0) mbar_arrive(&qempty[xb]);
    }
    __syncwarp();
    if (!cluster_ready) cluster_wait();
    cluster_sync_all();
}

template <typename T, int D, int G, bool SM>
cudaError_t decode_prepare(size_t smem) {
    const void* kern = reinterpret_cast<const void*>(k_decode<T, D, G, SM>);
    cudaError_t e = func_smem_optin(kern, smem);
    if (e != cudaSuccess) return e;
    return func_allow_nonportable_clusters(kern);
}

template <typename T, int D, int G>
cudaLaunchConfig_t decode_config(int cs, int n_clusters, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs, (unsigned)n_clusters, 1);
    cfg.blockDim = dim3(dec_threads<T, D, G>(), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

// Clusters of `cs` CTAs with `smem` bytes each that can be resident at once
// (clusters must fit in one GPC each); cached per (kernel, device, cs, smem).
template <typename T, int D, int G, bool SM>
int decode_active_clusters(int cs, size_t smem) {
    if (decode_prepare<T, D, G, SM>(smem) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = decode_config<T, D, G>(cs, 1, smem, nullptr, attr);
    cfg.numAttrs = 1;   // the cluster shape alone decides residency
    return func_active_clusters(reinterpret_cast<const void*>(k_decode<T, D, G, SM>), cs, cfg);
}

template <typename T, int D, int G, bool SM>
cudaError_t decode_launch_one(const DecodeArgs& a, const CUtensorMap& tmap, size_t smem, cudaStream_t s) {
    cudaError_t e = decode_prepare<T, D, G, SM>(smem);
    if (e != cudaSuccess) return e;
    // The clusters are persistent: launch no more than can be resident at
    // once, or the surplus would run as a second wave after the others had
    // finished all their units.
    DecodeArgs b = a;
    const int active = decode_active_clusters<T, D, G, SM>(a.cs, smem);
    if (active > 0 && b.n_clusters > active) b.n_clusters = active;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = decode_config<T, D, G>(b.cs, b.n_clusters, smem, s, attr);
    return cudaLaunchKernelEx(&cfg, k_decode<T, D, G, SM>, b, tmap);
}

template <typename T, int D, bool SM>
cudaError_t decode_launch_g(const DecodeArgs& a, const CUtensorMap& tmap, int group, size_t smem,
                            cudaStream_t s) {
    switch (group) {
        case 1: return decode_launch_one<T, D, 1, SM>(a, tmap, smem, s);
        case 2: return decode_launch_one<T, D, 2, SM>(a, tmap, smem, s);
        case 4: return decode_launch_one<T, D, 4, SM>(a, tmap, smem, s);
        case 8: return decode_launch_one<T, D, 8, SM>(a, tmap, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int D, bool SM>
int decode_active_g(int group, int cs, size_t smem) {
    switch (group) {
        case 1: return decode_active_clusters<T, D, 1, SM>(cs, smem);
        case 2: return decode_active_clusters<T, D, 2, SM>(cs, smem);
        case 4: return decode_active_clusters<T, D, 4, SM>(cs, smem);
        case 8: return decode_active_clusters<T, D, 8, SM>(cs, smem);
        default: return 0;
    }
}

template <typename T, int D>
size_t decode_smem_t(int group, bool smem_path, int chunk_cap) {
    switch (group) {
        case 1: return dec_layout<T, D, 1>(smem_path, chunk_cap).total;
        case 2: return dec_layout<T, D, 2>(smem_path, chunk_cap).total;
        case 4: return dec_layout<T, D, 4>(smem_path, chunk_cap).total;
        case 8: return dec_layout<T, D, 8>(smem_path, chunk_cap).total;
        default: return 0;
    }
}

}  // namespace hikv

#define HIKV_DECODE_INSTANTIATE(T, D, NAME)                                                         \
    namespace hikv {                                                                                \
    cudaError_t decode_launch_##NAME(const DecodeArgs& a, const CUtensorMap& tmap, int group,       \
                                     bool smem_path, size_t smem, cudaStream_t s) {                 \
        return smem_path ? decode_launch_g<T, D, true>(a, tmap, group, smem, s)                     \
                         : decode_launch_g<T, D, false>(a, tmap, group, smem, s);                   \
    }                                                                                               \
    size_t decode_smem_##NAME(int group, bool smem_path, int chunk_cap) {                           \
        return decode_smem_t<T, D>(group, smem_path, chunk_cap);                                    \
    }                                                                                               \
    int decode_active_##NAME(int group, bool smem_path, int cs, size_t smem) {                      \
        return smem_path ? decode_active_g<T, D, true>(group, cs, smem)                             \
                         : decode_active_g<T, D, false>(group, cs, smem);                           \
    }                                                                                               \
    cudaError_t decode_small_launch_##NAME(const SmallArgs& a, const CUtensorMap& tmap, int group,  \
                                           int n_ctas, cudaStream_t s) {                            \
        return decode_small_launch_g<T, D>(a, tmap, group, n_ctas, s);                              \
    }                                                                                               \
    }
