// Prefill importance from an observation window of queries, bf16 K/V on the
// tensor cores (setup step).
//
// Same result as the CUDA-core kernels of k_window.cu: the importance of each
// prompt token starts as its causal attention column summed over the last nq
// prompt queries and the G query heads of its group (HiKV sec. III-D
// initialises importance from prefill attention over a window of late
// queries; SnapKV's observation window, blog sec. 3), the queries applied in
// position order.  The logits of a unit are the product of its window
// queries [G*nq x d] with its keys [d x n], a dense contraction, so they are
// formed with mma.sync m16n8k16 (bf16 in, fp32 accumulate; a bf16 product is
// exact in fp32).
//
//   pass 1  per chunk of kWinChunk tokens: per query vector, the running max
//           and sum of 2^(s'-m) over the tokens it may see -> partials;
//   pass 2  merge the unit's partials, recompute the logits, and add
//           sum_h 2^(s'-m)/l per query, in query order, to each token.
//
// A CTA (8 warps) takes one chunk of one unit.  K tiles of 64 tokens come in
// by TMA through the pool's tensor map (16-row x 128-byte boxes with the
// 128-byte swizzle), double-buffered on two mbarriers.  Warp w computes rows
// [16 (w mod RB), +16) of the query block against a 64/NCS-token slice of
// the tile (RB = NQV/16 row blocks, NCS = 8/RB column slices); its A
// fragments (the queries) stay in registers for the whole chunk.  Rows are
// query-major (row = query * G + head), so the G heads of a query sit in
// lanes that differ only in lane bits 2.. and pass 2 sums them with G - 1
// shuffles before staging one increment per (query, token).
#include <type_traits>

#include "hikv_internal.cuh"

namespace hikv {
namespace {

constexpr int kTcThreads = 256;
constexpr int kTcTok = 64;                 // tokens per tile
constexpr int kMaxTcChunk = 1024;          // tokens per CTA at most
constexpr int kMaxChunkPages = kMaxTcChunk / 16 + 1;   // pages such a chunk can touch (pages hold >= 16 tokens)
constexpr int kTcGroups = kTcTok / 16;     // 16-row TMA row groups per tile

template <int D, int NQV>
struct WinTc {
    static constexpr int RB = NQV / 16;            // row blocks
    static constexpr int NCS = 8 / RB;             // column slices
    static constexpr int COLS = kTcTok / NCS;      // tokens per warp and tile
    static constexpr int NB = COLS / 8;            // n8 blocks per warp
    static constexpr int KS = D / 16;              // k16 steps
    static constexpr int NBOX = D * 2 / 128;       // 128-byte boxes per row
    static constexpr int TILE = kTcGroups * NBOX * 2048;   // bytes of one K tile
    static_assert(RB * NCS == 8 && NB >= 1, "warp tiling");
    static_assert(KS % 2 == 0, "ldmatrix.x4 covers two k16 steps");
    // TMA ring depth: three CTAs per SM with 3 stages up to 64 query rows, two with 4 above
    static constexpr int STAGES = NQV <= 64 ? 3 : 4;
    // shared memory (from a 1024-aligned base)
    static constexpr int OFF_TILE = 0;                         // [STAGES][TILE]
    static constexpr int OFF_BAR = STAGES * TILE;           // STAGES mbarriers, then a status word
    static constexpr int OFF_POS = OFF_BAR + 8 * STAGES + 16;   // [2][kTcTok] int32
    static constexpr int OFF_ML = OFF_POS + 2 * kTcTok * 4;    // [NCS][NQV][2] (pass 1) / MF,LI [NQV][2]
    static constexpr int OFF_P = OFF_ML + NCS * NQV * 2 * 4;   // [NQV][kTcTok + 4] fp32 increments (pass 2)
    static constexpr int OFF_PG = OFF_P + NQV * (kTcTok + 4) * 4;   // [kMaxChunkPages] page ids of the chunk
    static constexpr int BYTES = OFF_PG + kMaxChunkPages * 4 + 1024;
};

// byte offset of element e of tile row r in a tile loaded as row groups of
// [NBOX][16 rows][128 bytes], 16-byte chunks swizzled by (row mod 8)
template <int NBOX>
__device__ __forceinline__ uint32_t tile_off(int r, int e) {
    const int byte = e * 2, c = byte >> 4, rr = r & 15;
    return (uint32_t)((r >> 4) * (NBOX * 2048) + (c >> 3) * 2048 + rr * 128 + ((((c & 7) ^ (rr & 7)) << 4) | (byte & 15)));
}

// Queue the TMA loads of tile [s0, s0 + 64) of unit u into `dst`; returns the
// bytes that will arrive on `bar` (row groups wholly past the chunk end are
// not loaded).  pgs: the page ids of the chunk starting at c0.
template <int NBOX>
__device__ uint32_t issue_tile(const View& v, const CUtensorMap* tmap, const int32_t* pgs, int32_t c0, int32_t s0,
                               int32_t c1, uint8_t* dst, uint64_t* bar) {
    uint32_t bytes = 0;
    int32_t ys[kTcGroups];
#pragma unroll
    for (int j = 0; j < kTcGroups; ++j) {
        ys[j] = -1;
        const int32_t s = s0 + 16 * j;
        if (s >= c1) continue;
        const int32_t pg = pgs[(s >> v.page_shift) - (c0 >> v.page_shift)];   // the chunk's page ids, staged
        if (pg < 0 || pg >= v.pool_pages) {
            atomicOr(v.err, DEVERR_PAGE);
            continue;
        }
        ys[j] = pg * 2 * v.page_tokens + (s & (v.page_tokens - 1));   // K rows of the page
        bytes += NBOX * 2048;
    }
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int j = 0; j < kTcGroups; ++j) {
        if (ys[j] < 0) continue;
#pragma unroll
        for (int bx = 0; bx < NBOX; ++bx)
            tma_load_2d(dst + j * NBOX * 2048 + bx * 2048, tmap, bx * 64, ys[j], bar);
    }
    return bytes;
}

template <int D, int NQV, bool PASS2>
__global__ void __launch_bounds__(kTcThreads, NQV <= 64 ? 3 : 2) k_window_tc(const WindowArgs a, const __grid_constant__ CUtensorMap tmap) {
    using C = WinTc<D, NQV>;
    extern __shared__ __align__(128) uint8_t wsm_raw[];
    uint8_t* smem = wsm_raw + ((1024u - (smem_u32(wsm_raw) & 1023u)) & 1023u);
    const View& v = a.v;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rb = warp % C::RB, cslice = warp / C::RB;
    const int32_t u = a.u0 + blockIdx.y;
    const int32_t n = v.len[u];
    const int32_t c0 = blockIdx.x * a.chunk;
    const int nq = a.nq, nqv = v.group * nq;
    float* part_u = a.part + ((int64_t)u * a.nchunks_max) * nqv * 2;
    if (c0 >= n) {
        if (!PASS2)
            for (int q = tid; q < nqv; q += kTcThreads) {
                part_u[((int64_t)blockIdx.x * nqv + q) * 2] = -INFINITY;
                part_u[((int64_t)blockIdx.x * nqv + q) * 2 + 1] = 0.f;
            }
        return;
    }
    const int32_t c1 = min(n, c0 + a.chunk);
    const int32_t tnew = v.next_pos[u] - 1;
    uint8_t* tiles = smem + C::OFF_TILE;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    volatile int32_t* landed = reinterpret_cast<volatile int32_t*>(smem + C::OFF_BAR + 8 * C::STAGES);
    int32_t* Ps = reinterpret_cast<int32_t*>(smem + C::OFF_POS);
    float* ML = reinterpret_cast<float*>(smem + C::OFF_ML);
    float* Pt = reinterpret_cast<float*>(smem + C::OFF_P);
    int32_t* pgs = reinterpret_cast<int32_t*>(smem + C::OFF_PG);
    constexpr int PT = kTcTok + 4;   // row stride of Pt

    if (tid == 0) {
#pragma unroll
        for (int st = 0; st < C::STAGES; ++st) mbar_init(&bar[st], 1);
        fence_mbar_init();
        prefetch_tensormap(&tmap);
    }
    {   // the chunk's page ids, once (the refills then need no global round trip)
        const int p0 = c0 >> v.page_shift, np = ((c1 - 1) >> v.page_shift) - p0 + 1;
        for (int i = tid; i < np; i += kTcThreads) pgs[i] = v.page_table[(int64_t)u * v.max_pages + p0 + i];
    }
    __syncthreads();
    const int ntiles = ceil_div(c1 - c0, kTcTok);
    // the first C::STAGES - 1 tiles go out at once; each iteration then queues
    // the tile C::STAGES - 1 ahead into the stage the previous tile released
    if (tid == 0)
        for (int j = 0; j < C::STAGES - 1 && j < ntiles; ++j)
            issue_tile<C::NBOX>(v, &tmap, pgs, c0, c0 + j * kTcTok, c1, tiles + j * C::TILE, &bar[j]);
    // positions of tile 0, then one tile ahead in a register (threads < kTcTok)
    int32_t pnext = (tid < kTcTok && c0 + tid < c1) ? v.pos[(int64_t)u * v.cap + c0 + tid] : INT32_MAX;
    // pass 2: the importance of this thread's token of the next tile, likewise
    float inext = (PASS2 && tid < kTcTok && c0 + tid < c1) ? v.imp[(int64_t)u * v.cap + c0 + tid] : 0.f;

    // A fragments: query rows rb*16 + g and + 8 (rows past nqv are zero), raw bf16
    const int per_layer = v.batch * v.hkv;
    const int li = u / per_layer - a.layer0, b = (u / v.hkv) % v.batch, gh = u % v.hkv;
    const uint16_t* qb = reinterpret_cast<const uint16_t*>(a.q) +
                         (((int64_t)li * v.batch + b) * v.hq + (int64_t)gh * v.group) * nq * D;
    const int G = v.group;
    const int row0 = rb * 16 + g, row1 = row0 + 8;   // row = query * G + head
    auto qrow = [&](int row) { return (int64_t)((row % G) * nq + row / G) * D; };   // q is [G][nq][d]
    uint32_t af[C::KS][4];
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
        const int k0 = ks * 16 + 2 * t;
        auto ld = [&](int row, int k) -> uint32_t {
            return row < nqv ? *reinterpret_cast<const uint32_t*>(qb + qrow(row) + k) : 0u;
        };
        af[ks][0] = ld(row0, k0);
        af[ks][1] = ld(row1, k0);
        af[ks][2] = ld(row0, k0 + 8);
        af[ks][3] = ld(row1, k0 + 8);
    }
    // causal limit of each of this lane's two rows (query i sits at tnew - nq + 1 + i)
    const int32_t qfirst = tnew - nq + 1;
    const int32_t qpos0 = row0 < nqv ? tnew - nq + 1 + row0 / G : INT32_MIN;
    const int32_t qpos1 = row1 < nqv ? tnew - nq + 1 + row1 / G : INT32_MIN;

    float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};   // pass 1: this warp's slice
    float mf[2] = {0.f, 0.f}, lif[2] = {0.f, 0.f};              // pass 2: final per row
    if (PASS2) {
        // final (m, 1/l) of every query vector from the unit's chunk partials
        const int nch = ceil_div(n, a.chunk);
        for (int q = tid; q < nqv; q += kTcThreads) {
            float m = -INFINITY;
            for (int cc = 0; cc < nch; ++cc) m = fmaxf(m, part_u[((int64_t)cc * nqv + q) * 2]);
            float l = 0.f;
            for (int cc = 0; cc < nch; ++cc) {
                const float lc = part_u[((int64_t)cc * nqv + q) * 2 + 1];
                if (lc > 0.f) l += lc * exp2f(part_u[((int64_t)cc * nqv + q) * 2] - m);
            }
            ML[2 * q] = m;
            ML[2 * q + 1] = 1.0f / l;
        }
        __syncthreads();
        if (row0 < nqv) { mf[0] = ML[2 * row0]; lif[0] = ML[2 * row0 + 1]; }
        if (row1 < nqv) { mf[1] = ML[2 * row1]; lif[1] = ML[2 * row1 + 1]; }
    }
    const float qscale = a.qscale;

    for (int i = 0; i < ntiles; ++i) {
        const int32_t s0 = c0 + i * kTcTok;
        const int st = i % C::STAGES;
        int32_t* Pi = Ps + (i & 1) * kTcTok;   // read by tile i - 2 last: released two barriers ago
        float icur = 0.f;
        if (tid < kTcTok) {
            Pi[tid] = pnext;
            icur = inext;
            const int32_t sn = s0 + kTcTok + tid;
            pnext = sn < c1 ? v.pos[(int64_t)u * v.cap + sn] : INT32_MAX;   // lands during tile i
            if (PASS2) inext = sn < c1 ? v.imp[(int64_t)u * v.cap + sn] : 0.f;
        }
        if (tid == 0 && i + C::STAGES - 1 < ntiles) {   // its stage held tile i - 1, released at its end
            const int j = i + C::STAGES - 1;
            issue_tile<C::NBOX>(v, &tmap, pgs, c0, c0 + j * kTcTok, c1, tiles + (j % C::STAGES) * C::TILE,
                                &bar[j % C::STAGES]);
        }
        // one thread waits for the tile (bounded); the CTA barrier then orders
        // every thread's reads after the copy, and all take the same branch
        if (tid == 0) *landed = mbar_wait_bounded(&bar[st], (uint32_t)(i / C::STAGES) & 1u, v.err, kWaitFull, (uint32_t)i);
        // a full tile whose tokens all precede the first window query is seen
        // whole by every query: no causal mask (all tiles but the last few).
        // Only with 128 query rows: with fewer, the two compiled bodies cost
        // more in register spills than the mask does (measured on the 32-layer
        // stack's 64 rows)
        bool all_vis = false;
        if constexpr (NQV >= 128) all_vis = __syncthreads_and(tid >= kTcTok || Pi[tid] <= qfirst) != 0;
        else __syncthreads();
        if (!*landed) {
            // give up; let the copies already queued for the following tiles land first
            if (tid == 0)
                for (int j = i + 1; j < ntiles && j < i + C::STAGES; ++j)
                    mbar_wait_bounded(&bar[j % C::STAGES], (uint32_t)(j / C::STAGES) & 1u, v.err, kWaitDrain, (uint32_t)i);
            __syncthreads();
            break;
        }
        const uint8_t* tile = tiles + st * C::TILE;

        // S = Q K^T for rows [rb*16, +16) x tokens [cslice*COLS, +COLS) of the tile
        float acc[C::NB][4];
#pragma unroll
        for (int nb = 0; nb < C::NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
        // B fragments by ldmatrix.x4: matrices (k16 step ks, low 8 dims), (ks,
        // high 8), (ks + 1, low), (ks + 1, high) of token block nb; this lane
        // addresses row (lane mod 8) of matrix lane / 8
        {
            const uint32_t tbase = smem_u32(tile);
            const int mi = lane >> 3, rrow = lane & 7;
#pragma unroll
            for (int ks = 0; ks < C::KS; ks += 2) {
#pragma unroll
                for (int nb = 0; nb < C::NB; ++nb) {
                    const int row = cslice * C::COLS + nb * 8 + rrow;
                    const int k0 = (ks + (mi >> 1)) * 16 + (mi & 1) * 8;
                    uint32_t b[4];
                    ldmatrix_x4(b, tbase + tile_off<C::NBOX>(row, k0));
                    mma_bf16_16816(acc[nb], af[ks], b[0], b[1]);
                    mma_bf16_16816(acc[nb], af[ks + 1], b[2], b[3]);
                }
            }
        }
        // logits (log2 domain) and causal visibility: value j of block nb is
        // row (j < 2 ? row0 : row1), token cslice*COLS + nb*8 + 2t + (j & 1)
        auto tile_math = [&](auto masked_tag) {
        constexpr bool kMasked = decltype(masked_tag)::value;
        float s[C::NB][4];
        bool vis[C::NB][4];
#pragma unroll
        for (int nb = 0; nb < C::NB; ++nb)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = cslice * C::COLS + nb * 8 + 2 * t + (j & 1);
                vis[nb][j] = kMasked ? Pi[col] <= (j < 2 ? qpos0 : qpos1) : true;
                s[nb][j] = acc[nb][j] * qscale;
            }
        if (!PASS2) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float tm = -INFINITY;
#pragma unroll
                for (int nb = 0; nb < C::NB; ++nb)
#pragma unroll
                    for (int j = 2 * hr; j < 2 * hr + 2; ++j)
                        if (vis[nb][j]) tm = fmaxf(tm, s[nb][j]);
                tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
                tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
                const float mn = fmaxf(mr[hr], tm);
                float sum = 0.f;
                if (mn > -INFINITY) {
#pragma unroll
                    for (int nb = 0; nb < C::NB; ++nb)
#pragma unroll
                        for (int j = 2 * hr; j < 2 * hr + 2; ++j)
                            if (vis[nb][j]) sum += exp2f(s[nb][j] - mn);
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if (mn > -INFINITY) {
                    lr[hr] = (lr[hr] > 0.f ? lr[hr] * exp2f(mr[hr] - mn) : 0.f) + sum;
                    mr[hr] = mn;
                }
            }
        } else {
            // probabilities summed over the G heads of each query: the heads of
            // a query are rows q*G .. q*G+G-1, held by lanes that differ in
            // lane bits 2 .. 2+log2(G)-1 (row = rb*16 + lane/4)
#pragma unroll
            for (int nb = 0; nb < C::NB; ++nb) {
                float pr[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float m = j < 2 ? mf[0] : mf[1], li_ = j < 2 ? lif[0] : lif[1];
                    pr[j] = vis[nb][j] ? exp2f(s[nb][j] - m) * li_ : 0.f;
                }
                for (int o = 4; o < 4 * G; o <<= 1)
#pragma unroll
                    for (int j = 0; j < 4; ++j) pr[j] += __shfl_xor_sync(0xffffffffu, pr[j], o);
                const int col = cslice * C::COLS + nb * 8 + 2 * t;
                if (g % G == 0) {   // the head-0 lane of each query writes its increments
                    if (row0 < nqv) *reinterpret_cast<float2*>(&Pt[(row0 / G) * PT + col]) = make_float2(pr[0], pr[1]);
                    if (row1 < nqv) *reinterpret_cast<float2*>(&Pt[(row1 / G) * PT + col]) = make_float2(pr[2], pr[3]);
                }
            }
            __syncthreads();
            // per token (thread r < kTcTok): queries in position order, onto
            // the importance loaded one tile ahead (no other CTA touches it)
            static_assert(kTcTok <= kTcThreads, "one token per thread");
            if (tid < kTcTok && s0 + tid < c1) {
                float imp = icur;
                for (int qi = 0; qi < nq; ++qi) imp = imp + Pt[qi * PT + tid];
                v.imp[(int64_t)u * v.cap + s0 + tid] = imp;
            }
        }
        };
        if constexpr (NQV >= 128) {
            if (all_vis) tile_math(std::integral_constant<bool, false>{});
            else tile_math(std::integral_constant<bool, true>{});
        } else {
            tile_math(std::integral_constant<bool, true>{});
        }
        __syncthreads();   // the tile buffer, Ps and Pt are free again
    }

    if (!PASS2) {
        // merge the column slices' (m, l) of every row, then store the chunk's partials
        if (t == 0) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int row = hr ? row1 : row0;
                if (row < nqv) {
                    ML[(cslice * NQV + row) * 2] = mr[hr];
                    ML[(cslice * NQV + row) * 2 + 1] = lr[hr];
                }
            }
        }
        __syncthreads();
        for (int q = tid; q < nqv; q += kTcThreads) {
            float m = -INFINITY;
            for (int cs = 0; cs < C::NCS; ++cs) m = fmaxf(m, ML[(cs * NQV + q) * 2]);
            float l = 0.f;
            for (int cs = 0; cs < C::NCS; ++cs) {
                const float lc = ML[(cs * NQV + q) * 2 + 1];
                if (lc > 0.f) l += lc * exp2f(ML[(cs * NQV + q) * 2] - m);
            }
            part_u[((int64_t)blockIdx.x * nqv + q) * 2] = m;
            part_u[((int64_t)blockIdx.x * nqv + q) * 2 + 1] = l;
        }
    }
}

template <int D, int NQV>
cudaError_t launch_tc(const WindowArgs& a, const CUtensorMap& tmap, cudaStream_t s) {
    constexpr int smem = WinTc<D, NQV>::BYTES;
    cudaError_t e0 = func_smem_optin(reinterpret_cast<const void*>(k_window_tc<D, NQV, false>), smem);
    if (e0 == cudaSuccess) e0 = func_smem_optin(reinterpret_cast<const void*>(k_window_tc<D, NQV, true>), smem);
    if (e0 != cudaSuccess) return e0;
    dim3 grid(a.nchunks_grid, a.nunits);
    k_window_tc<D, NQV, false><<<grid, kTcThreads, smem, s>>>(a, tmap);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_window_tc<D, NQV, true><<<grid, kTcThreads, smem, s>>>(a, tmap);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_tc_d(const WindowArgs& a, const CUtensorMap& tmap, int nqv, cudaStream_t s) {
    if (nqv <= 16) return launch_tc<D, 16>(a, tmap, s);
    if (nqv <= 32) return launch_tc<D, 32>(a, tmap, s);
    if (nqv <= 64) return launch_tc<D, 64>(a, tmap, s);
    return launch_tc<D, 128>(a, tmap, s);
}

}  // namespace

bool window_tc_supported(int dtype, int d, int nqv) { return dtype == 1 && (d == 64 || d == 128) && nqv <= 128; }

cudaError_t launch_window_tc(const WindowArgs& a, const CUtensorMap& tmap, int d, int nqv, cudaStream_t s) {
    if (a.chunk > kMaxTcChunk || a.chunk % kTcTok) return cudaErrorInvalidValue;
    return d == 64 ? launch_tc_d<64>(a, tmap, nqv, s) : launch_tc_d<128>(a, tmap, nqv, s);
}

}  // namespace hikv
